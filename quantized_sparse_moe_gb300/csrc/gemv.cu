// Dense batch-1 Q8_0 GEMV y[n] = sum_c q[n,c] * d[n,c/32] * x[c].
//
// "Optimizing on-device inference for Apple Silicon", section "Optimizing
// the single-row weight path": one row of activations, weights read in
// parallel by cooperating lanes; the Q8_0 rows of "Ember: packed Q8 decode"
// (32 int8 codes and one fp16 scale per block).  Ember's 16-row VNNI
// interleave is a CPU layout; here rows stay row-contiguous and every warp
// streams a 16-row tile with coalesced 8-byte loads per lane (32 contiguous
// bytes per row per quad), the products summed by mma.sync (gemv_core.cuh).
// K is cut into fixed 512-wide segments; each segment's partial sum is
// accumulated by one warp from zero and the segment partials are added in
// segment order.  KS warps share the segments of a tile when the rows alone
// give too few warps to keep HBM busy, but the summation order depends on K
// only, so a row's result does not depend on N: the rows of a [gate; up]
// concatenation come out bit-identical to those of the separate matrices
// (the property the oMLX gate/up fusion relies on).
#include "gemv_core.cuh"

namespace qsm {
namespace {

using namespace gemv;

constexpr int kSeg = 512;  // K per segment

template <int KS>
__global__ void __launch_bounds__((KS > 8 ? KS : 8) * 32)
q8_gemv_kernel(const uint16_t* __restrict__ x, const int8_t* __restrict__ q8,
               const __half* __restrict__ d, int N, int K,
               uint16_t* __restrict__ y) {
  constexpr int W = KS > 8 ? KS : 8;  // warps per CTA
  constexpr int TPC = W / KS;         // 16-row tiles per CTA
  extern __shared__ float red[];      // [segments][TPC][16]
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int kw = warp % KS, tl = warp / KS;
  const int n0 = (blockIdx.x * TPC + tl) * 16;
  QW w;
  w.codes = reinterpret_cast<const uint8_t*>(q8);
  w.scales = d;
  w.biases = nullptr;
  w.cols = K;
  const int rg = min(n0 + g, N - 1), rh = min(n0 + g + 8, N - 1);
  const int nseg = (K + kSeg - 1) / kSeg;
  for (int seg = kw; seg < nseg; seg += KS) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int kend = min(K, (seg + 1) * kSeg);
#pragma unroll 4
    for (int k0 = seg * kSeg; k0 < kend; k0 += 64) {
      RawA r;
      load_a<QSM_Q8_0>(r, w, rg, rh, k0, q);
      uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
      if (g == 0) {
        X0 = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(x + k0 + 8 * q)));
        X1 = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(x + k0 + 32 + 8 * q)));
      }
      chunk_mma<QSM_Q8_0>(acc, r, X0, X1);
    }
    if (q == 0) {  // column 0 of the MMA tile: rows g and g + 8
      red[(seg * TPC + tl) * 16 + g] = acc[0];
      red[(seg * TPC + tl) * 16 + g + 8] = acc[2];
    }
  }
  __syncthreads();
  if (threadIdx.x < TPC * 16) {
    const int t2 = threadIdx.x / 16, r = threadIdx.x % 16;
    float s = 0.f;
    for (int seg = 0; seg < nseg; ++seg) s += red[(seg * TPC + t2) * 16 + r];
    const int n = (blockIdx.x * TPC + t2) * 16 + r;
    if (n < N) y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
  }
}

template <int KS>
cudaError_t launch_ks(const uint16_t* x, const int8_t* q, const uint16_t* d,
                      int N, int K, uint16_t* y, cudaStream_t s) {
  constexpr int W = KS > 8 ? KS : 8;
  constexpr int TPC = W / KS;
  const int tiles = (N + 15) / 16;
  const int grid = (tiles + TPC - 1) / TPC;
  const size_t smem = (size_t)((K + kSeg - 1) / kSeg) * TPC * 16 * sizeof(float);
  return launch_pdl(q8_gemv_kernel<KS>, dim3(grid), dim3(W * 32), smem, s, x, q,
                    reinterpret_cast<const __half*>(d), N, K, y);
}

}  // namespace
}  // namespace qsm

extern "C" qsm_status q8_gemv(const uint16_t* x, const int8_t* q,
                              const uint16_t* d, int32_t N, int32_t K,
                              uint16_t* y, int32_t* dev_status,
                              cudaStream_t stream) {
  using namespace qsm;
  (void)dev_status;  // nothing device-side to report for a dense GEMV
  if (N < 1 || K < 64 || K % 64 || !x || !q || !d || !y)
    return QSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(q) || !aligned16(d) || !aligned16(y))
    return QSM_ERR_INVALID_ARGUMENT;
  if ((size_t)N * K >= ((size_t)1 << 40) || K > 16384) return QSM_ERR_UNSUPPORTED;
  // Split K until there are enough warps in flight (about 24 per SM).
  const long tiles = (N + 15) / 16;
  int ks = 1;
  const int nseg = (K + kSeg - 1) / kSeg;
  while (ks < 32 && ks < nseg && tiles * ks < 152L * 24) ks *= 2;
  cudaError_t err;
  switch (ks) {
    case 1: err = launch_ks<1>(x, q, d, N, K, y, stream); break;
    case 2: err = launch_ks<2>(x, q, d, N, K, y, stream); break;
    case 4: err = launch_ks<4>(x, q, d, N, K, y, stream); break;
    case 8: err = launch_ks<8>(x, q, d, N, K, y, stream); break;
    case 16: err = launch_ks<16>(x, q, d, N, K, y, stream); break;
    default: err = launch_ks<32>(x, q, d, N, K, y, stream); break;
  }
  return err == cudaSuccess ? QSM_OK : QSM_ERR_CUDA;
}
