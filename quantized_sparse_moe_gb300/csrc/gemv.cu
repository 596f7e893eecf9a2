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
#include "tc_common.cuh"

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

// ------------------------------------------ int8-activation mode (i8 x i8)
//
// "Ember: packed Q8 decode": the projections that read the same activation
// share one quantization of it, and the dot products run on 8-bit groups.
// q8_quantize_x turns x into blocks of 32 int8 codes with an fp32 scale
// max|x| / 127 (codes round half away from zero); q8_gemv_i8 then takes
// each 32-wide block's dot product exactly as an int8 tensor-core MMA
// (m16n8k32, one block per MMA, the activation in column 0) and scales it
// by weight scale * activation scale in fp32.  Same tiling and K-segment
// order as the f16 GEMV, so results do not depend on N.

__global__ void __launch_bounds__(256)
q8_quantize_x_kernel(const uint16_t* __restrict__ x, int K, int8_t* __restrict__ qx,
                     float* __restrict__ dx) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // block of 32
  if (b >= K / 32) return;
  const float v = __uint_as_float((uint32_t)x[32 * b + lane] << 16);
  const float amax = warp_max(fabsf(v));
  const float db = amax / 127.0f;
  float r = 0.f;
  if (db != 0.f) r = fminf(fmaxf(roundf(v / db), -127.f), 127.f);
  qx[32 * b + lane] = (int8_t)r;
  if (lane == 0) dx[b] = db;
}

// D(16x8, s32) = A(16x32, s8, row) * B(32x8, s8, col).
__device__ __forceinline__ void mma_16832_s8(int (&d)[4], const uint32_t (&a)[4],
                                             uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

template <int KS>
__global__ void __launch_bounds__((KS > 8 ? KS : 8) * 32)
q8_gemv_i8_kernel(const int8_t* __restrict__ qx, const float* __restrict__ dx,
                  const int8_t* __restrict__ q8, const __half* __restrict__ d, int N,
                  int K, uint16_t* __restrict__ y) {
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
    float ag = 0.f, ah = 0.f;  // rows g and g + 8 (lanes with q == 0)
    const int kend = min(K, (seg + 1) * kSeg);
#pragma unroll 4
    for (int k0 = seg * kSeg; k0 < kend; k0 += 64) {
      RawA r;
      load_a<QSM_Q8_0>(r, w, rg, rh, k0, q);
      // lane (g, q) holds codes k0 + 8q .. + 7 of its rows; the MMA's k
      // groups 4q.. and 16 + 4q.. take the low and high halves, and the
      // activation codes (column 0, lanes g == 0) follow the same mapping
      uint2 x0 = make_uint2(0u, 0u), x1 = x0;
      if (g == 0) {
        x0 = __ldg(reinterpret_cast<const uint2*>(qx + k0 + 8 * q));
        x1 = __ldg(reinterpret_cast<const uint2*>(qx + k0 + 32 + 8 * q));
      }
      int s0[4], s1[4];
      const uint32_t a0[4] = {r.g0.x, r.h0.x, r.g0.y, r.h0.y};
      const uint32_t a1[4] = {r.g1.x, r.h1.x, r.g1.y, r.h1.y};
      mma_16832_s8(s0, a0, x0.x, x0.y);
      mma_16832_s8(s1, a1, x1.x, x1.y);
      if (q == 0) {
        const float d0 = __ldg(dx + k0 / 32), d1 = __ldg(dx + k0 / 32 + 1);
        const float sg0 = __half2float(__ushort_as_half((unsigned short)(r.sg & 0xffffu)));
        const float sg1 = __half2float(__ushort_as_half((unsigned short)(r.sg >> 16)));
        const float sh0 = __half2float(__ushort_as_half((unsigned short)(r.sh & 0xffffu)));
        const float sh1 = __half2float(__ushort_as_half((unsigned short)(r.sh >> 16)));
        ag = fmaf((float)s0[0], sg0 * d0, ag);
        ag = fmaf((float)s1[0], sg1 * d1, ag);
        ah = fmaf((float)s0[2], sh0 * d0, ah);
        ah = fmaf((float)s1[2], sh1 * d1, ah);
      }
    }
    if (q == 0) {
      red[(seg * TPC + tl) * 16 + g] = ag;
      red[(seg * TPC + tl) * 16 + g + 8] = ah;
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
cudaError_t launch_i8_ks(const int8_t* qx, const float* dx, const int8_t* q,
                         const uint16_t* d, int N, int K, uint16_t* y, cudaStream_t s) {
  constexpr int W = KS > 8 ? KS : 8;
  constexpr int TPC = W / KS;
  const int tiles = (N + 15) / 16;
  const int grid = (tiles + TPC - 1) / TPC;
  const size_t smem = (size_t)((K + kSeg - 1) / kSeg) * TPC * 16 * sizeof(float);
  return launch_pdl(q8_gemv_i8_kernel<KS>, dim3(grid), dim3(W * 32), smem, s, qx, dx, q,
                    reinterpret_cast<const __half*>(d), N, K, y);
}

// ------------------------------------------ TMA-fed tiles (K % 256 == 0)
//
// One CTA = one 16-row tile x `spc` consecutive 512-wide segments, one warp
// per segment.  A segment's codes (16 rows x 512 bytes) arrive by a single
// TMA copy of the 3D row view (128-byte swizzle, so the fragment reads of the
// 8 rows g land in 8 different 16-byte units and are free of bank
// conflicts), its block scales by a second copy, both issued before the
// programmatic-launch wait since the weights are static.  When one CTA does
// not take all of K, the CTAs of a tile form a cluster along x and store
// their segment partials into the rank-0 CTA's shared memory, which adds
// them in segment order.  Every TMA-fed kernel sums a row in the same order
// (fixed by K alone, see segment_partial), so a row's bits do not depend on N
// or on which of them ran.  Rows past N and chunks past K arrive as zeros
// (TMA fill) and are never stored.

constexpr int kTmaSegBytes = 16 * kSeg;              // codes of one segment
constexpr int kTmaScaleBytes = 16 * (kSeg / 32) * 2;  // its 16 x 16 fp16 scales
constexpr int kTmaMaxSpc = 4;
constexpr int kTmaMaxSeg = 32;                        // K <= 16384

// 8 bytes at byte b (a multiple of 8) of 128-byte line `line` of a tile
// written with the 128-byte swizzle.
__device__ __forceinline__ uint2 lds_sw128(const unsigned char* tile, int line, int b) {
  return *reinterpret_cast<const uint2*>(
      tile + line * 128 + ((((b >> 4) ^ (line & 7)) << 4) | (b & 15)));
}

// One 64-chunk of a 16-row tile (TMA-written codes, 3D row view with the
// 128-byte swizzle, and scales in shared memory) into the accumulators of
// rows g and g + 8: acc[0] / acc[2] (valid in lanes q == 0).  The activation
// comes from global memory (bf16, kXs false) or from shared memory (fp16,
// kXs true); in the int8 mode its codes and block scales likewise.
template <bool kI8, bool kXs>
__device__ __forceinline__ void tile_chunk(float (&acc)[4], const unsigned char* cs,
                                           const uint32_t* ss, const void* xa,
                                           const float* xd, int kb, int ch, int g, int q) {
  RawA r;
  const int lg = (ch >> 1) * 16 + g;  // line of row g in 128-byte chunk ch / 2
  const int b = (ch & 1) * 64 + 8 * q;
  r.g0 = lds_sw128(cs, lg, b);
  r.g1 = lds_sw128(cs, lg, b + 32);
  r.h0 = lds_sw128(cs, lg + 8, b);
  r.h1 = lds_sw128(cs, lg + 8, b + 32);
  r.sg = ss[g * 8 + ch];
  r.sh = ss[(g + 8) * 8 + ch];
  const int k0 = kb + 64 * ch;
  if constexpr (!kI8) {
    uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
    if (g == 0) {
      if constexpr (kXs) {
        const __half* xs = static_cast<const __half*>(xa);
        X0 = *reinterpret_cast<const uint4*>(xs + k0 + 8 * q);
        X1 = *reinterpret_cast<const uint4*>(xs + k0 + 32 + 8 * q);
      } else {
        const uint16_t* x = static_cast<const uint16_t*>(xa);
        X0 = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(x + k0 + 8 * q)));
        X1 = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(x + k0 + 32 + 8 * q)));
      }
    }
    chunk_mma<QSM_Q8_0>(acc, r, X0, X1);
  } else {
    const int8_t* qx = static_cast<const int8_t*>(xa);
    uint2 x0 = make_uint2(0u, 0u), x1 = x0;
    if (g == 0) {
      x0 = *reinterpret_cast<const uint2*>(qx + k0 + 8 * q);
      x1 = *reinterpret_cast<const uint2*>(qx + k0 + 32 + 8 * q);
    }
    int s0[4], s1[4];
    const uint32_t a0[4] = {r.g0.x, r.h0.x, r.g0.y, r.h0.y};
    const uint32_t a1[4] = {r.g1.x, r.h1.x, r.g1.y, r.h1.y};
    mma_16832_s8(s0, a0, x0.x, x0.y);
    mma_16832_s8(s1, a1, x1.x, x1.y);
    if (q == 0) {
      const float d0 = xd[k0 / 32], d1 = xd[k0 / 32 + 1];
      const float sg0 = __half2float(__ushort_as_half((unsigned short)(r.sg & 0xffffu)));
      const float sg1 = __half2float(__ushort_as_half((unsigned short)(r.sg >> 16)));
      const float sh0 = __half2float(__ushort_as_half((unsigned short)(r.sh & 0xffffu)));
      const float sh1 = __half2float(__ushort_as_half((unsigned short)(r.sh >> 16)));
      acc[0] = fmaf((float)s0[0], sg0 * d0, acc[0]);
      acc[0] = fmaf((float)s1[0], sg1 * d1, acc[0]);
      acc[2] = fmaf((float)s0[2], sh0 * d0, acc[2]);
      acc[2] = fmaf((float)s1[2], sh1 * d1, acc[2]);
    }
  }
}

// The partial of a 512-wide segment is (chain over chunks 0..3) + (chain
// over chunks 4..7), each chain accumulated from zero in chunk order; the
// TMA-fed kernels all follow this order, so a row's bits depend on K only.
constexpr int kChain = 4;  // chunks per chain

// Both chains of the segment at kb in one warp, interleaved (independent
// accumulators, so the chains' latencies overlap).
template <bool kI8, bool kXs>
__device__ __forceinline__ void segment_partial(const unsigned char* cs,
                                                const unsigned char* scl, const void* xa,
                                                const float* xd, int kb, int K, int g, int q,
                                                float& pg, float& ph) {
  const uint32_t* ss = reinterpret_cast<const uint32_t*>(scl);
  const int nch = min(kSeg, K - kb) / 64;
  float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kChain; ++i) {
    if (i < nch) tile_chunk<kI8, kXs>(a, cs, ss, xa, xd, kb, i, g, q);
    if (kChain + i < nch) tile_chunk<kI8, kXs>(b, cs, ss, xa, xd, kb, kChain + i, g, q);
  }
  pg = a[0] + b[0];
  ph = a[2] + b[2];
}

// One chain (half = 0: chunks 0..3, 1: chunks 4..7) of the segment at kb.
template <bool kI8, bool kXs>
__device__ __forceinline__ void chain_partial(const unsigned char* cs, const unsigned char* scl,
                                              const void* xa, const float* xd, int kb, int K,
                                              int half, int g, int q, float& pg, float& ph) {
  const uint32_t* ss = reinterpret_cast<const uint32_t*>(scl);
  const int nch = min(kSeg, K - kb) / 64;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kChain; ++i)
    if (kChain * half + i < nch) tile_chunk<kI8, kXs>(a, cs, ss, xa, xd, kb, kChain * half + i, g, q);
  pg = a[0];
  ph = a[2];
}

template <bool kI8>
__global__ void __launch_bounds__(kTmaMaxSpc * 32)
q8_gemv_tma_kernel(const __grid_constant__ CUtensorMap cmap,
                   const __grid_constant__ CUtensorMap smap,
                   const uint16_t* __restrict__ x, const int8_t* __restrict__ qx,
                   const float* __restrict__ dx, int N, int K, int spc, int tiles,
                   uint16_t* __restrict__ y, int32_t* dev_status) {
  extern __shared__ unsigned char gemv_dyn[];
  __shared__ __align__(8) uint64_t bar[kTmaMaxSpc];
  __shared__ float red[kTmaMaxSeg][16];  // [segment][row], used in rank 0
  const int tile = blockIdx.y + gridDim.y * blockIdx.z;
  if (tile >= tiles) return;  // the whole cluster shares the tile
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int n0 = tile * 16;
  const int nseg = (K + kSeg - 1) / kSeg;
  const int seg0 = blockIdx.x * spc;
  const int mine = min(spc, nseg - seg0);
  const uint32_t pad = (1024u - (smem_u32(gemv_dyn) & 1023u)) & 1023u;
  unsigned char* codes = gemv_dyn + pad;               // [spc][4][16][128]
  unsigned char* scl = codes + spc * kTmaSegBytes;     // [spc][16][16] fp16
  if (threadIdx.x == 0) {
    for (int s = 0; s < mine; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < mine; ++s) {
      mbar_arrive_expect_tx(&bar[s], kTmaSegBytes + kTmaScaleBytes);
      tc::tma_load_3d(codes + s * kTmaSegBytes, &cmap, 0, n0, (seg0 + s) * (kSeg / 128),
                      &bar[s]);
      tc::tma_load_2d(scl + s * kTmaScaleBytes, &smap, (seg0 + s) * (kSeg / 32), n0,
                      &bar[s]);
    }
  }
  pdl_wait();  // x (or its codes) come from the preceding launch
  pdl_launch_dependents();
  float pg = 0.f, ph = 0.f;  // rows g and g + 8 (lanes q == 0)
  if (warp < mine) {
    if (!mbar_wait_bounded(&bar[warp], 0, kWaitIters)) {
      if (lane == 0 && dev_status) set_status(dev_status, QSM_DEV_TIMEOUT);
      mbar_wait_bounded(&bar[warp], 0, kWaitIters);  // let the copy land
    } else {
      if constexpr (kI8)
        segment_partial<true, false>(codes + warp * kTmaSegBytes, scl + warp * kTmaScaleBytes,
                                     qx, dx, (seg0 + warp) * kSeg, K, g, q, pg, ph);
      else
        segment_partial<false, false>(codes + warp * kTmaSegBytes, scl + warp * kTmaScaleBytes,
                                      x, nullptr, (seg0 + warp) * kSeg, K, g, q, pg, ph);
    }
  }
  if (warp < mine && q == 0) {
    const int seg = seg0 + warp;
    if (gridDim.x == 1) {
      red[seg][g] = pg;
      red[seg][g + 8] = ph;
    } else {
      dsmem_st_f32(dsmem_addr(&red[seg][g], 0), pg);
      dsmem_st_f32(dsmem_addr(&red[seg][g + 8], 0), ph);
    }
  }
  if (gridDim.x > 1) cluster_sync_all();
  else __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x < 16) {
    float s = 0.f;
    for (int seg = 0; seg < nseg; ++seg) s += red[seg][threadIdx.x];
    const int n = n0 + threadIdx.x;
    if (n < N) y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
  }
}

// ------------------------------------------ persistent streaming (large N)
//
// With many tiles, one CTA per SM walks tiles t = blockIdx.x, t + gridDim.x,
// ...; a tile's segments stream through a ring of kStreamS stages (up to 4
// segments each) filled by one producer thread, so every SM keeps ~170 KB of
// weights in flight for the whole call instead of relaunching a CTA per tile.
// The activation is staged once in shared memory (fp16, or the int8 codes
// and block scales).  Two groups of eight consumer warps take alternate
// tiles (a tile of one stage) or alternate stages (a tile of several
// stages); in a group each warp takes one chain (half a segment) of a
// stage, and a tile's chains and segments are added in the order above.

constexpr int kStreamS = 5;
constexpr int kStreamSeg = 4;  // segments per stage
constexpr int kStageBytes = kStreamSeg * (kTmaSegBytes + kTmaScaleBytes);  // 34 KB
constexpr int kStreamGW = 2 * kStreamSeg;  // warps of a consumer group: one per chain
constexpr int kStreamCW = 2 * kStreamGW;   // two groups, alternate tiles
constexpr int kStreamWarps = kStreamCW + 1;

template <bool kI8, bool kByTile>  // kByTile: one stage per tile (K <= 2048)
__global__ void __launch_bounds__(kStreamWarps * 32, 1)
q8_gemv_stream_kernel(const __grid_constant__ CUtensorMap cmap,
                      const __grid_constant__ CUtensorMap smap,
                      const uint16_t* __restrict__ x, const int8_t* __restrict__ qx,
                      const float* __restrict__ dx, int N, int K, int tiles,
                      uint16_t* __restrict__ y, int32_t* dev_status) {
  extern __shared__ unsigned char gemv_dyn[];
  __shared__ __align__(8) uint64_t full[kStreamS], empty[kStreamS];
  // [buffer][tile parity][seg][chain][row]; buffer = the tile's group when
  // tiles alternate, 0 when stages alternate
  __shared__ float red[2][2][kTmaMaxSeg][2][16];
  __shared__ volatile int s_bad;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int nseg = (K + kSeg - 1) / kSeg;
  const int nst = (nseg + kStreamSeg - 1) / kStreamSeg;  // stages per tile
  const int G = gridDim.x;
  const int ntile = (tiles - (int)blockIdx.x + G - 1) / G;
  const int total = ntile * nst;
  const uint32_t pad = (1024u - (smem_u32(gemv_dyn) & 1023u)) & 1023u;
  unsigned char* ring = gemv_dyn + pad;  // stage: [4][8 KB] codes, then [4][512] scales
  unsigned char* xsm = ring + kStreamS * kStageBytes;  // fp16 x [K], or int8 codes + scales
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStreamS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kStreamGW);  // the stage's consumer group
    }
    s_bad = 0;
    fence_mbar_init();
  }
  __syncthreads();
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (mbar_wait_bounded(bar, parity, s_bad ? 1024u : kWaitIters)) return;
    s_bad = 1;
    if (dev_status) set_status(dev_status, QSM_DEV_TIMEOUT);
  };

  if (warp == kStreamCW) {  // producer
    if (lane != 0) return;
    auto issue = [&](int p) {
      const int slot = p % kStreamS;
      unsigned char* st = ring + slot * kStageBytes;
      const int tile = (int)blockIdx.x + (p / nst) * G, seg0 = (p % nst) * kStreamSeg;
      const int cnt = min(kStreamSeg, nseg - seg0);
      mbar_arrive_expect_tx(&full[slot], (uint32_t)cnt * (kTmaSegBytes + kTmaScaleBytes));
      for (int j = 0; j < cnt; ++j) {
        tc::tma_load_3d(st + j * kTmaSegBytes, &cmap, 0, tile * 16, (seg0 + j) * (kSeg / 128),
                        &full[slot]);
        tc::tma_load_2d(st + kStreamSeg * kTmaSegBytes + j * kTmaScaleBytes, &smap,
                        (seg0 + j) * (kSeg / 32), tile * 16, &full[slot]);
      }
    };
    int p = 0;
    for (; p < total && p < kStreamS; ++p) issue(p);  // static weights: before the wait
    pdl_wait();
    pdl_launch_dependents();
    for (; p < total; ++p) {
      wait(&empty[p % kStreamS], ((p / kStreamS) - 1) & 1);
      issue(p);
    }
    if (s_bad)  // let the last copy of every stage land
      for (int s = 0; s < kStreamS && s < total; ++s)
        mbar_wait_bounded(&full[s], (((s + ((total - 1 - s) / kStreamS) * kStreamS)) /
                                     kStreamS) & 1, kWaitIters);
    return;
  }

  pdl_wait();  // x (or its codes) come from the preceding launch
  pdl_launch_dependents();
  constexpr int nct = kStreamCW * 32;
  if constexpr (!kI8) {  // x -> fp16 in shared memory, once
    for (int i = threadIdx.x; i < K / 8; i += nct)
      reinterpret_cast<uint4*>(xsm)[i] =
          bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(x) + i));
  } else {
    for (int i = threadIdx.x; i < K / 16; i += nct)
      reinterpret_cast<uint4*>(xsm)[i] = __ldg(reinterpret_cast<const uint4*>(qx) + i);
    for (int i = threadIdx.x; i < K / 32; i += nct)
      reinterpret_cast<float*>(xsm + K)[i] = __ldg(dx + i);
  }
  asm volatile("barrier.sync 1, %0;" ::"r"(nct) : "memory");
  const void* xa = xsm;
  const float* xd = kI8 ? reinterpret_cast<const float*>(xsm + K) : nullptr;
  const int grp = warp / kStreamGW, gw = warp % kStreamGW;
  const int sw = gw >> 1, half = gw & 1;  // segment of the stage, chain of the segment
  constexpr bool by_tile = kByTile;       // groups alternate tiles, else stages
  for (int p = 0; p < total; ++p) {
    const int slot = p % kStreamS, i = p / nst, seg = (p % nst) * kStreamSeg + sw;
    const int b = by_tile ? grp : 0, par = by_tile ? (i >> 1) & 1 : i & 1;
    if (((by_tile ? i : p) & 1) == grp) {  // this group's stage
      wait(&full[slot], (p / kStreamS) & 1);
      const unsigned char* st = ring + slot * kStageBytes;
      if (seg < nseg) {
        float pg, ph;
        chain_partial<kI8, true>(st + sw * kTmaSegBytes,
                                 st + kStreamSeg * kTmaSegBytes + sw * kTmaScaleBytes, xa, xd,
                                 seg * kSeg, K, half, g, q, pg, ph);
        if (q == 0) {
          red[b][par][seg][half][g] = pg;
          red[b][par][seg][half][g + 8] = ph;
        }
        consumed(pg);
        consumed(ph);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
    }
    if (p % nst == nst - 1 && (!by_tile || (i & 1) == grp)) {  // tile end: add its segments
      // alternating tiles: the tile's group; alternating stages: both groups
      if (by_tile)
        asm volatile("barrier.sync %0, %1;" ::"r"(2 + grp), "r"(kStreamGW * 32) : "memory");
      else
        asm volatile("barrier.sync 1, %0;" ::"r"(nct) : "memory");
      if (gw == 0 && lane < 16 && (by_tile || grp == 0)) {
        const float(*rr)[2][16] = red[b][par];
        float sum = 0.f;
        for (int s2 = 0; s2 < nseg; ++s2) sum += rr[s2][0][lane] + rr[s2][1][lane];
        const int n = ((int)blockIdx.x + i * G) * 16 + lane;
        if (n < N) y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
      }
    }
  }
}

// Segments per CTA: as many as possible (at most 4) while the grid keeps at
// least ~1024 CTAs, and few enough that a tile's CTAs fit one cluster of 8.
int gemv_tma_spc(long tiles, int nseg) {
  const int lo = (nseg + 7) / 8;
  int spc = nseg < kTmaMaxSpc ? nseg : kTmaMaxSpc;
  while (spc / 2 >= lo && tiles * ((nseg + spc - 1) / spc) < 1024) spc /= 2;
  return spc;
}

// Launches the TMA-fed kernel; false when the shape or the tensor maps do
// not allow it (the caller then uses the register-fed kernels).
template <bool kI8>
bool launch_tma(const uint16_t* x, const int8_t* qx, const float* dx, const int8_t* q,
                const uint16_t* d, int N, int K, uint16_t* y, int32_t* status,
                cudaStream_t s, cudaError_t* err) {
  if (K % 256) return false;
  CUtensorMap cmap, smap;
  if (!tc::make_map_rows3d(&cmap, q, (uint64_t)N, (uint64_t)K, 16, kSeg / 128)) return false;
  if (!tc::make_map_2d(&smap, d, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)N,
                       (uint64_t)K / 32, kSeg / 32, 16, CU_TENSOR_MAP_SWIZZLE_NONE))
    return false;
  const long tiles = (N + 15) / 16;
  const int nseg = (K + kSeg - 1) / kSeg;
  int nsm = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (nsm > 0 && tiles >= 16 && tiles < (1L << 30)) {  // persistent streaming
    static bool attr[2][2] = {{false, false}, {false, false}};  // sized for K <= 16384
    const size_t smem = 1024 + (size_t)kStreamS * kStageBytes + (size_t)K * 2;
    const bool by_tile = nseg <= kStreamSeg;  // one stage per tile
    auto* kern = by_tile ? q8_gemv_stream_kernel<kI8, true> : q8_gemv_stream_kernel<kI8, false>;
    if (!attr[kI8][by_tile]) {
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(1024 + (size_t)kStreamS * kStageBytes + 16384 * 2));
      attr[kI8][by_tile] = true;
    }
    *err = launch_pdl(kern, dim3(tiles < nsm ? (int)tiles : nsm), dim3(kStreamWarps * 32),
                      smem, s, cmap, smap, x, qx, dx, N, K, (int)tiles, y, status);
    return true;
  }
  const int spc = gemv_tma_spc(tiles, nseg);
  const int slices = (nseg + spc - 1) / spc;
  const long gy = tiles < 65535 ? tiles : 65535;
  const dim3 grid(slices, (unsigned)gy, (unsigned)((tiles + gy - 1) / gy));
  const size_t smem = 1024 + (size_t)spc * (kTmaSegBytes + kTmaScaleBytes);
  *err = launch_pdl_cluster(q8_gemv_tma_kernel<kI8>, grid, dim3(spc * 32), slices, smem, s,
                            cmap, smap, x, qx, dx, N, K, spc, (int)tiles, y, status);
  return true;
}

int gemv_split(int N, int K) {  // K segments per tile: about 24 warps per SM
  const long tiles = (N + 15) / 16;
  int ks = 1;
  const int nseg = (K + kSeg - 1) / kSeg;
  while (ks < 32 && ks < nseg && tiles * ks < 152L * 24) ks *= 2;
  return ks;
}

}  // namespace
}  // namespace qsm

extern "C" qsm_status q8_gemv(const uint16_t* x, const int8_t* q,
                              const uint16_t* d, int32_t N, int32_t K,
                              uint16_t* y, int32_t* dev_status,
                              cudaStream_t stream) {
  using namespace qsm;
  if (N < 1 || K < 64 || K % 64 || !x || !q || !d || !y)
    return QSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(q) || !aligned16(d) || !aligned16(y))
    return QSM_ERR_INVALID_ARGUMENT;
  if ((size_t)N * K >= ((size_t)1 << 40) || K > 16384) return QSM_ERR_UNSUPPORTED;
  cudaError_t err;
  if (launch_tma<false>(x, nullptr, nullptr, q, d, N, K, y, dev_status, stream, &err))
    return err == cudaSuccess ? QSM_OK : QSM_ERR_CUDA;
  // Split K until there are enough warps in flight (about 24 per SM).
  switch (gemv_split(N, K)) {
    case 1: err = launch_ks<1>(x, q, d, N, K, y, stream); break;
    case 2: err = launch_ks<2>(x, q, d, N, K, y, stream); break;
    case 4: err = launch_ks<4>(x, q, d, N, K, y, stream); break;
    case 8: err = launch_ks<8>(x, q, d, N, K, y, stream); break;
    case 16: err = launch_ks<16>(x, q, d, N, K, y, stream); break;
    default: err = launch_ks<32>(x, q, d, N, K, y, stream); break;
  }
  return err == cudaSuccess ? QSM_OK : QSM_ERR_CUDA;
}

extern "C" qsm_status q8_quantize_x(const uint16_t* x, int32_t K, int8_t* qx, float* dx,
                                    int32_t* dev_status, cudaStream_t stream) {
  using namespace qsm;
  (void)dev_status;
  if (K < 32 || K % 32 || !x || !qx || !dx) return QSM_ERR_INVALID_ARGUMENT;
  const int blocks = K / 32;
  QSM_CUDA_TRY(launch_pdl(q8_quantize_x_kernel, dim3((blocks + 7) / 8), dim3(256), 0,
                          stream, x, (int)K, qx, dx));
  return QSM_OK;
}

extern "C" qsm_status q8_gemv_i8(const int8_t* qx, const float* dx, const int8_t* q,
                                 const uint16_t* d, int32_t N, int32_t K, uint16_t* y,
                                 int32_t* dev_status, cudaStream_t stream) {
  using namespace qsm;
  if (N < 1 || K < 64 || K % 64 || !qx || !dx || !q || !d || !y)
    return QSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(qx) || !aligned4(dx) || !aligned16(q) || !aligned16(d) || !aligned16(y))
    return QSM_ERR_INVALID_ARGUMENT;
  if ((size_t)N * K >= ((size_t)1 << 40) || K > 16384) return QSM_ERR_UNSUPPORTED;
  cudaError_t err;
  if (launch_tma<true>(nullptr, qx, dx, q, d, N, K, y, dev_status, stream, &err))
    return err == cudaSuccess ? QSM_OK : QSM_ERR_CUDA;
  switch (gemv_split(N, K)) {
    case 1: err = launch_i8_ks<1>(qx, dx, q, d, N, K, y, stream); break;
    case 2: err = launch_i8_ks<2>(qx, dx, q, d, N, K, y, stream); break;
    case 4: err = launch_i8_ks<4>(qx, dx, q, d, N, K, y, stream); break;
    case 8: err = launch_i8_ks<8>(qx, dx, q, d, N, K, y, stream); break;
    case 16: err = launch_i8_ks<16>(qx, dx, q, d, N, K, y, stream); break;
    default: err = launch_i8_ks<32>(qx, dx, q, d, N, K, y, stream); break;
  }
  return err == cudaSuccess ? QSM_OK : QSM_ERR_CUDA;
}
