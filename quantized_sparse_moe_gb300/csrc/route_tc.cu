// Router for many tokens on the tcgen05 tensor cores.
//
// Same result as the CUDA-core router (route.cu): logits = x W_r^T + bias
// with fp32 accumulation, top k by logit (ties to the lower expert index),
// softmax weights.  For a long prompt the logit matmul (2*T*E*H FLOPs) is
// too large for CUDA cores, so it runs as one bf16 GEMM over an exact
// three-way split of the fp32 router weight: w = hi + mid + lo with
// hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid) (fp32 has a
// 24-bit significand, three bf16 parts hold 3 x 8 bits).  x is bf16, so
// every product x * part is exact in fp32 and the tensor core's fp32
// accumulation gives fp32-accurate logits.
//
// The reduction over H is split in KS slices: CTA (tile, q) computes a tile
// of 128 tokens x all E experts (E <= 256) over slice q of H in tensor
// memory, D[token][expert], summing the lo, mid and hi parts (small ones
// first).  Few tensor-core accumulation steps per accumulator keep the logit
// error near plain fp32 accumulation, and the KS CTAs of a tile run on KS
// SMs.  Warp 0 streams x tiles and split-weight tiles by TMA (128-byte
// swizzle), lane 0 of warp 1 issues the MMAs, and warps 4-7 (one
// tensor-memory lane = one token each) write the slice's partial logits
// into the CTA's own shared memory.  The KS CTAs of a tile form a cluster:
// after a cluster barrier, CTA q adds, for its 128/KS tokens, the KS slices
// in slice order, reading the others' shared memory (distributed shared
// memory), and its eight warps select each token's experts with the
// router's warp selection (route_select_warp: one warp per token, ties to
// the lower index, the routing flags' weights).
#include "route_select.cuh"
#include "tc_common.cuh"

namespace qsm {
namespace route_tc {

constexpr int BM = 128;  // tokens per tile
constexpr int BK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxE = 256;

struct Params {
  CUtensorMap xa;  // x [T, H] bf16, box {64, 128}
  CUtensorMap wb;  // split router weight [3E, H] bf16, box {64, E}
  const float* bias;
  int T, H, E, k, renorm, ntiles, ks;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* status;
};

__device__ __forceinline__ uint32_t bf16_split3(float v, uint32_t& mid, uint32_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(m);
  mid = __bfloat16_as_ushort(m);
  lo = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
  return __bfloat16_as_ushort(h);
}

// out[p*n + i] = part p of w[i] (hi, mid, lo); n % 4 == 0.
__global__ void __launch_bounds__(256)
split_kernel(const float* __restrict__ w, __nv_bfloat16* __restrict__ out, size_t n) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t n4 = n / 4;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  uint2* o = reinterpret_cast<uint2*>(out);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(w) + i);
    uint32_t m0, m1, m2, m3, l0, l1, l2, l3;
    const uint32_t h0 = bf16_split3(v.x, m0, l0), h1 = bf16_split3(v.y, m1, l1);
    const uint32_t h2 = bf16_split3(v.z, m2, l2), h3 = bf16_split3(v.w, m3, l3);
    o[i] = make_uint2(h0 | (h1 << 16), h2 | (h3 << 16));
    o[n4 + i] = make_uint2(m0 | (m1 << 16), m2 | (m3 << 16));
    o[2 * n4 + i] = make_uint2(l0 | (l1 << 16), l2 | (l3 << 16));
  }
}

// Instruction descriptor, kind::f16 with bf16 A and B (K-major), fp32 D.
__device__ __forceinline__ uint32_t idesc_bf16_m128(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}

template <int KS>  // slices of H (p.ks == KS)
__global__ void __launch_bounds__(kThreads, 1)
route_tc_kernel(const __grid_constant__ Params p) {
  constexpr int A_BYTES = BM * BK * 2;
  constexpr int B_MAX = 256 * BK * 2;
  constexpr int STAGE = A_BYTES + B_MAX;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], accf_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / KS, q = blockIdx.x - tile * KS;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&accf_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_map(&p.xa);
    tc::prefetch_map(&p.wb);
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, 256);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  pdl_wait();
  pdl_launch_dependents();
  volatile int* abort_p = &abort_flag;
  const int kq = p.H / BK / KS;  // K steps of 64 per slice and part
  const int steps = 3 * kq;
  auto wait = [&](uint64_t* bar, uint32_t par) {
    for (uint32_t i = 0; i < kWaitIters; ++i) {
      if (mbar_try_wait(bar, par)) return true;
      if (*abort_p) return false;
    }
    *abort_p = 1;
    set_status(p.status, QSM_DEV_TIMEOUT);
    return false;
  };

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t bytes = A_BYTES + (uint32_t)p.E * BK * 2;
      for (int st = 0, s = 0; st < steps && !*abort_p; ++st) {
        if (st >= kStages && !wait(&empty_bar[s], ((st / kStages) - 1) & 1)) break;
        const int pi = st / kq, kk = q * kq + (st - pi * kq);
        const int part = 2 - pi;  // lo, mid, hi
        unsigned char* sb = smem + s * STAGE;
        mbar_arrive_expect_tx(&full_bar[s], bytes);
        tc::tma_load_2d(sb, &p.xa, kk * BK, tile * BM, &full_bar[s]);
        tc::tma_load_2d(sb + A_BYTES, &p.wb, kk * BK, part * p.E, &full_bar[s]);
        s = (s + 1 == kStages) ? 0 : s + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_m128(p.E);
      bool ok = true;
      for (int st = 0, s = 0; st < steps; ++st) {
        if (!wait(&full_bar[s], (st / kStages) & 1)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t a0 = smem_u32(smem + s * STAGE);
        const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc::mma_f16(tmem, tc::sw128_desc(a0 + kk * 32), tc::sw128_desc(b0 + kk * 32),
                      idesc, (st > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(&empty_bar[s]);
        s = (s + 1 == kStages) ? 0 : s + 1;
      }
      if (ok) tc::mma_commit(&accf_bar);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;  // token row of the tile = TMEM lane
    const bool ok = wait(&accf_bar, 0);
    tc::tc_fence_after();
    // this slice's partial logits -> this CTA's shared memory [row][E + 4]
    // (the pipeline stages are free: every MMA has completed)
    const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16);
    float* prow = reinterpret_cast<float*>(smem) + row * (p.E + 4);
    if (ok) {
      for (int c0 = 0; c0 < p.E; c0 += 16) {
        float v[16];
        tc::tmem_ld16(taddr + c0, v);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<float4*>(prow + c0 + 4 * u) =
              make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every slice of the tile is in its CTA's shared memory

  // CTA q: tokens [q * rpc, (q + 1) * rpc) of the tile.  Their logits: the
  // KS slices added in slice order (the bias is added at selection).  All
  // slices of a position are read before its sum is written.
  const int ld = p.E + 4;
  const int rpc = BM / KS, r0 = q * rpc;
  const int rows = min(BM, p.T - tile * BM);
  const float* pl = reinterpret_cast<const float*>(smem);  // [BM][ld], every CTA
  // the sums overwrite this CTA's own rows in place: the other CTAs read only
  // the rows of their own token ranges from this CTA
  float* lg = reinterpret_cast<float*>(smem) + r0 * ld;      // [rpc][ld]
  const int e4 = p.E / 4;
#pragma unroll 4
  for (int pos = threadIdx.x; pos < rpc * e4; pos += kThreads) {
    const int rr = pos / e4, c = pos - rr * e4;
    const uint32_t off = smem_u32(pl + (r0 + rr) * ld + 4 * c);
    float4 sl[KS];
#pragma unroll
    for (int s2 = 0; s2 < KS; ++s2) sl[s2] = dsmem_ld_f4(dsmem_addr_u32(off, s2));
    float4 a = sl[0];
#pragma unroll
    for (int s2 = 1; s2 < KS; ++s2) {
      a.x += sl[s2].x;
      a.y += sl[s2].y;
      a.z += sl[s2].z;
      a.w += sl[s2].w;
    }
    *reinterpret_cast<float4*>(lg + rr * ld + 4 * c) = a;
  }
  __syncthreads();
  // one warp per token: top k, routing weights
  if (!*abort_p) {
    for (int rr = warp; rr < rpc; rr += kThreads / 32) {
      if (r0 + rr >= rows) break;
      int my_e;
      float my_l, my_w;
      route_select_warp<kMaxE / 32, true>(lg + rr * ld, p.bias, p.E, p.k, p.renorm, p.status,
                                          my_e, my_l, my_w);
      const size_t t = (size_t)tile * BM + r0 + rr;
      if (lane < p.k) {
        p.topk_idx[t * p.k + lane] = my_e;
        p.topk_w[t * p.k + lane] = my_w;
      }
    }
  }
  cluster_sync_all();  // no CTA leaves while another still reads its slices
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 256);
}

int sm_count_route() {
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  return v > 0 ? v : 148;
}

}  // namespace route_tc

bool route_tc_supported(int T, int H, int E, int k) {
  return T > 64 && H % 128 == 0 && E % 16 == 0 && E >= 16 && E <= 256 && k <= 8;
}

namespace route_tc {
// H slices: 4 when H allows it (every slice a whole number of 64-wide steps)
int k_slices(int H) { return H % (4 * BK) == 0 ? 4 : (H % (2 * BK) == 0 ? 2 : 1); }
inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }
}  // namespace route_tc

// [256-byte header, zero][split router weight 3*E*H bf16]
size_t route_tc_workspace_bytes(int T, int H, int E) {
  using namespace route_tc;
  (void)T;
  return 256 + up256((size_t)3 * E * H * 2);
}

qsm_status route_tc_launch(const uint16_t* x, const float* w_router,
                           const float* logit_bias, int T, int H, int E, int k,
                           int renormalize, int32_t* topk_idx, float* topk_w,
                           void* split_buf, int32_t* dev_status,
                           cudaStream_t stream) {
  using namespace route_tc;
  const size_t n = (size_t)E * H;
  const int ntiles = (T + BM - 1) / BM;
  char* ws = static_cast<char*>(split_buf);
  __nv_bfloat16* split = reinterpret_cast<__nv_bfloat16*>(ws + 256);
  const int nsm = sm_count_route();
  QSM_CUDA_TRY(launch_pdl(split_kernel, dim3(nsm), dim3(256), 0, stream, w_router,
                          split, n));
  Params p = {};
  if (!tc::make_map_2d(&p.xa, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, BK, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_map_2d(&p.wb, split, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                       (uint64_t)3 * E, H, BK, E, CU_TENSOR_MAP_SWIZZLE_128B))
    return QSM_ERR_CUDA;
  p.bias = logit_bias;
  p.T = T;
  p.H = H;
  p.E = E;
  p.k = k;
  p.renorm = renormalize;
  p.ntiles = ntiles;
  p.ks = k_slices(H);
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  p.status = dev_status;
  const size_t smem = (size_t)kStages * (BM * BK * 2 + 256 * BK * 2) + 1024;
  auto* kern = p.ks == 4 ? route_tc_kernel<4>
                         : (p.ks == 2 ? route_tc_kernel<2> : route_tc_kernel<1>);
  QSM_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem));
  // the ks CTAs of a tile are one cluster (they exchange their slices)
  QSM_CUDA_TRY(
      launch_pdl_cluster(kern, dim3(ntiles * p.ks), dim3(kThreads), p.ks, smem, stream, p));
  return QSM_OK;
}

}  // namespace qsm
