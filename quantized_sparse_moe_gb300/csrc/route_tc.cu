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
// One CTA computes a tile of 128 tokens x all E experts (E <= 256) in tensor
// memory: D[token][expert], in two accumulators, one per half of H, each
// summing the lo, mid and hi parts (small ones first); the epilogue adds the
// halves in fp32.  Fewer tensor-core accumulation steps per accumulator keep
// the logit error near plain fp32 accumulation.  Warp 0 streams x tiles and split-weight tiles
// by TMA (128-byte swizzle), lane 0 of warp 1 issues the MMAs over K =
// 3 * H, and warps 4-7 (one tensor-memory lane = one token each) read the
// E logits of their token, keep the top k in registers and write the
// routing weights.
#include "tc_common.cuh"

namespace qsm {
namespace route_tc {

constexpr int BM = 128;  // tokens per tile
constexpr int BK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kMaxTopK = 8;

struct Params {
  CUtensorMap xa;  // x [T, H] bf16, box {64, 128}
  CUtensorMap wb;  // split router weight [3E, H] bf16, box {64, E}
  const float* bias;
  int T, H, E, k, renorm, ntiles;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* status;
};

// out[p*E*H + i] = part p of w[i] (hi, mid, lo).
__global__ void __launch_bounds__(256)
split_kernel(const float* __restrict__ w, __nv_bfloat16* __restrict__ out, size_t n) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const float v = __ldg(w + i);
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

// Instruction descriptor, kind::f16 with bf16 A and B (K-major), fp32 D.
__device__ __forceinline__ uint32_t idesc_bf16_m128(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}

__global__ void __launch_bounds__(kThreads, 1)
route_tc_kernel(const __grid_constant__ Params p) {
  constexpr int A_BYTES = BM * BK * 2;
  constexpr int B_MAX = 256 * BK * 2;
  constexpr int STAGE = A_BYTES + B_MAX;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], accf_bar,
      acce_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&accf_bar, 1);
    mbar_init(&acce_bar, 128);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_map(&p.xa);
    tc::prefetch_map(&p.wb);
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  pdl_wait();
  pdl_launch_dependents();
  volatile int* abort_p = &abort_flag;
  const int kh = p.H / BK;
  const int steps = 3 * kh;
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
      int s = 0, fill = 0;
      const uint32_t bytes = A_BYTES + (uint32_t)p.E * BK * 2;
      for (int tile = blockIdx.x; tile < p.ntiles && !*abort_p; tile += gridDim.x) {
        for (int st = 0; st < steps; ++st) {
          if (fill >= kStages && !wait(&empty_bar[s], ((fill / kStages) - 1) & 1)) break;
          const int pi = st / kh, ks = st - pi * kh;
          const int part = 2 - pi;  // lo, mid, hi
          unsigned char* sb = smem + s * STAGE;
          mbar_arrive_expect_tx(&full_bar[s], bytes);
          tc::tma_load_2d(sb, &p.xa, ks * BK, tile * BM, &full_bar[s]);
          tc::tma_load_2d(sb + A_BYTES, &p.wb, ks * BK, part * p.E, &full_bar[s]);
          ++fill;
          s = (s + 1 == kStages) ? 0 : s + 1;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int s = 0, fill = 0, j = 0;
      const uint32_t idesc = idesc_bf16_m128(p.E);
      for (int tile = blockIdx.x; tile < p.ntiles && !*abort_p; tile += gridDim.x, ++j) {
        if (j > 0 && !wait(&acce_bar, (j - 1) & 1)) break;
        tc::tc_fence_after();
        bool ok = true;
        for (int st = 0; st < steps; ++st) {
          if (!wait(&full_bar[s], (fill / kStages) & 1)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * STAGE);
          const uint32_t b0 = a0 + A_BYTES;
          const int pi = st / kh, ks = st - pi * kh;
          const int acc = ks < kh / 2 ? 0 : 1;  // accumulator of this half of H
          const bool first = pi == 0 && (ks == 0 || ks == kh / 2);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_f16(tmem + acc * 256, tc::sw128_desc(a0 + kk * 32),
                        tc::sw128_desc(b0 + kk * 32), idesc,
                        (!first || kk > 0) ? 1u : 0u);
          tc::mma_commit(&empty_bar[s]);
          ++fill;
          s = (s + 1 == kStages) ? 0 : s + 1;
        }
        if (!ok) break;
        tc::mma_commit(&accf_bar);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int q4 = warp & 3;
    int j = 0;
    bool bad = false;
    for (int tile = blockIdx.x; tile < p.ntiles && !*abort_p; tile += gridDim.x, ++j) {
      if (!wait(&accf_bar, j & 1)) break;
      tc::tc_fence_after();
      const int t = tile * BM + 32 * q4 + lane;
      const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16);
      float val[kMaxTopK];
      int idx[kMaxTopK];
#pragma unroll
      for (int i = 0; i < kMaxTopK; ++i) {
        val[i] = -INFINITY;
        idx[i] = 0x7fffffff;
      }
      for (int c0 = 0; c0 < p.E; c0 += 16) {
        float v[16], v2[16];
        tc::tmem_ld16(taddr + c0, v);
        tc::tmem_ld16(taddr + 256 + c0, v2);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float l = v[c] + v2[c] + (p.bias ? __ldg(p.bias + c0 + c) : 0.f);
          if (!isfinite(l)) {
            bad = bad || t < p.T;
            l = -INFINITY;
          }
          int ci = c0 + c;
          // keep the best kMaxTopK (value desc, index asc); indices arrive
          // in ascending order, so an equal value never displaces
          if (l > val[kMaxTopK - 1] || (l == val[kMaxTopK - 1] && ci < idx[kMaxTopK - 1])) {
#pragma unroll
            for (int i = 0; i < kMaxTopK; ++i) {
              if (l > val[i] || (l == val[i] && ci < idx[i])) {
                const float tv = val[i];
                const int ti = idx[i];
                val[i] = l;
                idx[i] = ci;
                l = tv;
                ci = ti;
              }
            }
          }
        }
      }
      const float top = val[0];
      float denom = 0.f;
      if (p.renorm) {
#pragma unroll
        for (int i = 0; i < kMaxTopK; ++i)
          if (i < p.k) denom += __expf(val[i] - top);
      } else {
        for (int c0 = 0; c0 < p.E; c0 += 16) {
          float v[16], v2[16];
          tc::tmem_ld16(taddr + c0, v);
          tc::tmem_ld16(taddr + 256 + c0, v2);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float l = v[c] + v2[c] + (p.bias ? __ldg(p.bias + c0 + c) : 0.f);
            if (isfinite(l)) denom += __expf(l - top);
          }
        }
      }
      const float inv = 1.0f / denom;
      if (t < p.T) {
#pragma unroll
        for (int i = 0; i < kMaxTopK; ++i) {
          if (i < p.k) {
            p.topk_idx[(size_t)t * p.k + i] = idx[i];
            p.topk_w[(size_t)t * p.k + i] = __expf(val[i] - top) * inv;
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acce_bar);
    }
    if (bad) set_status(p.status, QSM_DEV_NONFINITE);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
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

size_t route_tc_split_bytes(int H, int E) { return (size_t)3 * E * H * 2; }

qsm_status route_tc_launch(const uint16_t* x, const float* w_router,
                           const float* logit_bias, int T, int H, int E, int k,
                           int renormalize, int32_t* topk_idx, float* topk_w,
                           void* split_buf, int32_t* dev_status,
                           cudaStream_t stream) {
  using namespace route_tc;
  const size_t n = (size_t)E * H;
  __nv_bfloat16* split = static_cast<__nv_bfloat16*>(split_buf);
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
  p.ntiles = (T + BM - 1) / BM;
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  p.status = dev_status;
  const size_t smem = (size_t)kStages * (BM * BK * 2 + 256 * BK * 2) + 1024;
  QSM_CUDA_TRY(cudaFuncSetAttribute(route_tc_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem));
  const int grid = p.ntiles < nsm ? p.ntiles : nsm;
  QSM_CUDA_TRY(launch_pdl(route_tc_kernel, dim3(grid), dim3(kThreads), smem, stream, p));
  return QSM_OK;
}

}  // namespace qsm
