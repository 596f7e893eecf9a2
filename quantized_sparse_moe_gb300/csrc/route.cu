// Router: logits, top-k selection and routing weights in one launch.
//
// "Optimizing on-device inference for Apple Silicon", section "Qwen creates
// three distinct workload shapes": the router scores every expert for each
// token and keeps the best eight.  Readings: ties go to the lower expert
// index; the weights are the softmax over the selected logits
// (renormalize != 0) or the full softmax taken at the selected ones.
//
// Layout of the work: blockIdx.x owns kExpertsPerCta experts, blockIdx.y a
// block of kTokPerCta tokens.  Each expert's dot products are split over
// 128 threads (float4 slices of the router row, 8-byte bf16 slices of x).
// The logits land in the workspace; the CTA that finishes last for a token
// block (a per-block arrival counter, no waiting) selects the top k for
// those tokens, one warp per token, and re-arms the counter to zero.
#include "qsm_common.cuh"

namespace qsm {
namespace {

constexpr int kThreads = 256;
constexpr int kExpertsPerCta = 2;
constexpr int kThreadsPerExpert = kThreads / kExpertsPerCta;  // 128
constexpr int kTokPerCta = 8;
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;

size_t counters_offset(int T, int E) {
  size_t b = (size_t)T * E * sizeof(float);
  return (b + 255) & ~size_t(255);
}

__global__ void __launch_bounds__(kThreads)
route_kernel(const uint16_t* __restrict__ x, const float* __restrict__ w,
             const float* __restrict__ bias, int T, int H, int E, int k,
             int renormalize, int32_t* __restrict__ topk_idx,
             float* __restrict__ topk_w, float* __restrict__ logits,
             unsigned int* __restrict__ counters, int32_t* dev_status) {
  __shared__ float red[kExpertsPerCta][kThreadsPerExpert / 32][kTokPerCta];
  __shared__ int is_last;

  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int sub = tid / kThreadsPerExpert;          // expert within the CTA
  const int st = tid % kThreadsPerExpert;           // thread within expert
  const int e = blockIdx.x * kExpertsPerCta + sub;
  const int t0 = blockIdx.y * kTokPerCta;
  const int nt = min(kTokPerCta, T - t0);

  // Router row slice is read-only model data: fetch before the wait.
  const float4* wrow = reinterpret_cast<const float4*>(w + (size_t)min(e, E - 1) * H);
  const int H4 = H / 4;
  pdl_wait();

  float acc[kTokPerCta];
#pragma unroll
  for (int i = 0; i < kTokPerCta; ++i) acc[i] = 0.f;
  if (e < E) {
    for (int h4 = st; h4 < H4; h4 += kThreadsPerExpert) {
      const float4 wv = __ldg(wrow + h4);
#pragma unroll
      for (int i = 0; i < kTokPerCta; ++i) {
        if (i < nt) {
          const uint2 xv = __ldg(reinterpret_cast<const uint2*>(
              x + (size_t)(t0 + i) * H + 4 * h4));
          float a = acc[i];
          a = fmaf(wv.x, bf16_lo(xv.x), a);
          a = fmaf(wv.y, bf16_hi(xv.x), a);
          a = fmaf(wv.z, bf16_lo(xv.y), a);
          a = fmaf(wv.w, bf16_hi(xv.y), a);
          acc[i] = a;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kTokPerCta; ++i) {
    const float s = warp_sum(acc[i]);
    if (lane == 0) red[sub][st / 32][i] = s;
  }
  __syncthreads();
  if (tid < kExpertsPerCta * kTokPerCta) {
    const int s2 = tid / kTokPerCta, i = tid % kTokPerCta;
    const int e2 = blockIdx.x * kExpertsPerCta + s2;
    if (e2 < E && i < nt) {
      float v = 0.f;
#pragma unroll
      for (int wq = 0; wq < kThreadsPerExpert / 32; ++wq) v += red[s2][wq][i];
      if (bias) v += bias[e2];
      logits[(size_t)(t0 + i) * E + e2] = v;
    }
  }

  // Arrival: the last CTA of this token block selects the experts.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&counters[blockIdx.y], 1u);
    is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  const int warp = tid / 32;
  if (warp < nt) {
    const int t = t0 + warp;
    constexpr int kPer = kMaxE / 32;
    float v[kPer];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int ee = lane + 32 * i;
      float l = -INFINITY;
      if (ee < E) {
        l = __ldcg(logits + (size_t)t * E + ee);
        if (!isfinite(l)) {
          bad = true;
          l = -INFINITY;
        }
      }
      v[i] = l;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0)
      set_status(dev_status, QSM_DEV_NONFINITE);
    uint32_t taken = 0;  // bit i: candidate lane + 32 i already selected
    float top = 0.f, sel_l[kMaxK];
    int sel_e[kMaxK];
    for (int j = 0; j < k; ++j) {
      // local best among this lane's untaken candidates (value desc, index asc)
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int ee = lane + 32 * i;
        if (ee < E && !((taken >> i) & 1u)) {
          if (v[i] > bv || (v[i] == bv && ee < be)) {
            bv = v[i];
            be = ee;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (j == 0) top = bv;
      sel_l[j < kMaxK ? j : 0] = bv;
      sel_e[j < kMaxK ? j : 0] = be;
    }
    float denom = 0.f;
    if (renormalize) {
      for (int j = 0; j < k; ++j) denom += __expf(sel_l[j] - top);
    } else {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (lane + 32 * i < E) part += __expf(v[i] - top);
      denom = warp_sum(part);
    }
    const float inv = 1.0f / denom;
    for (int j = lane; j < k; j += 32) {
      // sel_l / sel_e are uniform across the warp; index them by j
      topk_idx[(size_t)t * k + j] = sel_e[j];
      topk_w[(size_t)t * k + j] = __expf(sel_l[j] - top) * inv;
    }
  }
  if (tid == 0) counters[blockIdx.y] = 0u;  // re-arm for the next call
}

}  // namespace
}  // namespace qsm

extern "C" size_t moe_route_workspace_bytes(int32_t T, int32_t E) {
  if (T < 0 || E <= 0) return 0;
  const size_t nblk = (size_t)(T + qsm::kTokPerCta - 1) / qsm::kTokPerCta;
  return qsm::counters_offset(T, E) + ((nblk * 4 + 255) & ~size_t(255));
}

extern "C" qsm_status moe_route(const uint16_t* x, const float* w_router,
                                const float* logit_bias, int32_t T, int32_t H,
                                int32_t E, int32_t k, int32_t renormalize,
                                int32_t* topk_idx, float* topk_w,
                                void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, cudaStream_t stream) {
  using namespace qsm;
  if (T < 0 || H <= 0 || H % 64 || E < 1 || E > kMaxE || k < 1 || k > E ||
      k > kMaxK)
    return QSM_ERR_INVALID_ARGUMENT;
  if (T == 0) return QSM_OK;
  if (!x || !w_router || !topk_idx || !topk_w || !workspace || !dev_status)
    return QSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace) ||
      !aligned4(topk_idx) || !aligned4(topk_w) || !aligned4(dev_status) ||
      (logit_bias && !aligned4(logit_bias)))
    return QSM_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < moe_route_workspace_bytes(T, E))
    return QSM_ERR_WORKSPACE_TOO_SMALL;
  float* logits = static_cast<float*>(workspace);
  unsigned* counters = reinterpret_cast<unsigned*>(
      static_cast<char*>(workspace) + counters_offset(T, E));
  dim3 grid((E + kExpertsPerCta - 1) / kExpertsPerCta,
            (T + kTokPerCta - 1) / kTokPerCta);
  QSM_CUDA_TRY(launch_pdl(route_kernel, grid, dim3(kThreads), 0, stream, x,
                          w_router, logit_bias, T, H, E, k, renormalize,
                          topk_idx, topk_w, logits, counters, dev_status));
  return QSM_OK;
}
