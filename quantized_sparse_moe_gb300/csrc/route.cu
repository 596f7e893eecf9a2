// Router: logits, top-k selection and routing weights in one launch.
//
// "Optimizing on-device inference for Apple Silicon", section "Qwen creates
// three distinct workload shapes": the router scores every expert for each
// token and keeps the best eight.  Readings: ties go to the lower expert
// index; the weights are the softmax over the selected logits
// (QSM_ROUTE_RENORMALIZE) or the full softmax taken at the selected ones;
// with QSM_ROUTE_BIAS_SELECT_ONLY the logit bias decides the selection but
// the weights use the logits without it.  The workspace holds the logits
// without the bias; the selecting CTA adds it.
//
// Layout of the work: blockIdx.x owns kExpertsPerCta experts, blockIdx.y a
// block of kTokPerCta tokens.  Each expert's dot products are split over
// 128 threads (float4 slices of the router row, 8-byte bf16 slices of x).
// The logits land in the workspace; the CTA that finishes last for a token
// block (a per-block arrival counter, no waiting) selects the top k for
// those tokens, one warp per token, and re-arms the counter to zero.
//
// With kGroup (one token block, E <= 256) that same last CTA also groups
// the T*k assignments ("Keeping expert routing on the GPU": histogram,
// prefix scan, stable scatter, block map) from the ids it holds in shared
// memory, so routing plus grouping is one launch for decode batches.
#include "route_select.cuh"

namespace qsm {
namespace {

constexpr int kThreads = 256;
constexpr int kExpertsPerCta = 2;
constexpr int kThreadsPerExpert = kThreads / kExpertsPerCta;  // 128
constexpr int kTokPerCta = 8;
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kRouteFlags = QSM_ROUTE_RENORMALIZE | QSM_ROUTE_BIAS_SELECT_ONLY;

// CUDA-core path workspace: [arrival counters][logits T x E fp32]
size_t counters_bytes(int T) {
  const size_t nblk = (size_t)(T + kTokPerCta - 1) / kTokPerCta;
  return (nblk * 4 + 255) & ~size_t(255);
}

constexpr int kWPer = 4;  // float4 of the router row per thread and batch

// Grouping outputs of the fused variant (see qsm_grouping).
struct GroupOut {
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* tile_map;
  int32_t* n_tiles;
  int tile_rows;
  int max_tiles;
};

// Groups the A = T*k assignments a = t*k + j whose experts sit in
// sel_e[t][j]: thread e counts expert e, two block scans give the start
// offsets and first block of every expert, and each thread scatters its
// expert's assignments in increasing a (a stable sort by expert).  Needs
// E <= blockDim.x == kThreads.
__device__ void group_in_cta(const int (*sel_e)[kMaxK], int T, int k, int E,
                             const GroupOut& g, int* s_cnt, int* s_blk) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int A = T * k, BM = g.tile_rows;
  int cnt = 0;
  if (tid < E)
    for (int a = 0; a < A; ++a) cnt += (sel_e[a / k][a % k] == tid);
  const int nb = (cnt + BM - 1) / BM;
  int ic = cnt, ib = nb;  // inclusive warp scans
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int c2 = __shfl_up_sync(0xffffffffu, ic, o);
    const int b2 = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ic += c2;
      ib += b2;
    }
  }
  if (lane == 31) {
    s_cnt[warp] = ic;
    s_blk[warp] = ib;
  }
  __syncthreads();
  int cbase = 0, bbase = 0, ctot = 0, btot = 0;
#pragma unroll
  for (int w2 = 0; w2 < kThreads / 32; ++w2) {
    if (w2 < warp) {
      cbase += s_cnt[w2];
      bbase += s_blk[w2];
    }
    ctot += s_cnt[w2];
    btot += s_blk[w2];
  }
  const int off = cbase + ic - cnt, b0 = bbase + ib - nb;
  if (tid < E) {
    g.counts[tid] = cnt;
    g.offsets[tid] = off;
    for (int m = 0; m < nb && b0 + m < g.max_tiles; ++m) {
      g.tile_map[2 * (b0 + m)] = tid;
      g.tile_map[2 * (b0 + m) + 1] = off + m * BM;
    }
    int pos = off;
    for (int a = 0; a < A && pos < off + cnt; ++a) {
      if (sel_e[a / k][a % k] == tid) {
        g.perm[pos] = a;
        g.inv_perm[a] = pos;
        ++pos;
      }
    }
  }
  if (tid == 0) {
    g.offsets[E] = ctot;
    g.n_tiles[0] = btot < g.max_tiles ? btot : g.max_tiles;
  }
  for (int i = btot + tid; i < g.max_tiles; i += kThreads) {  // sentinels
    g.tile_map[2 * i] = -1;
    g.tile_map[2 * i + 1] = -1;
  }
}

template <int kPer, bool kGroup>  // kPer: top-k candidates per lane, ceil(E/32)
__global__ void __launch_bounds__(kThreads)
route_kernel(const uint16_t* __restrict__ x, const float* __restrict__ w,
             const float* __restrict__ bias, int T, int H, int E, int k,
             int renormalize, int32_t* __restrict__ topk_idx,
             float* __restrict__ topk_w, float* __restrict__ logits,
             unsigned int* __restrict__ counters, int32_t* dev_status,
             GroupOut gout) {
  __shared__ float red[kExpertsPerCta][kThreadsPerExpert / 32][kTokPerCta];
  __shared__ float sel_l[kThreads / 32][kMaxK];
  __shared__ int sel_e[kThreads / 32][kMaxK];
  __shared__ int is_last;
  __shared__ int s_cnt[kThreads / 32], s_blk[kThreads / 32];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int sub = tid / kThreadsPerExpert;          // expert within the CTA
  const int st = tid % kThreadsPerExpert;           // thread within expert
  const int e = blockIdx.x * kExpertsPerCta + sub;
  const int t0 = blockIdx.y * kTokPerCta;
  const int nt = min(kTokPerCta, T - t0);
  const int H4 = H / 4;

  // The router row is model data no launch writes: fetch it before waiting.
  const float4* wrow = reinterpret_cast<const float4*>(w + (size_t)min(e, E - 1) * H);
  float4 wv[kWPer];
#pragma unroll
  for (int i = 0; i < kWPer; ++i) {
    const int h4 = st + i * kThreadsPerExpert;
    wv[i] = h4 < H4 ? __ldg(wrow + h4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();
  pdl_launch_dependents();

  float acc[kTokPerCta];
#pragma unroll
  for (int i = 0; i < kTokPerCta; ++i) acc[i] = 0.f;
  for (int hb = 0; hb < H4; hb += kWPer * kThreadsPerExpert) {
    if (hb > 0) {
#pragma unroll
      for (int i = 0; i < kWPer; ++i) {
        const int h4 = hb + st + i * kThreadsPerExpert;
        wv[i] = h4 < H4 ? __ldg(wrow + h4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int tt = 0; tt < kTokPerCta; ++tt) {
      if (tt < nt) {
        const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)(t0 + tt) * H);
        uint2 xv[kWPer];
#pragma unroll
        for (int i = 0; i < kWPer; ++i) {
          const int h4 = hb + st + i * kThreadsPerExpert;
          xv[i] = h4 < H4 ? __ldg(xr + h4) : make_uint2(0u, 0u);
        }
        float a = acc[tt];
#pragma unroll
        for (int i = 0; i < kWPer; ++i) {
          a = fmaf(wv[i].x, bf16_lo(xv[i].x), a);
          a = fmaf(wv[i].y, bf16_hi(xv[i].x), a);
          a = fmaf(wv[i].z, bf16_lo(xv[i].y), a);
          a = fmaf(wv[i].w, bf16_hi(xv[i].y), a);
        }
        acc[tt] = a;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kTokPerCta; ++i) {
    if (i < nt) {
      const float s2 = warp_sum(acc[i]);
      if (lane == 0) red[sub][st / 32][i] = s2;
    }
  }
  __syncthreads();
  if (tid < kExpertsPerCta * kTokPerCta) {
    const int s2 = tid / kTokPerCta, i = tid % kTokPerCta;
    const int e2 = blockIdx.x * kExpertsPerCta + s2;
    if (e2 < E && i < nt) {
      float v = 0.f;
#pragma unroll
      for (int wq = 0; wq < kThreadsPerExpert / 32; ++wq) v += red[s2][wq][i];
      logits[(size_t)(t0 + i) * E + e2] = v;
    }
  }

  // Arrival: the last CTA of this token block selects the experts.  The
  // writers make their logits visible device-wide, one thread per CTA
  // counts the arrival, and the last arrival reads the others' logits.
  if (tid < kExpertsPerCta * kTokPerCta) __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&counters[blockIdx.y], 1u);
    is_last = (prev == gridDim.x - 1);
    if (is_last) __threadfence();
  }
  __syncthreads();
  if (!is_last) return;

  const int warp = tid / 32;
  if (warp < nt) {
    const int t = t0 + warp;
    int my_e;
    float my_l, my_w;
    route_select_warp<kPer>(logits + (size_t)t * E, bias, E, k, renormalize, dev_status,
                            my_e, my_l, my_w);
    if (lane < k) {
      sel_l[warp][lane] = my_l;
      sel_e[warp][lane] = my_e;
      topk_idx[(size_t)t * k + lane] = my_e;
      topk_w[(size_t)t * k + lane] = my_w;
    }
    __syncwarp();
  }
  if (tid == 0) counters[blockIdx.y] = 0u;  // re-arm for the next call
  if constexpr (kGroup) {
    __syncthreads();
    group_in_cta(sel_e, nt, k, E, gout, s_cnt, s_blk);
  }
}

}  // namespace
}  // namespace qsm

namespace qsm {
bool route_tc_supported(int T, int H, int E, int k);
size_t route_tc_workspace_bytes(int T, int H, int E);
qsm_status route_tc_launch(const uint16_t* x, const float* w_router,
                           const float* logit_bias, int T, int H, int E, int k,
                           int renormalize, int32_t* topk_idx, float* topk_w,
                           void* split_buf, int32_t* dev_status,
                           cudaStream_t stream);
}  // namespace qsm

extern "C" size_t moe_route_workspace_bytes(int32_t T, int32_t H, int32_t E) {
  if (T < 0 || H <= 0 || E <= 0) return 0;
  if (qsm::route_tc_supported(T, H, E, 1)) return qsm::route_tc_workspace_bytes(T, H, E);
  return qsm::counters_bytes(T) + (((size_t)T * E * sizeof(float) + 255) & ~size_t(255));
}

extern "C" qsm_status moe_route(const uint16_t* x, const float* w_router,
                                const float* logit_bias, int32_t T, int32_t H,
                                int32_t E, int32_t k, int32_t renormalize,
                                int32_t* topk_idx, float* topk_w,
                                void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, cudaStream_t stream) {
  using namespace qsm;
  if (T < 0 || H <= 0 || H % 64 || E < 1 || E > kMaxE || k < 1 || k > E ||
      k > kMaxK || (renormalize & ~kRouteFlags))
    return QSM_ERR_INVALID_ARGUMENT;
  if (T == 0) return QSM_OK;
  if (!x || !w_router || !topk_idx || !topk_w || !workspace || !dev_status)
    return QSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace) ||
      !aligned4(topk_idx) || !aligned4(topk_w) || !aligned4(dev_status) ||
      (logit_bias && !aligned4(logit_bias)))
    return QSM_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < moe_route_workspace_bytes(T, H, E))
    return QSM_ERR_WORKSPACE_TOO_SMALL;
  if (route_tc_supported(T, H, E, k))  // many tokens: tensor-core logits
    return route_tc_launch(x, w_router, logit_bias, T, H, E, k, renormalize,
                           topk_idx, topk_w, workspace, dev_status, stream);
  unsigned* counters = static_cast<unsigned*>(workspace);
  float* logits = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           counters_bytes(T));
  dim3 grid((E + kExpertsPerCta - 1) / kExpertsPerCta,
            (T + kTokPerCta - 1) / kTokPerCta);
  const GroupOut none = {};
  if (E <= 256)
    QSM_CUDA_TRY(launch_pdl(route_kernel<8, false>, grid, dim3(kThreads), 0, stream,
                            x, w_router, logit_bias, T, H, E, k, renormalize,
                            topk_idx, topk_w, logits, counters, dev_status, none));
  else
    QSM_CUDA_TRY(launch_pdl(route_kernel<kMaxE / 32, false>, grid, dim3(kThreads), 0,
                            stream, x, w_router, logit_bias, T, H, E, k,
                            renormalize, topk_idx, topk_w, logits, counters,
                            dev_status, none));
  return QSM_OK;
}

extern "C" qsm_status moe_route_group(const uint16_t* x, const float* w_router,
                                      const float* logit_bias, int32_t T,
                                      int32_t H, int32_t E, int32_t k,
                                      int32_t renormalize, int32_t* topk_idx,
                                      float* topk_w, const qsm_grouping* g,
                                      void* workspace, size_t workspace_bytes,
                                      int32_t* dev_status, cudaStream_t stream) {
  using namespace qsm;
  if (renormalize & ~kRouteFlags) return QSM_ERR_INVALID_ARGUMENT;
  if (T < 1 || T > kTokPerCta || H <= 0 || H % 64 || E < 1 || E > kThreads ||
      k < 1 || k > E || k > kMaxK)
    return QSM_ERR_UNSUPPORTED;
  if (!x || !w_router || !topk_idx || !topk_w || !workspace || !dev_status || !g ||
      !g->counts || !g->offsets || !g->perm || !g->inv_perm || !g->tile_map ||
      !g->n_tiles || g->tile_rows < 1 ||
      g->max_tiles < moe_group_max_tiles(T, k, E, g->tile_rows))
    return QSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace) ||
      !aligned4(topk_idx) || !aligned4(topk_w) || !aligned4(dev_status) ||
      (logit_bias && !aligned4(logit_bias)))
    return QSM_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < moe_route_workspace_bytes(T, H, E))
    return QSM_ERR_WORKSPACE_TOO_SMALL;
  unsigned* counters = static_cast<unsigned*>(workspace);
  float* logits = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           counters_bytes(T));
  const GroupOut gout = {g->counts, g->offsets, g->perm, g->inv_perm,
                         g->tile_map, g->n_tiles, g->tile_rows, g->max_tiles};
  const dim3 grid((E + kExpertsPerCta - 1) / kExpertsPerCta, 1);
  QSM_CUDA_TRY(launch_pdl(route_kernel<8, true>, grid, dim3(kThreads), 0, stream, x,
                          w_router, logit_bias, T, H, E, k, renormalize, topk_idx,
                          topk_w, logits, counters, dev_status, gout));
  return QSM_OK;
}
