// Token grouping: histogram, exclusive scan, stable scatter and block map.
//
// "Optimizing on-device inference for Apple Silicon", section "Keeping
// expert routing on the GPU": the grouped matmul needs each expert's rows
// stored together; a histogram counts the assignments per expert, a prefix
// scan turns the counts into start offsets, a scatter places the rows and a
// block map lists the fixed-size blocks to process, with no host round trip.
// Reading: inside an expert the rows keep assignment order (stable), so the
// permutation is unique.
//
// One CTA of 1024 threads does it all (T*k is at most a few ten thousand on
// this path).  Warp w owns a contiguous range of assignments; a pass with
// __match_any_sync counts its per-expert histogram without atomics, the CTA
// turns the 32 histograms into per-(warp, expert) start positions, and a
// second pass scatters with in-warp ranks, which keeps the order stable.
// The permutation is staged in shared memory when it fits and written out
// coalesced.
#include "qsm_common.cuh"

namespace qsm {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 1024;
constexpr size_t kSmemLimit = 227 * 1024 - 1024;  // leave room for static smem

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot,
                                                    int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nwarps) warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + incl - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
group_kernel(const int32_t* __restrict__ topk_idx, int A, int E, int BM,
             int max_tiles, int stage, int32_t* __restrict__ counts,
             int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
             int32_t* __restrict__ inv_perm, int32_t* __restrict__ tile_map,
             int32_t* __restrict__ n_tiles, int32_t* dev_status) {
  extern __shared__ int smem[];
  int* hist = smem;                       // [kWarps][E]
  int* sperm = smem + kWarps * E;         // [A] when staged
  __shared__ int warp_tot[32];
  __shared__ int s_total, s_tiles;
  pdl_launch_dependents();
  pdl_wait();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kWarps * E; i += kThreads) hist[i] = 0;
  __syncthreads();

  const int chunk = ((A + kWarps - 1) / kWarps + 31) & ~31;
  const int beg = min(A, warp * chunk), end = min(A, beg + chunk);
  int* myhist = hist + warp * E;
  bool bad = false;
  // pass 1: per-warp histogram
  for (int base = beg; base < end; base += 32) {
    const int a = base + lane;
    int key = -1;
    if (a < end) {
      const int e = topk_idx[a];
      if (e >= 0 && e < E) key = e; else bad = true;
    }
    const unsigned m = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && lane == __ffs(m) - 1) myhist[key] += __popc(m);
    __syncwarp();
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0)
    set_status(dev_status, QSM_DEV_BAD_EXPERT_ID);
  __syncthreads();

  // counts, offsets, per-(warp, expert) bases, block map
  {
    const int e = tid;
    int cnt = 0;
    if (e < E)
      for (int w = 0; w < kWarps; ++w) cnt += hist[w * E + e];
    const int off = block_exclusive_scan(e < E ? cnt : 0, warp_tot, &s_total);
    const int nt = (e < E) ? (cnt + BM - 1) / BM : 0;
    const int t0 = block_exclusive_scan(nt, warp_tot, &s_tiles);
    if (e < E) {
      counts[e] = cnt;
      offsets[e] = off;
      int run = off;
      for (int w = 0; w < kWarps; ++w) {
        const int c = hist[w * E + e];
        hist[w * E + e] = run;
        run += c;
      }
      for (int m = 0; m < nt && t0 + m < max_tiles; ++m) {
        tile_map[2 * (t0 + m)] = e;
        tile_map[2 * (t0 + m) + 1] = off + m * BM;
      }
    }
    if (tid == 0) {
      offsets[E] = s_total;
      n_tiles[0] = min(s_tiles, max_tiles);
    }
  }
  __syncthreads();
  for (int i = s_tiles + tid; i < max_tiles; i += kThreads) {
    tile_map[2 * i] = -1;
    tile_map[2 * i + 1] = -1;
  }

  // pass 2: stable scatter
  const unsigned lt = (1u << lane) - 1u;
  for (int base = beg; base < end; base += 32) {
    const int a = base + lane;
    int key = -1;
    if (a < end) {
      const int e = topk_idx[a];
      if (e >= 0 && e < E) key = e;
    }
    const unsigned m = __match_any_sync(0xffffffffu, key);
    if (key >= 0) {
      const int pos = myhist[key] + __popc(m & lt);
      if (stage) sperm[pos] = a; else perm[pos] = a;
      inv_perm[a] = pos;
    } else if (a < end) {
      inv_perm[a] = -1;
    }
    __syncwarp();
    if (key >= 0 && lane == __ffs(m) - 1) myhist[key] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  const int valid = s_total;
  if (stage)
    for (int i = tid; i < valid; i += kThreads) perm[i] = sperm[i];
  for (int i = valid + tid; i < A; i += kThreads) perm[i] = -1;
}

// Few assignments (decode): the per-warp histogram machinery above costs
// more than the work.  Thread e owns expert e and walks the (at most
// kSmallA) assignments in shared memory twice: once to count, once to place
// its rows in assignment order (stable by construction).
constexpr int kSmallA = 1024;

template <int NT>  // threads: a multiple of 32 and >= E
__global__ void __launch_bounds__(NT, 1)
group_small_kernel(const int32_t* __restrict__ topk_idx, int A, int E, int BM,
                   int max_tiles, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                   int32_t* __restrict__ inv_perm,
                   int32_t* __restrict__ tile_map,
                   int32_t* __restrict__ n_tiles, int32_t* dev_status) {
  __shared__ int sidx[kSmallA];
  __shared__ int warp_tot[32];
  __shared__ int s_total, s_tiles;
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  bool bad = false;
  for (int a = tid; a < A; a += NT) {
    int v = __ldcg(topk_idx + a);
    if (v < 0 || v >= E) {
      bad = true;
      v = -1;
      inv_perm[a] = -1;
    }
    sidx[a] = v;
  }
  if (__syncthreads_or(bad) && tid == 0)
    set_status(dev_status, QSM_DEV_BAD_EXPERT_ID);
  const int e = tid;
  int cnt = 0;
  if (e < E)
    for (int a = 0; a < A; ++a) cnt += (sidx[a] == e);
  const int off = block_exclusive_scan(e < E ? cnt : 0, warp_tot, &s_total);
  const int nt = (e < E) ? (cnt + BM - 1) / BM : 0;
  const int t0 = block_exclusive_scan(nt, warp_tot, &s_tiles);
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = off;
    for (int m = 0; m < nt && t0 + m < max_tiles; ++m) {
      tile_map[2 * (t0 + m)] = e;
      tile_map[2 * (t0 + m) + 1] = off + m * BM;
    }
    int pos = off;
    for (int a = 0; a < A && pos < off + cnt; ++a) {
      if (sidx[a] == e) {
        perm[pos] = a;
        inv_perm[a] = pos;
        ++pos;
      }
    }
  }
  if (tid == 0) {
    offsets[E] = s_total;
    n_tiles[0] = min(s_tiles, max_tiles);
  }
  for (int i = s_tiles + tid; i < max_tiles; i += NT) {
    tile_map[2 * i] = -1;
    tile_map[2 * i + 1] = -1;
  }
  for (int i = s_total + tid; i < A; i += NT) perm[i] = -1;
}

}  // namespace
}  // namespace qsm

extern "C" int32_t moe_group_max_tiles(int32_t T, int32_t k, int32_t E,
                                       int32_t tile_rows) {
  if (T < 0 || k < 1 || E < 1 || tile_rows < 1) return 0;
  // n non-empty experts hold A rows: sum ceil(c_e / BM) <= n + (A - n) / BM,
  // largest at n = min(E, A).
  const int64_t A = (int64_t)T * k;
  const int64_t n = A < E ? A : E;
  return (int32_t)(n + (A - n) / tile_rows);
}

extern "C" qsm_status moe_group_tokens(const int32_t* topk_idx, int32_t T,
                                       int32_t k, int32_t E,
                                       const qsm_grouping* g,
                                       int32_t* dev_status,
                                       cudaStream_t stream) {
  using namespace qsm;
  if (!g || T < 0 || k < 1 || E < 1 || E > kMaxE || g->tile_rows < 1)
    return QSM_ERR_INVALID_ARGUMENT;
  const int64_t A = (int64_t)T * k;
  if (A > (1 << 24)) return QSM_ERR_UNSUPPORTED;
  if (!g->counts || !g->offsets || !g->n_tiles || !dev_status ||
      (A > 0 && (!topk_idx || !g->perm || !g->inv_perm)) ||
      (g->max_tiles > 0 && !g->tile_map))
    return QSM_ERR_INVALID_ARGUMENT;
  if (g->max_tiles < moe_group_max_tiles(T, k, E, g->tile_rows))
    return QSM_ERR_INVALID_ARGUMENT;
  if (A <= kSmallA) {
    if (E <= 256)
      QSM_CUDA_TRY(launch_pdl(group_small_kernel<256>, dim3(1), dim3(256), 0,
                              stream, topk_idx, (int)A, (int)E,
                              (int)g->tile_rows, (int)g->max_tiles, g->counts,
                              g->offsets, g->perm, g->inv_perm, g->tile_map,
                              g->n_tiles, dev_status));
    else
      QSM_CUDA_TRY(launch_pdl(group_small_kernel<kThreads>, dim3(1), dim3(kThreads),
                              0, stream, topk_idx, (int)A, (int)E,
                              (int)g->tile_rows, (int)g->max_tiles, g->counts,
                              g->offsets, g->perm, g->inv_perm, g->tile_map,
                              g->n_tiles, dev_status));
    return QSM_OK;
  }
  const size_t hist_bytes = (size_t)kWarps * E * sizeof(int);
  const int stage = hist_bytes + (size_t)A * sizeof(int) <= kSmemLimit;
  const size_t smem = hist_bytes + (stage ? (size_t)A * sizeof(int) : 0);
  QSM_CUDA_TRY(cudaFuncSetAttribute(group_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemLimit));
  QSM_CUDA_TRY(launch_pdl(group_kernel, dim3(1), dim3(kThreads), smem, stream,
                          topk_idx, (int)A, (int)E, (int)g->tile_rows,
                          (int)g->max_tiles, stage, g->counts, g->offsets,
                          g->perm, g->inv_perm, g->tile_map, g->n_tiles,
                          dev_status));
  return QSM_OK;
}
