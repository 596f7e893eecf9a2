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
// Many assignments: CTA c of the grid owns a contiguous chunk of them.  It
// histograms ALL the ids (shared-memory atomics; the ids are few and stay in
// L2), which gives it the global counts, offsets and block map and the
// counts of the chunks before its own, with no scratch memory and no
// waiting on other CTAs.  Warp w of the CTA owns a contiguous run of groups
// of 32 inside the chunk; per-(warp, expert) start positions follow from a
// scan, and each group is scattered with in-group ranks (the number of
// lower lanes holding the same expert, from 31 shuffles), which keeps the
// order stable.  CTA 0 writes the counts, offsets and block map.
#include "qsm_common.cuh"

namespace qsm {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 1024;
constexpr int kBatch = 8;
constexpr int kMaxCtas = 64;

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
group_kernel(const int32_t* __restrict__ topk_idx, int A, int E, int BM, int max_tiles,
             int G, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
             int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm,
             int32_t* __restrict__ tile_map, int32_t* __restrict__ n_tiles,
             int32_t* dev_status) {
  extern __shared__ int smem[];
  int* tot = smem;          // [E] all assignments per expert
  int* bef = smem + E;      // [E] those before this CTA's chunk
  int* wh = smem + 2 * E;   // [kWarps][E] this CTA's groups, per warp
  __shared__ int warp_tot[32];
  __shared__ int s_total, s_tiles;
  pdl_wait();
  pdl_launch_dependents();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < (2 + kWarps) * E; i += kThreads) smem[i] = 0;
  __syncthreads();
  const int c0 = blockIdx.x * G * kThreads;  // first assignment of the chunk
  for (int b = 0; b < A; b += kThreads * kBatch) {
    int ids[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int a = b + u * kThreads + tid;
      ids[u] = a < A ? __ldcg(topk_idx + a) : -1;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int a = b + u * kThreads + tid;
      if (ids[u] >= 0 && ids[u] < E) {
        atomicAdd(&tot[ids[u]], 1);
        if (a < c0) atomicAdd(&bef[ids[u]], 1);
      }
    }
  }
  const int wbeg = c0 + warp * G * 32;  // this warp's G groups of 32
  bool bad = false;
  for (int g = 0; g < G; ++g) {
    const int a = wbeg + 32 * g + lane;
    if (a < A) {
      const int e = __ldcg(topk_idx + a);
      if (e >= 0 && e < E) atomicAdd(&wh[warp * E + e], 1);
      else bad = true;
    }
  }
  if (__syncthreads_or(bad) && tid == 0) set_status(dev_status, QSM_DEV_BAD_EXPERT_ID);

  // offsets and block map (thread e owns expert e), per-(warp, expert) starts
  {
    const int e = tid;
    const int cnt = e < E ? tot[e] : 0;
    const int off = block_exclusive_scan(cnt, warp_tot, &s_total);
    const int nt = (e < E) ? (cnt + BM - 1) / BM : 0;
    const int t0 = block_exclusive_scan(nt, warp_tot, &s_tiles);
    if (e < E) {
      int run = off + bef[e];
      for (int w = 0; w < kWarps; ++w) {
        const int c = wh[w * E + e];
        wh[w * E + e] = run;
        run += c;
      }
      if (blockIdx.x == 0) {
        counts[e] = cnt;
        offsets[e] = off;
        for (int m = 0; m < nt && t0 + m < max_tiles; ++m) {
          tile_map[2 * (t0 + m)] = e;
          tile_map[2 * (t0 + m) + 1] = off + m * BM;
        }
      }
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    if (tid == 0) {
      offsets[E] = s_total;
      n_tiles[0] = min(s_tiles, max_tiles);
    }
    for (int i = s_tiles + tid; i < max_tiles; i += kThreads) {
      tile_map[2 * i] = -1;
      tile_map[2 * i + 1] = -1;
    }
    for (int i = s_total + tid; i < A; i += kThreads) perm[i] = -1;
  }

  // stable scatter of this warp's groups
  for (int g = 0; g < G; ++g) {
    const int a = wbeg + 32 * g + lane;
    int key = a < A ? __ldcg(topk_idx + a) : -1;
    if (key >= E) key = -1;
    int rank = 0;  // lower lanes of this group with the same expert
#pragma unroll
    for (int d = 1; d < 32; ++d) {
      const int o = __shfl_up_sync(0xffffffffu, key, d);
      rank += (lane >= d && o == key) ? 1 : 0;
    }
    if (key >= 0) {
      const int pos = wh[warp * E + key] + rank;
      perm[pos] = a;
      inv_perm[a] = pos;
    } else if (a < A) {
      inv_perm[a] = -1;
    }
    __syncwarp();
    if (key >= 0) atomicAdd(&wh[warp * E + key], 1);
    __syncwarp();
  }
}

// Few assignments (decode): one CTA.  The ids go to shared memory, the
// threads count them with shared-memory atomics, a block scan gives the
// offsets and the block map (thread e owns expert e), and one warp places
// the assignments 32 at a time in assignment order: the lanes holding the
// same expert (match.any) take consecutive positions in lane order after
// those the earlier groups placed, which keeps the permutation stable.
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
  __shared__ int scnt[NT];   // per expert: count, then the next free position
  __shared__ int warp_tot[32];
  __shared__ int s_total, s_tiles;
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31;
  scnt[tid] = 0;
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
  for (int a = tid; a < A; a += NT)
    if (sidx[a] >= 0) atomicAdd(&scnt[sidx[a]], 1);
  __syncthreads();
  const int e = tid;
  const int cnt = e < E ? scnt[e] : 0;
  const int off = block_exclusive_scan(cnt, warp_tot, &s_total);
  const int nt = (e < E) ? (cnt + BM - 1) / BM : 0;
  const int t0 = block_exclusive_scan(nt, warp_tot, &s_tiles);
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = off;
    for (int m = 0; m < nt && t0 + m < max_tiles; ++m) {
      tile_map[2 * (t0 + m)] = e;
      tile_map[2 * (t0 + m) + 1] = off + m * BM;
    }
    scnt[e] = off;
  }
  __syncthreads();
  if (tid < 32) {
    const unsigned lower = (1u << lane) - 1u;
    for (int a0 = 0; a0 < A; a0 += 32) {
      const int a = a0 + lane;
      const int key = a < A ? sidx[a] : -2;  // -1: bad id, -2: past the end
      const unsigned same = __match_any_sync(0xffffffffu, key);
      const int base = key >= 0 ? scnt[key] : 0;
      __syncwarp();  // every lane has read its expert's position
      if (key >= 0) {
        const int pos = base + __popc(same & lower);
        perm[pos] = a;
        inv_perm[a] = pos;
        if (lane == 31 - __clz(same)) scnt[key] = base + __popc(same);
      }
      __syncwarp();
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
  // chunks of G groups of 32 per warp, at most kMaxCtas CTAs
  const int G = (int)((A + (int64_t)kThreads * kMaxCtas - 1) / ((int64_t)kThreads * kMaxCtas));
  const int nblk = (int)((A + (int64_t)G * kThreads - 1) / ((int64_t)G * kThreads));
  const size_t smem = (size_t)(2 + kWarps) * E * sizeof(int);
  QSM_CUDA_TRY(cudaFuncSetAttribute(group_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem));
  QSM_CUDA_TRY(launch_pdl(group_kernel, dim3(nblk), dim3(kThreads), smem, stream,
                          topk_idx, (int)A, (int)E, (int)g->tile_rows,
                          (int)g->max_tiles, G, g->counts, g->offsets, g->perm,
                          g->inv_perm, g->tile_map, g->n_tiles, dev_status));
  return QSM_OK;
}
