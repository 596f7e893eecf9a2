// Prefill path of the MoE FFN (many tokens): grouped GEMMs on the tcgen05
// tensor cores with the weights dequantised tile by tile on chip.
//
// "Optimizing on-device inference for Apple Silicon", section "Dequantizing
// weights during matrix multiplication": the grouped GEMM rebuilds small
// tiles of the quantized weights in on-chip memory just long enough to
// multiply them with the routed activation rows, accumulates in fp32, and
// never writes the expanded weight matrix to memory; section "Keeping
// expert routing on the GPU": the block map of the grouping drives the
// tiles, with no host round trip; "oMLX MoE gate/up 融合优化", "融合原理":
// one pass over the fused [gate; up] weight.
//
// Launch sequence (stream ordered, programmatic dependent launch):
//   prep      x -> fp16 copy (exact for the bf16 inputs), zero the fp32
//             output accumulator
//   gate_up   per work item (block of <= 128 token rows of one expert,
//             128 intermediate indices): D_gate, D_up (128 x N fp32 each, in
//             tensor memory) += W_gate/up tile x token rows; epilogue
//             h = silu(gate) * up, stored fp16 (scaled by 1/16) per sorted row
//   down      per work item (same token block, 128 output rows):
//             D (128 x N) = W_down tile x h rows; epilogue
//             y_acc[token] += routing weight * D (fp32 reduce-add)
//   finalize  y = bf16(y_acc) (and the fp32 copy)
//
// Roles in a persistent CTA (one per SM, 16 warps):
//   warp 0       TMA producer: int8 code tiles (2D tensor map) and the token
//                rows (tile::gather4 from the fp16 x copy, or 2D tiles of h)
//   warp 1       allocates tensor memory; lane 0 issues the MMAs
//   warps 4-11   dequantise the code tiles: fp16(code * block scale) written
//                in the 128-byte-swizzled K-major layout the MMA reads
//   warps 12-15  epilogue, one warp per quarter of the tensor-memory lanes
// A ring of shared-memory stages (mbarriers: full / dequantised / empty)
// connects producer, dequant and MMA; two accumulator buffers in tensor
// memory (mbarriers: full / empty) connect MMA and epilogue.
//
// Precision: weights are fp16(code * scale) (relative rounding 2^-11),
// tokens are exact; products are accumulated in fp32.
#include "tc_common.cuh"

namespace qsm {
namespace prefill {

constexpr int BM = 128;   // weight rows per MMA tile (M)
constexpr int BK = 64;    // K per stage: 128 bytes of fp16
constexpr int BN = 128;   // token rows per tile (N <= BN) = the path's tile_rows
constexpr int kThreads = 512;
constexpr int kDeqThreads = 256;  // warps 4..11
constexpr float kHScale = 1.0f / 16.0f;
constexpr float kHScaleInv = 16.0f;

enum { kGateUp = 1, kDown = 2 };

struct Params {
  CUtensorMap codes;      // routed experts' codes [E*R, K] u8, box {64, 128}
  CUtensorMap codes_sh;   // shared expert's codes [R, K] u8, box {64, 128}
  CUtensorMap bmap;       // gate_up: x16 [T, H] box {64, 1} (gather4)
                          // down:    h [rows, I] box {64, 128}
  CUtensorMap bmap_tile;  // gate_up: x16 [T, H] box {64, 128} (shared tiles)
  const __half* scales;   // [E*R, K/32]
  const __half* scales_sh;
  int R, K;               // rows per expert and reduction length
  int T, k, I, H;
  const int32_t* perm;
  const int32_t* offsets;
  const int32_t* tile_map;
  const int32_t* n_tiles;
  const float* topk_w;
  int shared_tiles;       // ceil(T / BN)
  int nsub;               // 128-row sub-blocks per tile
  __half* hbuf;           // [T*k + T, I]
  float* yacc;            // [T, H]
  int32_t* status;
};

struct TileInfo {
  int e;     // expert, -1 = shared expert
  int row0;  // first sorted row (routed) or first token (shared)
  int cnt;   // rows in the tile
  int n;     // MMA N: cnt rounded up to 16
};

__device__ __forceinline__ TileInfo tile_info(const Params& p, int tau) {
  TileInfo t;
  if (tau < p.shared_tiles) {
    t.e = -1;
    t.row0 = tau * BN;
    t.cnt = min(BN, p.T - t.row0);
  } else {
    const int2 te = __ldcg(reinterpret_cast<const int2*>(p.tile_map) + (tau - p.shared_tiles));
    t.e = te.x;
    t.row0 = te.y;
    t.cnt = min(BN, __ldcg(p.offsets + t.e + 1) - t.row0);
  }
  t.n = (t.cnt + 15) & ~15;
  return t;
}

// Bounded mbarrier wait shared by all roles: gives up when the CTA-wide
// abort flag is set or the iteration limit runs out (then sets the flag and
// the device status).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity,
                                         volatile int* abort_flag,
                                         int32_t* status) {
  for (uint32_t i = 0; i < kWaitIters; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  set_status(status, QSM_DEV_TIMEOUT);
  return false;
}

template <int MODE, int RAW, int AST>
__global__ void __launch_bounds__(kThreads, 1)
moe_prefill_gemm(const __grid_constant__ Params p) {
  constexpr int NA = MODE == kGateUp ? 2 : 1;  // A tiles per K step
  constexpr int A_BYTES = BM * BK * 2;         // fp16, 128B swizzle
  constexpr int B_BYTES = BN * BK * 2;
  constexpr int C_BYTES = BM * BK;             // int8 codes
  constexpr int A_STAGE = NA * A_BYTES;        // dequantised ring
  constexpr int RAW_STAGE = B_BYTES + NA * C_BYTES;  // TMA ring
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* aring = smem;                     // [AST][A_STAGE]
  unsigned char* rring = smem + AST * A_STAGE;     // [RAW][RAW_STAGE]
  __shared__ __align__(8) uint64_t raw_full[RAW], raw_empty[RAW], a_full[AST],
      a_empty[AST], accf_bar[2], acce_bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_tok[2][BN];
  __shared__ float s_w[2][BN];
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kDeqThreads + 1);  // dequant threads + MMA commit
    }
    for (int s = 0; s < AST; ++s) {
      mbar_init(&a_full[s], kDeqThreads);
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 128);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_map(&p.codes);
    tc::prefetch_map(&p.codes_sh);
    tc::prefetch_map(&p.bmap);
    if (MODE == kGateUp) tc::prefetch_map(&p.bmap_tile);
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;

  pdl_wait();
  pdl_launch_dependents();
  const int n_tiles = __ldcg(p.n_tiles);
  const int total = (p.shared_tiles + n_tiles) * p.nsub;
  const int ksteps = p.K / BK;
  volatile int* abort_p = &abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int r = 0, f = 0;
    for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x) {
      const int tau = item / p.nsub, sub = item - tau * p.nsub;
      const TileInfo ti = tile_info(p, tau);
      const bool gather = MODE == kGateUp && ti.e >= 0;
      int tr[4] = {0, 0, 0, 0};
      if (gather) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int rr = min(4 * lane + j, ti.cnt - 1);
          tr[j] = __ldcg(p.perm + ti.row0 + rr) / p.k;
        }
      }
      const CUtensorMap* cm = ti.e < 0 ? &p.codes_sh : &p.codes;
      const int ebase = ti.e < 0 ? 0 : ti.e * p.R;
      int arow[2];
      arow[0] = ebase + sub * BM;
      arow[1] = ebase + p.I + sub * BM;  // gate_up: the up rows
      const int brow = MODE == kGateUp ? ti.row0
                                       : (ti.e < 0 ? p.T * p.k + ti.row0 : ti.row0);
      const uint32_t bbytes = gather ? (uint32_t)ti.n * (BK * 2) : (uint32_t)B_BYTES;
      for (int ks = 0; ks < ksteps; ++ks) {
        bool ok = true;
        if (f >= RAW && lane == 0)
          ok = wait_bar(&raw_empty[r], ((f / RAW) - 1) & 1, abort_p, p.status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        unsigned char* bdst = rring + r * RAW_STAGE;
        if (lane == 0) {
          mbar_arrive_expect_tx(&raw_full[r], NA * C_BYTES + bbytes);
#pragma unroll
          for (int a = 0; a < NA; ++a)
            tc::tma_load_2d(bdst + B_BYTES + a * C_BYTES, cm, ks * BK, arow[a], &raw_full[r]);
          if (!gather)
            tc::tma_load_2d(bdst, MODE == kGateUp ? &p.bmap_tile : &p.bmap, ks * BK,
                            brow, &raw_full[r]);
        }
        __syncwarp();
        if (gather && lane < ti.n / 4)
          tc::tma_gather4(bdst + lane * 4 * (BK * 2), &p.bmap, ks * BK, tr[0], tr[1],
                          tr[2], tr[3], &raw_full[r]);
        ++f;
        r = (r + 1 == RAW) ? 0 : r + 1;
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int r = 0, a = 0, f = 0, j = 0;
      for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x, ++j) {
        const int tau = item / p.nsub;
        const TileInfo ti = tile_info(p, tau);
        const int b = j & 1;
        if (j >= 2 && !wait_bar(&acce_bar[b], ((j >> 1) - 1) & 1, abort_p, p.status)) break;
        tc::tc_fence_after();
        const uint32_t idesc = tc::idesc_f16_m128(ti.n);
        const uint32_t dbase = tmem + b * 256;
        bool ok = true;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!wait_bar(&raw_full[r], (f / RAW) & 1, abort_p, p.status) ||
              !wait_bar(&a_full[a], (f / AST) & 1, abort_p, p.status)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a0 = smem_u32(aring + a * A_STAGE);
          const uint32_t b0 = smem_u32(rring + r * RAW_STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
            for (int m = 0; m < NA; ++m)
              tc::mma_f16(dbase + m * 128, tc::sw128_desc(a0 + m * A_BYTES + kk * 32),
                          tc::sw128_desc(b0 + kk * 32), idesc,
                          (ks > 0 || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit(&raw_empty[r]);
          tc::mma_commit(&a_empty[a]);
          ++f;
          r = (r + 1 == RAW) ? 0 : r + 1;
          a = (a + 1 == AST) ? 0 : a + 1;
        }
        if (!ok) break;
        tc::mma_commit(&accf_bar[b]);
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------- dequant
    const int d = threadIdx.x - 128;
    const int am = MODE == kGateUp ? (d >> 7) : 0;
    const int rw = MODE == kGateUp ? (d & 127) : (d >> 1);
    const int half = MODE == kGateUp ? 0 : (d & 1);
    constexpr int kInChunks = MODE == kGateUp ? 4 : 2;  // 16 codes per chunk
    int r = 0, a = 0, f = 0;
    for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x) {
      const int tau = item / p.nsub, sub = item - tau * p.nsub;
      const TileInfo ti = tile_info(p, tau);
      const int ebase = ti.e < 0 ? 0 : ti.e * p.R;
      const int row = ebase + (am ? p.I : 0) + sub * BM + rw;
      // this row's block scales: one 4-byte pair per K step (4-byte aligned
      // for any K % 64 == 0), fetched one group of 8 K steps ahead
      const uint32_t* sc = reinterpret_cast<const uint32_t*>(
          (ti.e < 0 ? p.scales_sh : p.scales) + (size_t)row * (p.K / 32));
      uint32_t nx[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) nx[jj] = jj < ksteps ? __ldg(sc + jj) : 0u;
      bool ok = true;
      for (int kg = 0; kg < ksteps && ok; kg += 8) {
        uint32_t cur[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          cur[jj] = nx[jj];
          nx[jj] = kg + 8 + jj < ksteps ? __ldg(sc + kg + 8 + jj) : 0u;
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (kg + jj >= ksteps) break;
          if (!wait_bar(&raw_full[r], (f / RAW) & 1, abort_p, p.status) ||
              (f >= AST && !wait_bar(&a_empty[a], ((f / AST) - 1) & 1, abort_p, p.status))) {
            ok = false;
            break;
          }
          const uint32_t sc2 = cur[jj];
          const unsigned char* codes = rring + r * RAW_STAGE + B_BYTES + am * C_BYTES + rw * BK;
          unsigned char* arow_s = aring + a * A_STAGE + am * A_BYTES + (rw >> 3) * 1024 +
                                  (rw & 7) * 128;
#pragma unroll
          for (int j = 0; j < kInChunks; ++j) {
            // rotate the chunk order by row to spread shared-memory banks
            const int ci = half * kInChunks + ((j + rw) & (kInChunks - 1));
            const uint4 v = *reinterpret_cast<const uint4*>(codes + ci * 16);
            const uint32_t sbits = (ci < 2) ? (sc2 & 0xffffu) : (sc2 >> 16);
            const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)sbits));
            uint32_t o[8];
            s8x4_to_f16x2x2(v.x, o[0], o[1]);
            s8x4_to_f16x2x2(v.y, o[2], o[3]);
            s8x4_to_f16x2x2(v.z, o[4], o[5]);
            s8x4_to_f16x2x2(v.w, o[6], o[7]);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              __half2 h = __hmul2(*reinterpret_cast<__half2*>(&o[t]), s2);
              o[t] = *reinterpret_cast<uint32_t*>(&h);
            }
            const int oc0 = 2 * ci, oc1 = 2 * ci + 1;  // 16-byte output chunks
            *reinterpret_cast<uint4*>(arow_s + ((oc0 ^ (rw & 7)) << 4)) =
                make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(arow_s + ((oc1 ^ (rw & 7)) << 4)) =
                make_uint4(o[4], o[5], o[6], o[7]);
          }
          tc::fence_async_smem();
          tc::mbar_arrive(&a_full[a]);
          tc::mbar_arrive(&raw_empty[r]);
          ++f;
          r = (r + 1 == RAW) ? 0 : r + 1;
          a = (a + 1 == AST) ? 0 : a + 1;
        }
      }
      if (!ok) break;
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int et = threadIdx.x - 384;  // 0..127
    int j = 0;
    bool bad = false;
    for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x, ++j) {
      const int tau = item / p.nsub, sub = item - tau * p.nsub;
      const TileInfo ti = tile_info(p, tau);
      const int b = j & 1;
      if (MODE == kDown) {
        if (et < ti.cnt) {
          if (ti.e < 0) {
            s_tok[b][et] = ti.row0 + et;
            s_w[b][et] = kHScaleInv;
          } else {
            const int asg = __ldcg(p.perm + ti.row0 + et);
            s_tok[b][et] = asg / p.k;
            s_w[b][et] = __ldcg(p.topk_w + asg) * kHScaleInv;
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
      if (!wait_bar(&accf_bar[b], (j >> 1) & 1, abort_p, p.status)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16) + b * 256;
      if (MODE == kGateUp) {
        const int i = sub * BM + 32 * q4 + lane;  // intermediate index
        for (int c0 = 0; c0 < ti.n; c0 += 16) {
          float gv[16], uv[16];
          tc::tmem_ld16(taddr + c0, gv);
          tc::tmem_ld16(taddr + 128 + c0, uv);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int col = c0 + c;
            if (col < ti.cnt) {
              const float h = silu(gv[c]) * uv[c] * kHScale;
              if (!(fabsf(h) <= 65504.f)) bad = true;
              const int hrow = ti.e < 0 ? p.T * p.k + ti.row0 + col : ti.row0 + col;
              p.hbuf[(size_t)hrow * p.I + i] = __float2half_rn(h);
            }
          }
        }
      } else {
        const int n = sub * BM + 32 * q4 + lane;  // output row
        for (int c0 = 0; c0 < ti.n; c0 += 16) {
          float dv[16];
          tc::tmem_ld16(taddr + c0, dv);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int col = c0 + c;
            if (col < ti.cnt)
              atomicAdd(p.yacc + (size_t)s_tok[b][col] * p.H + n, s_w[b][col] * dv[c]);
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acce_bar[b]);
      if (MODE == kDown) asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    if (bad) set_status(p.status, QSM_DEV_FP16_RANGE);
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// x (bf16) -> fp16 copy; zero the fp32 output accumulator.
__global__ void __launch_bounds__(256)
prep_kernel(const uint16_t* __restrict__ x, __half* __restrict__ x16,
            float* __restrict__ yacc, size_t n8, int32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  bool bad = false;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + i);
    const uint4 h = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                               bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
    const uint32_t* hw = reinterpret_cast<const uint32_t*>(&h);
#pragma unroll
    for (int t = 0; t < 4; ++t)  // an all-ones exponent: out of fp16 range
      if ((hw[t] & 0x7c00u) == 0x7c00u || (hw[t] & 0x7c000000u) == 0x7c000000u)
        bad = true;
    reinterpret_cast<uint4*>(x16)[i] = h;
    reinterpret_cast<float4*>(yacc)[2 * i] = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(yacc)[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (bad) set_status(status, QSM_DEV_FP16_RANGE);
}

// y = bf16(y_acc) (and the fp32 copy).
__global__ void __launch_bounds__(256)
finalize_kernel(const float* __restrict__ yacc, uint16_t* __restrict__ y,
                float* __restrict__ y32, size_t n4) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(yacc) + i);
    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y)) << 16);
    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w)) << 16);
    reinterpret_cast<uint2*>(y)[i] = make_uint2(lo, hi);
    if (y32) reinterpret_cast<float4*>(y32)[i] = v;
  }
}

// (TMA ring, dequantised ring) depths
constexpr int kGateUpRaw = 4, kGateUpA = 2;
constexpr int kDownRaw = 6, kDownA = 2;

template <int MODE, int RAW, int AST>
constexpr size_t gemm_smem() {
  constexpr int NA = MODE == kGateUp ? 2 : 1;
  return (size_t)AST * NA * BM * BK * 2 + (size_t)RAW * (BN * BK * 2 + NA * BM * BK) +
         1024;
}

int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (n[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

struct WsLayout {
  size_t x16, hbuf, yacc, total;
};

inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

WsLayout ws_layout(const qsm_moe_layer* L, int T) {
  WsLayout w;
  w.x16 = 0;
  w.hbuf = up256((size_t)T * L->H * 2);
  w.yacc = w.hbuf + up256(((size_t)T * L->k + T) * L->I * 2);
  w.total = w.yacc + up256((size_t)T * L->H * 4);
  return w;
}

}  // namespace prefill

bool prefill_supported(const qsm_moe_layer* L) {
  return L->gate_up.qtype == QSM_Q8_0 && L->H % 128 == 0 && L->I % 128 == 0;
}

size_t prefill_ffn_workspace_bytes(const qsm_moe_layer* L, int T) {
  return prefill::ws_layout(L, T).total;
}

qsm_status prefill_ffn_launch(const qsm_moe_layer* L, const uint16_t* x, int T,
                              const float* topk_w, const qsm_grouping* g,
                              uint16_t* y, float* y32, void* ws,
                              int32_t* dev_status, cudaStream_t stream) {
  using namespace prefill;
  const int H = L->H, I = L->I, E = L->E, k = L->k;
  const WsLayout wl = ws_layout(L, T);
  char* wsb = static_cast<char*>(ws);
  __half* x16 = reinterpret_cast<__half*>(wsb + wl.x16);
  __half* hbuf = reinterpret_cast<__half*>(wsb + wl.hbuf);
  float* yacc = reinterpret_cast<float*>(wsb + wl.yacc);
  const int nsm = sm_count();
  const size_t rows_h = (size_t)T * k + T;

  QSM_CUDA_TRY(launch_pdl(prep_kernel, dim3(2 * nsm), dim3(256), 0, stream, x, x16,
                          yacc, (size_t)T * H / 8, dev_status));

  Params p1 = {};
  bool ok = true;
  ok &= tc::make_map_2d(&p1.codes, L->gate_up.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                        (uint64_t)E * 2 * I, H, BK, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok &= tc::make_map_2d(&p1.codes_sh, L->shared_gate_up.codes,
                        CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 2 * I, H, BK, BM,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  ok &= tc::make_map_2d(&p1.bmap, x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, T, H, BK, 1,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  ok &= tc::make_map_2d(&p1.bmap_tile, x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, T, H,
                        BK, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return QSM_ERR_CUDA;
  p1.scales = reinterpret_cast<const __half*>(L->gate_up.scales);
  p1.scales_sh = reinterpret_cast<const __half*>(L->shared_gate_up.scales);
  p1.R = 2 * I;
  p1.K = H;
  p1.T = T;
  p1.k = k;
  p1.I = I;
  p1.H = H;
  p1.perm = g->perm;
  p1.offsets = g->offsets;
  p1.tile_map = g->tile_map;
  p1.n_tiles = g->n_tiles;
  p1.topk_w = topk_w;
  p1.shared_tiles = (T + BN - 1) / BN;
  p1.nsub = I / BM;
  p1.hbuf = hbuf;
  p1.yacc = yacc;
  p1.status = dev_status;

  Params p2 = p1;
  ok &= tc::make_map_2d(&p2.codes, L->down.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                        (uint64_t)E * H, I, BK, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok &= tc::make_map_2d(&p2.codes_sh, L->shared_down.codes,
                        CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, H, I, BK, BM,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  ok &= tc::make_map_2d(&p2.bmap, hbuf, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows_h, I,
                        BK, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return QSM_ERR_CUDA;
  p2.scales = reinterpret_cast<const __half*>(L->down.scales);
  p2.scales_sh = reinterpret_cast<const __half*>(L->shared_down.scales);
  p2.R = H;
  p2.K = I;
  p2.nsub = H / BM;

  constexpr size_t smem1 = gemm_smem<kGateUp, kGateUpRaw, kGateUpA>();
  constexpr size_t smem2 = gemm_smem<kDown, kDownRaw, kDownA>();
  auto* k1 = moe_prefill_gemm<kGateUp, kGateUpRaw, kGateUpA>;
  auto* k2 = moe_prefill_gemm<kDown, kDownRaw, kDownA>;
  QSM_CUDA_TRY(cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem1));
  QSM_CUDA_TRY(cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem2));
  QSM_CUDA_TRY(launch_pdl(k1, dim3(nsm), dim3(kThreads), smem1, stream, p1));
  QSM_CUDA_TRY(launch_pdl(k2, dim3(nsm), dim3(kThreads), smem2, stream, p2));
  QSM_CUDA_TRY(launch_pdl(finalize_kernel, dim3(2 * nsm), dim3(256), 0, stream,
                          (const float*)yacc, y, y32, (size_t)T * H / 4));
  return QSM_OK;
}

}  // namespace qsm
