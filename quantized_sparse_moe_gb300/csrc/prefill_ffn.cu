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
//   prep      the token operand of gate_up as one fp16 matrix (exact for
//             the bf16 inputs): the routed rows in grouped order (sorted
//             row r holds the token of assignment perm[r]), then the T
//             tokens in order for the shared expert; zero the fp32 output
//             accumulator
//   gate_up   per work item (block of <= 128 token rows of one expert,
//             128 intermediate indices): D (128 token rows x 256, fp32 in
//             tensor memory) += token rows x [W_gate tile; W_up tile]^T, one
//             N = 256 MMA per 16-wide K step; epilogue (one token row per
//             thread) h = silu(gate) * up, stored fp16 (scaled by 1/16) in
//             16-byte pieces per sorted row
//   down      per work item (same token block, 256 output rows):
//             D (128 token rows x 256) = h rows x W_down tiles^T; epilogue
//             y_acc[token] += routing weight * D row (8-byte fp32
//             reduce-adds, four threads on 32 contiguous bytes of a row)
// Rows of a short tile beyond its tokens hold stale data: their D rows are
// never read.
//   finalize  y = bf16(y_acc) (and the fp32 copy)
//
// Roles in a persistent CTA (one per SM, 16 warps):
//   warp 0       TMA producer of the int8 code tiles (2D tensor map)
//   warp 1       allocates tensor memory; lane 0 issues the MMAs
//   warp 2       TMA producer of the token-row tiles: 2D boxes of the
//                grouped fp16 x (gate_up) or of h (down), 128 rows or a
//                64/32/16-row decomposition of a short tile's rows
//   warps 4-11   dequantise the code tiles: fp16(code * block scale) written
//                in the 128-byte-swizzled K-major layout the MMA reads
//   warps 12-15  epilogue, one warp per quarter of the tensor-memory lanes
// Three shared-memory rings, each with full / empty mbarriers: code tiles
// (freed as soon as the dequantising warps have read them), token tiles
// (freed by the MMA commit) and dequantised weight tiles (freed by the MMA
// commit).  Keeping the rings apart lets each run as many stages ahead as
// its own latency needs.  Two accumulator buffers in tensor memory
// (mbarriers: full / empty) connect MMA and epilogue.
//
// Weights: Q8_0 (int8 codes, an fp16 scale per 32) or affine-4 (8 codes
// per 32-bit word, lowest nibble first along K, fp16 scale and bias per 64:
// "Dequantizing weights during matrix multiplication").  A 64-wide K step
// is 64 bytes of Q8_0 codes or 32 bytes of affine-4 codes per row.
//
// Precision: weights are fp16(code * scale) or fp16(code * scale + bias)
// (one rounding, relative 2^-11), tokens are exact; products are
// accumulated in fp32.
#include "tc_common.cuh"

namespace qsm {
namespace prefill {

constexpr int BM = 128;   // weight rows per weight tile (two tiles form the MMA's N = 256)
constexpr int BK = 64;    // K per stage: 128 bytes of fp16
constexpr int BN = 128;   // token rows per tile (the MMA's M) = the path's tile_rows
constexpr int kThreads = 512;
constexpr int kDeqThreads = 256;  // warps 4..11
constexpr float kHScale = 1.0f / 16.0f;
constexpr float kHScaleInv = 16.0f;

enum { kGateUp = 1, kDown = 2 };

struct Params {
  CUtensorMap codes;      // routed experts' codes [E*R, K] u8, box {64, 128}
  CUtensorMap codes_sh;   // shared expert's codes [R, K] u8, box {64, 128}
  CUtensorMap bmap[4];    // token rows [T*k + T, K] fp16 (gate_up: grouped
                          // x; down: h), boxes {64, 128 / 64 / 32 / 16}
  const __half* scales;   // [E*R, K/32] (Q8_0) or [E*R, K/64] (affine-4)
  const __half* scales_sh;
  const __half* biases;   // [E*R, K/64] (affine-4)
  const __half* biases_sh;
  int R, K;               // rows per expert and reduction length
  int T, k, I, H;
  const int32_t* perm;
  const int32_t* offsets;
  const int32_t* tile_map;
  const int32_t* n_tiles;
  const float* topk_w;
  int shared_tiles;       // ceil(T / BN)
  int nsub;               // weight blocks (two 128-row tiles each) per tile
  __half* hbuf;           // [T*k + T, I]
  float* yacc;            // [T, H]
  const float* gate;      // [T] shared-expert gates, or NULL (weight 1)
  float* gu_dump;         // test hook: [T*k + T, 2I] fp32 gate and up values, or NULL
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

// The abort flag as one decision for the whole warp (roles whose lanes run
// .sync.aligned tensor-memory instructions together).
__device__ __forceinline__ bool warp_aborted(volatile int* abort_flag) {
  return __any_sync(0xffffffffu, *abort_flag != 0);
}

// A producer's last copies: wait (briefly bounded) until the up to `depth`
// most recent of its f issued stages have landed, so that no copy is still
// writing shared memory when the CTA exits after an abort.  Immediate on
// the normal path, where consumers already waited for every stage.
__device__ __forceinline__ void drain_stages(uint64_t* full, int depth, uint32_t f) {
  const uint32_t n = f < (uint32_t)depth ? f : (uint32_t)depth;
  for (uint32_t i = 0; i < n; ++i) {
    const uint32_t g = f - 1 - i;
    mbar_wait_bounded(&full[g % depth], (g / depth) & 1, 1u << 16);
  }
}

// First row (within the expert) of weight tile a in {0, 1} of work item sub:
// gate_up pairs the gate rows and the up rows of intermediates sub*128..,
// down takes output rows sub*256 + a*128...
__device__ __forceinline__ int weight_row0(const Params& p, int mode, int sub, int a) {
  return mode == kGateUp ? a * p.I + sub * BM : (2 * sub + a) * BM;
}

// y[0..1] += v0, v1 in one 8-byte reduction (8-byte aligned address).
__device__ __forceinline__ void red_add_v2(float* y, float v0, float v1) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(y), "f"(v0), "f"(v1) : "memory");
}

// 16 lanes from the lane in taddr, 32 columns: thread t gets, for j = 0..3,
// columns 8j + 2(t % 4) and + 1 of lane t / 4 (registers 4j, 4j + 1) and of
// lane t / 4 + 8 (registers 4j + 2, 4j + 3).
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// One 32-bit word of affine-4 codes (K order k..k+7, lowest nibble first)
// -> eight fp16 s*q + b in K order (one rounding each: q is exact in fp16).
__device__ __forceinline__ uint4 a4_word_to_f16x8(uint32_t w, __half2 s2, __half2 b2) {
  const uint32_t lo = w & 0x0F0F0F0Fu;         // q0 q2 q4 q6
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // q1 q3 q5 q7
  const uint32_t t0 = __byte_perm(lo, hi, 0x5140);  // q0 q1 q2 q3
  const uint32_t t1 = __byte_perm(lo, hi, 0x7362);  // q4 q5 q6 q7
  // each code under the fp16 exponent of 1024: 1024 + q
  uint32_t v[4] = {__byte_perm(t0, 0x64646464u, 0x4140), __byte_perm(t0, 0x64646464u, 0x4342),
                   __byte_perm(t1, 0x64646464u, 0x4140), __byte_perm(t1, 0x64646464u, 0x4342)};
  const __half2 k1024 = __half2half2(__ushort_as_half(0x6400));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&v[i]), k1024);
    h = __hfma2(h, s2, b2);
    v[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(v[0], v[1], v[2], v[3]);
}

template <int MODE, int QT, int CR, int BR, int AST>
__global__ void __launch_bounds__(kThreads, 1)
moe_prefill_gemm(const __grid_constant__ Params p) {
  constexpr int NA = 2;                        // weight tiles per K step
  constexpr int A_BYTES = BM * BK * 2;         // fp16, 128B swizzle
  constexpr int B_BYTES = BN * BK * 2;
  constexpr int KB = QT == QSM_Q8_0 ? BK : BK / 2;  // code bytes per row and K step
  constexpr int C_BYTES = BM * KB;
  constexpr int A_STAGE = NA * A_BYTES;        // dequantised ring
  constexpr int C_STAGE = NA * C_BYTES;        // code ring
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* aring = smem;                     // [AST][A_STAGE]
  unsigned char* bring = aring + AST * A_STAGE;    // [BR][B_BYTES]
  unsigned char* cring = bring + BR * B_BYTES;     // [CR][C_STAGE]
  __shared__ __align__(8) uint64_t c_full[CR], c_empty[CR], b_full[BR], b_empty[BR],
      a_full[AST], a_empty[AST], accf_bar[2], acce_bar[2], mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < CR; ++s) {
      mbar_init(&c_full[s], 1);
      mbar_init(&c_empty[s], kDeqThreads);
    }
    for (int s = 0; s < BR; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);  // MMA commit
    }
    for (int s = 0; s < AST; ++s) {
      mbar_init(&a_full[s], kDeqThreads);
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 128);
    }
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_map(&p.codes);
    tc::prefetch_map(&p.codes_sh);
#pragma unroll
    for (int m = 0; m < 4; ++m) tc::prefetch_map(&p.bmap[m]);
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
    // ------------------------------------------------- producer: code tiles
    if (lane == 0) {
      int c = 0;
      uint32_t f = 0;
      for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x) {
        const int tau = item / p.nsub, sub = item - tau * p.nsub;
        const TileInfo ti = tile_info(p, tau);
        const CUtensorMap* cm = ti.e < 0 ? &p.codes_sh : &p.codes;
        const int ebase = ti.e < 0 ? 0 : ti.e * p.R;
        int arow[2];
        for (int a = 0; a < NA; ++a) arow[a] = ebase + weight_row0(p, MODE, sub, a);
        bool ok = true;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (f >= CR && !wait_bar(&c_empty[c], ((f / CR) - 1) & 1, abort_p, p.status)) {
            ok = false;
            break;
          }
          unsigned char* cdst = cring + c * C_STAGE;
          mbar_arrive_expect_tx(&c_full[c], C_STAGE);
#pragma unroll
          for (int a = 0; a < NA; ++a)
            tc::tma_load_2d(cdst + a * C_BYTES, cm, ks * KB, arow[a], &c_full[c]);
          ++f;
          c = (c + 1 == CR) ? 0 : c + 1;
        }
        if (!ok) break;
      }
      drain_stages(c_full, CR, f);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------ producer: token tiles
    if (lane == 0) {
      int b = 0;
      uint32_t f = 0;
      for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x) {
        const int tau = item / p.nsub;
        const TileInfo ti = tile_info(p, tau);
        const int brow = (ti.e < 0 ? p.T * p.k : 0) + ti.row0;
        bool ok = true;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (f >= BR && !wait_bar(&b_empty[b], ((f / BR) - 1) & 1, abort_p, p.status)) {
            ok = false;
            break;
          }
          unsigned char* bdst = bring + b * B_BYTES;
          mbar_arrive_expect_tx(&b_full[b], (uint32_t)ti.n * (BK * 2));
          if (ti.n == BN) {
            tc::tma_load_2d(bdst, &p.bmap[0], ks * BK, brow, &b_full[b]);
          } else {  // n = 16 * (4a + 2b + c): boxes of 64, 32 and 16 rows
            int r0 = 0;
#pragma unroll
            for (int m = 1; m < 4; ++m) {
              const int rows = BN >> m;
              if (ti.n & rows) {
                tc::tma_load_2d(bdst + r0 * (BK * 2), &p.bmap[m], ks * BK, brow + r0,
                                &b_full[b]);
                r0 += rows;
              }
            }
          }
          ++f;
          b = (b + 1 == BR) ? 0 : b + 1;
        }
        if (!ok) break;
      }
      drain_stages(b_full, BR, f);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int b = 0, a = 0, j = 0;
      uint32_t f = 0;
      for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x, ++j) {
        const int tau = item / p.nsub;
        const TileInfo ti = tile_info(p, tau);
        const int ab = j & 1;  // accumulator buffer
        if (j >= 2 && !wait_bar(&acce_bar[ab], ((j >> 1) - 1) & 1, abort_p, p.status)) break;
        tc::tc_fence_after();
        // D[token row, weight row]: M = 128 token rows, N = 256 weight rows
        const uint32_t idesc = tc::idesc_f16_m128(NA * BM);
        const uint32_t dbase = tmem + ab * 256;
        bool ok = true;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!wait_bar(&b_full[b], (f / BR) & 1, abort_p, p.status) ||
              !wait_bar(&a_full[a], (f / AST) & 1, abort_p, p.status)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a0 = smem_u32(aring + a * A_STAGE);
          const uint32_t b0 = smem_u32(bring + b * B_BYTES);
          // the two weight tiles of a stage are one 256-row K-major operand
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_f16(dbase, tc::sw128_desc(b0 + kk * 32), tc::sw128_desc(a0 + kk * 32),
                        idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(&b_empty[b]);
          tc::mma_commit(&a_empty[a]);
          ++f;
          b = (b + 1 == BR) ? 0 : b + 1;
          a = (a + 1 == AST) ? 0 : a + 1;
        }
        if (!ok) break;
        tc::mma_commit(&accf_bar[ab]);
      }
      // every MMA issued has completed before tensor memory is freed
      tc::mma_commit(&mma_done);
      mbar_wait_bounded(&mma_done, 0, kWaitIters);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------- dequant
    const int d = threadIdx.x - 128;
    const int am = d >> 7;   // weight tile
    const int rw = d & 127;  // row of the tile
    constexpr int kInChunks = 4;  // 16 codes per chunk
    int c = 0, a = 0;
    uint32_t f = 0;
    for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x) {
      const int tau = item / p.nsub, sub = item - tau * p.nsub;
      const TileInfo ti = tile_info(p, tau);
      const int ebase = ti.e < 0 ? 0 : ti.e * p.R;
      const int row = ebase + weight_row0(p, MODE, sub, am) + rw;
      // this row's block constants, one 32-bit word per K step, fetched one
      // group of 8 K steps ahead: Q8_0 the two block scales (4-byte aligned
      // for any K % 64 == 0), affine-4 the group's scale | bias << 16
      const __half* scb = (ti.e < 0 ? p.scales_sh : p.scales) +
                          (size_t)row * (p.K / (QT == QSM_Q8_0 ? 32 : 64));
      const __half* bib = QT == QSM_Q8_0 ? nullptr
                                         : (ti.e < 0 ? p.biases_sh : p.biases) +
                                               (size_t)row * (p.K / 64);
      auto consts = [&](int ks) -> uint32_t {
        if (QT == QSM_Q8_0) return __ldg(reinterpret_cast<const uint32_t*>(scb) + ks);
        return (uint32_t)__half_as_ushort(__ldg(scb + ks)) |
               ((uint32_t)__half_as_ushort(__ldg(bib + ks)) << 16);
      };
      uint32_t nx[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) nx[jj] = jj < ksteps ? consts(jj) : 0u;
      bool ok = true;
      for (int kg = 0; kg < ksteps && ok; kg += 8) {
        uint32_t cur[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          cur[jj] = nx[jj];
          nx[jj] = kg + 8 + jj < ksteps ? consts(kg + 8 + jj) : 0u;
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (kg + jj >= ksteps) break;
          if (!wait_bar(&c_full[c], (f / CR) & 1, abort_p, p.status) ||
              (f >= AST && !wait_bar(&a_empty[a], ((f / AST) - 1) & 1, abort_p, p.status))) {
            ok = false;
            break;
          }
          const uint32_t sc2 = cur[jj];
          const unsigned char* codes = cring + c * C_STAGE + am * C_BYTES + rw * KB;
          unsigned char* arow_s = aring + a * A_STAGE + am * A_BYTES + (rw >> 3) * 1024 +
                                  (rw & 7) * 128;
          if (QT == QSM_AFFINE4_G64) {
            // word i holds K 8i..8i+7: one 16-byte output chunk each
            const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)(sc2 & 0xffffu)));
            const __half2 b2 = __half2half2(__ushort_as_half((unsigned short)(sc2 >> 16)));
            const uint4 w0 = *reinterpret_cast<const uint4*>(codes);
            const uint4 w1 = *reinterpret_cast<const uint4*>(codes + 16);
            const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(arow_s + ((i ^ (rw & 7)) << 4)) =
                  a4_word_to_f16x8(wv[i], s2, b2);
          } else {
#pragma unroll
          for (int j = 0; j < kInChunks; ++j) {
            // chunk order per row: conflict-free shared-memory banks for the
            // code reads (8 rows per quarter warp, 64-byte row pitch) and the
            // swizzled fp16 writes alike
            const int ci = j ^ (int)((0x5FA0u >> (2 * (rw & 7))) & 3u);
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
          }
          tc::mbar_arrive(&c_empty[c]);
          tc::fence_async_smem();
          tc::mbar_arrive(&a_full[a]);
          ++f;
          c = (c + 1 == CR) ? 0 : c + 1;
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
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++j) {
      if (warp_aborted(abort_p)) break;
      const int tau = item / p.nsub, sub = item - tau * p.nsub;
      const TileInfo ti = tile_info(p, tau);
      const int b = j & 1;
      // this thread's token row of the tile: its sorted row (gate_up) or
      // its token and routing weight (down)
      const bool live = et < ti.cnt;
      const int srow = (ti.e < 0 ? p.T * p.k : 0) + ti.row0 + et;
      int tok = 0;
      float wt = 0.f;
      if (MODE == kDown && live) {
        if (ti.e < 0) {  // shared expert: weight 1, or its gate
          tok = ti.row0 + et;
          wt = (p.gate ? __ldcg(p.gate + tok) : 1.f) * kHScaleInv;
        } else {
          const int asg = __ldcg(p.perm + ti.row0 + et);
          tok = asg / p.k;
          wt = __ldcg(p.topk_w + asg) * kHScaleInv;
        }
      }
      if (!__all_sync(0xffffffffu, wait_bar(&accf_bar[b], (j >> 1) & 1, abort_p, p.status)))
        break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16) + b * 256;
      if (MODE == kGateUp) {
        // columns 0..127 gate, 128..255 up of intermediates sub*128 + c
        __half* dst = p.hbuf + (size_t)srow * p.I + sub * BM;
        for (int c0 = 0; c0 < BM; c0 += 16) {
          float gv[16], uv[16];
          tc::tmem_ld16(taddr + c0, gv);
          tc::tmem_ld16(taddr + BM + c0, uv);
          if (live) {
            uint32_t hw[8];
            if (p.gu_dump) {  // test hook: the fused projection's values per h row
              float* dr = p.gu_dump + (size_t)srow * 2 * p.I + sub * BM + c0;
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                dr[c] = gv[c];
                dr[p.I + c] = uv[c];
              }
            }
#pragma unroll
            for (int c = 0; c < 16; c += 2) {
              const float h0 = silu(gv[c]) * uv[c] * kHScale;
              const float h1 = silu(gv[c + 1]) * uv[c + 1] * kHScale;
              if (!(fabsf(h0) <= 65504.f) || !(fabsf(h1) <= 65504.f)) bad = true;
              const __half2 hh = __floats2half2_rn(h0, h1);
              hw[c / 2] = *reinterpret_cast<const uint32_t*>(&hh);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
            d4[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            d4[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          }
        }
      } else {
        // The accumulator read in 16-lane halves with the 16x256b shape:
        // four consecutive threads hold 8 consecutive output rows of one
        // token, so a warp's reduce-add covers 32 contiguous bytes of each
        // of 8 tokens (half the L2 transactions of 16 bytes of 32 tokens).
        // Thread t handles warp rows t / 4 + 8 i (i = 0..3): their tokens and
        // weights come from the rows' own threads.
        const int rq = lane >> 2, cq = 2 * (lane & 3);
        float* rdst[4];
        float rwt[4];
        bool rlive[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int src = rq + 8 * i;
          const int t2 = __shfl_sync(0xffffffffu, tok, src);
          rwt[i] = __shfl_sync(0xffffffffu, wt, src);
          rlive[i] = 32 * q4 + src < ti.cnt;
          rdst[i] = p.yacc + (size_t)t2 * p.H + sub * (NA * BM) + cq;
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          for (int c0 = 0; c0 < NA * BM; c0 += 32) {
            uint32_t r[16];
            tmem_ld_16x256b_x4(taddr + ((uint32_t)(16 * hh) << 16) + c0, r);
            tc::tmem_wait_ld(r);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int i0 = 2 * hh, i1 = 2 * hh + 1;
              if (rlive[i0])
                red_add_v2(rdst[i0] + c0 + 8 * jj, rwt[i0] * __uint_as_float(r[4 * jj]),
                           rwt[i0] * __uint_as_float(r[4 * jj + 1]));
              if (rlive[i1])
                red_add_v2(rdst[i1] + c0 + 8 * jj, rwt[i1] * __uint_as_float(r[4 * jj + 2]),
                           rwt[i1] * __uint_as_float(r[4 * jj + 3]));
            }
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acce_bar[b]);
    }
    if (bad) set_status(p.status, QSM_DEV_FP16_RANGE);
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// The token operand of gate_up, fp16 [A + T, H] with A = T*k: row r < A
// holds the token of assignment perm[r] (zero if that assignment has no
// valid expert), row A + t holds token t.  One warp per row, its 16-byte
// chunks loaded four at a time before they are converted and stored.  With
// a shared-expert gate, the warp of row A + t also forms sigmoid(x[t] .
// shared_gate) in fp32.  Also zeroes the fp32 output accumulator.
__global__ void __launch_bounds__(256)
prep_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, int T,
            int k, int H, __half* __restrict__ xall, float* __restrict__ yacc,
            const float* __restrict__ sgate, float* __restrict__ gbuf,
            int32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  bool bad = false;
  const int A = T * k, rows = A + T;
  const int cpr = H / 8;  // 16-byte chunks per row
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    int t = r - A;
    if (r < A) {
      const int a = __ldcg(perm + r);
      t = a >= 0 ? a / k : -1;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(t < 0 ? 0 : t) * H);
    uint4* dst = reinterpret_cast<uint4*>(xall + (size_t)r * H);
    const bool gate_row = sgate != nullptr && r >= A;
    float z = 0.f;
    for (int c0 = lane; c0 < cpr; c0 += 4 * 32) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u;
        v[u] = (c < cpr && t >= 0) ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u;
        if (c >= cpr) break;
        const uint4 h = make_uint4(bf16x2_to_f16x2(v[u].x), bf16x2_to_f16x2(v[u].y),
                                   bf16x2_to_f16x2(v[u].z), bf16x2_to_f16x2(v[u].w));
        if (gate_row) {
          const float4 w0 = __ldg(reinterpret_cast<const float4*>(sgate) + 2 * c);
          const float4 w1 = __ldg(reinterpret_cast<const float4*>(sgate) + 2 * c + 1);
          z = fmaf(bf16_lo(v[u].x), w0.x, z);
          z = fmaf(bf16_hi(v[u].x), w0.y, z);
          z = fmaf(bf16_lo(v[u].y), w0.z, z);
          z = fmaf(bf16_hi(v[u].y), w0.w, z);
          z = fmaf(bf16_lo(v[u].z), w1.x, z);
          z = fmaf(bf16_hi(v[u].z), w1.y, z);
          z = fmaf(bf16_lo(v[u].w), w1.z, z);
          z = fmaf(bf16_hi(v[u].w), w1.w, z);
        }
        const uint32_t* hw = reinterpret_cast<const uint32_t*>(&h);
#pragma unroll
        for (int q = 0; q < 4; ++q)  // an all-ones exponent: out of fp16 range
          if ((hw[q] & 0x7c00u) == 0x7c00u || (hw[q] & 0x7c000000u) == 0x7c000000u)
            bad = true;
        dst[c] = h;
      }
    }
    if (gate_row) {
      z = warp_sum(z);
      if (lane == 0) gbuf[t] = 1.0f / (1.0f + __expf(-z));
    }
  }
  const size_t ny = (size_t)T * H / 4;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < ny; i += stride)
    reinterpret_cast<float4*>(yacc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (bad) set_status(status, QSM_DEV_FP16_RANGE);
}

// y = bf16(y_acc) (and the fp32 copy).  Four 16-byte loads per thread in
// flight per step.
__device__ __forceinline__ void finalize_one(float4 v, size_t i, uint16_t* __restrict__ y,
                                             float* __restrict__ y32) {
  const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y)) << 16);
  const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w)) << 16);
  reinterpret_cast<uint2*>(y)[i] = make_uint2(lo, hi);
  if (y32) reinterpret_cast<float4*>(y32)[i] = v;
}

__global__ void __launch_bounds__(256)
finalize_kernel(const float* __restrict__ yacc, uint16_t* __restrict__ y,
                float* __restrict__ y32, size_t n4) {
  pdl_wait();
  pdl_launch_dependents();
  const float4* src = reinterpret_cast<const float4*>(yacc);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcg(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) finalize_one(v[u], i + u * stride, y, y32);
  }
  for (; i < n4; i += stride) finalize_one(__ldcg(src + i), i, y, y32);
}

// (code ring, token ring, dequantised ring) depths
constexpr int kGateUpC = 4, kGateUpB = 3, kGateUpA = 3;
constexpr int kDownC = 4, kDownB = 3, kDownA = 3;

template <int QT, int CR, int BR, int AST>
constexpr size_t gemm_smem() {
  constexpr int NA = 2;
  constexpr int KB = QT == QSM_Q8_0 ? BK : BK / 2;
  return (size_t)AST * NA * BM * BK * 2 + (size_t)BR * BN * BK * 2 +
         (size_t)CR * NA * BM * KB + 1024;
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

template <int QT>
qsm_status launch_gemms(const Params& p1, const Params& p2, cudaStream_t stream) {
  constexpr size_t smem1 = gemm_smem<QT, kGateUpC, kGateUpB, kGateUpA>();
  constexpr size_t smem2 = gemm_smem<QT, kDownC, kDownB, kDownA>();
  static_assert(smem1 <= 225 * 1024 && smem2 <= 225 * 1024, "shared memory");
  auto* k1 = moe_prefill_gemm<kGateUp, QT, kGateUpC, kGateUpB, kGateUpA>;
  auto* k2 = moe_prefill_gemm<kDown, QT, kDownC, kDownB, kDownA>;
  QSM_CUDA_TRY(cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem1));
  QSM_CUDA_TRY(cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem2));
  const int nsm = sm_count();
  QSM_CUDA_TRY(launch_pdl(k1, dim3(nsm), dim3(kThreads), smem1, stream, p1));
  QSM_CUDA_TRY(launch_pdl(k2, dim3(nsm), dim3(kThreads), smem2, stream, p2));
  return QSM_OK;
}

struct WsLayout {
  size_t xall, hbuf, yacc, gate, total;
};

inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

WsLayout ws_layout(const qsm_moe_layer* L, int T) {
  WsLayout w;
  const size_t rows = (size_t)T * L->k + T;  // grouped rows, then shared
  w.xall = 0;
  w.hbuf = up256(rows * L->H * 2);
  w.yacc = w.hbuf + up256(rows * L->I * 2);
  w.gate = w.yacc + up256((size_t)T * L->H * 4);
  w.total = w.gate + up256((size_t)T * 4);
  return w;
}

}  // namespace prefill

bool prefill_supported(const qsm_moe_layer* L) {
  return (L->gate_up.qtype == QSM_Q8_0 || L->gate_up.qtype == QSM_AFFINE4_G64) &&
         L->H % 256 == 0 && L->I % 128 == 0;
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
  __half* xall = reinterpret_cast<__half*>(wsb + wl.xall);
  __half* hbuf = reinterpret_cast<__half*>(wsb + wl.hbuf);
  float* yacc = reinterpret_cast<float*>(wsb + wl.yacc);
  float* gbuf = reinterpret_cast<float*>(wsb + wl.gate);
  const int nsm = sm_count();
  const size_t rows_h = (size_t)T * k + T;
  float* dump = nullptr;
  if (g_gu_dump) {
    if (g_gu_dump_floats < rows_h * 2 * I) return QSM_ERR_INVALID_ARGUMENT;
    dump = g_gu_dump;
  }

  QSM_CUDA_TRY(launch_pdl(prep_kernel, dim3(4 * nsm), dim3(256), 0, stream, x,
                          (const int32_t*)g->perm, T, k, H, xall, yacc, L->shared_gate,
                          gbuf, dev_status));

  // code tiles: 64 K per step = 64 bytes (Q8_0) or 32 bytes (affine-4) a row
  const bool a4 = L->gate_up.qtype == QSM_AFFINE4_G64;
  const int kb = a4 ? BK / 2 : BK;
  auto code_cols = [&](int K) { return (uint64_t)(a4 ? K / 2 : K); };
  Params p1 = {};
  bool ok = true;
  ok &= tc::make_map_2d(&p1.codes, L->gate_up.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                        (uint64_t)E * 2 * I, code_cols(H), kb, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok &= tc::make_map_2d(&p1.codes_sh, L->shared_gate_up.codes,
                        CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 2 * I, code_cols(H), kb, BM,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  for (int m = 0; m < 4; ++m)
    ok &= tc::make_map_2d(&p1.bmap[m], xall, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows_h, H,
                          BK, BN >> m, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return QSM_ERR_CUDA;
  p1.scales = reinterpret_cast<const __half*>(L->gate_up.scales);
  p1.scales_sh = reinterpret_cast<const __half*>(L->shared_gate_up.scales);
  p1.biases = reinterpret_cast<const __half*>(L->gate_up.biases);
  p1.biases_sh = reinterpret_cast<const __half*>(L->shared_gate_up.biases);
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
  p1.gate = L->shared_gate ? gbuf : nullptr;
  p1.gu_dump = dump;
  p1.status = dev_status;

  Params p2 = p1;
  ok &= tc::make_map_2d(&p2.codes, L->down.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                        (uint64_t)E * H, code_cols(I), kb, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok &= tc::make_map_2d(&p2.codes_sh, L->shared_down.codes,
                        CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, H, code_cols(I), kb, BM,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  for (int m = 0; m < 4; ++m)
    ok &= tc::make_map_2d(&p2.bmap[m], hbuf, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows_h, I,
                          BK, BN >> m, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return QSM_ERR_CUDA;
  p2.scales = reinterpret_cast<const __half*>(L->down.scales);
  p2.scales_sh = reinterpret_cast<const __half*>(L->shared_down.scales);
  p2.biases = reinterpret_cast<const __half*>(L->down.biases);
  p2.biases_sh = reinterpret_cast<const __half*>(L->shared_down.biases);
  p2.R = H;
  p2.K = I;
  p2.nsub = H / (2 * BM);
  p2.gu_dump = nullptr;

  const qsm_status st = a4 ? launch_gemms<QSM_AFFINE4_G64>(p1, p2, stream)
                           : launch_gemms<QSM_Q8_0>(p1, p2, stream);
  if (st != QSM_OK) return st;
  QSM_CUDA_TRY(launch_pdl(finalize_kernel, dim3(4 * nsm), dim3(256), 0, stream,
                          (const float*)yacc, y, y32, (size_t)T * H / 4));
  return QSM_OK;
}

}  // namespace qsm
