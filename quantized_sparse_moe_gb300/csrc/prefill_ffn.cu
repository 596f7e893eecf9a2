// Prefill path of the MoE FFN (many tokens): grouped GEMMs on the tcgen05
// tensor cores with the weights dequantised tile by tile on chip.
//
// "Optimizing on-device inference for Apple Silicon", section "Dequantizing
// weights during matrix multiplication": the grouped GEMM rebuilds small
// tiles of the quantized weights in on-chip memory just long enough to
// multiply them with the routed activation rows, accumulates in fp32, and
// never writes the expanded weight matrix to memory; section "Keeping
// expert routing on the GPU": the block map of the grouping drives the
// tiles, with no host round trip; section "Matching tile size to expert
// load": the MMA's token dimension is sized to each expert's block; "oMLX
// MoE gate/up 融合优化", "融合原理": one pass over the fused [gate; up]
// weight.
//
// Launch sequence (stream ordered, programmatic dependent launch):
//   prep      the token operand of gate_up as one fp16 matrix (exact for
//             the bf16 inputs): the routed rows in grouped order (sorted
//             row r holds the token of assignment perm[r]), then the T
//             tokens in order for the shared expert; with a gated shared
//             expert, its gates
//   gate_up   per work item (a block of <= 128 token rows of one expert and
//             128 intermediate indices): two accumulators D_gate, D_up
//             (128 weight rows x N tokens, fp32 in tensor memory) +=
//             [W_gate tile | W_up tile] x token rows^T, N = the block's
//             rows rounded up to 16; epilogue (one intermediate index per
//             thread) h = silu(gate) * up, stored fp16 (scaled by 1/16) per
//             sorted row.  Warp 3 zeroes the fp32 output accumulator.
//   down      per work item (same token block, 256 output rows as two
//             128-row tiles): D = W_down tiles x h rows^T; epilogue
//             y_acc[token][row] += routing weight * D (fp32 reduce-adds, a
//             warp's 32 rows of one token in one 128-byte request)
//   finalize  y = bf16(y_acc) (and the fp32 copy)
//
// Roles in a persistent CTA (one per SM, 16 warps):
//   warp 0       TMA producer of the int8 / uint4 code tiles (2D tensor map,
//                64- or 32-byte swizzle)
//   warp 1       allocates tensor memory; lane 0 issues the MMAs
//   warp 2       TMA producer of the token tiles: 2D boxes of the grouped
//                fp16 x (gate_up) or of h (down), 128 rows or a 64/32/16-row
//                decomposition of a short block, 128-byte swizzled, K-major
//   warp 3       gate_up: zeroes its slice of y_acc
//   warps 4-11   dequantise the code tiles, one weight row per thread, into
//                the A operand in tensor memory (tcgen05.st): fp16(code *
//                block scale) (Q8_0) or fp16(scale * code + bias) (affine-4)
//   warps 12-15  epilogue, one warp per quarter of the tensor-memory lanes
// Rings: code tiles in shared memory (freed once dequantised), token tiles
// in shared memory (freed by the MMA commit), dequantised weight tiles in
// tensor memory (freed by the MMA commit).  The weights are the MMA's A
// operand and never pass through shared memory, which leaves its bandwidth
// to the token tiles.  One accumulator pair (tensor-memory columns 0..255)
// connects MMA and epilogue; the dequantised ring (columns 256..511) runs
// ahead into the next item while the epilogue drains.
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

constexpr int BW = 128;   // weight rows per MMA tile (the MMA's M)
constexpr int BK = 64;    // K per stage: 128 bytes of fp16 token row
constexpr int BN = 128;   // token rows per block (the MMA's N <= BN) = the path's tile_rows
constexpr int kThreads = 512;
constexpr int kDeqThreads = 256;  // warps 4..11
constexpr int kEpiThreads = 128;  // warps 12..15
constexpr float kHScale = 1.0f / 16.0f;
constexpr float kHScaleInv = 16.0f;
// Tensor memory: the two accumulators at columns 0 and BN, then the ring of
// dequantised weight stages (two 128-row tiles of 64 K = 2 x 32 columns).
constexpr int kAst = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 2 * BN;
static_assert(kAcol + kAst * 64 <= kTmemCols, "tensor memory columns");

enum { kGateUp = 1, kDown = 2 };

struct Params {
  CUtensorMap codes;      // routed experts' codes [E*R, K code bytes] u8, box {KB, 128}
  CUtensorMap codes_sh;   // shared expert's codes [R, K code bytes]
  CUtensorMap bmap[4];    // token rows [T*k + T, K] fp16 (gate_up: grouped x; down:
                          // h), boxes {64, 128 / 64 / 32 / 16}
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
  int nsub;               // weight-tile pairs per block
  __half* hbuf;           // [T*k + T, I]
  float* yacc;            // [T, H]
  const float* gate;      // [T] shared-expert gates, or NULL (weight 1)
  float* gu_dump;         // test hook: [T*k + T, 2I] fp32 gate and up values, or NULL
  int32_t* status;
};

struct TileInfo {
  int e;     // expert, -1 = shared expert
  int row0;  // first sorted row (routed) or first token (shared)
  int cnt;   // rows in the block
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
  t.cnt = max(t.cnt, 0);
  t.n = max(16, (t.cnt + 15) & ~15);  // an empty block still issues a valid MMA
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
// .sync.aligned tensor-memory instructions or warp shuffles together).
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
  return mode == kGateUp ? a * p.I + sub * BW : (2 * sub + a) * BW;
}

__device__ __forceinline__ void red_add(float* y, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(y), "f"(v) : "memory");
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

template <int MODE, int QT, int CR, int BR>
__global__ void __launch_bounds__(kThreads, 1)
moe_prefill_gemm(const __grid_constant__ Params p) {
  constexpr int KB = QT == QSM_Q8_0 ? BK : BK / 2;  // code bytes per row and K step
  constexpr int C_BYTES = BW * KB;                  // one weight tile's codes
  constexpr int C_STAGE = 2 * C_BYTES;
  constexpr int B_BYTES = BN * BK * 2;              // token tile, fp16, 128B swizzle
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* bring = smem;                     // [BR][B_BYTES]
  unsigned char* cring = bring + BR * B_BYTES;     // [CR][C_STAGE]
  __shared__ __align__(8) uint64_t c_full[CR], c_empty[CR], b_full[BR], b_empty[BR],
      a_full[kAst], a_empty[kAst], acc_full, acc_empty, mma_done;
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
    for (int s = 0; s < kAst; ++s) {
      mbar_init(&a_full[s], kDeqThreads);
      mbar_init(&a_empty[s], 1);  // MMA commit
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kEpiThreads);
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
  if (warp == 1) tc::tmem_alloc(&tmem_base, kTmemCols);
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
        const int arow0 = ebase + weight_row0(p, MODE, sub, 0);
        const int arow1 = ebase + weight_row0(p, MODE, sub, 1);
        bool ok = true;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (f >= CR && !wait_bar(&c_empty[c], ((f / CR) - 1) & 1, abort_p, p.status)) {
            ok = false;
            break;
          }
          unsigned char* cdst = cring + c * C_STAGE;
          mbar_arrive_expect_tx(&c_full[c], C_STAGE);
          tc::tma_load_2d(cdst, cm, ks * KB, arow0, &c_full[c]);
          tc::tma_load_2d(cdst + C_BYTES, cm, ks * KB, arow1, &c_full[c]);
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
  } else if (warp == 3) {
    // ---------------------------------------- gate_up: zero the accumulator
    if (MODE == kGateUp) {
      float4* y4 = reinterpret_cast<float4*>(p.yacc);
      const size_t n4 = (size_t)p.T * p.H / 4;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      for (size_t i = (size_t)blockIdx.x * 32 + lane; i < n4; i += (size_t)gridDim.x * 32)
        y4[i] = z;
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      uint32_t f = 0;
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort_p; item += gridDim.x, ++j) {
        const int tau = item / p.nsub;
        const TileInfo ti = tile_info(p, tau);
        if (j >= 1 && !wait_bar(&acc_empty, (j - 1) & 1, abort_p, p.status)) break;
        tc::tc_fence_after();
        // D[weight row, token]: M = 128 weight rows per tile, N = the block
        const uint32_t idesc = tc::idesc_f16_m128(ti.n);
        bool ok = true;
        for (int ks = 0; ks < ksteps; ++ks) {
          const int b = (int)(f % BR), s = (int)(f % kAst);
          if (!wait_bar(&b_full[b], (f / BR) & 1, abort_p, p.status) ||
              !wait_bar(&a_full[s], (f / kAst) & 1, abort_p, p.status)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t b0 = smem_u32(bring + b * B_BYTES);
          const uint32_t a0 = tmem + kAcol + (uint32_t)s * 64;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = tc::sw128_desc(b0 + kk * 32);
            const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
            tc::mma_f16_tmem_a(tmem, a0 + kk * 8, bd, idesc, acc);
            tc::mma_f16_tmem_a(tmem + BN, a0 + 32 + kk * 8, bd, idesc, acc);
          }
          tc::mma_commit(&b_empty[b]);
          tc::mma_commit(&a_empty[s]);
          ++f;
        }
        if (!ok) break;
        tc::mma_commit(&acc_full);
      }
      // every MMA issued has completed before tensor memory is freed
      tc::mma_commit(&mma_done);
      mbar_wait_bounded(&mma_done, 0, kWaitIters);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------- dequant
    const int d = threadIdx.x - 128;
    const int am = d >> 7;        // weight tile
    const int m = d & 127;        // row of the tile = tensor-memory lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int c = 0;
    uint32_t f = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      if (warp_aborted(abort_p)) break;
      const int tau = item / p.nsub, sub = item - tau * p.nsub;
      const TileInfo ti = tile_info(p, tau);
      const int ebase = ti.e < 0 ? 0 : ti.e * p.R;
      const int row = ebase + weight_row0(p, MODE, sub, am) + m;
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
          const int s = (int)(f % kAst);
          const bool got =
              wait_bar(&c_full[c], (f / CR) & 1, abort_p, p.status) &&
              (f < kAst || wait_bar(&a_empty[s], ((f / kAst) - 1) & 1, abort_p, p.status));
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t sc2 = cur[jj];
          const unsigned char* tile = cring + c * C_STAGE + am * C_BYTES;
          uint32_t w[32];
          if (QT == QSM_AFFINE4_G64) {
            // 32 bytes a row, 32-byte swizzle: 16-byte unit u at u ^ ((m >> 2) & 1)
            const unsigned char* rp = tile + m * 32;
            const int sw = (m >> 2) & 1;
            const uint4 w0 = *reinterpret_cast<const uint4*>(rp + ((0 ^ sw) << 4));
            const uint4 w1 = *reinterpret_cast<const uint4*>(rp + ((1 ^ sw) << 4));
            const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)(sc2 & 0xffffu)));
            const __half2 b2 = __half2half2(__ushort_as_half((unsigned short)(sc2 >> 16)));
            const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 o = a4_word_to_f16x8(wv[i], s2, b2);
              w[4 * i] = o.x;
              w[4 * i + 1] = o.y;
              w[4 * i + 2] = o.z;
              w[4 * i + 3] = o.w;
            }
          } else {
            // 64 bytes a row, 64-byte swizzle: 16-byte unit u at u ^ ((m >> 1) & 3)
            const unsigned char* rp = tile + m * 64;
            const int sw = (m >> 1) & 3;
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const uint4*>(rp + ((u ^ sw) << 4));
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t sbits = (u < 2) ? (sc2 & 0xffffu) : (sc2 >> 16);
              const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)sbits));
              s8x4_to_f16x2x2(v[u].x, w[8 * u + 0], w[8 * u + 1]);
              s8x4_to_f16x2x2(v[u].y, w[8 * u + 2], w[8 * u + 3]);
              s8x4_to_f16x2x2(v[u].z, w[8 * u + 4], w[8 * u + 5]);
              s8x4_to_f16x2x2(v[u].w, w[8 * u + 6], w[8 * u + 7]);
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                __half2 h = __hmul2(*reinterpret_cast<__half2*>(&w[8 * u + t]), s2);
                w[8 * u + t] = *reinterpret_cast<uint32_t*>(&h);
              }
            }
          }
          tc::tmem_st32(tmem + lane_base + kAcol + (uint32_t)s * 64 + (uint32_t)am * 32, w);
          tc::tmem_wait_st(w);
          // The code slot is released only after the store, whose operands
          // are computed from every byte this thread loaded from it: an
          // arrive placed right after the loads could be issued while a
          // load is still in flight, and the next copy into the slot would
          // then overwrite its first rows under the reader.
          tc::mbar_arrive(&c_empty[c]);
          tc::tc_fence_before();
          tc::mbar_arrive(&a_full[s]);
          ++f;
          c = (c + 1 == CR) ? 0 : c + 1;
        }
      }
      if (!ok) break;
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16);
    int j = 0;
    bool bad = false;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++j) {
      if (warp_aborted(abort_p)) break;
      const int tau = item / p.nsub, sub = item - tau * p.nsub;
      const TileInfo ti = tile_info(p, tau);
      if (!__all_sync(0xffffffffu, wait_bar(&acc_full, j & 1, abort_p, p.status))) break;
      tc::tc_fence_after();
      if (MODE == kGateUp) {
        // lane = intermediate index; columns = the block's tokens
        const int ji = sub * BW + 32 * q4 + lane;
        const int srow0 = (ti.e < 0 ? p.T * p.k : 0) + ti.row0;
        for (int c0 = 0; c0 < ti.n; c0 += 16) {
          uint32_t gr[16], ur[16];
          tc::tmem_ld16_nowait(taddr + c0, gr);
          tc::tmem_ld16_nowait(taddr + BN + c0, ur);
          tc::tmem_wait_ld(gr, ur);
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            if (c0 + t < ti.cnt) {
              const float g = __uint_as_float(gr[t]), u = __uint_as_float(ur[t]);
              const float h = silu(g) * u * kHScale;
              if (!(fabsf(h) <= 65504.f)) bad = true;
              const size_t r = (size_t)(srow0 + c0 + t);
              p.hbuf[r * p.I + ji] = __float2half_rn(h);
              if (p.gu_dump) {
                p.gu_dump[r * 2 * p.I + ji] = g;
                p.gu_dump[r * 2 * p.I + p.I + ji] = u;
              }
            }
          }
        }
      } else {
        // lane = output row of each tile; columns = the block's tokens
        const int r0 = 2 * sub * BW + 32 * q4 + lane;
        for (int c0 = 0; c0 < ti.n; c0 += 16) {
          // token and routing weight (x16: h is stored / 16) of block row
          // c0 + lane, for lanes < 16, then shared across the warp
          int tok_l = 0;
          float wt_l = 0.f;
          if (lane < 16 && c0 + lane < ti.cnt) {
            const int i = c0 + lane;
            if (ti.e < 0) {  // shared expert: weight 1, or its gate
              tok_l = ti.row0 + i;
              wt_l = (p.gate ? __ldcg(p.gate + tok_l) : 1.f) * kHScaleInv;
            } else {
              const int asg = __ldcg(p.perm + ti.row0 + i);
              tok_l = asg >= 0 ? min(asg / p.k, p.T - 1) : 0;
              wt_l = asg >= 0 ? __ldcg(p.topk_w + asg) * kHScaleInv : 0.f;
            }
          }
          uint32_t d0[16], d1[16];
          tc::tmem_ld16_nowait(taddr + c0, d0);
          tc::tmem_ld16_nowait(taddr + BN + c0, d1);
          tc::tmem_wait_ld(d0, d1);
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int tok = __shfl_sync(0xffffffffu, tok_l, t);
            const float wt = __shfl_sync(0xffffffffu, wt_l, t);
            if (c0 + t < ti.cnt) {
              float* yr = p.yacc + (size_t)tok * p.H + r0;
              red_add(yr, wt * __uint_as_float(d0[t]));
              red_add(yr + BW, wt * __uint_as_float(d1[t]));
            }
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acc_empty);
    }
    if (bad) set_status(p.status, QSM_DEV_FP16_RANGE);
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// The token operand of gate_up, fp16 [A + T, H] with A = T*k: row r < A
// holds the token of assignment perm[r] (zero if that assignment has no
// valid expert), row A + t holds token t.  One warp per row, its 16-byte
// chunks loaded four at a time before they are converted and stored.  With
// a shared-expert gate, the warp of row A + t also forms sigmoid(x[t] .
// shared_gate) in fp32.
__global__ void __launch_bounds__(256)
prep_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, int T,
            int k, int H, __half* __restrict__ xall, const float* __restrict__ sgate,
            float* __restrict__ gbuf, int32_t* status) {
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
      t = a >= 0 ? min(a / k, T - 1) : -1;
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

// (code ring, token ring) depths in shared memory; the dequantised ring is
// kAst stages of tensor memory
constexpr int kGateUpC = 6, kGateUpB = 4;
constexpr int kDownC = 6, kDownB = 4;

template <int QT, int CR, int BR>
constexpr size_t gemm_smem() {
  constexpr int KB = QT == QSM_Q8_0 ? BK : BK / 2;
  return (size_t)BR * BN * BK * 2 + (size_t)CR * 2 * BW * KB + 1024;
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
  constexpr size_t smem1 = gemm_smem<QT, kGateUpC, kGateUpB>();
  constexpr size_t smem2 = gemm_smem<QT, kDownC, kDownB>();
  static_assert(smem1 <= 220 * 1024 && smem2 <= 220 * 1024, "shared memory");
  auto* k1 = moe_prefill_gemm<kGateUp, QT, kGateUpC, kGateUpB>;
  auto* k2 = moe_prefill_gemm<kDown, QT, kDownC, kDownB>;
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
                          (const int32_t*)g->perm, T, k, H, xall, L->shared_gate, gbuf,
                          dev_status));

  // code tiles: 64 K per step = 64 bytes (Q8_0, 64-byte swizzle) or 32 bytes
  // (affine-4, 32-byte swizzle) a row, 128 rows
  const bool a4 = L->gate_up.qtype == QSM_AFFINE4_G64;
  const int kb = a4 ? BK / 2 : BK;
  const CUtensorMapSwizzle csw = a4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
  auto code_cols = [&](int K) { return (uint64_t)(a4 ? K / 2 : K); };
  Params p1 = {};
  bool ok = true;
  ok &= tc::make_map_2d(&p1.codes, L->gate_up.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                        (uint64_t)E * 2 * I, code_cols(H), kb, BW, csw);
  ok &= tc::make_map_2d(&p1.codes_sh, L->shared_gate_up.codes,
                        CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 2 * I, code_cols(H), kb, BW, csw);
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
  p1.nsub = I / BW;
  p1.hbuf = hbuf;
  p1.yacc = yacc;
  p1.gate = L->shared_gate ? gbuf : nullptr;
  p1.gu_dump = dump;
  p1.status = dev_status;

  Params p2 = p1;
  ok &= tc::make_map_2d(&p2.codes, L->down.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                        (uint64_t)E * H, code_cols(I), kb, BW, csw);
  ok &= tc::make_map_2d(&p2.codes_sh, L->shared_down.codes,
                        CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, H, code_cols(I), kb, BW, csw);
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
  p2.nsub = H / (2 * BW);
  p2.gu_dump = nullptr;

  const qsm_status st = a4 ? launch_gemms<QSM_AFFINE4_G64>(p1, p2, stream)
                           : launch_gemms<QSM_Q8_0>(p1, p2, stream);
  if (st != QSM_OK) return st;
  QSM_CUDA_TRY(launch_pdl(finalize_kernel, dim3(4 * nsm), dim3(256), 0, stream,
                          (const float*)yacc, y, y32, (size_t)T * H / 4));
  return QSM_OK;
}

}  // namespace qsm
