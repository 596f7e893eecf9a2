// Decode path, more than 8 tokens: the gate_up matmul + SwiGLU as one
// persistent streaming pass over the touched experts' weights.
//
// "Optimizing on-device inference for Apple Silicon", section "Reducing
// intermediate and state traffic": the two input projections with their
// gated activation in one kernel; over the fused [gate; up] weight of "oMLX
// MoE gate/up 融合优化", section "融合原理".  The work slots are those of the
// short-batch kernel (blocks of at most 8 tokens of one expert, the shared
// expert's first); a work item is one slot x 8 intermediate indices, i.e. a
// 16-row weight tile (gate rows i0..i0+7 over up rows i0..i0+7), so SwiGLU
// stays thread-local as in the short-batch kernel.
//
// One CTA per SM takes a contiguous run of the items in slot order.  Its
// producer thread streams the tiles through a ring of TMA stages (3D row
// view of the codes, 128-byte swizzle, 8 rows per copy; the rows' block
// constants as 8-row boxes with the swizzle of their row width) and copies
// the x rows of each new slot into one of two buffers, which the consumers
// convert to fp16 in place: an expert's tokens are staged once per CTA
// rather than once per 16 weight rows.  Four groups of four consumer warps
// take the items in turn; the warps of a group split the tile's 64-wide K
// chunks, add their partials in warp order and the group's first warp
// applies SwiGLU and stores h.  A stage is waited for and released by the
// warps of the group that owns its position only.
//
// Fewer instructions per weight than dequantising each one: the codes go
// into the MMA still biased under an fp16 exponent (Q8_0: 1152 + c from the
// byte's sign flip, affine-4: 1024 + c from the nibble), both exact, and the
// bias and the block constants are applied once per block and token from the
// block sums of x, staged with the slot:
//   Q8_0      sum_k s c_k x_k          = s (P - 1152 X)
//   affine-4  sum_k (s c_k + b) x_k    = s (P - 1024 X) + b X
// with P the MMA's fp32 sum over the block and X = sum_k x_k in fp32.  The
// cancellation in P - 1152 X costs about 2^-24 of |P| (a few 1e-4 of the
// block's code sum), far inside the path's tolerance; weights are never
// rounded to fp16, unlike the short-batch kernel.  For affine-4 the staged
// x rows are stored with each 8-group in the order 0 4 1 5 2 6 3 7, the K
// order in which the nibble extraction yields code pairs, so the MMA's B
// registers are whole words.
//
// h has the short-batch kernel's layout: routed rows at their sorted
// position, the shared expert's rows after the T*k routed ones.
#include "decode_stream.cuh"

#include "gemv_core.cuh"
#include "tc_common.cuh"

namespace qsm {
namespace dstream {

using namespace gemv;

constexpr int kGW = 4;                  // warps of a consumer group
constexpr int kNG = 4;                  // consumer groups
constexpr int kCW = kGW * kNG;          // consumer warps
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kMaxS = 8;                // ring stages at most (a multiple of kNG)
static_assert(kMaxS % kNG == 0, "stages per consumer group");
constexpr int kTok = 8;                 // tokens per slot (the MMA's N)
constexpr uint32_t kShortWait = 1u << 10;  // waits after a timeout
constexpr float kHScale = 1.0f / 16.0f;
constexpr size_t kSmemBudget = 208 * 1024;  // dynamic shared memory
constexpr int kBarAll = 15;             // named barrier of all consumer warps (groups: 1..kNG)

// Padding (fp16 elements) after each staged x row: the eight rows of an MMA's
// B fragment then fall in different shared-memory banks for the K offsets
// each weight type reads.
__host__ __device__ constexpr int x_pad(int qt) { return qt == QSM_Q8_0 ? 32 : 8; }

struct Params {
  CUtensorMap gu;      // routed codes [E*2I, hb] u8, 3D row view, 8-row boxes
  CUtensorMap gu_sh;   // shared expert's codes [2I, hb]
  // block scales and (affine-4) biases [rows, hsb / 2] u16, 8-row boxes of
  // whole rows with the swizzle of the row's width (hsb = 32, 64 or 128 B),
  // so that the eight rows of a tile read one group each without bank
  // conflicts
  CUtensorMap sc, sc_sh, bi, bi_sh;
  const uint16_t* x;   // [T, H] bf16
  const int32_t* perm;
  const int32_t* offsets;
  const int32_t* tile_map;
  const int32_t* n_tiles;
  const float* sgate;  // [H] shared-expert gate weights, or NULL
  float* gbuf;         // [T] sigmoid(x . sgate)
  __half* hbuf;        // [T*k + T, I] fp16 h / 16
  float* gu_dump;      // test hook: [T*k + T, 2I] fp32 gate and up values, or NULL
  int32_t* status;
  int T, H, I, k, shared_slots;
  int hb, hsb;         // code bytes and block-constant bytes per weight row
  int ns, slot_bytes, x_off, xsum_off;
};

struct Slot {
  int e;     // -1 = shared expert
  int row0;  // first sorted row (routed) or first token (shared)
  int cnt;   // tokens of the slot (1..8)
};

__device__ __forceinline__ Slot slot_at(const Params& p, int s, int n_tiles) {
  Slot r;
  if (s < p.shared_slots) {
    r.e = -1;
    r.row0 = kTok * s;
    r.cnt = min(kTok, p.T - r.row0);
  } else {
    const int tau = s - p.shared_slots;
    const int2 te = __ldcg(reinterpret_cast<const int2*>(p.tile_map) + tau);
    r.e = te.x;
    r.row0 = te.y;
    r.cnt = tau < n_tiles && te.x >= 0 ? min(kTok, __ldcg(p.offsets + te.x + 1) - te.y) : 0;
  }
  return r;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// 8 bytes at byte b (a multiple of 8) of 128-byte line `line`, 128-byte swizzle.
__device__ __forceinline__ uint2 lds_sw(const unsigned char* t, int line, int b) {
  return *reinterpret_cast<const uint2*>(
      t + line * 128 + ((((b >> 4) ^ (line & 7)) << 4) | (b & 15)));
}

// Byte offset of byte `bo` of row r in a tile of rows of `pitch` bytes
// (32, 64 or 128) written by TMA with the swizzle of that width: the 16-byte
// unit index is XORed with the row's position in the swizzle pattern.
__device__ __forceinline__ int swz(int r, int bo, int pitch) {
  const int a = r * pitch + bo;
  const int k = pitch == 128 ? 7 : (pitch == 64 ? 3 : 1);  // unit-index mask
  return a ^ (((a >> 7) & k) << 4);
}

// Raw A fragment of 64-chunk ch of a staged tile: gate rows at `cg`, up rows
// at `cu` (each [hb / 128 chunks][8 rows][128 B], 128-byte swizzle); block
// constants as swizzled tiles of 8 rows x hsb bytes: gate scales, up scales
// (, gate biases, up biases).
template <int QT>
__device__ __forceinline__ void tile_a(RawA& r, const unsigned char* cg,
                                       const unsigned char* cu, const unsigned char* ss,
                                       int hsb, int g, int ch, int q) {
  const int cb = 8 * hsb;  // bytes of one constants tile
  if (QT == QSM_Q8_0) {
    const int c = ch >> 1, b = (ch & 1) * 64 + 8 * q;
    r.g0 = lds_sw(cg, c * 8 + g, b);
    r.g1 = lds_sw(cg, c * 8 + g, b + 32);
    r.h0 = lds_sw(cu, c * 8 + g, b);
    r.h1 = lds_sw(cu, c * 8 + g, b + 32);
    r.sg = *reinterpret_cast<const uint32_t*>(ss + swz(g, 4 * ch, hsb));
    r.sh = *reinterpret_cast<const uint32_t*>(ss + cb + swz(g, 4 * ch, hsb));
  } else {
    const int c = ch >> 2, b = (ch & 3) * 32 + 8 * q;
    r.g0 = lds_sw(cg, c * 8 + g, b);
    r.h0 = lds_sw(cu, c * 8 + g, b);
    const int o = swz(g, 2 * ch, hsb);
    const uint32_t sgv = *reinterpret_cast<const uint16_t*>(ss + o);
    const uint32_t suv = *reinterpret_cast<const uint16_t*>(ss + cb + o);
    const uint32_t bgv = *reinterpret_cast<const uint16_t*>(ss + 2 * cb + o);
    const uint32_t buv = *reinterpret_cast<const uint16_t*>(ss + 3 * cb + o);
    r.sg = sgv | (bgv << 16);
    r.sh = suv | (buv << 16);
  }
}

// Q8_0: 4 codes -> fp16 (1152 + c) pairs, lo = (c0, c1), hi = (c2, c3): the
// sign-flipped byte under the exponent of 1024.
__device__ __forceinline__ void q8_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
}

// affine-4: the word of K 8i'..8i'+7 -> fp16 (1024 + c_n, 1024 + c_{n+4}),
// n = 0..3: nibble n (low half) and n + 4 (high half) under the exponent.
__device__ __forceinline__ void a4_biased(uint32_t w, uint32_t (&v)[4]) {
#pragma unroll
  for (int n = 0; n < 4; ++n) v[n] = ((w >> (4 * n)) & 0x000F000Fu) | 0x64006400u;
}

__device__ __forceinline__ float f16lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
}
__device__ __forceinline__ float f16hi(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// acc (rows g, g, g+8, g+8 x tokens 2q, 2q+1) += the tile's 64-chunk times
// the staged x (X0, X1 as the weight type's B layout wants them); xs: the
// chunk's x block sums [block][token] (two 32-blocks).
template <int QT>
__device__ __forceinline__ void chunk_biased(float (&acc)[4], const RawA& r, const uint4& X0,
                                             const uint4& X1, const float* xs, int q) {
  if (QT == QSM_Q8_0) {
    float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const uint2 wg = blk ? r.g1 : r.g0, wh = blk ? r.h1 : r.h0;
        uint32_t a[4], b0, b1;
        q8_biased(jj ? wg.y : wg.x, a[0], a[2]);
        q8_biased(jj ? wh.y : wh.x, a[1], a[3]);
        b_frag<QT>(X0, X1, 2 * blk + jj, b0, b1);
        mma_16816(d[blk], a, b0, b1);
      }
    }
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const float2 X = *reinterpret_cast<const float2*>(xs + blk * kTok + 2 * q);
      const float sg = blk ? f16hi(r.sg) : f16lo(r.sg);
      const float sh = blk ? f16hi(r.sh) : f16lo(r.sh);
      acc[0] = fmaf(sg, fmaf(-1152.f, X.x, d[blk][0]), acc[0]);
      acc[1] = fmaf(sg, fmaf(-1152.f, X.y, d[blk][1]), acc[1]);
      acc[2] = fmaf(sh, fmaf(-1152.f, X.x, d[blk][2]), acc[2]);
      acc[3] = fmaf(sh, fmaf(-1152.f, X.y, d[blk][3]), acc[3]);
    }
  } else {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
      uint32_t vg[4], vh[4];
      a4_biased(wi ? r.g0.y : r.g0.x, vg);
      a4_biased(wi ? r.h0.y : r.h0.x, vh);
      const uint4& X = wi ? X1 : X0;  // (x0,x4) (x1,x5) (x2,x6) (x3,x7)
#pragma unroll
      for (int par = 0; par < 2; ++par) {
        const uint32_t a[4] = {vg[2 * par], vh[2 * par], vg[2 * par + 1], vh[2 * par + 1]};
        mma_16816(d, a, par ? X.z : X.x, par ? X.w : X.y);
      }
    }
    const float2 X0s = *reinterpret_cast<const float2*>(xs + 2 * q);
    const float2 X1s = *reinterpret_cast<const float2*>(xs + kTok + 2 * q);
    const float xa = X0s.x + X1s.x, xb = X0s.y + X1s.y;
    const float sg = f16lo(r.sg), bg = f16hi(r.sg), sh = f16lo(r.sh), bh = f16hi(r.sh);
    acc[0] = fmaf(sg, fmaf(-1024.f, xa, d[0]), fmaf(bg, xa, acc[0]));
    acc[1] = fmaf(sg, fmaf(-1024.f, xb, d[1]), fmaf(bg, xb, acc[1]));
    acc[2] = fmaf(sh, fmaf(-1024.f, xa, d[2]), fmaf(bh, xa, acc[2]));
    acc[3] = fmaf(sh, fmaf(-1024.f, xb, d[3]), fmaf(bh, xb, acc[3]));
  }
}

template <int QT>
__global__ void __launch_bounds__(kThreads, 1)
gate_up_stream_kernel(const __grid_constant__ Params p) {
  extern __shared__ unsigned char ds_dyn[];
  __shared__ __align__(8) uint64_t full[kMaxS], empty[kMaxS], xfull[2], xempty[2];
  __shared__ float red[2][kCW][32][4];
  __shared__ volatile int s_bad;
  constexpr int kBi = QT == QSM_Q8_0 ? 1 : 2;  // constant planes (scales, biases)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int T = p.T, H = p.H, I = p.I, ns = p.ns;
  const int tps = I / 8;  // items (16-row tiles) per slot
  const uint32_t pad = (1024u - (smem_u32(ds_dyn) & 1023u)) & 1023u;
  unsigned char* ring = ds_dyn + pad;                                  // [ns][slot_bytes]
  uint16_t* xs = reinterpret_cast<uint16_t*>(ring + p.x_off);  // [2][8][xp] bf16, then fp16
  const int xp = H + x_pad(QT);                                 // elements per staged row
  float* xsum = reinterpret_cast<float*>(ring + p.xsum_off);    // [2][H/32][8] block sums

  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGW);  // the owning group's warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xfull[b], 1);
      mbar_init(&xempty[b], kCW);
    }
    s_bad = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Every wait is bounded; after one runs out the kernel keeps going on
  // short waits (results invalid, status set) so that it always ends.
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (mbar_wait_bounded(bar, parity, s_bad ? kShortWait : kWaitIters)) return;
    s_bad = 1;
    set_status(p.status, QSM_DEV_TIMEOUT);
  };

  // The slots come from the grouping launch.
  pdl_wait();
  pdl_launch_dependents();
  const int n_tiles = __ldcg(p.n_tiles);
  const int total = (p.shared_slots + n_tiles) * tps;
  const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
  const int p0 = min(total, (int)blockIdx.x * per);
  const int n = min(total, p0 + per) - p0;

  // ================================================================ producer
  if (warp == kCW) {
    if (lane != 0) return;
    int prev = -1, xuse = 0;
    Slot sl = {0, 0, 0};
    for (int pos = 0; pos < n; ++pos) {
      const int it = p0 + pos, s = it / tps, j = it - s * tps;
      if (s != prev) {  // the slot's x rows into the next buffer
        sl = slot_at(p, s, n_tiles);
        const int b = xuse & 1;
        if (xuse >= 2) wait(&xempty[b], ((xuse >> 1) - 1) & 1);
        uint16_t* xb = xs + (size_t)b * kTok * xp;
        mbar_arrive_expect_tx(&xfull[b], (uint32_t)sl.cnt * H * 2);
        for (int c = 0; c < sl.cnt; ++c) {
          int tok = sl.row0 + c;
          if (sl.e >= 0) {
            const int a = __ldcg(p.perm + sl.row0 + c);
            tok = a >= 0 ? min(a / p.k, T - 1) : 0;
          }
          bulk_g2s(xb + (size_t)c * xp, p.x + (size_t)tok * H, (uint32_t)H * 2, &xfull[b]);
        }
        ++xuse;
        prev = s;
      }
      const int st = pos % ns;
      if (pos >= ns) wait(&empty[st], ((pos / ns) - 1) & 1);
      unsigned char* sb = ring + st * p.slot_bytes;
      const bool sh = sl.e < 0;
      const int rg = (sh ? 0 : sl.e * 2 * I) + 8 * j, ru = rg + I;
      mbar_arrive_expect_tx(&full[st], 16u * p.hb + 16u * p.hsb * kBi);
      tc::tma_load_3d(sb, sh ? &p.gu_sh : &p.gu, 0, rg, 0, &full[st]);
      tc::tma_load_3d(sb + 8 * p.hb, sh ? &p.gu_sh : &p.gu, 0, ru, 0, &full[st]);
      unsigned char* ss = sb + 16 * p.hb;
      const CUtensorMap* scm = sh ? &p.sc_sh : &p.sc;
      tc::tma_load_2d(ss, scm, 0, rg, &full[st]);
      tc::tma_load_2d(ss + 8 * p.hsb, scm, 0, ru, &full[st]);
      if (QT != QSM_Q8_0) {
        const CUtensorMap* bim = sh ? &p.bi_sh : &p.bi;
        tc::tma_load_2d(ss + 16 * p.hsb, bim, 0, rg, &full[st]);
        tc::tma_load_2d(ss + 24 * p.hsb, bim, 0, ru, &full[st]);
      }
    }
    // normally every copy has been consumed; after a timeout, let the last
    // copy of each buffer land before the CTA's shared memory goes away
    if (s_bad) {
      for (int s = 0; s < ns && s < n; ++s) {
        const int last = s + ((n - 1 - s) / ns) * ns;
        mbar_wait_bounded(&full[s], (last / ns) & 1, kWaitIters);
      }
      for (int b = 0; b < 2 && b < xuse; ++b) {
        const int last = b + ((xuse - 1 - b) / 2) * 2;
        mbar_wait_bounded(&xfull[b], (last >> 1) & 1, kWaitIters);
      }
    }
    return;
  }

  // ================================================================ consumers
  const int gi = warp / kGW, wg = warp % kGW;
  const int nch = H / 64;
  int prev = -1, xuse = 0, jg = 0;
  Slot sl = {0, 0, 0};
  uint16_t* xb = xs;
  bool range_bad = false;
  for (int pos = 0; pos < n; ++pos) {
    const int it = p0 + pos, s = it / tps, j = it - s * tps;
    if (s != prev) {
      if (xuse >= 1) {  // done with the previous slot's x rows
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&xempty[(xuse - 1) & 1]);
      }
      sl = slot_at(p, s, n_tiles);
      const int b = xuse & 1;
      wait(&xfull[b], (xuse >> 1) & 1);
      xb = xs + (size_t)b * kTok * xp;
      // gated shared expert: sigmoid(x . sgate) of the slot's tokens, by the
      // warps (one per token) that see the slot's first tile, from the bf16 rows
      if (p.sgate && sl.e < 0 && j == 0 && warp < sl.cnt) {
        const uint16_t* xr = xb + (size_t)warp * xp;
        float z = 0.f;
        for (int h8 = lane; h8 < H / 8; h8 += 32) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xr + 8 * h8);
          const float4 w0 = __ldg(reinterpret_cast<const float4*>(p.sgate) + 2 * h8);
          const float4 w1 = __ldg(reinterpret_cast<const float4*>(p.sgate) + 2 * h8 + 1);
          z = fmaf(bf16_lo(xv.x), w0.x, z);
          z = fmaf(bf16_hi(xv.x), w0.y, z);
          z = fmaf(bf16_lo(xv.y), w0.z, z);
          z = fmaf(bf16_hi(xv.y), w0.w, z);
          z = fmaf(bf16_lo(xv.z), w1.x, z);
          z = fmaf(bf16_hi(xv.z), w1.y, z);
          z = fmaf(bf16_lo(xv.w), w1.z, z);
          z = fmaf(bf16_hi(xv.w), w1.w, z);
        }
        z = warp_sum(z);
        if (lane == 0) p.gbuf[sl.row0 + warp] = 1.0f / (1.0f + __expf(-z));
      }
      // once per slot, by all consumer warps: the rows to fp16 in place (in
      // the weight type's K order) and their 32-block sums (fp32, in K
      // order); tokens past the slot's count get zero sums
      named_bar(kBarAll, kCW * 32);
      float* xsb = xsum + (size_t)b * (H / 32) * kTok;
      for (int i = tid; i < kTok * (H / 32); i += kCW * 32) {
        const int c = i / (H / 32), blk = i - c * (H / 32);
        float sum = 0.f;
        if (c < sl.cnt) {
          uint4* v = reinterpret_cast<uint4*>(xb + (size_t)c * xp + 32 * blk);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 raw = v[u];
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              sum += bf16_lo(w[e]);
              sum += bf16_hi(w[e]);
            }
            uint4 h = bf16x8_to_f16x8(raw);
            if (QT != QSM_Q8_0) {  // (x0,x1)(x2,x3)(x4,x5)(x6,x7) -> (x0,x4)(x1,x5)(x2,x6)(x3,x7)
              const uint4 o = h;
              h.x = __byte_perm(o.x, o.z, 0x5410);
              h.y = __byte_perm(o.x, o.z, 0x7632);
              h.z = __byte_perm(o.y, o.w, 0x5410);
              h.w = __byte_perm(o.y, o.w, 0x7632);
            }
            v[u] = h;
          }
        }
        xsb[blk * kTok + c] = sum;
      }
      named_bar(kBarAll, kCW * 32);
      ++xuse;
      prev = s;
    }
    // the group's own positions only.  The stage count is a multiple of the
    // group count, so every use of a stage belongs to the same group, which
    // waits for the stage's phases in order: a parity wait never meets a
    // phase two ahead of the one it asks for, and an arrival never counts
    // toward another use of the stage
    if (pos % kNG != gi) continue;
    const int st = pos % ns;
    wait(&full[st], (pos / ns) & 1);
    const unsigned char* sb = ring + st * p.slot_bytes;
    const unsigned char* ss = sb + 16 * p.hb;
    const bool has_tok = g < sl.cnt;
    const __half* xr = reinterpret_cast<const __half*>(xb) + (size_t)(has_tok ? g : 0) * xp;
    const float* xsb = xsum + (size_t)((xuse - 1) & 1) * (H / 32) * kTok;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto chunk = [&](int ch) {
      RawA r;
      tile_a<QT>(r, sb, sb + 8 * p.hb, ss, p.hsb, g, ch, q);
      uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
      if (has_tok) {
        X0 = *reinterpret_cast<const uint4*>(xr + 64 * ch + b_off0<QT>(q));
        X1 = *reinterpret_cast<const uint4*>(xr + 64 * ch + b_off1<QT>(q));
      }
      chunk_biased<QT>(acc, r, X0, X1, xsb + 2 * ch * kTok, q);
    };
    if (nch == 4 * kGW) {  // H = 2048: four chunks per warp, unrolled
#pragma unroll
      for (int u = 0; u < 4; ++u) chunk(wg + u * kGW);
    } else {
      for (int ch = wg; ch < nch; ch += kGW) chunk(ch);
    }
    consumed(acc);
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&empty[st]);
    // the group's partials, buffered by the group's item parity so that the
    // first warp still reading the previous ones is not overwritten
    float(*gred)[32][4] = red[jg & 1] + gi * kGW;
#pragma unroll
    for (int i = 0; i < 4; ++i) gred[wg][lane][i] = acc[i];
    named_bar(1 + gi, kGW * 32);
    if (wg == 0) {
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kGW; ++w) sum += gred[w][lane][i];
        a[i] = sum;
      }
      const int i0 = 8 * j;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * q + cc;
        if (c < sl.cnt) {
          const float h = silu(a[cc]) * a[2 + cc] * kHScale;
          if (!(fabsf(h) <= 65504.f)) range_bad = true;
          const size_t hrow = sl.e < 0 ? (size_t)T * p.k + sl.row0 + c : (size_t)sl.row0 + c;
          p.hbuf[hrow * I + i0 + g] = __float2half_rn(h);
          if (p.gu_dump) {  // test hook: the fused projection's values per h row
            p.gu_dump[hrow * 2 * I + i0 + g] = a[cc];
            p.gu_dump[hrow * 2 * I + I + i0 + g] = a[2 + cc];
          }
        }
      }
    }
    ++jg;
  }
  if (range_bad) set_status(p.status, QSM_DEV_FP16_RANGE);
}

// Ring stages for the layer: as many as the budget holds beside the two x
// buffers (at most kMaxS); 0 when fewer than 2 fit.
struct Geo {
  int hb, hsb, slot_bytes, ns, x_off, xsum_off;
  size_t smem;
};

bool geo_of(int qt, int H, Geo* g) {
  g->hb = qt == QSM_Q8_0 ? H : H / 2;
  g->hsb = (qt == QSM_Q8_0 ? H / 32 : H / 64) * 2;
  if (g->hb % 128 || g->hb / 128 > 256) return false;
  if (g->hsb != 32 && g->hsb != 64 && g->hsb != 128) return false;  // one swizzled box per row
  const int bi = qt == QSM_Q8_0 ? 1 : 2;
  g->slot_bytes = (16 * g->hb + 16 * g->hsb * bi + 1023) & ~1023;
  const size_t xrows = (size_t)2 * kTok * (H + x_pad(qt)) * 2;
  const size_t xbytes = xrows + (size_t)2 * (H / 32) * kTok * 4;
  if (1024 + 2 * (size_t)g->slot_bytes + xbytes > kSmemBudget) return false;
  g->ns = (int)((kSmemBudget - 1024 - xbytes) / g->slot_bytes);
  if (g->ns > kMaxS) g->ns = kMaxS;
  g->ns -= g->ns % kNG;  // every use of a stage by the same consumer group
  if (g->ns < kNG) return false;
  g->x_off = g->ns * g->slot_bytes;
  g->xsum_off = g->x_off + (int)xrows;
  g->smem = 1024 + (size_t)g->x_off + xbytes;
  return true;
}

int sm_count_ds() {
  static int n[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (n[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

template <int QT>
qsm_status launch_qt(const qsm_moe_layer* L, const uint16_t* x, int T, const qsm_grouping* grp,
                     int shared_slots, __half* hbuf, float* gbuf, float* gu_dump,
                     int32_t* dev_status, cudaStream_t stream) {
  Geo geo;
  if (!geo_of(QT, L->H, &geo)) return QSM_ERR_UNSUPPORTED;
  Params p;
  const int E = L->E, H = L->H, I = L->I;
  if (!tc::make_map_rows3d(&p.gu, L->gate_up.codes, (uint64_t)E * 2 * I, geo.hb, 8,
                           geo.hb / 128) ||
      !tc::make_map_rows3d(&p.gu_sh, L->shared_gate_up.codes, (uint64_t)2 * I, geo.hb, 8,
                           geo.hb / 128))
    return QSM_ERR_UNSUPPORTED;
  auto swz_of = [](int bytes) {
    return bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                        : (bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  };
  const int G = geo.hsb / 2;  // block constants per row
  bool ok = tc::make_map_2d(&p.sc, L->gate_up.scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                            (uint64_t)E * 2 * I, G, G, 8, swz_of(geo.hsb)) &&
            tc::make_map_2d(&p.sc_sh, L->shared_gate_up.scales, CU_TENSOR_MAP_DATA_TYPE_UINT16,
                            2, (uint64_t)2 * I, G, G, 8, swz_of(geo.hsb));
  if (QT != QSM_Q8_0)
    ok = ok &&
         tc::make_map_2d(&p.bi, L->gate_up.biases, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                         (uint64_t)E * 2 * I, G, G, 8, swz_of(geo.hsb)) &&
         tc::make_map_2d(&p.bi_sh, L->shared_gate_up.biases, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                         (uint64_t)2 * I, G, G, 8, swz_of(geo.hsb));
  if (!ok) return QSM_ERR_UNSUPPORTED;
  p.x = x;
  p.perm = grp->perm;
  p.offsets = grp->offsets;
  p.tile_map = grp->tile_map;
  p.n_tiles = grp->n_tiles;
  p.sgate = L->shared_gate;
  p.gbuf = gbuf;
  p.hbuf = hbuf;
  p.gu_dump = gu_dump;
  p.status = dev_status;
  p.T = T;
  p.H = H;
  p.I = I;
  p.k = L->k;
  p.shared_slots = shared_slots;
  p.hb = geo.hb;
  p.hsb = geo.hsb;
  p.ns = geo.ns;
  p.slot_bytes = geo.slot_bytes;
  p.x_off = geo.x_off;
  p.xsum_off = geo.xsum_off;
  auto* kern = gate_up_stream_kernel<QT>;
  QSM_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)geo.smem));
  QSM_CUDA_TRY(launch_pdl(kern, dim3(sm_count_ds()), dim3(kThreads), geo.smem, stream, p));
  return QSM_OK;
}

}  // namespace dstream

bool gate_up_stream_supported(const qsm_moe_layer* L) {
  dstream::Geo g;
  return L->I % 8 == 0 && dstream::geo_of(L->gate_up.qtype, L->H, &g);
}

qsm_status gate_up_stream_launch(const qsm_moe_layer* L, const uint16_t* x, int T,
                                 const qsm_grouping* grp, int shared_slots, __half* hbuf,
                                 float* gbuf, float* gu_dump, int32_t* dev_status,
                                 cudaStream_t stream) {
  if (L->gate_up.qtype == QSM_Q8_0)
    return dstream::launch_qt<QSM_Q8_0>(L, x, T, grp, shared_slots, hbuf, gbuf, gu_dump,
                                        dev_status, stream);
  return dstream::launch_qt<QSM_AFFINE4_G64>(L, x, T, grp, shared_slots, hbuf, gbuf, gu_dump,
                                             dev_status, stream);
}

}  // namespace qsm
