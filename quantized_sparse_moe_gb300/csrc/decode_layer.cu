// The MoE layer for a few tokens (T <= 8) in one launch: router, expert
// selection, gate_up + SwiGLU, down + routing weights + shared expert.
//
// "Optimizing on-device inference for Apple Silicon": section "Keeping
// expert routing on the GPU" (the routing never leaves the device), section
// "Reducing intermediate and state traffic" (the input projections with
// their gated activation, then the output projection with its routing score
// and the shared expert's result, summed per token) and section
// "Overlapping independent GPU work"; the fused [gate; up] rows of "oMLX MoE
// gate/up 融合优化", section "融合原理".  The dependent launches of the
// decode path (router + grouping, gate_up, down) become three phases of one
// launch: an exchange of call-tagged logits after the router, and
// call-tagged h between gate_up and down.  No grouping is needed: every CTA
// derives its work from the selection itself.
//
//   A  CTA c computes the logits of its experts for the T tokens, with the
//      arithmetic of moe_route (router rows fetched before the
//      programmatic-launch wait), into the workspace, tagged with the call.
//   B  Every CTA waits for the tagged logits of all experts, selects each
//      token's experts from them with the code of moe_route (ids and
//      weights bit-identical to it), forms the sorted set U of selected
//      experts and computes gate_up + SwiGLU for its tiles.  Tile tau =
//      (slot, 8 intermediates): slot 0 is the shared expert, slot s >= 1
//      the s-th expert of U; a tile covers all T tokens (pairs that are not
//      routed are computed and never read).  h goes to the workspace as
//      64-bit words (call tag, two fp16 values).
//   C  CTA c < H / 16 computes rows 16c..16c+15 of y: for every slot, the
//      down rows times the slot's h, times the token's weight for the
//      slot's expert (the shared expert's gate, or 1; pairs with weight 0
//      are skipped), summed over the slots in a fixed order.  The slots go
//      a few at a time (C items); the consumers read an item's h from the
//      workspace, waiting until its words carry this call's tag (the data
//      and its readiness in one round trip), so a CTA with fewer tiles
//      starts on the first slots while others still compute the last
//      gate_up tiles.  (Placing items
//      between a CTA's own tiles, as soon as those they need are done, made
//      every item a grid-wide wait and was slower.)
//
// Weights stream through a shared-memory ring of up to five slots, filled
// by TMA from one producer thread: B tiles (gate and up halves of 8 rows,
// each one copy of the 3D row view with the 128-byte swizzle) and then C
// items (the down tiles of up to m slots, 16 rows each).  As soon as the
// selection is known the producer requests into L2 the weights of the next
// ~320 KB of its sequence past the ring (all of them for a few tokens), so
// HBM streams the layer at once and the ring mostly reads L2.  The shared
// expert's first tile and its down rows are requested before the wait; x
// is loaded by the consumer threads themselves (through L2: the previous
// launch wrote it), which is quicker than a bulk copy's round trip.
// For the gate_up tiles the consumer warps form two groups that take
// alternate ring positions, so two tiles are in flight at once; for the
// down items they form four smaller groups, so that the items of a layer
// run at once, each as soon as its slots' h is there.
//
// The grid has one CTA per SM (fewer when the layer has fewer gate_up
// tiles): CTAs c < H / 16 also own rows of y, the others only gate_up tiles,
// so that the tiles spread over every SM.  The logit exchange and the h
// hand-off need all G CTAs resident at once: G is at most the SM count and
// a launch's CTAs are all running once the launch lets its dependents start
// (every CTA triggers).  Every wait is bounded; when one runs out the kernel
// sets QSM_DEV_TIMEOUT, keeps its control flow (later waits are short), lets
// its own copies land and returns.  A 64-bit ticket in the workspace counts
// calls: every CTA adds 1 per call, so before its own arrival it reads
// (calls so far) * G plus the arrivals of this call, and the call's tag is
// calls so far + 1 (calls that share a workspace must have the same layer
// shape).  A logit travels as one 64-bit word (tag, value): a reader waits
// until every word of its token carries this call's tag, which is the
// barrier and the data in one round trip; h travels the same way.  Every h
// word a call reads is written by that call (a gate_up tile covers all T
// tokens of its slot), so a word of an earlier call never passes.
//
// Every phase runs once per launch, so code size matters: loops that run
// once are not unrolled, and the selection's code is warmed by idle warps
// while the token warps wait for the logits.  The hottest pieces have a
// second copy for the common shape (the selection for all 32 kPer
// candidates and top 8, the chunk loops for H = 2048 and for four chunks of
// a down slot), with the same arithmetic in the same order.
#include <algorithm>
#include <mutex>
#include <vector>

#include "gemv_core.cuh"
#include "route_select.cuh"
#include "tc_common.cuh"

namespace qsm {
namespace dlayer {

using namespace gemv;

// consumer warps: 16 when the top-k keeps few candidates per lane (E <= 256;
// the registers then allow 17 warps), else 8; plus one producer warp
template <int kPer>
constexpr int consumer_warps() { return kPer <= 8 ? 16 : 8; }
constexpr int kMaxS = 5;                  // ring slots (at most)
constexpr int kMaxT = 8;
constexpr int kMaxE = 1024;
constexpr int kTPE = 128;                 // router threads per expert
constexpr int kWPer = 4;                  // float4 of a router row per thread and batch
constexpr float kHScale = 1.0f / 16.0f;
constexpr float kHScaleInv = 16.0f;
constexpr int kBarCons = 1;               // named barrier of the consumer warps
constexpr int kBarGrp = 2;                // + group: named barriers of the gate_up groups
constexpr int kGW = 8;                    // warps per gate_up group
constexpr int kGWC = 4;                   // warps per down group (ids kBarGrp + 2 + group)
constexpr int kMaxGC = 4;                 // down groups at most
constexpr int kMaxM = 3;                  // down tiles (slots) per C item at most
constexpr uint32_t kShortWait = 1u << 10; // waits after a timeout

struct Params {
  CUtensorMap gu, gu_sh;  // gate_up codes, 3D row views, box {128, 8, hb/128}
  CUtensorMap dn, dn_sh;  // down codes, box {128, 16, ib/128}
  const uint8_t* gu_c;
  const uint8_t* gush_c;
  const uint8_t* dn_c;
  const uint8_t* dnsh_c;
  const __half* gu_s;     // scales (and affine-4 biases) per row
  const __half* gu_b;
  const __half* gush_s;
  const __half* gush_b;
  const __half* dn_s;
  const __half* dn_b;
  const __half* dnsh_s;
  const __half* dnsh_b;
  const uint16_t* x;      // [T, H] bf16
  const float* wr;        // [E, H]
  const float* bias;      // [E] or null
  const float* sgate;     // [H] or null
  int T, H, I, E, k, flags, G, epc;
  int GC;                 // CTAs c < GC own rows 16c..16c+15 of y (GC = H / 16)
  int hb, hsb, ib, isb;   // code / scale bytes per gate_up row and per down row
  int m;                  // down tiles per C item
  int ns;                 // ring slots
  int slot_bytes, xs_off, sg_off, wr_off, hs_off, hs_bytes, ul_off, wm_off;
  unsigned long long* gbar;  // call ticket: G arrivals per call
  unsigned long long* logits;  // [kMaxT, E] (call tag << 32) | logit bits
  unsigned long long* hbuf;  // [slots, T, I / 2]: (call tag << 32) | fp16 pair of h / 16
  int32_t* topk_idx;
  float* topk_w;
  uint16_t* y;
  float* y32;
  int32_t* status;
  int skew;               // test hook: added to the awaited call tag (0)
  float* gu_dump;         // test hook: [slots * T, 2I] gate and up values, or null
};

// Barrier over n threads (a multiple of 32) of the CTA; the non-aligned form,
// so lanes of one warp may reach it apart.
__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}


// One thread's share of an item's h: words src[i] for i = first, first +
// stride, ... < n, each (call tag << 32) | fp16 pair, into dst[i] once it
// carries tag `want`; eight loads in flight at a time, the stale ones
// reloaded.  False when the wait ran out (dst then holds what arrived).
__device__ __forceinline__ bool stage_h(const unsigned long long* src, uint32_t* dst, int n,
                                        int first, int stride, uint32_t want, uint32_t iters) {
  bool ok = true;
  for (int i0 = first; i0 < n; i0 += 8 * stride) {
    unsigned long long v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * stride;
      v[u] = i < n ? ld_relaxed_u64(src + i) : ((unsigned long long)want << 32);
    }
    uint32_t stale = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if ((uint32_t)(v[u] >> 32) != want) stale |= 1u << u;
    for (uint32_t k = 0; stale; ++k) {
      if (k >= iters) {
        ok = false;
        break;
      }
      if (k > 8) __nanosleep(32);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (stale & (1u << u)) {
          v[u] = ld_relaxed_u64(src + i0 + u * stride);
          if ((uint32_t)(v[u] >> 32) == want) stale &= ~(1u << u);
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * stride;
      if (i < n) dst[i] = (uint32_t)v[u];
    }
  }
  return ok;
}

// One warp: the E tagged logits of a token into dst (shared memory), once
// every word carries tag `want`.  All loads of a pass are in flight together;
// later passes reload only the words that were stale.  False when the wait
// ran out (dst then holds whatever arrived).
template <int kPer>
__device__ __forceinline__ bool gather_tagged(const unsigned long long* src, float* dst, int E,
                                              uint32_t want, uint32_t iters) {
  const int lane = threadIdx.x & 31;
  unsigned long long v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    v[i] = lane + 32 * i < E ? ld_relaxed_u64(src + lane + 32 * i) : 0ull;
  uint32_t stale = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      if ((uint32_t)(v[i] >> 32) == want) dst[e] = __uint_as_float((uint32_t)v[i]);
      else stale |= 1u << i;
    }
  }
  for (uint32_t n = 0; __any_sync(0xffffffffu, stale != 0); ++n) {
    if (n >= iters) return false;
    if (n > 16) __nanosleep(32);
    for (uint32_t m = stale; m; m &= m - 1) {
      const int i = __ffs(m) - 1, e = lane + 32 * i;
      const unsigned long long w = ld_relaxed_u64(src + e);
      if ((uint32_t)(w >> 32) == want) {
        dst[e] = __uint_as_float((uint32_t)w);
        stale &= ~(1u << i);
      }
    }
  }
  return true;
}

// 8 bytes at byte b (a multiple of 8) of 128-byte line `line`, 128-byte swizzle.
__device__ __forceinline__ uint2 lds_sw(const unsigned char* t, int line, int b) {
  return *reinterpret_cast<const uint2*>(
      t + line * 128 + ((((b >> 4) ^ (line & 7)) << 4) | (b & 15)));
}

// Raw A fragment of the 64-chunk ch of a tile whose rows g / g + 8 are lines
// lg / lh (+ 128-byte chunk index x rows per chunk) of `codes`, with scales
// (and biases) as fp16 rows of `spitch` bytes.
template <int QT>
__device__ __forceinline__ void load_tile_a(RawA& r, const unsigned char* codes_g,
                                            const unsigned char* codes_h, int rows_per_chunk,
                                            int g, int gh, const unsigned char* sc_g,
                                            const unsigned char* sc_h, const unsigned char* bi_g,
                                            const unsigned char* bi_h, int ch, int q) {
  if (QT == QSM_Q8_0) {
    const int c = ch >> 1, b = (ch & 1) * 64 + 8 * q;
    const int lg = c * rows_per_chunk + g, lh = c * rows_per_chunk + gh;
    r.g0 = lds_sw(codes_g, lg, b);
    r.g1 = lds_sw(codes_g, lg, b + 32);
    r.h0 = lds_sw(codes_h, lh, b);
    r.h1 = lds_sw(codes_h, lh, b + 32);
    r.sg = reinterpret_cast<const uint32_t*>(sc_g)[ch];
    r.sh = reinterpret_cast<const uint32_t*>(sc_h)[ch];
  } else {
    const int c = ch >> 2, b = (ch & 3) * 32 + 8 * q;
    r.g0 = lds_sw(codes_g, c * rows_per_chunk + g, b);
    r.h0 = lds_sw(codes_h, c * rows_per_chunk + gh, b);
    const uint16_t* sg = reinterpret_cast<const uint16_t*>(sc_g);
    const uint16_t* sh = reinterpret_cast<const uint16_t*>(sc_h);
    const uint16_t* bg = reinterpret_cast<const uint16_t*>(bi_g);
    const uint16_t* bh = reinterpret_cast<const uint16_t*>(bi_h);
    r.sg = (uint32_t)sg[ch] | ((uint32_t)bg[ch] << 16);
    r.sh = (uint32_t)sh[ch] | ((uint32_t)bh[ch] << 16);
  }
}

template <int QT, int kPer, int kCW = consumer_warps<kPer>()>
__global__ void __launch_bounds__((kCW + 1) * 32, 1)
decode_layer_kernel(const __grid_constant__ Params p) {
  constexpr int kThreads = (kCW + 1) * 32;
  constexpr int kSubs = kCW * 32 / kTPE;  // experts per router pass
  extern __shared__ unsigned char dl_dyn[];
  __shared__ __align__(8) uint64_t full[kMaxS], empty[kMaxS];
  __shared__ __align__(8) uint64_t xbar, rdy;
  __shared__ float red[2][kCW][32][4];
  __shared__ float rsum[kSubs][kTPE / 32][kMaxT];
  __shared__ int sel_e[kMaxT][32];
  __shared__ float sel_w[kMaxT][32];
  __shared__ unsigned bm[kMaxE / 32];
  __shared__ float szero[kPer * 32];  // the selection's warm-up input
  __shared__ float sgv[kMaxT];
  __shared__ int s_nu;
  __shared__ uint32_t s_tag;  // this call's tag
  __shared__ volatile int s_bad;  // a wait ran out: later waits are short

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int c = blockIdx.x;
  const int n0 = 16 * c;
  const int T = p.T, H = p.H, I = p.I, E = p.E, k = p.k, G = p.G;
  const int tps = I / 8;  // B tiles per slot
  const int ns = p.ns;
  const uint32_t pad = (1024u - (smem_u32(dl_dyn) & 1023u)) & 1023u;
  unsigned char* ring = dl_dyn + pad;
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(ring + p.xs_off);  // bf16 [T][H]
  const float* sgs = reinterpret_cast<const float*>(ring + p.sg_off);       // [H]
  const float* wrs = reinterpret_cast<const float*>(ring + p.wr_off);       // [epc][H]
  int* ulist = reinterpret_cast<int*>(ring + p.ul_off);
  float* wmat = reinterpret_cast<float*>(ring + p.wm_off);  // [(slots)][T]
  constexpr int kBi = QT == QSM_Q8_0 ? 1 : 2;  // scale planes (scales, biases)

  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    mbar_init(&xbar, 1);
    mbar_init(&rdy, 1);
    s_bad = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < kMaxE / 32; i += kThreads) bm[i] = 0u;
  for (int i = tid; i < kPer * 32; i += kThreads) szero[i] = 0.f;
  __syncthreads();

  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (mbar_wait_bounded(bar, parity, s_bad ? kShortWait : kWaitIters)) return;
    s_bad = 1;
    set_status(p.status, QSM_DEV_TIMEOUT);
  };

  // ================================================================ producer
  if (warp == kCW) {
    if (lane != 0) return;
    int nu = 0, nB = 0, items = 0;
    auto expert_of_slot = [&](int s) { return s == 0 ? 0 : ulist[s - 1]; };
    // B tile tau -> ring buffer sb, barrier bar
    auto issue_b = [&](int tau, unsigned char* sb, uint64_t* bar) {
      const int s = tau / tps, i0 = 8 * (tau % tps);
      const int e = expert_of_slot(s);
      const int rg = (s == 0 ? 0 : e * 2 * I) + i0, ru = rg + I;
      const CUtensorMap* map = s == 0 ? &p.gu_sh : &p.gu;
      const __half* sc = s == 0 ? p.gush_s : p.gu_s;
      const __half* bi = s == 0 ? p.gush_b : p.gu_b;
      mbar_arrive_expect_tx(bar, 16u * p.hb + 16u * p.hsb * kBi);
      tc::tma_load_3d(sb, map, 0, rg, 0, bar);
      tc::tma_load_3d(sb + 8 * p.hb, map, 0, ru, 0, bar);
      unsigned char* ss = sb + 16 * p.hb;
      bulk_g2s(ss, sc + (size_t)rg * (p.hsb / 2), 8 * p.hsb, bar);
      bulk_g2s(ss + 8 * p.hsb, sc + (size_t)ru * (p.hsb / 2), 8 * p.hsb, bar);
      if (QT != QSM_Q8_0) {
        bulk_g2s(ss + 16 * p.hsb, bi + (size_t)rg * (p.hsb / 2), 8 * p.hsb, bar);
        bulk_g2s(ss + 24 * p.hsb, bi + (size_t)ru * (p.hsb / 2), 8 * p.hsb, bar);
      }
    };
    auto down_row = [&](int s) { return (s == 0 ? 0 : expert_of_slot(s) * H) + n0; };
    auto issue_c = [&](int it, unsigned char* sb, uint64_t* bar) {
      const int cnt = min(p.m, nu + 1 - p.m * it);
      mbar_arrive_expect_tx(bar, (uint32_t)cnt * (16u * p.ib + 16u * p.isb * kBi));
#pragma unroll 1
      for (int j = 0; j < cnt; ++j) {
        const int s = p.m * it + j, r = down_row(s);
        tc::tma_load_3d(sb + j * 16 * p.ib, s == 0 ? &p.dn_sh : &p.dn, 0, r, 0, bar);
        unsigned char* ss = sb + p.m * 16 * p.ib + j * 16 * p.isb;
        bulk_g2s(ss, (s == 0 ? p.dnsh_s : p.dn_s) + (size_t)r * (p.isb / 2), 16 * p.isb, bar);
        if (QT != QSM_Q8_0)
          bulk_g2s(ss + p.m * 16 * p.isb, (s == 0 ? p.dnsh_b : p.dn_b) + (size_t)r * (p.isb / 2),
                   16 * p.isb, bar);
      }
    };
    // the same weights into L2 only
    auto prefetch_b = [&](int tau) {
      const int s = tau / tps, i0 = 8 * (tau % tps);
      const int rg = (s == 0 ? 0 : expert_of_slot(s) * 2 * I) + i0, ru = rg + I;
      const uint8_t* cd = s == 0 ? p.gush_c : p.gu_c;
      const __half* sc = s == 0 ? p.gush_s : p.gu_s;
      const __half* bi = s == 0 ? p.gush_b : p.gu_b;
      bulk_prefetch_l2(cd + (size_t)rg * p.hb, 8 * p.hb);
      bulk_prefetch_l2(cd + (size_t)ru * p.hb, 8 * p.hb);
      bulk_prefetch_l2(sc + (size_t)rg * (p.hsb / 2), 8 * p.hsb);
      bulk_prefetch_l2(sc + (size_t)ru * (p.hsb / 2), 8 * p.hsb);
      if (QT != QSM_Q8_0) {
        bulk_prefetch_l2(bi + (size_t)rg * (p.hsb / 2), 8 * p.hsb);
        bulk_prefetch_l2(bi + (size_t)ru * (p.hsb / 2), 8 * p.hsb);
      }
    };
    auto prefetch_c = [&](int it) {
      const int cnt = min(p.m, nu + 1 - p.m * it);
#pragma unroll 1
      for (int j = 0; j < cnt; ++j) {
        const int s = p.m * it + j, r = down_row(s);
        bulk_prefetch_l2((s == 0 ? p.dnsh_c : p.dn_c) + (size_t)r * p.ib, 16 * p.ib);
        bulk_prefetch_l2((s == 0 ? p.dnsh_s : p.dn_s) + (size_t)r * (p.isb / 2), 16 * p.isb);
        if (QT != QSM_Q8_0)
          bulk_prefetch_l2((s == 0 ? p.dnsh_b : p.dn_b) + (size_t)r * (p.isb / 2),
                           16 * p.isb);
      }
    };
    auto issue_pos = [&](int pos) {
      unsigned char* sb = ring + (pos % ns) * p.slot_bytes;
      if (pos < nB) issue_b(c + pos * G, sb, &full[pos % ns]);
      else issue_c(pos - nB, sb, &full[pos % ns]);
    };
    // before the wait: static weights only (the shared expert's tiles at the
    // head of this CTA's sequence, its down rows, the shared-expert gate)
    int pre = 0;
#pragma unroll 1
    while (pre < ns && c + pre * G < tps) {
      issue_b(c + pre * G, ring + pre * p.slot_bytes, &full[pre]);
      ++pre;
    }
    if (c < p.GC) {
      bulk_prefetch_l2(p.dnsh_c + (size_t)n0 * p.ib, 16 * p.ib);
      bulk_prefetch_l2(p.dnsh_s + (size_t)n0 * (p.isb / 2), 16 * p.isb);
    }
    {  // this CTA's router rows; counted in xbar's phase without arriving
      const int ea = c * p.epc, ne = min(E, ea + p.epc) - ea;
      if (ne > 0) {
        mbar_expect_tx(&xbar, (uint32_t)ne * H * 4);
        bulk_g2s(ring + p.wr_off, p.wr + (size_t)ea * H, ne * H * 4, &xbar);
      }
    }
    if (p.sgate) {  // counted in xbar's phase without arriving
      mbar_expect_tx(&xbar, (uint32_t)H * 4);
      bulk_g2s(ring + p.sg_off, p.sgate, H * 4, &xbar);
    }
    pdl_wait();
    pdl_launch_dependents();
    tc::mbar_arrive(&xbar);  // x: the consumers load it

    wait(&rdy, 0);  // the selection: s_nu, ulist (and s_tag)
    nu = s_nu;
    const int NT = (nu + 1) * tps;
    nB = c < NT ? (NT - c + G - 1) / G : 0;
    items = c < p.GC ? (nu + 1 + p.m - 1) / p.m : 0;
    const int total = nB + items;
    int pos = pre;
#pragma unroll 1
    for (; pos < total && pos < ns; ++pos) issue_pos(pos);
    // the positions past the first fill go to L2 now, up to a window of
    // about 320 KB ahead of the ring (all of them for a few tokens)
    const int win = max(2, 327680 / p.slot_bytes);
    int fpos = pos;
    auto prefetch_to = [&](int end) {
#pragma unroll 1
      for (; fpos < total && fpos < end; ++fpos) {
        if (fpos < nB) prefetch_b(c + fpos * G);
        else prefetch_c(fpos - nB);
      }
    };
    prefetch_to(ns + win);
#pragma unroll 1
    for (; pos < total; ++pos) {
      wait(&empty[pos % ns], ((pos / ns) - 1) & 1);
      issue_pos(pos);
      prefetch_to(pos + 1 + win);
    }
    // normally every copy has been consumed; after a timeout, let the last
    // copy of each buffer land before the CTA's shared memory goes away
    if (s_bad) {
#pragma unroll 1
      for (int s = 0; s < ns && s < total; ++s) {
        const int last = s + ((total - 1 - s) / ns) * ns;
        mbar_wait_bounded(&full[s], (last / ns) & 1, kWaitIters);
      }
    }
    return;
  }

  // ================================================================ consumers
  // ---- A: logits of experts [ea, eb), kSubs experts per pass, 128 threads each
  const int sub = tid / kTPE, st = tid % kTPE;
  const int ea = c * p.epc, eb = min(E, ea + p.epc);
  const int H4 = H / 4;
  pdl_wait();
  pdl_launch_dependents();
  // the call's tag: every earlier call on this workspace has completed, so
  // before this CTA's arrival the ticket holds (calls so far) * G plus
  // arrivals of this call
  if (tid == 0) {
    const unsigned long long t = ld_relaxed_u64(p.gbar);
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], 1;" ::"l"(p.gbar) : "memory");
    s_tag = (uint32_t)(t / (unsigned long long)G) + 1u;
  }
  {  // x into shared memory through L2 (the previous launch wrote it)
    const uint4* src = reinterpret_cast<const uint4*>(p.x);
    uint4* dst = reinterpret_cast<uint4*>(ring + p.xs_off);
    for (int i = tid; i < T * H / 8; i += kCW * 32) dst[i] = __ldcg(src + i);
  }
  wait(&xbar, 0);  // router rows (and the shared-expert gate vector)
  named_bar(kBarCons, kCW * 32);  // s_tag
  const uint32_t tag = s_tag;
  for (int e0 = ea; e0 < eb; e0 += kSubs) {
    const int e = e0 + sub;
    const bool mine = e < eb;
    const float4* wrow = reinterpret_cast<const float4*>(wrs + (size_t)(mine ? e - ea : 0) * H);
    // one token at a time (a runtime loop: the kernel's code stays small);
    // per token the products and sums in the order of moe_route
#pragma unroll 1
    for (int tt = 0; tt < T; ++tt) {
      const uint2* xr = reinterpret_cast<const uint2*>(xs + (size_t)tt * H);
      float a = 0.f;
      for (int hb = 0; hb < H4; hb += kWPer * kTPE) {
        float4 wv[kWPer];
        uint2 xv[kWPer];
#pragma unroll
        for (int i = 0; i < kWPer; ++i) {
          const int h4 = hb + st + i * kTPE;
          wv[i] = (mine && h4 < H4) ? wrow[h4] : make_float4(0.f, 0.f, 0.f, 0.f);
          xv[i] = h4 < H4 ? xr[h4] : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kWPer; ++i) {
          a = fmaf(wv[i].x, bf16_lo(xv[i].x), a);
          a = fmaf(wv[i].y, bf16_hi(xv[i].x), a);
          a = fmaf(wv[i].z, bf16_lo(xv[i].y), a);
          a = fmaf(wv[i].w, bf16_hi(xv[i].y), a);
        }
      }
      const float s2 = warp_sum(a);
      if (lane == 0) rsum[sub][st / 32][tt] = s2;
    }
    named_bar(kBarCons, kCW * 32);
    // all kMaxT token rows carry this call's tag (rows i >= T the value
    // 0), so that every word of the region holds the previous call's tag
    // when a call starts: none can pass for the current one
    if (tid < kSubs * kMaxT) {
      const int s2 = tid / kMaxT, i = tid % kMaxT;
      const int e2 = e0 + s2;
      if (e2 < eb) {
        float v = 0.f;
        if (i < T) {
#pragma unroll
          for (int wq = 0; wq < kTPE / 32; ++wq) v += rsum[s2][wq][i];
        }
        st_relaxed_u64(p.logits + (size_t)i * E + e2,
                       ((unsigned long long)tag << 32) | __float_as_uint(v));
      }
    }
    named_bar(kBarCons, kCW * 32);
  }
  // the shared expert's gate sigmoid(x . shared_gate), one warp per token
  if (p.sgate) {
    for (int t = warp; t < T; t += kCW) {
      const uint16_t* xr = xs + (size_t)t * H;
      float z = 0.f;
      for (int h = lane; h < H; h += 32)
        z = fmaf(__uint_as_float((uint32_t)xr[h] << 16), sgs[h], z);
      z = warp_sum(z);
      if (lane == 0) sgv[t] = 1.0f / (1.0f + __expf(-z));
    }
  }

  // ---- B: selection (one warp per token), the set U, weights per slot
  // the logits go where the router rows were (phase A's last CTA barrier
  // ordered every read of those before)
  float* lsm = reinterpret_cast<float*>(ring + p.wr_off);  // [T][E]
  // Warps T..T+3 (one per scheduler) run the same selection code on a row
  // of zeros while the token warps wait for the logits: the code is then in
  // the instruction caches when the token warps reach it (every phase of
  // this kernel runs once per launch, so its code is otherwise fetched
  // cold).  Their results and status are dropped.
  if (warp < min(kCW, T + 4)) {
    const bool real = warp < T;
    if (real && !gather_tagged<kPer>(p.logits + (size_t)warp * E, lsm + (size_t)warp * E, E,
                                     tag + (uint32_t)p.skew, s_bad ? kShortWait : kWaitIters)) {
      s_bad = 1;
      set_status(p.status, QSM_DEV_TIMEOUT);
    }
    __syncwarp();
    int my_e;
    float my_l, my_w;
    // the common shape (all 32 kPer candidates, top 8) with its sizes known
    // to the compiler: the rounds unroll and the bounds checks fold away
    const float* lrow = real ? lsm + (size_t)warp * E : szero;
    if (E == 32 * kPer && k == 8)
      route_select_warp<kPer, true>(lrow, p.bias, 32 * kPer, 8, p.flags,
                                    real ? p.status : nullptr, my_e, my_l, my_w);
    else
      route_select_warp<kPer, true>(lrow, p.bias, E, k, p.flags, real ? p.status : nullptr,
                                    my_e, my_l, my_w);
    if (real && lane < k) {
      sel_e[warp][lane] = my_e;
      sel_w[warp][lane] = my_w;
      if (c == 0) {
        p.topk_idx[(size_t)warp * k + lane] = my_e;
        p.topk_w[(size_t)warp * k + lane] = my_w;
      }
    }
    if (T == 1 && warp == 0) {
      // one token: its k experts are distinct; the warp ranks them, writes
      // the sorted set, the slot weights and the count, and lets the
      // producer start (no bitmap, no scan, no CTA barriers)
      int rank = 0;
      for (int j = 0; j < k; ++j) {
        const int ej = __shfl_sync(0xffffffffu, my_e, j);
        rank += ej < my_e ? 1 : 0;
      }
      if (lane < k) {
        ulist[rank] = my_e;
        wmat[rank + 1] = my_w;
      }
      if (lane == 0) {
        wmat[0] = p.sgate ? sgv[0] : 1.f;
        s_nu = k;
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&rdy);  // the producer may start: s_nu, ulist
    }
  }
  named_bar(kBarCons, kCW * 32);
  if (T > 1 && tid < T * k) {
    const int e = sel_e[tid / k][tid % k];
    atomicOr(&bm[e >> 5], 1u << (e & 31));
  }
  if (T > 1) named_bar(kBarCons, kCW * 32);
  if (T > 1 && warp == 0) {  // sorted distinct ids: prefix popcounts of the bitmap
    const unsigned word = lane < (E + 31) / 32 ? bm[lane] : 0u;
    const int cnt = __popc(word);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int pos = incl - cnt;
    for (unsigned w = word; w; w &= w - 1) ulist[pos++] = 32 * lane + (__ffs(w) - 1);
    if (lane == 31) s_nu = incl;
  }
  if (T > 1) {
    named_bar(kBarCons, kCW * 32);
    if (tid == 0) tc::mbar_arrive(&rdy);  // the producer may start: s_nu, ulist
  }
  const int nu = s_nu;
  for (int i = tid; T > 1 && i < (nu + 1) * T; i += kCW * 32) {
    const int s = i / T, t = i - s * T;
    float w = 0.f;
    if (s == 0) {
      w = p.sgate ? sgv[t] : 1.f;
    } else {
      const int e = ulist[s - 1];
      for (int j = 0; j < k; ++j)
        if (sel_e[t][j] == e) w = sel_w[t][j];
    }
    wmat[i] = w;
  }
  if (T > 1) named_bar(kBarCons, kCW * 32);

  const int NT = (nu + 1) * tps;
  const int nB = c < NT ? (NT - c + G - 1) / G : 0;

  const int items = c < p.GC ? (nu + 1 + p.m - 1) / p.m : 0;  // C items (rows of y)
  const int nch = H / 64, ich = I / 64;
  bool range_bad = false;
  float yp[4] = {0.f, 0.f, 0.f, 0.f};
  // ---- B: gate_up + SwiGLU tiles.  The warps form groups of kGW; group gi
  // owns the gate_up ring positions p with p % ngr == gi, so ngr of them
  // are in flight at once.  A tile's kGW warps take nch / kGW chunks each
  // and reduce behind the group's own named barrier.  Every warp still waits
  // for every position in order (gate_up tiles, then the down items) and
  // arrives on its empty barrier, the others right away: a ring slot's next
  // phase then waits for all warps, and no warp waits on a phase two ahead
  // of the barrier's (a parity wait would take that one as done).
  constexpr int ngr = kCW / kGW;
  const int gi = warp / kGW, wg = warp % kGW;
  for (int j = 0; j < nB; ++j) {
    const int sl = j % ns;
    wait(&full[sl], (j / ns) & 1);
    if (j % ngr != gi) {
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[sl]);
      continue;
    }
    const unsigned char* sb = ring + sl * p.slot_bytes;
    const unsigned char* ss = sb + 16 * p.hb;  // gate scales, up scales (, biases)
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto chunk = [&](int ch) {
      RawA r;
      load_tile_a<QT>(r, sb, sb + 8 * p.hb, 8, g, g, ss + g * p.hsb,
                      ss + 8 * p.hsb + g * p.hsb, ss + 16 * p.hsb + g * p.hsb,
                      ss + 24 * p.hsb + g * p.hsb, ch, q);
      uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
      if (g < T) {
        const uint16_t* xr = xs + (size_t)g * H + 64 * ch;
        X0 = bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(xr + b_off0<QT>(q)));
        X1 = bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(xr + b_off1<QT>(q)));
      }
      chunk_mma<QT>(acc, r, X0, X1);
    };
    if (nch == 4 * kGW) {  // H = 2048: four chunks per warp, unrolled
#pragma unroll
      for (int u = 0; u < 4; ++u) chunk(wg + u * kGW);
    } else {
      for (int ch = wg; ch < nch; ch += kGW) chunk(ch);
    }
    consumed(acc);
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&empty[sl]);
    // the group's partials: buffer by the group's tile parity, so that the
    // group's leader still reading the previous one is not overwritten
    float (*gred)[32][4] = red[(j / ngr) & 1] + gi * kGW;
#pragma unroll
    for (int i = 0; i < 4; ++i) gred[wg][lane][i] = acc[i];
    named_bar(kBarGrp + gi, kGW * 32);
    if (wg == 0) {
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kGW; ++w) s += gred[w][lane][i];
        a[i] = s;
      }
      const int tau = c + j * G, s = tau / tps, i0 = 8 * (tau % tps);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int t = 2 * q + cc;
        const float h = silu(a[cc]) * a[2 + cc] * kHScale;
        const uint32_t hv = __half_as_ushort(__float2half_rn(h));
        // intermediates i0 + g (g even) and i0 + g + 1 (lane + 4) share a word
        const uint32_t hn = __shfl_down_sync(0xffffffffu, hv, 4);
        if (t < T) {
          if (!(fabsf(h) <= 65504.f)) range_bad = true;
          if ((g & 1) == 0)
            st_relaxed_u64(p.hbuf + (((size_t)s * T + t) * I + i0 + g) / 2,
                           ((unsigned long long)tag << 32) | (hn << 16) | hv);
          if (p.gu_dump) {  // test hook: the fused projection's values per h row
            p.gu_dump[((size_t)s * T + t) * 2 * I + i0 + g] = a[cc];
            p.gu_dump[((size_t)s * T + t) * 2 * I + I + i0 + g] = a[2 + cc];
          }
        }
      }
      __syncwarp();  // converged before the next MMAs
    }
  }
  // ---- C: down rows n0..n0+15 of every slot, weighted per token.  The
  // warps form smaller groups of kGWC here, so that several items (a few
  // slots each) are worked on at once, each as soon as its slots' h is
  // there; a group's own items, their (slot, chunk) pairs cut evenly over
  // its warps
  constexpr int ngc = kCW / kGWC;
  static_assert(ngc <= kMaxGC && kBarGrp + ngr + ngc <= 16, "down groups");
  const int gc = warp / kGWC, wc = warp % kGWC;
  for (int it = 0; it < items; ++it) {
    const int pos = nB + it, sl = pos % ns;
    wait(&full[sl], (pos / ns) & 1);
    const unsigned char* sb = ring + sl * p.slot_bytes;
    if (it % ngc != gc) {
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[sl]);
      continue;
    }
    const int cnt = min(p.m, nu + 1 - p.m * it);
    // the item's h (its slots' words are contiguous) into the group's
    // buffer as fp16, by all of the group's warps, once this call wrote it:
    // the group's barrier first, so no warp still reads the previous item's
    uint32_t* hsw = reinterpret_cast<uint32_t*>(ring + p.hs_off + gc * p.hs_bytes);
    named_bar(kBarGrp + ngr + gc, kGWC * 32);
    if (!stage_h(p.hbuf + (size_t)p.m * it * T * (I / 2), hsw, cnt * T * (I / 2), wc * 32 + lane,
                 kGWC * 32, tag, s_bad ? kShortWait : kWaitIters)) {
      s_bad = 1;
      set_status(p.status, QSM_DEV_TIMEOUT);
    }
    named_bar(kBarGrp + ngr + gc, kGWC * 32);
    const __half* hb = reinterpret_cast<const __half*>(hsw);
    // the (slot, chunk) pairs of the item, flattened and cut over the group
    const int tot = cnt * ich, per = (tot + kGWC - 1) / kGWC;
    const int lo = min(tot, wc * per), hi = min(tot, lo + per);
    for (int j = lo / ich; j * ich < hi; ++j) {
      const int s = p.m * it + j;
      const int c0 = max(lo, j * ich) - j * ich, c1 = min(hi, (j + 1) * ich) - j * ich;
      const unsigned char* cd = sb + j * 16 * p.ib;
      const unsigned char* ss = sb + p.m * 16 * p.ib + j * 16 * p.isb;
      const unsigned char* bs = ss + p.m * 16 * p.isb;
      const __half* hr = hb + ((size_t)j * T + min(g, T - 1)) * I;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      auto dchunk = [&](int ch) {
        RawA r;
        load_tile_a<QT>(r, cd, cd, 16, g, g + 8, ss + g * p.isb, ss + (g + 8) * p.isb,
                        bs + g * p.isb, bs + (g + 8) * p.isb, ch, q);
        uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
        if (g < T) {
          X0 = *reinterpret_cast<const uint4*>(hr + 64 * ch + b_off0<QT>(q));
          X1 = *reinterpret_cast<const uint4*>(hr + 64 * ch + b_off1<QT>(q));
        }
        chunk_mma<QT>(acc, r, X0, X1);
      };
      if (c1 - c0 == 4) {  // the common share: four chunks of one slot, unrolled
#pragma unroll
        for (int u = 0; u < 4; ++u) dchunk(c0 + u);
      } else {
#pragma unroll 1
        for (int ch = c0; ch < c1; ++ch) dchunk(ch);
      }
      consumed(acc);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int t = 2 * q + cc;
        const float w = t < T ? wmat[s * T + t] : 0.f;
        if (w != 0.f) {
          yp[cc] = fmaf(w * kHScaleInv, acc[cc], yp[cc]);
          yp[2 + cc] = fmaf(w * kHScaleInv, acc[2 + cc], yp[2 + cc]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&empty[sl]);
    __syncwarp();
  }
  if (range_bad) set_status(p.status, QSM_DEV_FP16_RANGE);
  // per-warp partials, summed in warp order (after every group's leader has
  // read its last gate_up partials)
  named_bar(kBarCons, kCW * 32);
#pragma unroll
  for (int i = 0; i < 4; ++i) red[0][warp][lane][i] = yp[i];
  named_bar(kBarCons, kCW * 32);
  if (c < p.GC && tid < 16 * T) {
    const int r = tid & 15, t = tid >> 4;
    const int ln = 4 * (r & 7) + (t >> 1), ii = (r >= 8 ? 2 : 0) + (t & 1);
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) s += red[0][w][ln][ii];
    const size_t o = (size_t)t * H + n0 + r;
    p.y[o] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
    if (p.y32) p.y32[o] = s;
  }
}

// ------------------------------------------------------------------ host

inline size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int sm_count_dl() {
  static int n[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev];
}

// dynamic shared memory per CTA: the per-block maximum minus the static part
constexpr size_t kSmemBudget = 227 * 1024 - 20 * 1024;

struct Geo {
  int hb, hsb, ib, isb, m, ns, slot_bytes, xs_off, sg_off, wr_off, hs_off, hs_bytes, ul_off,
      wm_off;
  size_t smem;
  int numax;
};

// One CTA per SM, or as many as the most gate_up tiles a call of up to 8
// tokens can have, but at least one per 16 rows of y.  Independent of T, so
// that calls of any T share a workspace (the call tag divides by it).
int grid_of(const qsm_moe_layer* L, int nsm) {
  const int numax = kMaxT * L->k < L->E ? kMaxT * L->k : L->E;
  const int nt = (numax + 1) * (L->I / 8), gc = L->H / 16;
  return std::max(gc, std::min(nsm, nt));
}

// The logit exchange and the h hand-off need every CTA of the grid
// resident at once: G CTAs on nsm SMs holding blocks_per_sm CTAs each.
bool grid_fits(int G, int nsm, int blocks_per_sm) {
  return G >= 1 && nsm >= 1 && blocks_per_sm >= 1 && (long long)G <= (long long)nsm * blocks_per_sm;
}

bool geo_of(const qsm_moe_layer* L, int T, int nsm, Geo* o) {
  const int qt = L->gate_up.qtype;
  const int H = L->H, I = L->I, E = L->E, k = L->k;
  if (T < 1 || T > kMaxT || E < 1 || E > kMaxE || k < 1 || k > 32 || k > E) return false;
  if (qt != QSM_Q8_0 && qt != QSM_AFFINE4_G64) return false;
  if (L->down.qtype != qt || L->shared_gate_up.qtype != qt || L->shared_down.qtype != qt)
    return false;
  if (H % 256 || I % (qt == QSM_Q8_0 ? 128 : 256)) return false;
  if (H / 16 > nsm || H > 16384 || I > 16384) return false;
  const int bi = qt == QSM_Q8_0 ? 1 : 2;
  Geo g;
  g.hb = qt == QSM_Q8_0 ? H : H / 2;
  g.hsb = (qt == QSM_Q8_0 ? H / 32 : H / 64) * 2;
  g.ib = qt == QSM_Q8_0 ? I : I / 2;
  g.isb = (qt == QSM_Q8_0 ? I / 32 : I / 64) * 2;
  const size_t btile = 16 * (size_t)g.hb + 16 * (size_t)g.hsb * bi;
  const size_t dtile = 16 * (size_t)g.ib + 16 * (size_t)g.isb * bi;
  g.slot_bytes = (int)up(btile > dtile ? btile : dtile, 1024);
  g.numax = T * k < E ? T * k : E;
  const int G = grid_of(L, nsm), epc = (E + G - 1) / G;
  // the deepest ring (then the largest C items) that fits
  const int mmax = std::min(kMaxM, (int)(g.slot_bytes / dtile));
  bool fit = false;
  for (g.ns = kMaxS; g.ns >= 2 && !fit; --g.ns) {
    for (g.m = mmax; g.m >= 1; --g.m) {
      size_t off = (size_t)g.ns * g.slot_bytes;
      g.xs_off = (int)off;
      off = up(off + (size_t)T * H * 2, 128);
      g.sg_off = (int)off;
      off = up(off + (L->shared_gate ? (size_t)H * 4 : 0), 128);
      // the router rows (phase A), then the logits and the two groups' h
      // staging buffers share a region
      g.wr_off = g.hs_off = (int)off;
      g.hs_bytes = (int)((size_t)g.m * T * I * 2);
      const size_t wr = (size_t)epc * H * 4, lg = (size_t)T * E * 4,
                   hsz = kMaxGC * (size_t)g.hs_bytes;
      off = up(off + std::max(wr, std::max(lg, hsz)), 128);
      g.ul_off = (int)off;
      off = up(off + (size_t)g.numax * 4, 16);
      g.wm_off = (int)off;
      off = up(off + (size_t)(g.numax + 1) * T * 4, 16);
      g.smem = 1024 + off;
      if (g.smem <= kSmemBudget) {
        fit = true;
        break;
      }
    }
  }
  if (!fit) return false;
  ++g.ns;  // undo the loop's last decrement
  *o = g;
  return true;
}

int g_barrier_skew = 0;  // qsm_debug_barrier_skew

// The call ticket and the tagged logits (sized for the largest T, so that
// their place does not depend on T and the logit words never share bytes
// with h of another call), then the tagged h words.

struct WsLayout {
  size_t logits, hbuf, total;
};

WsLayout ws_layout(const qsm_moe_layer* L, int T, const Geo& g) {
  WsLayout w;
  w.logits = 256;
  w.hbuf = w.logits + up((size_t)kMaxT * L->E * 8, 256);
  w.total = w.hbuf + up((size_t)(g.numax + 1) * T * (L->I / 2) * 8, 256);
  return w;
}

// The kernel instance for the layer's weight type and expert count.
template <int QT, int kPer>
void* kernel_ptr() {
  return reinterpret_cast<void*>(decode_layer_kernel<QT, kPer>);
}
void* kernel_of(const qsm_moe_layer* L) {
  const bool a4 = L->gate_up.qtype == QSM_AFFINE4_G64;
  if (L->E <= 256) return a4 ? kernel_ptr<QSM_AFFINE4_G64, 8>() : kernel_ptr<QSM_Q8_0, 8>();
  return a4 ? kernel_ptr<QSM_AFFINE4_G64, 32>() : kernel_ptr<QSM_Q8_0, 32>();
}
int threads_of(const qsm_moe_layer* L) {
  return ((L->E <= 256 ? consumer_warps<8>() : consumer_warps<32>()) + 1) * 32;
}

// CTAs of the kernel that fit one SM of the current device at `smem` bytes
// of dynamic shared memory (the occupancy calculator; cached per device,
// kernel and size).  0 when the query fails.
int blocks_per_sm(void* kernel, int threads, size_t smem) {
  struct Key {
    int dev;
    void* k;
    size_t smem;
  };
  static std::mutex mu;
  static std::vector<std::pair<Key, int>> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& c : cache)
    if (c.first.dev == dev && c.first.k == kernel && c.first.smem == smem) return c.second;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBudget) != cudaSuccess)
    return 0;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem) != cudaSuccess)
    nb = 0;
  cache.push_back({Key{dev, kernel, smem}, nb});
  return nb;
}

// The layer and T are supported on the current device, and the whole grid
// can be resident at once.
bool supported_here(const qsm_moe_layer* L, int T, Geo* g) {
  const int nsm = sm_count_dl();
  if (!geo_of(L, T, nsm, g)) return false;
  return grid_fits(grid_of(L, nsm), nsm, blocks_per_sm(kernel_of(L), threads_of(L), g->smem));
}

template <int QT, int kPer>
cudaError_t launch(const Params& prm, size_t smem, cudaStream_t stream) {
  return launch_pdl(decode_layer_kernel<QT, kPer>, dim3(prm.G),
                    dim3((consumer_warps<kPer>() + 1) * 32), smem, stream,
                    prm);
}

}  // namespace dlayer
}  // namespace qsm

extern "C" qsm_status qsm_debug_barrier_skew(int32_t skew) {
  if (skew < 0 || skew > 1024) return QSM_ERR_INVALID_ARGUMENT;
  qsm::dlayer::g_barrier_skew = skew;
  return QSM_OK;
}

extern "C" size_t moe_decode_layer_workspace_bytes(const qsm_moe_layer* L, int32_t T) {
  qsm::dlayer::Geo g;
  if (!L || !qsm::dlayer::supported_here(L, T, &g)) return 0;
  return qsm::dlayer::ws_layout(L, T, g).total;
}

extern "C" int32_t qsm_decode_layer_fits(const qsm_moe_layer* L, int32_t T, int32_t sm_count,
                                         int32_t blocks_per_sm) {
  qsm::dlayer::Geo g;
  if (!L || !qsm::dlayer::geo_of(L, T, sm_count, &g)) return 0;
  return qsm::dlayer::grid_fits(qsm::dlayer::grid_of(L, sm_count), sm_count, blocks_per_sm)
             ? 1
             : 0;
}

extern "C" qsm_status moe_decode_layer(const qsm_moe_layer* L, const uint16_t* x, int32_t T,
                                       const float* w_router, const float* logit_bias,
                                       int32_t flags, int32_t* topk_idx, float* topk_w,
                                       uint16_t* y, float* y_f32, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status,
                                       cudaStream_t stream) {
  using namespace qsm;
  using namespace qsm::dlayer;
  if (!L || T < 0 || (flags & ~(QSM_ROUTE_RENORMALIZE | QSM_ROUTE_BIAS_SELECT_ONLY)))
    return QSM_ERR_INVALID_ARGUMENT;
  if (T == 0) return QSM_OK;
  if (!x || !w_router || !topk_idx || !topk_w || !y || !workspace || !dev_status)
    return QSM_ERR_INVALID_ARGUMENT;
  Geo g;
  if (!supported_here(L, T, &g)) return QSM_ERR_UNSUPPORTED;
  const WsLayout wl = ws_layout(L, T, g);
  if (workspace_bytes < wl.total) return QSM_ERR_WORKSPACE_TOO_SMALL;
  const qsm_qweights *gu = &L->gate_up, *gs = &L->shared_gate_up, *dn = &L->down,
                     *ds = &L->shared_down;
  const bool a4 = gu->qtype == QSM_AFFINE4_G64;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace) || !aligned4(topk_idx) ||
      !aligned4(topk_w) || !aligned4(y) || (y_f32 && !aligned4(y_f32)) ||
      (logit_bias && !aligned4(logit_bias)) || (L->shared_gate && !aligned16(L->shared_gate)))
    return QSM_ERR_INVALID_ARGUMENT;
  for (const qsm_qweights* w : {gu, gs, dn, ds}) {
    if (!w->codes || !w->scales || !aligned16(w->codes) || !aligned16(w->scales) ||
        (a4 && (!w->biases || !aligned16(w->biases))))
      return QSM_ERR_INVALID_ARGUMENT;
  }
  if (gu->experts != L->E || gu->rows != 2 * L->I || gu->cols != L->H || dn->experts != L->E ||
      dn->rows != L->H || dn->cols != L->I || gs->rows != 2 * L->I || gs->cols != L->H ||
      ds->rows != L->H || ds->cols != L->I)
    return QSM_ERR_INVALID_ARGUMENT;
  Params prm;
  const int H = L->H, I = L->I, E = L->E;
  bool ok = tc::make_map_rows3d(&prm.gu, gu->codes, (uint64_t)E * 2 * I, g.hb, 8, g.hb / 128) &&
            tc::make_map_rows3d(&prm.gu_sh, gs->codes, (uint64_t)2 * I, g.hb, 8, g.hb / 128) &&
            tc::make_map_rows3d(&prm.dn, dn->codes, (uint64_t)E * H, g.ib, 16, g.ib / 128) &&
            tc::make_map_rows3d(&prm.dn_sh, ds->codes, (uint64_t)H, g.ib, 16, g.ib / 128);
  if (!ok) return QSM_ERR_UNSUPPORTED;
  prm.gu_c = static_cast<const uint8_t*>(gu->codes);
  prm.gush_c = static_cast<const uint8_t*>(gs->codes);
  prm.dn_c = static_cast<const uint8_t*>(dn->codes);
  prm.dnsh_c = static_cast<const uint8_t*>(ds->codes);
  prm.gu_s = reinterpret_cast<const __half*>(gu->scales);
  prm.gu_b = reinterpret_cast<const __half*>(gu->biases);
  prm.gush_s = reinterpret_cast<const __half*>(gs->scales);
  prm.gush_b = reinterpret_cast<const __half*>(gs->biases);
  prm.dn_s = reinterpret_cast<const __half*>(dn->scales);
  prm.dn_b = reinterpret_cast<const __half*>(dn->biases);
  prm.dnsh_s = reinterpret_cast<const __half*>(ds->scales);
  prm.dnsh_b = reinterpret_cast<const __half*>(ds->biases);
  prm.x = x;
  prm.wr = w_router;
  prm.bias = logit_bias;
  prm.sgate = L->shared_gate;
  prm.T = T;
  prm.H = H;
  prm.I = I;
  prm.E = E;
  prm.k = L->k;
  prm.flags = flags;
  prm.G = grid_of(L, sm_count_dl());
  prm.GC = H / 16;
  prm.epc = (E + prm.G - 1) / prm.G;
  prm.hb = g.hb;
  prm.hsb = g.hsb;
  prm.ib = g.ib;
  prm.isb = g.isb;
  prm.m = g.m;
  prm.ns = g.ns;
  prm.slot_bytes = g.slot_bytes;
  prm.xs_off = g.xs_off;
  prm.sg_off = g.sg_off;
  prm.wr_off = g.wr_off;
  prm.hs_off = g.hs_off;
  prm.hs_bytes = g.hs_bytes;
  prm.ul_off = g.ul_off;
  prm.wm_off = g.wm_off;
  char* ws = static_cast<char*>(workspace);
  prm.gbar = reinterpret_cast<unsigned long long*>(ws);
  prm.logits = reinterpret_cast<unsigned long long*>(ws + wl.logits);
  prm.hbuf = reinterpret_cast<unsigned long long*>(ws + wl.hbuf);
  prm.topk_idx = topk_idx;
  prm.topk_w = topk_w;
  prm.y = y;
  prm.y32 = y_f32;
  prm.status = dev_status;
  prm.skew = g_barrier_skew;
  prm.gu_dump = nullptr;
  if (g_gu_dump) {
    if (g_gu_dump_floats < (size_t)(g.numax + 1) * T * 2 * I) return QSM_ERR_INVALID_ARGUMENT;
    prm.gu_dump = g_gu_dump;
  }
  cudaError_t err;
  if (E <= 256)
    err = a4 ? launch<QSM_AFFINE4_G64, 8>(prm, g.smem, stream)
             : launch<QSM_Q8_0, 8>(prm, g.smem, stream);
  else
    err = a4 ? launch<QSM_AFFINE4_G64, 32>(prm, g.smem, stream)
             : launch<QSM_Q8_0, 32>(prm, g.smem, stream);
  return err == cudaSuccess ? QSM_OK : QSM_ERR_CUDA;
}
