// Decode path of the MoE FFN (few tokens): stream the selected experts'
// quantized bytes once, with coalesced loads, in two fused kernels
//   d1: gate_up matmul + SwiGLU                          -> h (fp16)
//   d2: down matmul x routing weight + shared expert, summed per token -> y
// following "Optimizing on-device inference for Apple Silicon", section
// "Reducing intermediate and state traffic" (the two input projections with
// their gated activation; the output projection with its routing score and
// the shared expert's result), over the fused [gate; up] weight of "oMLX
// MoE gate/up 融合优化", section "融合原理".
//
// The dot products run on the tensor pipe with mma.sync m16n8k16 (fp16 in,
// fp32 accumulate): a warp holds a 16-row weight tile and up to 8 tokens.
// Not for throughput (the path is bound by HBM) but to keep instructions per
// weight low: int8 -> fp16 costs 1.25 instructions per weight and the
// multiply-adds one MMA per 256 weights, where fp32 FMAs need ~4.
//
// d1 tile rows: gate rows i0..i0+7 are MMA rows 0..7 and up rows i0..i0+7
// MMA rows 8..15, so each thread's accumulators hold the gate and the up
// value of the same (intermediate index, token) and SwiGLU is thread-local.
//
// K mapping and the MMA building blocks: gemv_core.cuh.
//
// Precision: x (bf16) is converted to fp16, exact for |x| in [2^-17, 65504];
// h is stored as fp16 after scaling by 1/16 (so |h| up to ~1e6 fits); a
// non-finite or out-of-range value sets QSM_DEV_FP16_RANGE.
#include <utility>

#include "decode_stream.cuh"
#include "gemv_core.cuh"

namespace qsm {
namespace decode {

constexpr float kHScale = 1.0f / 16.0f;
constexpr float kHScaleInv = 16.0f;
constexpr int kTok = 8;       // tokens per MMA (N = 8) = the path's tile_rows
constexpr int kD1Split = 4;   // d1: warps splitting K of one 16-row tile
constexpr int kD2Warps = 12;  // d2: max warps per 16-row output tile

using namespace gemv;

// Work slot -> (expert, token rows).  Slots [0, shared_slots) are blocks of
// 8 tokens for the shared expert; slot shared_slots + tau is block tau of
// the block map (at most 8 rows of one expert).
struct Slot {
  int e;     // -1 = shared expert
  int row0;  // first sorted row (routed) or first token (shared)
  int cnt;   // rows in the block (0 = nothing to do)
};

__device__ __forceinline__ Slot slot_of(int s, int shared_slots, int T,
                                        const int32_t* __restrict__ offsets,
                                        const int32_t* __restrict__ tile_map,
                                        int n_tiles) {
  Slot r;
  if (s < shared_slots) {
    r.e = -1;
    r.row0 = kTok * s;
    r.cnt = min(kTok, T - r.row0);
  } else {
    const int tau = s - shared_slots;
    if (tau >= n_tiles) {
      r.e = 0; r.row0 = 0; r.cnt = 0;
    } else {
      const int2 te = __ldcg(reinterpret_cast<const int2*>(tile_map) + tau);
      r.e = te.x;
      r.row0 = te.y;
      r.cnt = min(kTok, __ldcg(offsets + r.e + 1) - r.row0);
    }
  }
  return r;
}

// A warp keeps up to kPre 64-chunks of its weight slice in registers: all of
// their loads are issued before the first MMA, so each warp pays about one
// memory round trip per kPre chunks instead of one per chunk.
constexpr int kPre = 8;
constexpr int kXPad = 32;  // fp16 padding per staged x row (bank spread)

template <int QT>
__device__ __forceinline__ void load_batch(RawA (&r)[kPre], const QW& w, int rg,
                                           int rh, int first, int stride,
                                           int nch, int q) {
#pragma unroll
  for (int c = 0; c < kPre; ++c) {
    const int ci = first + c * stride;
    if (ci < nch) load_a<QT>(r[c], w, rg, rh, 64 * ci, q);
  }
}

// ----------------------------------------------------------------- d1
//
// One CTA = one work slot (an expert and its <= 8 tokens) x 8 intermediate
// indices: weight rows gate[i0..i0+7] and up[i0..i0+7].  The 16 code rows
// arrive by TMA bulk copies (one per row, into rows padded by kRowPad bytes
// so the MMA fragment reads are free of bank conflicts), tracked by one
// mbarrier; the shared expert's CTAs start their copies before waiting on
// the routing.  While the layer's weights fit in L2 beside each other, the
// CTA also asks L2 to prefetch its share of the expert's down-projection
// rows, which the next launch streams.

constexpr int kRowPad = 32;

template <int QT>
__device__ __forceinline__ int code_row_bytes(int cols) {
  return QT == QSM_Q8_0 ? cols : cols / 2;
}

// RawA of rows g and g + 8 of a staged 16-row tile, for the 64-chunk at k0.
template <int QT>
__device__ __forceinline__ void load_a_smem(RawA& r, const unsigned char* wsm,
                                            int pitch, const uint32_t* ssm,
                                            int spitch, int g, int k0, int q) {
  const unsigned char* rg = wsm + g * pitch;
  const unsigned char* rh = wsm + (g + 8) * pitch;
  if (QT == QSM_Q8_0) {
    r.g0 = *reinterpret_cast<const uint2*>(rg + k0 + 8 * q);
    r.g1 = *reinterpret_cast<const uint2*>(rg + k0 + 32 + 8 * q);
    r.h0 = *reinterpret_cast<const uint2*>(rh + k0 + 8 * q);
    r.h1 = *reinterpret_cast<const uint2*>(rh + k0 + 32 + 8 * q);
  } else {
    r.g0 = *reinterpret_cast<const uint2*>(rg + k0 / 2 + 8 * q);
    r.h0 = *reinterpret_cast<const uint2*>(rh + k0 / 2 + 8 * q);
  }
  r.sg = ssm[g * spitch + k0 / 64];
  r.sh = ssm[(g + 8) * spitch + k0 / 64];
}

template <int QT>
__global__ void __launch_bounds__(kD1Split * 32)
d1_gate_up_swiglu(qsm_qweights gu_w, qsm_qweights sgu_w, qsm_qweights dn_w,
                  qsm_qweights sdn_w, const uint16_t* __restrict__ x, int T,
                  int H, int I, int k, const int32_t* __restrict__ perm,
                  const int32_t* __restrict__ offsets,
                  const int32_t* __restrict__ tile_map, int shared_slots,
                  int xrows, __half* __restrict__ hbuf,
                  const float* __restrict__ sgate, float* __restrict__ gbuf,
                  float* __restrict__ gu_dump, int prefetch, int32_t* dev_status) {
  extern __shared__ __align__(128) unsigned char d1_smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ float red[kD1Split][32][4];
  __shared__ int s_tok[kTok];
  const int lane = threadIdx.x & 31, kw = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int i0 = kTok * blockIdx.x;  // 8 intermediate indices per CTA
  const int crow = code_row_bytes<QT>(H);
  const int pitch = crow + kRowPad;
  const int spitch = H / 64 + 1;     // u32 per staged scale row (+1: banks)
  unsigned char* wsm = d1_smem;                                   // [16][pitch]
  uint32_t* ssm = reinterpret_cast<uint32_t*>(d1_smem + 16 * pitch);  // [16][spitch]
  __half* xs = reinterpret_cast<__half*>(
      d1_smem + ((16 * pitch + 16 * spitch * 4 + 15) & ~15));     // [xrows][H+kXPad]
  const bool shared_slot = (int)blockIdx.y < shared_slots;

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue_copies = [&](const QW& w) {
    if (kw == 0) {
      if (lane == 0) mbar_arrive_expect_tx(&bar, 16u * crow);
      __syncwarp();
      if (lane < 16) {
        const int row = lane < 8 ? i0 + lane : I + i0 + (lane - 8);
        bulk_g2s(wsm + lane * pitch, w.codes + (size_t)row * crow, crow, &bar);
      }
    }
  };
  // L2 prefetch of this CTA's 1/gridDim.x share of the expert's down rows.
  auto prefetch_down = [&](const QW& d) {
    if (prefetch && kw == 1 && lane == 0) {
      const int drow = code_row_bytes<QT>(I);
      const int rows = H / gridDim.x;  // H is a multiple of 16, grid = I/8
      if (rows > 0 && (rows * drow) % 16 == 0) {
        const int r0 = blockIdx.x * rows;
        bulk_prefetch_l2(d.codes + (size_t)r0 * drow, rows * drow);
        const int sb = (QT == QSM_Q8_0 ? I / 32 : I / 64) * 2;
        if ((rows * sb) % 16 == 0) {
          bulk_prefetch_l2(d.scales + (size_t)r0 * (sb / 2), rows * sb);
          if (QT != QSM_Q8_0) bulk_prefetch_l2(d.biases + (size_t)r0 * (sb / 2), rows * sb);
        }
      }
    }
  };

  int e = -1, row0, cnt;
  QW w;
  if (shared_slot) {  // static weights: start the copies before the wait
    w = expert_of<QT>(sgu_w, 0);
    issue_copies(w);
    prefetch_down(expert_of<QT>(sdn_w, 0));
  }
  // The routing comes from the grouping launch: wait for it, then let the
  // down-projection launch start (it may read the routing right away).
  pdl_wait();
  pdl_launch_dependents();
  if (shared_slot) {
    row0 = kTok * blockIdx.y;
    cnt = min(kTok, T - row0);
  } else {
    const int tau = blockIdx.y - shared_slots;
    const int2 te = __ldcg(reinterpret_cast<const int2*>(tile_map) + tau);
    if (te.x < 0) return;  // no block map entry for this slot
    e = te.x;
    row0 = te.y;
    w = expert_of<QT>(gu_w, e);
    issue_copies(w);
    prefetch_down(expert_of<QT>(dn_w, e));
    cnt = min(kTok, __ldcg(offsets + e + 1) - row0);
  }

  // block scales (and biases) of the 16 rows -> shared, as u32 per 64-chunk
  for (int i = threadIdx.x; i < 16 * (H / 64); i += blockDim.x) {
    const int rr = i / (H / 64), j = i - rr * (H / 64);
    const int row = rr < 8 ? i0 + rr : I + i0 + (rr - 8);
    uint32_t v;
    if (QT == QSM_Q8_0) {
      v = __ldg(reinterpret_cast<const uint32_t*>(w.scales + (size_t)row * (H / 32)) + j);
    } else {
      const size_t gi = (size_t)row * (H / 64) + j;
      v = (uint32_t)__half_as_ushort(w.scales[gi]) |
          ((uint32_t)__half_as_ushort(w.biases[gi]) << 16);
    }
    ssm[rr * spitch + j] = v;
  }
  // this slot's token rows of x, as fp16
  if (threadIdx.x < kTok)
    s_tok[threadIdx.x] = threadIdx.x < cnt
        ? (shared_slot ? row0 + threadIdx.x : __ldcg(perm + row0 + threadIdx.x) / k)
        : 0;
  __syncthreads();
  const int xpitch = H + kXPad;
  const int v8 = H / 8;
  for (int i = threadIdx.x; i < cnt * v8; i += blockDim.x) {
    const int c = i / v8, j = i - c * v8;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)s_tok[c] * H) + j);
    *reinterpret_cast<uint4*>(xs + c * xpitch + 8 * j) = bf16x8_to_f16x8(v);
  }
  __syncthreads();
  // gated shared expert: sigmoid(x . shared_gate) of this slot's tokens,
  // computed by the slot's first CTA while its weight copies land
  if (sgate != nullptr && shared_slot && blockIdx.x == 0) {
    for (int c = kw; c < cnt; c += kD1Split) {
      const __half* xr = xs + c * xpitch;
      float z = 0.f;
      for (int h8 = lane; h8 < H / 8; h8 += 32) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xr + 8 * h8);
        const float4 w0 = __ldg(reinterpret_cast<const float4*>(sgate) + 2 * h8);
        const float4 w1 = __ldg(reinterpret_cast<const float4*>(sgate) + 2 * h8 + 1);
        const __half2* x2 = reinterpret_cast<const __half2*>(&xv);
        const float2 a = __half22float2(x2[0]), b = __half22float2(x2[1]);
        const float2 cc = __half22float2(x2[2]), d = __half22float2(x2[3]);
        z = fmaf(a.x, w0.x, z);
        z = fmaf(a.y, w0.y, z);
        z = fmaf(b.x, w0.z, z);
        z = fmaf(b.y, w0.w, z);
        z = fmaf(cc.x, w1.x, z);
        z = fmaf(cc.y, w1.y, z);
        z = fmaf(d.x, w1.z, z);
        z = fmaf(d.y, w1.w, z);
      }
      z = warp_sum(z);
      if (lane == 0) gbuf[row0 + c] = 1.0f / (1.0f + __expf(-z));
    }
  }
  // bounded wait for the weight rows; the CTA agrees on the outcome
  if (!__syncthreads_and(mbar_wait_bounded(&bar, 0, kWaitIters))) {
    if (threadIdx.x == 0) set_status(dev_status, QSM_DEV_TIMEOUT);
    mbar_wait_bounded(&bar, 0, kWaitIters);  // let our copies land first
    return;
  }

  const __half* xg = xs + min(g, xrows - 1) * xpitch;
  const bool has_tok = g < cnt;
  const int nch = H / 64;  // chunks dealt round-robin to the kD1Split warps
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int ci = kw; ci < nch; ci += kD1Split) {
    RawA r;
    load_a_smem<QT>(r, wsm, pitch, ssm, spitch, g, 64 * ci, q);
    uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
    if (has_tok) {
      X0 = *reinterpret_cast<const uint4*>(xg + 64 * ci + b_off0<QT>(q));
      X1 = *reinterpret_cast<const uint4*>(xg + 64 * ci + b_off1<QT>(q));
    }
    chunk_mma<QT>(acc, r, X0, X1);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) red[kw][lane][i] = acc[i];
  __syncthreads();
  if (kw != 0) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kD1Split; ++j) s += red[j][lane][i];
    acc[i] = s;
  }
  bool bad = false;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int c = 2 * q + cc;
    if (c < cnt) {
      const float gate = acc[cc], up = acc[2 + cc];
      const float h = silu(gate) * up * kHScale;
      if (!(fabsf(h) <= 65504.f)) bad = true;
      const int hrow = shared_slot ? T * k + row0 + c : row0 + c;
      hbuf[(size_t)hrow * I + i0 + g] = __float2half_rn(h);
      if (gu_dump) {  // test hook: the fused projection's values per h row
        gu_dump[(size_t)hrow * 2 * I + i0 + g] = gate;
        gu_dump[(size_t)hrow * 2 * I + I + i0 + g] = up;
      }
    }
  }
  if (bad) set_status(dev_status, QSM_DEV_FP16_RANGE);
}

// ----------------------------------------------------------------- d2
//
// One CTA = 16 output rows n0..n0+15 of y for every token.  Work items are
// the shared expert's blocks of 8 tokens and the block map's blocks; warp w
// takes items w, w + warps, ...  Each warp has two shared-memory slots for
// an item's 16 down rows (padded) and their block constants, filled by bulk
// copies on the slot's mbarrier, so the next item's rows are in flight while
// one is multiplied; the copies of a warp's first two items are issued
// before waiting on the gate_up launch (the routing was complete before that
// launch let this one start).  An item's h rows come from global memory (L2)
// straight into registers, requested as soon as the previous item is done,
// and each warp keeps its next item's slot, tokens and weights ahead of time
// so those dependent lookups overlap a copy's wait.  Each warp sums its items
// into its own [T][16] fp32 slab; the slabs are added in warp order.

constexpr int kD2HCh = 8;  // 64-wide chunks of an item's h held in registers

struct D2Geo {  // per-slot layout (bytes)
  int crow, pitch, wbytes, sbytes, slot;
};

template <int QT>
__host__ __device__ __forceinline__ D2Geo d2_geo(int I) {
  D2Geo g;
  g.crow = QT == QSM_Q8_0 ? I : I / 2;          // code bytes per row
  g.pitch = g.crow + kRowPad;
  g.wbytes = 16 * g.pitch;
  g.sbytes = QT == QSM_Q8_0 ? 16 * (I / 32) * 2 : 2 * 16 * (I / 64) * 2;
  g.slot = (g.wbytes + g.sbytes + 127) & ~127;
  return g;
}

template <int QT>
__global__ void __launch_bounds__(kD2Warps * 32)
d2_down_combine(qsm_qweights dn_w, qsm_qweights sdn_w,
                const __half* __restrict__ hbuf, int T, int H, int I, int k,
                const int32_t* __restrict__ perm,
                const int32_t* __restrict__ offsets,
                const int32_t* __restrict__ tile_map,
                const int32_t* __restrict__ n_tiles_p,
                const float* __restrict__ topk_w, int shared_slots,
                const float* __restrict__ gbuf, uint16_t* __restrict__ y,
                float* __restrict__ y32, int32_t* dev_status) {
  extern __shared__ __align__(128) unsigned char d2_smem[];
  __shared__ __align__(8) uint64_t bars[kD2Warps][2];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int n0 = 16 * blockIdx.x;
  const int nch = I / 64;
  const D2Geo geo = d2_geo<QT>(I);
  unsigned char* wslot = d2_smem + (size_t)wid * 2 * geo.slot;  // [2][slot]
  float* slab = reinterpret_cast<float*>(d2_smem + (size_t)nw * 2 * geo.slot);  // [nw][T][16]
  if (lane == 0) {
    mbar_init(&bars[wid][0], 1);
    mbar_init(&bars[wid][1], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Routing data and weights need no wait (see above).
  const int n_tiles = __ldcg(n_tiles_p);
  const int items = shared_slots + n_tiles;
  for (int i = threadIdx.x; i < nw * T * 16; i += blockDim.x) slab[i] = 0.f;

  auto issue_weights = [&](const Slot& sl, int b) {
    const QW w = sl.e < 0 ? expert_of<QT>(sdn_w, 0) : expert_of<QT>(dn_w, sl.e);
    unsigned char* slot = wslot + b * geo.slot;
    if (lane == 0) mbar_arrive_expect_tx(&bars[wid][b], 16u * geo.crow + geo.sbytes);
    __syncwarp();
    if (lane < 16)
      bulk_g2s(slot + lane * geo.pitch, w.codes + (size_t)(n0 + lane) * geo.crow, geo.crow,
               &bars[wid][b]);
    if (lane == 16) {
      if (QT == QSM_Q8_0) {
        bulk_g2s(slot + geo.wbytes, w.scales + (size_t)n0 * (I / 32), geo.sbytes, &bars[wid][b]);
      } else {
        bulk_g2s(slot + geo.wbytes, w.scales + (size_t)n0 * (I / 64), geo.sbytes / 2,
                 &bars[wid][b]);
        bulk_g2s(slot + geo.wbytes + geo.sbytes / 2, w.biases + (size_t)n0 * (I / 64),
                 geo.sbytes / 2, &bars[wid][b]);
      }
    }
  };
  auto h_row_of = [&](const Slot& sl, int c) {
    return sl.e < 0 ? T * k + sl.row0 + c : sl.row0 + c;
  };
  // this thread's B operands of the item's first kD2HCh chunks (token g)
  uint4 hx[2 * kD2HCh];
  auto load_h = [&](const Slot& sl) {
    const bool has = g < sl.cnt;
    const __half* hr = hbuf + (size_t)h_row_of(sl, has ? g : 0) * I;
#pragma unroll
    for (int ci = 0; ci < kD2HCh; ++ci) {
      const bool in = has && ci < nch;
      hx[2 * ci] = in ? __ldcg(reinterpret_cast<const uint4*>(hr + 64 * ci + b_off0<QT>(q)))
                      : make_uint4(0u, 0u, 0u, 0u);
      hx[2 * ci + 1] = in ? __ldcg(reinterpret_cast<const uint4*>(hr + 64 * ci + b_off1<QT>(q)))
                          : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // the item's columns 2q, 2q+1: token and routing weight (the shared
  // expert's gate is read after the wait: the gate_up launch writes it)
  int tok[2] = {-1, -1};
  float wt[2] = {0.f, 0.f};
  auto columns = [&](const Slot& sl, bool gates_ready) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * q + cc;
      tok[cc] = -1;
      wt[cc] = 0.f;
      if (c < sl.cnt) {
        if (sl.e < 0) {  // shared expert: weight 1, or its gate
          tok[cc] = sl.row0 + c;
          wt[cc] = (gbuf && gates_ready) ? __ldcg(gbuf + tok[cc]) : 1.f;
        } else {
          const int a = __ldcg(perm + sl.row0 + c);
          tok[cc] = a / k;
          wt[cc] = __ldcg(topk_w + a);
        }
      }
    }
  };

  Slot cur, nxt;
  if (wid < items) {
    cur = slot_of(wid, shared_slots, T, offsets, tile_map, n_tiles);
    issue_weights(cur, 0);
    columns(cur, false);
  }
  if (wid + nw < items) {
    nxt = slot_of(wid + nw, shared_slots, T, offsets, tile_map, n_tiles);
    issue_weights(nxt, 1);
  }
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();  // slab zeroed
  if (wid < items) {
    if (cur.e < 0 && gbuf) columns(cur, true);
    load_h(cur);
  }

  float* my = slab + (size_t)wid * T * 16;
  uint32_t ph[2] = {0u, 0u};
  int b = 0;
  bool ok_all = true;
  for (int it = wid; it < items; it += nw) {
    const bool ok = mbar_wait_bounded(&bars[wid][b], ph[b], kWaitIters);
    ph[b] ^= 1u;
    if (!ok) {  // copies did not land: skip, flag, let them (and the other slot's) finish
      ok_all = false;
      mbar_wait_bounded(&bars[wid][b], ph[b] ^ 1u, kWaitIters);
      if (it + nw < items) mbar_wait_bounded(&bars[wid][b ^ 1], ph[b ^ 1], kWaitIters);
      break;
    }
    const unsigned char* slot = wslot + b * geo.slot;
    const unsigned char* sc = slot + geo.wbytes;
    const bool has_tok = g < cur.cnt;
    const __half* hg = hbuf + (size_t)h_row_of(cur, has_tok ? g : 0) * I;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto chunk = [&](int ci, const uint4& X0, const uint4& X1) {
      const int k0 = 64 * ci;
      RawA r;
      const unsigned char* rg = slot + g * geo.pitch;
      const unsigned char* rh = slot + (g + 8) * geo.pitch;
      if (QT == QSM_Q8_0) {
        r.g0 = *reinterpret_cast<const uint2*>(rg + k0 + 8 * q);
        r.g1 = *reinterpret_cast<const uint2*>(rg + k0 + 32 + 8 * q);
        r.h0 = *reinterpret_cast<const uint2*>(rh + k0 + 8 * q);
        r.h1 = *reinterpret_cast<const uint2*>(rh + k0 + 32 + 8 * q);
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(sc);
        r.sg = s32[g * (I / 64) + ci];
        r.sh = s32[(g + 8) * (I / 64) + ci];
      } else {
        r.g0 = *reinterpret_cast<const uint2*>(rg + k0 / 2 + 8 * q);
        r.h0 = *reinterpret_cast<const uint2*>(rh + k0 / 2 + 8 * q);
        const uint16_t* s16 = reinterpret_cast<const uint16_t*>(sc);
        const uint16_t* b16 = s16 + 16 * (I / 64);
        r.sg = (uint32_t)s16[g * (I / 64) + ci] | ((uint32_t)b16[g * (I / 64) + ci] << 16);
        r.sh = (uint32_t)s16[(g + 8) * (I / 64) + ci] |
               ((uint32_t)b16[(g + 8) * (I / 64) + ci] << 16);
      }
      chunk_mma<QT>(acc, r, X0, X1);
    };
#pragma unroll
    for (int ci = 0; ci < kD2HCh; ++ci)
      if (ci < nch) chunk(ci, hx[2 * ci], hx[2 * ci + 1]);
    for (int ci = kD2HCh; ci < nch; ++ci) {  // I > 512: the rest straight from L2
      uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
      if (has_tok) {
        X0 = __ldcg(reinterpret_cast<const uint4*>(hg + 64 * ci + b_off0<QT>(q)));
        X1 = __ldcg(reinterpret_cast<const uint4*>(hg + 64 * ci + b_off1<QT>(q)));
      }
      chunk(ci, X0, X1);
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      if (tok[cc] >= 0) {
        const float s = wt[cc] * kHScaleInv;
        my[tok[cc] * 16 + g] += s * acc[cc];
        my[tok[cc] * 16 + g + 8] += s * acc[2 + cc];
      }
    }
    consumed(acc);
    __syncwarp();  // this slot free for the item after next
    if (it + nw < items) {  // next: its h and lookups now, the one after into this slot
      cur = nxt;
      columns(cur, true);
      load_h(cur);
      if (it + 2 * nw < items) {
        nxt = slot_of(it + 2 * nw, shared_slots, T, offsets, tile_map, n_tiles);
        issue_weights(nxt, b);
      }
      b ^= 1;
    }
  }
  if (!__syncthreads_and(ok_all)) {
    if (threadIdx.x == 0) set_status(dev_status, QSM_DEV_TIMEOUT);
    return;
  }
  for (int i = threadIdx.x; i < T * 16; i += blockDim.x) {
    float s = 0.f;
    for (int wv = 0; wv < nw; ++wv) s += slab[(size_t)wv * T * 16 + i];
    const int t = i / 16, rr = i % 16;
    const size_t o = (size_t)t * H + n0 + rr;
    y[o] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
    if (y32) y32[o] = s;
  }
}

}  // namespace decode

// Host launcher used by moe_ffn_forward for the decode path.
template <int QT>
static qsm_status decode_launch_qt(const qsm_moe_layer* L, const uint16_t* x,
                                   int T, const float* topk_w,
                                   const qsm_grouping* g, uint16_t* y,
                                   float* y32, __half* hbuf, float* gbuf,
                                   int32_t* dev_status, cudaStream_t stream) {
  using namespace decode;
  const int H = L->H, I = L->I, k = L->k;
  const int shared_slots = (T + kTok - 1) / kTok;
  float* gu_dump = nullptr;
  if (g_gu_dump) {
    if (g_gu_dump_floats < ((size_t)T * k + T) * 2 * I) return QSM_ERR_INVALID_ARGUMENT;
    gu_dump = g_gu_dump;
  }
  // d1 asks L2 for the down rows of its experts, which d2 streams next, only
  // while the layer's touched weights fit in L2 beside each other: past that
  // the gate_up stream evicts them before d2 runs and they are read twice.
  const size_t row_bytes_gu = QT == QSM_Q8_0 ? H + H / 32 * 2 : H / 2 + H / 64 * 4;
  const size_t row_bytes_dn = QT == QSM_Q8_0 ? I + I / 32 * 2 : I / 2 + I / 64 * 4;
  const size_t experts = (size_t)(T * k < L->E ? T * k : L->E) + 1;
  const size_t touched = experts * (2 * (size_t)I * row_bytes_gu + (size_t)H * row_bytes_dn);
  const int prefetch_down = touched <= ((size_t)48 << 20) ? 1 : 0;
  const dim3 g1(I / kTok, shared_slots + g->max_tiles);
  const int xrows = T < kTok ? T : kTok;
  const int crow = QT == QSM_Q8_0 ? H : H / 2;
  const size_t smem1 = ((size_t)16 * (crow + kRowPad) + 16 * (H / 64 + 1) * 4 + 15) / 16 * 16 +
                       (size_t)xrows * (H + kXPad) * sizeof(__half);
  const int max_items = shared_slots + g->max_tiles;
  const D2Geo geo = d2_geo<QT>(I);
  int w2 = max_items < kD2Warps ? max_items : kD2Warps;
  const size_t slab_bytes_per_warp = (size_t)T * 16 * sizeof(float);
  const size_t kSmemBudget = 200 * 1024;
  while (w2 > 1 && (size_t)w2 * (2 * geo.slot + slab_bytes_per_warp) > kSmemBudget) --w2;
  const size_t smem2 = (size_t)w2 * (2 * geo.slot + slab_bytes_per_warp);
  if (T > kTok && gate_up_stream_supported(L)) {
    // several slots: one persistent pass streams every touched expert's
    // gate_up rows once per slot, each slot's x rows staged once per CTA
    const qsm_status st = gate_up_stream_launch(L, x, T, g, shared_slots, hbuf, gbuf, gu_dump,
                                                dev_status, stream);
    if (st != QSM_OK) return st;
  } else {
    QSM_CUDA_TRY(cudaFuncSetAttribute(d1_gate_up_swiglu<QT>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem1));
    QSM_CUDA_TRY(launch_pdl(d1_gate_up_swiglu<QT>, g1, dim3(kD1Split * 32), smem1,
                            stream, L->gate_up, L->shared_gate_up, L->down,
                            L->shared_down, x, T, H, I, k, (const int32_t*)g->perm,
                            (const int32_t*)g->offsets, (const int32_t*)g->tile_map,
                            shared_slots, xrows, hbuf, L->shared_gate, gbuf, gu_dump,
                            prefetch_down, dev_status));
  }
  QSM_CUDA_TRY(cudaFuncSetAttribute(d2_down_combine<QT>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem2));
  QSM_CUDA_TRY(launch_pdl(d2_down_combine<QT>, dim3(H / 16), dim3(w2 * 32), smem2,
                          stream, L->down, L->shared_down, (const __half*)hbuf, T,
                          H, I, k, (const int32_t*)g->perm,
                          (const int32_t*)g->offsets, (const int32_t*)g->tile_map,
                          (const int32_t*)g->n_tiles, topk_w, shared_slots,
                          L->shared_gate ? (const float*)gbuf : nullptr, y, y32,
                          dev_status));
  return QSM_OK;
}

qsm_status decode_ffn_launch(const qsm_moe_layer* L, const uint16_t* x, int T,
                             const float* topk_w, const qsm_grouping* g,
                             uint16_t* y, float* y32, void* ws,
                             int32_t* dev_status, cudaStream_t stream) {
  // [h (T*k + T) x I fp16][shared-expert gates T fp32]
  __half* hbuf = static_cast<__half*>(ws);
  const size_t hbytes = (((size_t)T * L->k + T) * L->I * sizeof(__half) + 255) & ~size_t(255);
  float* gbuf = reinterpret_cast<float*>(static_cast<char*>(ws) + hbytes);
  if (L->gate_up.qtype == QSM_Q8_0)
    return decode_launch_qt<QSM_Q8_0>(L, x, T, topk_w, g, y, y32, hbuf, gbuf,
                                      dev_status, stream);
  return decode_launch_qt<QSM_AFFINE4_G64>(L, x, T, topk_w, g, y, y32, hbuf, gbuf,
                                           dev_status, stream);
}

size_t decode_ffn_workspace_bytes(const qsm_moe_layer* L, int T) {
  const size_t rows = (size_t)T * L->k + T;
  return (((rows * L->I * sizeof(__half)) + 255) & ~size_t(255)) +
         (((size_t)T * sizeof(float) + 255) & ~size_t(255));
}

}  // namespace qsm
