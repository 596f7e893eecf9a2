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

#include "gemv_core.cuh"

namespace qsm {
namespace decode {

constexpr float kHScale = 1.0f / 16.0f;
constexpr float kHScaleInv = 16.0f;
constexpr int kTok = 8;       // tokens per MMA (N = 8) = the path's tile_rows
constexpr int kD1Split = 4;   // d1: warps splitting K of one 16-row tile
constexpr int kD2Warps = 16;  // d2: warps per 16-row output tile

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
      r.e = tile_map[2 * tau];
      r.row0 = tile_map[2 * tau + 1];
      r.cnt = min(kTok, offsets[r.e + 1] - r.row0);
    }
  }
  return r;
}

// ----------------------------------------------------------------- d1

template <int QT>
__global__ void __launch_bounds__(kD1Split * 32)
d1_gate_up_swiglu(qsm_qweights gu_w, qsm_qweights sgu_w,
                  const uint16_t* __restrict__ x, int T, int H, int I, int k,
                  const int32_t* __restrict__ perm,
                  const int32_t* __restrict__ offsets,
                  const int32_t* __restrict__ tile_map,
                  const int32_t* __restrict__ n_tiles_p, int shared_slots,
                  __half* __restrict__ hbuf, int32_t* dev_status) {
  __shared__ float red[kD1Split][32][4];
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31, kw = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int i0 = kTok * blockIdx.x;  // 8 intermediate indices per CTA
  const Slot sl = slot_of(blockIdx.y, shared_slots, T, offsets, tile_map,
                          *n_tiles_p);
  if (sl.cnt <= 0) return;
  const QW w = sl.e < 0 ? expert_of<QT>(sgu_w, 0) : expert_of<QT>(gu_w, sl.e);
  // token of B column g, and the h rows of this thread's output columns
  int tok_g = -1;
  if (g < sl.cnt) tok_g = sl.e < 0 ? sl.row0 + g : perm[sl.row0 + g] / k;
  const uint16_t* xrow = x + (size_t)max(tok_g, 0) * H;

  // 64-wide chunks are dealt round-robin to the kD1Split warps
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
  for (int k0 = 64 * kw; k0 < H; k0 += 64 * kD1Split) {
    RawA r;
    load_a<QT>(r, w, i0 + g, I + i0 + g, k0, q);
    uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
    if (tok_g >= 0) {
      X0 = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(xrow + k0 + b_off0<QT>(q))));
      X1 = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(xrow + k0 + b_off1<QT>(q))));
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
    if (c < sl.cnt) {
      const float gate = acc[cc], up = acc[2 + cc];
      const float h = silu(gate) * up * kHScale;
      if (!(fabsf(h) <= 65504.f)) bad = true;
      const int hrow = sl.e < 0 ? T * k + sl.row0 + c : sl.row0 + c;
      hbuf[(size_t)hrow * I + i0 + g] = __float2half_rn(h);
    }
  }
  if (bad) set_status(dev_status, QSM_DEV_FP16_RANGE);
}

// ----------------------------------------------------------------- d2

template <int QT>
__global__ void __launch_bounds__(kD2Warps * 32)
d2_down_combine(qsm_qweights dn_w, qsm_qweights sdn_w,
                const __half* __restrict__ hbuf, int T, int H, int I, int k,
                const int32_t* __restrict__ perm,
                const int32_t* __restrict__ offsets,
                const int32_t* __restrict__ tile_map,
                const int32_t* __restrict__ n_tiles_p,
                const float* __restrict__ topk_w, int shared_slots,
                uint16_t* __restrict__ y, float* __restrict__ y32) {
  extern __shared__ float slab[];  // [kD2Warps][T][16]
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int n0 = 16 * blockIdx.x;
  for (int i = threadIdx.x; i < kD2Warps * T * 16; i += blockDim.x) slab[i] = 0.f;
  __syncthreads();
  float* my = slab + (size_t)wid * T * 16;
  const int items = shared_slots + *n_tiles_p;
  for (int it = wid; it < items; it += kD2Warps) {
    const Slot sl = slot_of(it, shared_slots, T, offsets, tile_map, items - shared_slots);
    if (sl.cnt <= 0) continue;
    const QW w = sl.e < 0 ? expert_of<QT>(sdn_w, 0) : expert_of<QT>(dn_w, sl.e);
    const int hrow_g = g < sl.cnt ? (sl.e < 0 ? T * k + sl.row0 + g : sl.row0 + g) : -1;
    int tok[2];
    float wt[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * q + cc;
      tok[cc] = -1;
      wt[cc] = 0.f;
      if (c < sl.cnt) {
        if (sl.e < 0) {
          tok[cc] = sl.row0 + c;
          wt[cc] = 1.f;
        } else {
          const int a = perm[sl.row0 + c];
          tok[cc] = a / k;
          wt[cc] = topk_w[a];
        }
      }
    }
    const __half* hrow = hbuf + (size_t)max(hrow_g, 0) * I;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int k0 = 0; k0 < I; k0 += 64) {
      RawA r;
      load_a<QT>(r, w, n0 + g, n0 + g + 8, k0, q);
      uint4 X0 = make_uint4(0, 0, 0, 0), X1 = X0;
      if (hrow_g >= 0) {
        X0 = __ldg(reinterpret_cast<const uint4*>(hrow + k0 + b_off0<QT>(q)));
        X1 = __ldg(reinterpret_cast<const uint4*>(hrow + k0 + b_off1<QT>(q)));
      }
      chunk_mma<QT>(acc, r, X0, X1);
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      if (tok[cc] >= 0) {
        const float s = wt[cc] * kHScaleInv;
        my[tok[cc] * 16 + g] += s * acc[cc];
        my[tok[cc] * 16 + g + 8] += s * acc[2 + cc];
      }
    }
    __syncwarp();
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * 16; i += blockDim.x) {
    float s = 0.f;
#pragma unroll 4
    for (int wv = 0; wv < kD2Warps; ++wv) s += slab[(size_t)wv * T * 16 + i];
    const int t = i / 16, r = i % 16;
    const size_t o = (size_t)t * H + n0 + r;
    y[o] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
    if (y32) y32[o] = s;
  }
}

}  // namespace decode

// Host launcher used by moe_ffn_forward for the decode path.
qsm_status decode_ffn_launch(const qsm_moe_layer* L, const uint16_t* x, int T,
                             const float* topk_w, const qsm_grouping* g,
                             uint16_t* y, float* y32, void* ws,
                             int32_t* dev_status, cudaStream_t stream) {
  using namespace decode;
  const int H = L->H, I = L->I, k = L->k;
  const int shared_slots = (T + kTok - 1) / kTok;
  __half* hbuf = static_cast<__half*>(ws);
  const dim3 g1(I / kTok, shared_slots + g->max_tiles);
  const size_t smem2 = (size_t)kD2Warps * T * 16 * sizeof(float);
  if (L->gate_up.qtype == QSM_Q8_0) {
    QSM_CUDA_TRY(launch_pdl(d1_gate_up_swiglu<QSM_Q8_0>, g1, dim3(kD1Split * 32), 0,
                            stream, L->gate_up, L->shared_gate_up, x, T, H, I, k,
                            (const int32_t*)g->perm, (const int32_t*)g->offsets,
                            (const int32_t*)g->tile_map, (const int32_t*)g->n_tiles,
                            shared_slots, hbuf, dev_status));
    QSM_CUDA_TRY(cudaFuncSetAttribute(d2_down_combine<QSM_Q8_0>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem2));
    QSM_CUDA_TRY(launch_pdl(d2_down_combine<QSM_Q8_0>, dim3(H / 16), dim3(kD2Warps * 32),
                            smem2, stream, L->down, L->shared_down, (const __half*)hbuf,
                            T, H, I, k, (const int32_t*)g->perm,
                            (const int32_t*)g->offsets, (const int32_t*)g->tile_map,
                            (const int32_t*)g->n_tiles, topk_w, shared_slots, y, y32));
  } else {
    QSM_CUDA_TRY(launch_pdl(d1_gate_up_swiglu<QSM_AFFINE4_G64>, g1, dim3(kD1Split * 32), 0,
                            stream, L->gate_up, L->shared_gate_up, x, T, H, I, k,
                            (const int32_t*)g->perm, (const int32_t*)g->offsets,
                            (const int32_t*)g->tile_map, (const int32_t*)g->n_tiles,
                            shared_slots, hbuf, dev_status));
    QSM_CUDA_TRY(cudaFuncSetAttribute(d2_down_combine<QSM_AFFINE4_G64>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem2));
    QSM_CUDA_TRY(launch_pdl(d2_down_combine<QSM_AFFINE4_G64>, dim3(H / 16),
                            dim3(kD2Warps * 32), smem2, stream, L->down, L->shared_down,
                            (const __half*)hbuf, T, H, I, k, (const int32_t*)g->perm,
                            (const int32_t*)g->offsets, (const int32_t*)g->tile_map,
                            (const int32_t*)g->n_tiles, topk_w, shared_slots, y, y32));
  }
  return QSM_OK;
}

size_t decode_ffn_workspace_bytes(const qsm_moe_layer* L, int T) {
  const size_t rows = (size_t)T * L->k + T;
  return ((rows * L->I * sizeof(__half)) + 255) & ~size_t(255);
}

}  // namespace qsm
