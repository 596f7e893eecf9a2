// Building blocks of the weight-streaming GEMV kernels (decode FFN and the
// dense Q8_0 GEMV): a warp multiplies a 16-row quantized weight tile by up to
// 8 activation columns with mma.sync m16n8k16 (fp16 in, fp32 accumulate),
// 64 inputs per step.
//
// K mapping inside a 64-wide chunk (the same for A and B, since MMA k slots
// {2q, 2q+1, 2q+8, 2q+9} belong to thread quad q in both operands):
//   Q8_0:    quad q holds bytes [8q, 8q+8) of each of the chunk's two
//            32-blocks; MMAs 0,1 cover block 0 and MMAs 2,3 block 1, so each
//            MMA stays in one block and the block's fp16 scale multiplies the
//            fp32 MMA result (exact integer codes x exact fp16 inputs).
//   AFFINE4: quad q holds inputs [16q, 16q+16); the chunk is one group of 64,
//            dequantised to fp16 as scale*code + bias (one rounding).
#pragma once

#include "qsm_common.cuh"

namespace qsm {
namespace gemv {

struct QW {  // one expert's quantized matrix [rows, cols]
  const uint8_t* codes;
  const __half* scales;
  const __half* biases;
  int cols;
};

template <int QT>
__device__ __forceinline__ QW expert_of(const qsm_qweights& w, int e) {
  QW r;
  const size_t nrow = (size_t)e * w.rows;
  const size_t row_bytes = QT == QSM_Q8_0 ? (size_t)w.cols : (size_t)w.cols / 2;
  const int groups = QT == QSM_Q8_0 ? w.cols / 32 : w.cols / 64;
  r.codes = static_cast<const uint8_t*>(w.codes) + nrow * row_bytes;
  r.scales = reinterpret_cast<const __half*>(w.scales) + nrow * groups;
  r.biases = QT == QSM_Q8_0 ? nullptr
                            : reinterpret_cast<const __half*>(w.biases) + nrow * groups;
  r.cols = w.cols;
  return r;
}

// Raw bytes of a 16-row tile (rows rg and rh = MMA rows g and g+8) for one
// 64-chunk, as thread (g, q) holds them.
struct RawA {
  uint2 g0, g1, h0, h1;  // Q8_0: block 0 / block 1 bytes; AFFINE4: g0/h0 only
  uint32_t sg, sh;       // Q8_0: 2 block scales; AFFINE4: scale | bias << 16
};

template <int QT>
__device__ __forceinline__ void load_a(RawA& r, const QW& w, int rg, int rh,
                                       int k0, int q) {
  if (QT == QSM_Q8_0) {
    const uint8_t* bg = w.codes + (size_t)rg * w.cols + k0 + 8 * q;
    const uint8_t* bh = w.codes + (size_t)rh * w.cols + k0 + 8 * q;
    r.g0 = ldg_nc_v2(bg);
    r.g1 = ldg_nc_v2(bg + 32);
    r.h0 = ldg_nc_v2(bh);
    r.h1 = ldg_nc_v2(bh + 32);
    r.sg = ldg_nc_u32(w.scales + (size_t)rg * (w.cols / 32) + k0 / 32);
    r.sh = ldg_nc_u32(w.scales + (size_t)rh * (w.cols / 32) + k0 / 32);
  } else {
    const size_t rb = (size_t)w.cols / 2;
    r.g0 = ldg_nc_v2(w.codes + (size_t)rg * rb + k0 / 2 + 8 * q);
    r.h0 = ldg_nc_v2(w.codes + (size_t)rh * rb + k0 / 2 + 8 * q);
    const size_t gg = (size_t)rg * (w.cols / 64) + k0 / 64;
    const size_t gh = (size_t)rh * (w.cols / 64) + k0 / 64;
    r.sg = (uint32_t)__half_as_ushort(w.scales[gg]) |
           ((uint32_t)__half_as_ushort(w.biases[gg]) << 16);
    r.sh = (uint32_t)__half_as_ushort(w.scales[gh]) |
           ((uint32_t)__half_as_ushort(w.biases[gh]) << 16);
  }
}

// Offsets (in elements, inside the chunk) of the two 8-element B runs that
// thread quad q supplies.
template <int QT>
__device__ __forceinline__ int b_off0(int q) { return QT == QSM_Q8_0 ? 8 * q : 16 * q; }
template <int QT>
__device__ __forceinline__ int b_off1(int q) { return QT == QSM_Q8_0 ? 32 + 8 * q : 16 * q + 8; }

// fp16 pairs of 8 consecutive K (X = {p01, p23, p45, p67}) -> B registers
// of MMA j.
template <int QT>
__device__ __forceinline__ void b_frag(const uint4& X0, const uint4& X1, int j,
                                       uint32_t& b0, uint32_t& b1) {
  const uint4& X = j < 2 ? X0 : X1;
  if (QT == QSM_Q8_0) {
    b0 = (j & 1) ? X.z : X.x;
    b1 = (j & 1) ? X.w : X.y;
  } else {  // pairs (c0,c4),(c1,c5) for even j, (c2,c6),(c3,c7) for odd j
    const uint32_t lo = (j & 1) ? X.y : X.x, hi = (j & 1) ? X.w : X.z;
    b0 = __byte_perm(lo, hi, 0x5410);
    b1 = __byte_perm(lo, hi, 0x7632);
  }
}

__device__ __forceinline__ void a4_deq(uint32_t w, uint32_t sb, uint32_t (&v)[4]) {
  const __half2 k1024 = __half2half2(__ushort_as_half(0x6400));
  const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)(sb & 0xffff)));
  const __half2 b2 = __half2half2(__ushort_as_half((unsigned short)(sb >> 16)));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t t = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
    __half2 h = __hsub2(*reinterpret_cast<__half2*>(&t), k1024);
    h = __hfma2(h, s2, b2);
    v[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

// acc (rows g, g, g+8, g+8 x cols 2q, 2q+1) += tile(64-chunk) * B
template <int QT>
__device__ __forceinline__ void chunk_mma(float (&acc)[4], const RawA& r,
                                          const uint4& X0, const uint4& X1) {
  if (QT == QSM_Q8_0) {
    // one fp32 partial per 32-block (its two MMAs accumulate in order); the
    // two blocks' MMA chains are interleaved so their latencies overlap
    float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const uint2 wg = blk ? r.g1 : r.g0, wh = blk ? r.h1 : r.h0;
        uint32_t a[4], b0, b1;
        s8x4_to_f16x2x2(jj ? wg.y : wg.x, a[0], a[2]);
        s8x4_to_f16x2x2(jj ? wh.y : wh.x, a[1], a[3]);
        b_frag<QT>(X0, X1, 2 * blk + jj, b0, b1);
        mma_16816(d[blk], a, b0, b1);
      }
    }
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const float sg = __half2float(__ushort_as_half(
          (unsigned short)(blk ? (r.sg >> 16) : (r.sg & 0xffff))));
      const float sh = __half2float(__ushort_as_half(
          (unsigned short)(blk ? (r.sh >> 16) : (r.sh & 0xffff))));
      acc[0] = fmaf(sg, d[blk][0], acc[0]);
      acc[1] = fmaf(sg, d[blk][1], acc[1]);
      acc[2] = fmaf(sh, d[blk][2], acc[2]);
      acc[3] = fmaf(sh, d[blk][3], acc[3]);
    }
  } else {
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
      uint32_t vg[4], vh[4];
      a4_deq(wi ? r.g0.y : r.g0.x, r.sg, vg);
      a4_deq(wi ? r.h0.y : r.h0.x, r.sh, vh);
#pragma unroll
      for (int par = 0; par < 2; ++par) {
        uint32_t a[4] = {vg[2 * par], vh[2 * par], vg[2 * par + 1], vh[2 * par + 1]};
        uint32_t b0, b1;
        b_frag<QT>(X0, X1, 2 * wi + par, b0, b1);
        mma_16816(acc, a, b0, b1);
      }
    }
  }
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& v) {
  return make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                    bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
}

}  // namespace gemv
}  // namespace qsm
