// Expert selection of one token by one warp, shared by the router's
// selecting CTA and the one-launch decode layer so that both give the same
// ids and weights bit for bit.
//
// "Optimizing on-device inference for Apple Silicon", section "Qwen creates
// three distinct workload shapes": keep the k best-scoring experts of the
// token.  Readings: ties go to the lower expert index; the weights are the
// softmax over the selected logits (QSM_ROUTE_RENORMALIZE) or the full
// softmax taken at the selected ones; with QSM_ROUTE_BIAS_SELECT_ONLY the
// bias decides the selection but the weights use the logits without it.
// A non-finite logit (after adding the bias) counts as -inf and sets
// QSM_DEV_NONFINITE.
#pragma once

#include "qsm_common.cuh"

namespace qsm {

// lt: the token's E logits without the bias, in global memory (read
// through L2: another CTA may have written them in this launch) or, with
// kShared, in this CTA's shared memory.  Lane j < k receives the j-th
// selected expert, its selection logit and its routing weight.
template <int kPer, bool kShared = false>
__device__ __forceinline__ void route_select_warp(const float* __restrict__ lt,
                                                  const float* __restrict__ bias, int E,
                                                  int k, int flags, int32_t* dev_status,
                                                  int& out_e, float& out_l, float& out_w) {
  const int lane = threadIdx.x & 31;
  const bool renorm = (flags & QSM_ROUTE_RENORMALIZE) != 0;
  const bool sel_only = (flags & QSM_ROUTE_BIAS_SELECT_ONLY) != 0 && bias;
  float v[kPer], u[kPer];  // selection logits (with the bias), weight logits
  // all loads first (logits, then the bias), so they are in flight together
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    u[i] = lane + 32 * i < E ? (kShared ? lt[lane + 32 * i] : __ldcg(lt + lane + 32 * i))
                             : -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    v[i] = (bias && lane + 32 * i < E) ? __ldg(bias + lane + 32 * i) : 0.f;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    float l = u[i], sl = bias ? l + v[i] : l;
    if (lane + 32 * i < E && (!isfinite(sl) || !isfinite(l))) {
      bad = true;
      l = sl = -INFINITY;
    }
    v[i] = sl;
    u[i] = sel_only ? l : sl;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(dev_status, QSM_DEV_NONFINITE);
  float my_l;
  int my_e;
  warp_topk<kPer>(v, E, k, my_l, my_e);
  // this lane's selection's weight logit, and the largest one the softmax
  // runs over (the selection, or all E)
  float my_w = my_l;
  if (sel_only && lane < k) {
    my_w = kShared ? lt[my_e] : __ldcg(lt + my_e);
    if (!isfinite(my_w)) my_w = -INFINITY;
  }
  float top = -INFINITY;
  if (renorm) {
    top = warp_max(lane < k ? my_w : -INFINITY);
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i < E) top = fmaxf(top, u[i]);
    top = warp_max(top);
  }
  float part = 0.f;
  if (renorm) {
    if (lane < k) part = __expf(my_w - top);
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i < E) part += __expf(u[i] - top);
  }
  const float inv = 1.0f / warp_sum(part);
  out_e = my_e;
  out_l = my_l;
  out_w = lane < k ? __expf(my_w - top) * inv : 0.f;
}

}  // namespace qsm
