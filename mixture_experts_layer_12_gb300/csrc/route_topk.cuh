// route_topk.cuh -- per-token TopK and gate weights of the tensor-core
// routers, computed by a group of 8 lanes (router_kernel, route_fused_kernel).
//
// "用Ascend C写一个MoE融合算子", section "1. Routing + Gating 合并": TopK of
// the token's expert scores, then Softmax over the top-k scores only; the
// first-maximum '>' scan of "CANN ops-transformer：MoE 路由算子的负载均衡策略",
// section "Top-K 路由的并行化", fixes ties to the lower expert index.
#pragma once

#include <math.h>

#include "tc_common.cuh"

namespace moe {

constexpr int kTopkGroup = 8;  // lanes per token

// Lane g of the group holds the 4-expert chunks g, g + 8, g + 16, ... of the
// token's logits: lv[4 cc + i] is expert 4 (g + 8 cc) + i, already with the
// bias added, NaN replaced by -inf, and entries past E at -inf with their
// bit set in `taken` (bit q: logit q unavailable).  Each of the k rounds
// scans the lane's untaken logits in ascending expert order (strictly larger
// replaces, so equal logits keep the lower index), a 3-step shuffle argmax
// over the 8 lanes picks the round's expert (larger value, then lower
// index), and its owner marks it taken.  Lane g < k ends with choice g (best
// first) and its gate weight: softmax over the k selected logits, or
// (gating != MOE_GATE_TOPK_SOFTMAX) softmax over all E logits then the k
// probabilities, renormalised for MOE_GATE_SOFTMAX_TOPK_RENORM.  The rounds
// stay a loop: this code runs once per launch, cold in the instruction
// cache, so its size is its cost.
template <int NCH>
__device__ __forceinline__ void topk_gate_group(const float (&lv)[NCH * 4], uint32_t taken, int g,
                                                unsigned gmask, int k, int E, int gating,
                                                int& my_id, float& my_w) {
  constexpr int GS = kTopkGroup;
  constexpr int NV = NCH * 4;
  static_assert(kMaxTopK <= GS, "lane g keeps choice g");
  static_assert(NV <= 32, "taken mask");
  my_id = 0;
  float my_v = -INFINITY;
  float mx = 0.f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bq = -1;
#pragma unroll
    for (int q = 0; q < NV; ++q)
      if (!((taken >> q) & 1u) && (bq < 0 || lv[q] > bv)) {
        bv = lv[q];
        bq = q;
      }
    // local index q = 4*cc + i  <->  expert 4*(g + 8*cc) + i
    int be = bq < 0 ? 0x7fffffff : ((g + (bq >> 2) * GS) << 2) + (bq & 3);
#pragma unroll
    for (int off = GS / 2; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(gmask, bv, off);
      const int oe = __shfl_xor_sync(gmask, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be != 0x7fffffff && ((be >> 2) & (GS - 1)) == g)
      taken |= 1u << (((be >> 5) << 2) | (be & 3));
    if (j == 0) mx = bv;
    if (j == g) {
      my_id = be;
      my_v = bv;
    }
  }
  // softmax over the k choices: lane g < k holds exp(l_g - l_0), the group
  // sums by butterfly
  float ex = g < k ? expf(my_v - mx) : 0.f;
  float z = ex;
#pragma unroll
  for (int off = GS / 2; off > 0; off >>= 1) z += __shfl_xor_sync(gmask, z, off);
  if (gating != MOE_GATE_TOPK_SOFTMAX) {
    // softmax over all E logits first: p_j = exp(l_j - max) / sum_e exp(l_e - max)
    float zall = 0.f;
#pragma unroll
    for (int cc = 0; cc < NCH; ++cc)
      if ((g + cc * GS) * 4 < E)
#pragma unroll
        for (int i = 0; i < 4; ++i) zall += expf(lv[cc * 4 + i] - mx);
#pragma unroll
    for (int off = GS / 2; off > 0; off >>= 1) zall += __shfl_xor_sync(gmask, zall, off);
    ex = ex / zall;
    float zsel = ex;
#pragma unroll
    for (int off = GS / 2; off > 0; off >>= 1) zsel += __shfl_xor_sync(gmask, zsel, off);
    z = gating == MOE_GATE_SOFTMAX_TOPK ? 1.f : zsel;
  }
  my_w = ex / z;
}

}  // namespace moe
