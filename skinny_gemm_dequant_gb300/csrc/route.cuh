// Softmax top-k routing of one token by one warp ([DSV4] §0.1, the M=1 routing fast path, and
// §0.3, the grouped batch MoE): the one routing rule every MoE launch uses.
//
// Selection: every expert becomes one 32-bit key, an order-preserving image of its bf16 logit
// above 65535 - e, so that the largest key is the largest logit and, among equal logits, the
// lowest expert id.  Each round of the top-k is one warp max (redux.sync) over the lanes' best
// keys.  Arithmetic: fp32 exponentials, their sum carried as a float-float pair (hi + lo, twice
// the precision of fp32 with fp32 instructions only; fp64 throughput on this part is a small
// fraction of fp32's).
//
// The fused router of the persistent MoE kernel runs this in every CTA, so its instruction
// count is paid on every SM: the loops are unrolled to E / 32 keys per lane, not to the largest
// E supported.
#pragma once

#include "common.cuh"

namespace ql {

// hi + lo, |lo| at most half an ulp of hi
struct FloatPair {
  float hi, lo;
};

// Knuth's TwoSum: s.hi + s.lo == a + b exactly (no overflow); symmetric in a and b
__device__ __forceinline__ FloatPair two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, err};
}

// Dekker's Fast2Sum, |a| >= |b|: s.hi + s.lo == a + b exactly
__device__ __forceinline__ FloatPair fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// x + y for non-negative terms (which keeps |hi| >= |lo| for the renormalisation)
__device__ __forceinline__ FloatPair pair_add(FloatPair x, FloatPair y) {
  const FloatPair s = two_sum(x.hi, y.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ FloatPair pair_add(FloatPair x, float y) {
  const FloatPair s = two_sum(x.hi, y);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}

__device__ __forceinline__ FloatPair warp_pair_sum(FloatPair v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = pair_add(v, FloatPair{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)});
  return v;  // the same in every lane: pair_add is symmetric in its operands
}

// e / (s.hi + s.lo) rounded to fp32: the quotient by hi, corrected by the exact remainder
// (one fma) less the quotient times lo
__device__ __forceinline__ float pair_div(float e, FloatPair s) {
  const float q = __fdiv_rn(e, s.hi);
  const float r = __fmaf_rn(-q, s.lo, __fmaf_rn(-q, s.hi, e));
  return __fadd_rn(q, __fdiv_rn(r, s.hi));
}

// order-preserving 16-bit image of a bf16 value, -0 taken as +0 (they compare equal): a larger
// image is a larger value.  bf16_from_order inverts it.
__device__ __forceinline__ uint32_t bf16_order(uint32_t b) {
  if (b == 0x8000u) b = 0u;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ float bf16_from_order(uint32_t o) {
  const uint32_t b = (o & 0x8000u) ? (o & 0x7FFFu) : (~o & 0xFFFFu);
  return __uint_as_float(b << 16);
}

// The routing of one token (row: its E bf16 logits; E <= 32 J).  p = exp(l - max) / sum over all
// experts of exp(l_e - max).  The topk largest logits are chosen in decreasing order, equal
// logits to the lower expert id; the weight of a chosen expert is its p, or with renorm
// p / (sum of the chosen p) = its exp / (sum of the chosen exps).  Lane k < topk receives the
// k-th choice in id and w; other lanes keep theirs.
template <int J>
__device__ __forceinline__ void route_token_warp_j(const uint16_t* __restrict__ row, int E, int topk, bool renorm,
                                                   int& id, float& w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[J];  // 0: no expert (past E, or already chosen)
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int e = lane + 32 * j;
    key[j] = e < E ? (bf16_order(row[e]) << 16) | (0xFFFFu - (uint32_t)e) : 0u;
  }
  uint32_t best = 0u;
#pragma unroll
  for (int j = 0; j < J; ++j) best = max(best, key[j]);
  const float mx = bf16_from_order(__reduce_max_sync(0xffffffffu, best) >> 16);
  FloatPair sum = {0.f, 0.f};
#pragma unroll
  for (int j = 0; j < J; ++j)
    if (key[j]) sum = pair_add(sum, expf(bf16_from_order(key[j] >> 16) - mx));
  sum = warp_pair_sum(sum);
  uint32_t mine = 0u;
  for (int k = 0; k < topk; ++k) {
    best = 0u;
#pragma unroll
    for (int j = 0; j < J; ++j) best = max(best, key[j]);
    const uint32_t win = __reduce_max_sync(0xffffffffu, best);
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (key[j] == win) key[j] = 0u;  // keys are distinct: only the owner's entry matches
    if (lane == k) mine = win;
  }
  const float x = lane < topk ? expf(bf16_from_order(mine >> 16) - mx) : 0.f;
  const FloatPair chosen = renorm ? warp_pair_sum(FloatPair{x, 0.f}) : sum;
  if (lane < topk) {
    id = (int)(0xFFFFu - (mine & 0xFFFFu));
    w = pair_div(x, chosen);
  }
}

__device__ __forceinline__ void route_token_warp(const uint16_t* __restrict__ row, int E, int topk, bool renorm,
                                                 int& id, float& w) {
  if (E <= 128)
    route_token_warp_j<4>(row, E, topk, renorm, id, w);
  else if (E <= 256)
    route_token_warp_j<8>(row, E, topk, renorm, id, w);
  else if (E <= 512)
    route_token_warp_j<16>(row, E, topk, renorm, id, w);
  else
    route_token_warp_j<32>(row, E, topk, renorm, id, w);
}

}  // namespace ql
