// Router top-k on a group of G lanes per token, shared by the stand-alone
// router kernel and the fused forward front ("Three axes of Parallelism",
// section "Expert Parallel (EP)" -> "Producing assignments": top-K experts per
// token and the probability with which each was chosen).
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving map of a finite float to an unsigned key; 0 is never a key.
// -0.0 and +0.0 share one key, so they tie.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f == 0.f) f = 0.f;   // -0.0 -> +0.0
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One token's top-K on a group of G lanes (G = 4, 8, 16 or 32; the group's
// lanes are consecutive lanes of the warp), lane g of the group holding experts
// g, g + G, ... (at most V <= 16 of them, E <= V * G). Each of the K rounds
// takes the lane's best untaken key (lowest id on equal keys), the group's max key by xor
// shuffles, then the lowest id holding it: the larger logit wins and equal
// logits go to the lower id. Slot j's id and logit stay with lane j % G
// (sid[j / G], sv[j / G]). top is the round-0 logit (the softmax max); den is
// the softmax denominator: over the K selected logits (renorm), summed in slot
// order, or over all E (the group's sum of its lanes' terms). Every lane of the
// warp must call it (dead groups pass live = false and follow along).
template <int G, int V>
__device__ __forceinline__ void group_topk(const float* __restrict__ row, bool live, int g, int E,
                                           int K, int renorm, float (&sv)[(32 + G - 1) / G],
                                           int (&sid)[(32 + G - 1) / G], float& top, float& den) {
  static_assert(G >= 4 && G <= 32 && (G & (G - 1)) == 0 && V >= 1 && V <= 16, "group shape");
  constexpr int SLOTS = (32 + G - 1) / G;   // slots per lane for K <= 32
  float v[V];
  uint32_t key[V];
  uint32_t avail = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = g + G * i;
    const bool ok = live && e < E;
    v[i] = ok ? __ldg(row + e) : 0.f;
    key[i] = ok ? order_key(v[i]) : 0u;
    if (ok) avail |= 1u << i;
  }
  top = 0.f;
  den = 0.f;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) { sv[s] = 0.f; sid[s] = 0; }
  for (int j = 0; j < K; ++j) {
    uint32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (((avail >> i) & 1u) && key[i] > bk) { bk = key[i]; bi = i; }
    uint32_t m = bk;
#pragma unroll
    for (int o = 1; o < G; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    uint32_t id = (bk == m && bk != 0u) ? static_cast<uint32_t>(g + G * bi) : 0xffffffffu;
#pragma unroll
    for (int o = 1; o < G; o <<= 1) id = min(id, __shfl_xor_sync(0xffffffffu, id, o));
    if (static_cast<int>(id % G) == g) avail &= ~(1u << (id / G));
    const float val = key_value(m);
    if (j == 0) top = val;
    if (renorm) den += expf(val - top);
    if ((j % G) == g) {
#pragma unroll
      for (int s = 0; s < SLOTS; ++s)
        if (s == j / G) { sv[s] = val; sid[s] = static_cast<int>(id); }
    }
  }
  if (!renorm) {   // softmax over all E: the group's sum of its lanes' terms
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (g + G * i < E) part += expf(v[i] - top);
#pragma unroll
    for (int o = 1; o < G; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    den = part;
  }
}

}  // namespace moe
