// Router top-k and its backward ("Three axes of Parallelism", section
// "Expert Parallel (EP)" -> "Producing assignments": scores [T,E] against all
// experts, top-K selection of expert_IDs and router_weights [T,K]).
//
// Forward: one warp per token; lane l holds experts l, l+32, ... Logits become
// order-preserving unsigned keys (-0.0 and +0.0 share one key, so they tie),
// and each of the K rounds is a warp-wide max over the lanes' best untaken
// keys followed by a warp-wide min over the ids that hold it: the larger logit
// wins, equal logits go to the lower id. The softmax max is the round-0
// winner. Backward: one warp per token.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

// Order-preserving map of a finite float to an unsigned key; 0 is never a key.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f == 0.f) f = 0.f;   // -0.0 -> +0.0
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// V = ceil(E / 32) logits per lane. Round j: each lane's best untaken key
// (lowest id on equal keys), the warp max M of those (redux.sync), then the
// lowest id among lanes whose best is M (redux.sync). Lane j keeps slot j's
// id and logit, and lanes 0..K-1 write the K slots with coalesced stores.
template <int V>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_topk_kernel(const float* __restrict__ logits, int T, int E, int K, int renorm,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;   // whole warps only
  const float* row = logits + t * E;
  float v[V];
  uint32_t key[V];
  uint32_t avail = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(row + e) : 0.f;
    key[i] = (e < E) ? order_key(v[i]) : 0u;
    if (e < E) avail |= 1u << i;
  }
  float top = 0.f, mine = 0.f;
  int mine_id = 0;
  for (int j = 0; j < K; ++j) {
    uint32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (((avail >> i) & 1u) && key[i] > bk) { bk = key[i]; bi = i; }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = (bk == m && bk != 0u) ? static_cast<uint32_t>(lane + 32 * bi) : 0xffffffffu;
    const uint32_t id = __reduce_min_sync(0xffffffffu, cand);
    if (static_cast<int>(id & 31u) == lane) avail &= ~(1u << (id >> 5));
    const float val = key_value(m);
    if (j == 0) top = val;
    if (lane == j) { mine = val; mine_id = static_cast<int>(id); }
  }
  // softmax over all E (max = top), or over the K selected when renormalising
  float part = 0.f;
  if (renorm) {
    if (lane < K) part = expf(mine - top);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (lane + 32 * i < E) part += expf(v[i] - top);
  }
  const float denom = warp_sum(part);
  if (lane < K) {
    topk_idx[t * K + lane] = mine_id;
    topk_w[t * K + lane] = expf(mine - top) / denom;
  }
}

template <int V>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_topk_backward_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                           const float* __restrict__ topk_w, const float* __restrict__ dtopk_w,
                           int T, int E, int K, int renorm, float* __restrict__ dlogits) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const size_t base = static_cast<size_t>(t) * K;
  int id = 0;
  float w = 0.f, dw = 0.f;
  if (lane < K) { id = topk_idx[base + lane]; w = topk_w[base + lane]; dw = dtopk_w[base + lane]; }
  float* out = dlogits + static_cast<size_t>(t) * E;
  if (renorm) {
    const float s = warp_sum(w * dw);
    for (int e = lane; e < E; e += 32) out[e] = 0.f;
    __syncwarp();
    if (lane < K) out[id] = w * (dw - s);
    return;
  }
  // renorm == 0: p = softmax(logits[t]); dl_i = p_i * (g_i - s), s = sum_j p_{e_j} dw_j
  const float* row = logits + static_cast<size_t>(t) * E;
  float v[V];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(row + e) : -INFINITY;
    mx = fmaxf(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    if (e < E) sum += expf(v[i] - mx);
  }
  sum = warp_sum(sum);
  const float inv = 1.f / sum;
  const float p_sel = (lane < K) ? expf(__ldg(row + id) - mx) * inv : 0.f;
  const float s = warp_sum(p_sel * dw);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    if (e < E) out[e] = -expf(v[i] - mx) * inv * s;
  }
  __syncwarp();
  if (lane < K) out[id] = p_sel * (dw - s);
}

template <template <int> class Launcher, typename... Args>
int dispatch_v(int E, Args... args) {
  if (E <= 32) return Launcher<1>::run(args...);
  if (E <= 64) return Launcher<2>::run(args...);
  if (E <= 128) return Launcher<4>::run(args...);
  if (E <= 256) return Launcher<8>::run(args...);
  if (E <= 512) return Launcher<16>::run(args...);
  return Launcher<32>::run(args...);
}

template <int V>
struct FwdLauncher {
  static int run(const float* logits, int T, int E, int K, int renorm, int32_t* idx, float* w,
                 cudaStream_t st) {
    const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
    ProfScope prof("route_topk", st);
    return launch_pdl(route_topk_kernel<V>, blocks, kWarpsPerBlock * 32, 0, st, 1, logits, T, E, K,
                      renorm, idx, w);
  }
};

template <int V>
struct BwdLauncher {
  static int run(const float* logits, const int32_t* idx, const float* w, const float* dw, int T,
                 int E, int K, int renorm, float* dl, cudaStream_t st) {
    const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
    ProfScope prof("route_topk_backward", st);
    return launch_pdl(route_topk_backward_kernel<V>, blocks, kWarpsPerBlock * 32, 0, st, 1, logits,
                      idx, w, dw, T, E, K, renorm, dl);
  }
};

}  // namespace
}  // namespace moe

extern "C" int moe_route_topk(const float* logits, int T, int E, int K, int renorm,
                              int32_t* topk_idx, float* topk_w, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(topk_w)) return MOE_ERR_MISALIGNED;
  return dispatch_v<FwdLauncher>(E, logits, T, E, K, renorm, topk_idx, topk_w, as_stream(stream));
}

extern "C" int moe_route_topk_backward(const float* logits, const int32_t* topk_idx,
                                       const float* topk_w, const float* dtopk_w, int T, int E,
                                       int K, int renorm, float* dlogits, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_idx || !topk_w || !dtopk_w || !dlogits || (!renorm && !logits))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(dtopk_w) || !aligned16(dlogits) ||
      (logits && !aligned16(logits)))
    return MOE_ERR_MISALIGNED;
  return dispatch_v<BwdLauncher>(E, logits, topk_idx, topk_w, dtopk_w, T, E, K, renorm, dlogits,
                                 as_stream(stream));
}
