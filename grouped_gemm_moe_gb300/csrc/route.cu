// Router top-k and its backward ("Three axes of Parallelism", section
// "Expert Parallel (EP)" -> "Producing assignments": scores [T,E] against all
// experts, top-K selection of expert_IDs and router_weights [T,K]).
//
// One warp per token. Lane l holds experts l, l+32, l+64, ... in registers.
// Each of the K rounds is a butterfly arg-max over (logit, -id) across the
// warp: the larger logit wins, equal logits go to the lower id (a float
// comparison, so -0.0 and +0.0 tie). The winner's owner lane marks it taken.
// The softmax max is the round-0 winner; its denominator is a warp sum.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

template <int V>  // V = ceil(E / 32) values per lane
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_topk_kernel(const float* __restrict__ logits, int T, int E, int K, int renorm,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + static_cast<size_t>(t) * E;
  float v[V];
  unsigned taken = 0;  // bit i: value i of this lane already selected
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(row + e) : 0.f;
    if (e >= E) taken |= 1u << i;          // padding never competes
  }
  float my_v = 0.f;
  int my_id = 0;
  float top = 0.f;
  for (int j = 0; j < K; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      if (taken & (1u << i)) continue;
      const int e = lane + 32 * i;
      if (bi == 0x7fffffff || v[i] > bv) { bv = v[i]; bi = e; }   // ids ascend with i
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const bool better = (oi != 0x7fffffff) &&
                          (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
      if (better) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) { my_v = bv; my_id = bi; }
    if (j == 0) top = bv;
  }
  // softmax over all E (max = top), then optional renormalisation over the K selected
  float s_all = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    if (e < E) s_all += expf(v[i] - top);
  }
  s_all = warp_sum(s_all);
  const float ex = (lane < K) ? expf(my_v - top) : 0.f;
  const float s_sel = warp_sum(ex);
  if (lane < K) {
    const size_t o = static_cast<size_t>(t) * K + lane;
    topk_idx[o] = my_id;
    topk_w[o] = renorm ? ex / s_sel : ex / s_all;
  }
}

template <int V>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_topk_backward_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                           const float* __restrict__ topk_w, const float* __restrict__ dtopk_w,
                           int T, int E, int K, int renorm, float* __restrict__ dlogits) {
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
    route_topk_kernel<V><<<blocks, kWarpsPerBlock * 32, 0, st>>>(logits, T, E, K, renorm, idx, w);
    return check_launch();
  }
};

template <int V>
struct BwdLauncher {
  static int run(const float* logits, const int32_t* idx, const float* w, const float* dw, int T,
                 int E, int K, int renorm, float* dl, cudaStream_t st) {
    const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
    ProfScope prof("route_topk_backward", st);
    route_topk_backward_kernel<V><<<blocks, kWarpsPerBlock * 32, 0, st>>>(logits, idx, w, dw, T,
                                                                           E, K, renorm, dl);
    return check_launch();
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
