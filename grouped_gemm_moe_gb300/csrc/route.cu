// Router top-k and its backward ("Three axes of Parallelism", section
// "Expert Parallel (EP)" -> "Producing assignments": scores [T,E] against all
// experts, top-K selection of expert_IDs and router_weights [T,K]).
//
// Forward: a group of G lanes per token (see route_topk_kernel). Each of the K
// rounds is a butterfly arg-max over (logit, -id) across the group: the larger
// logit wins, equal logits go to the lower id (a float comparison, so -0.0 and
// +0.0 tie). The softmax max is the round-0 winner; its denominators are group
// sums. Backward: one warp per token.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

// One group of G lanes per token (G in 4..32, a power of two); lane l of a
// group holds experts l, l+G, l+2G, ... (V values). Each of the K rounds is a
// local best over the lane's untaken values and a butterfly over the group on
// (logit, -id). The winner's owner marks it taken and remembers its slot; the
// weights are written per taken value at the end.
template <int G, int V>
__global__ void __launch_bounds__(256)
route_topk_kernel(const float* __restrict__ logits, int T, int E, int K, int renorm,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  const int gl = threadIdx.x & (G - 1);
  const long long tok = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / G;
  const bool active = tok < T;
  const float* row = logits + (active ? tok : 0) * static_cast<long long>(E);
  float v[V];
  int slot[V];
  unsigned taken = 0;  // bit i: value i of this lane is selected (or padding)
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = gl + G * i;
    v[i] = (e < E) ? __ldg(row + e) : 0.f;
    slot[i] = 0;
    if (e >= E) taken |= 1u << i;
  }
  float top = 0.f;
  for (int j = 0; j < K; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      if (taken & (1u << i)) continue;
      if (bi == 0x7fffffff || v[i] > bv) { bv = v[i]; bi = gl + G * i; }   // ids ascend with i
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const bool better = (oi != 0x7fffffff) &&
                          (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
      if (better) { bv = ov; bi = oi; }
    }
    if ((bi & (G - 1)) == gl) {
      const int wi = bi / G;
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (i == wi) { taken |= 1u << i; slot[i] = j; }
    }
    if (j == 0) top = bv;
  }
  // softmax over all E (max = top), optionally renormalised over the K selected
  float s_all = 0.f, s_sel = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = gl + G * i;
    if (e < E) {
      const float x = expf(v[i] - top);
      s_all += x;
      if (taken & (1u << i)) s_sel += x;
    }
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) {
    s_all += __shfl_xor_sync(0xffffffffu, s_all, o);
    s_sel += __shfl_xor_sync(0xffffffffu, s_sel, o);
  }
  if (!active) return;
  const float denom = renorm ? s_sel : s_all;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = gl + G * i;
    if (e < E && (taken & (1u << i))) {
      const long long o = tok * K + slot[i];
      topk_idx[o] = e;
      topk_w[o] = expf(v[i] - top) / denom;
    }
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

template <int G, int V>
int launch_fwd(const float* logits, int T, int E, int K, int renorm, int32_t* idx, float* w,
               cudaStream_t st) {
  const long long threads = static_cast<long long>(T) * G;
  const int blocks = static_cast<int>((threads + 255) / 256);
  ProfScope prof("route_topk", st);
  route_topk_kernel<G, V><<<blocks, 256, 0, st>>>(logits, T, E, K, renorm, idx, w);
  return check_launch();
}

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
  cudaStream_t st = as_stream(stream);
  // group width: at most 16 logits per lane up to E = 512, 32 beyond
  if (E <= 64) return launch_fwd<4, 16>(logits, T, E, K, renorm, topk_idx, topk_w, st);
  if (E <= 128) return launch_fwd<8, 16>(logits, T, E, K, renorm, topk_idx, topk_w, st);
  if (E <= 256) return launch_fwd<16, 16>(logits, T, E, K, renorm, topk_idx, topk_w, st);
  if (E <= 512) return launch_fwd<32, 16>(logits, T, E, K, renorm, topk_idx, topk_w, st);
  return launch_fwd<32, 32>(logits, T, E, K, renorm, topk_idx, topk_w, st);
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
