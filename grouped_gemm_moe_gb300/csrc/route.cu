// Router top-k and its backward ("Three axes of Parallelism", section
// "Expert Parallel (EP)" -> "Producing assignments": scores [T,E] against all
// experts, top-K selection of expert_IDs and router_weights [T,K]).
//
// Forward: a group of lanes per token (one warp per token above 256 experts);
// lane l of the group holds experts l, l + G, ... Logits become
// order-preserving unsigned keys (-0.0 and +0.0 share one key, so they tie),
// and each of the K rounds is a warp-wide max over the lanes' best untaken
// keys followed by a warp-wide min over the ids that hold it: the larger logit
// wins, equal logits go to the lower id. The softmax max is the round-0
// winner. Backward: one warp per token.
#include <algorithm>

#include "common.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

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

// Small expert counts (E <= 256): a group of G lanes per token (G = 4, 8 or 16,
// so 32 / G tokens share each warp instruction), lane g of the group holding
// experts g, g + G, ... (at most V = 16 each). Each round: the lane's best
// untaken key (lowest id on equal keys), the group's max key by shuffles, then
// the lowest id holding it by shuffles: the same rule as route_topk_kernel.
// Slot j's id and logit stay with lane j % G of the group, which also writes
// slot j; every lane accumulates the renormalised denominator in slot order.
// With one token per warp the kernel above issues about 500 warp instructions
// per token at E = 128, K = 8, and that issue rate, not memory, bounds it. Per
// token and round the lanes' scans cost E / 32 compares whatever G is, while
// the group's shuffles cost 2 G log2(G) / 32: small groups with 16 logits per
// lane issue the fewest instructions.
template <int G, int V>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
route_topk_group_kernel(const float* __restrict__ logits, int T, int E, int K, int renorm,
                        int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  constexpr int SLOTS = (32 + G - 1) / G;
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int g = lane & (G - 1);
  const long long t = (static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) *
                          (32 / G) + lane / G;
  const bool live = t < T;                  // dead groups follow along for the shuffles
  float sv[SLOTS], top, den;
  int sid[SLOTS];
  group_topk<G, V>(logits + (live ? t : 0) * E, live, g, E, K, renorm, sv, sid, top, den);
  if (!live) return;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    const int j = s * G + g;
    if (j < K) {
      topk_idx[t * K + j] = sid[s];
      topk_w[t * K + j] = expf(sv[s] - top) / den;
    }
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

// ----------------------------------------------------------------- load balance
// Partial sums of the router probabilities: CTA b (kLbBlocks of them, a fixed
// count, so the summation order does not depend on the device) gives each of
// its warps the tokens t = b*8 + w, + 8*kLbBlocks, ...; lane l accumulates
// softmax(logits[t]) at its experts l, l+32, ... in registers; the warps'
// sums are added in warp order into partial[b][e].
constexpr int kLbBlocks = 256;

template <int V>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
load_balance_partial_kernel(const float* __restrict__ logits, int T, int E,
                            float* __restrict__ partial) {
  pdl_enter();
  __shared__ float sums[kWarpsPerBlock][32 * V];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  for (long long t = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp; t < T;
       t += static_cast<long long>(gridDim.x) * kWarpsPerBlock) {
    const float* row = logits + t * E;
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
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      v[i] = (lane + 32 * i < E) ? expf(v[i] - mx) : 0.f;
      s += v[i];
    }
    s = warp_sum(s);
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] += v[i] / s;
  }
#pragma unroll
  for (int i = 0; i < V; ++i) sums[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float tot = 0.f;
    for (int w = 0; w < kWarpsPerBlock; ++w) tot += sums[w][e];
    partial[static_cast<size_t>(blockIdx.x) * E + e] = tot;
  }
}

// One CTA: P_e = (sum of the partials) / T, f_e = counts_e / TK, and the loss
// and metrics. The G = 1024 / E threads of expert e (e = tid % E) each sum the
// partials b = j, j + G, ... and the G sums are added in j order; the loss and
// metrics use fixed-shape block reductions, so every sum has a fixed order.
constexpr int kLbFinalThreads = 1024;

__global__ void __launch_bounds__(kLbFinalThreads)
load_balance_final_kernel(const float* __restrict__ partial, int nblk,
                          const int32_t* __restrict__ counts, int T, int E, int K,
                          float* __restrict__ load_frac, float* __restrict__ prob_mean,
                          float* __restrict__ stats) {
  pdl_enter();
  __shared__ float part[kLbFinalThreads];
  __shared__ float red[4][kLbFinalThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = kLbFinalThreads / E;   // >= 1 for E <= 1024
  if (tid < G * E) {
    const int e = tid % E, j = tid / E;
    float tot = 0.f;
    for (int b = j; b < nblk; b += G) tot += partial[static_cast<size_t>(b) * E + e];
    part[j * E + e] = tot;
  }
  __syncthreads();
  const float inv_t = 1.f / static_cast<float>(T);
  const float inv_tk = 1.f / (static_cast<float>(T) * static_cast<float>(K));
  float fp = 0.f, fmax = 0.f, nempty = 0.f, fsum = 0.f;
  if (tid < E) {
    const int e = tid;
    float tot = 0.f;
    for (int j = 0; j < G; ++j) tot += part[j * E + e];
    const float P = tot * inv_t;
    const int c = counts[e];
    const float f = static_cast<float>(c) * inv_tk;
    prob_mean[e] = P;
    load_frac[e] = f;
    fp = f * P;
    fmax = f;
    nempty = (c == 0) ? 1.f : 0.f;
    fsum = f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    fp += __shfl_xor_sync(0xffffffffu, fp, o);
    fmax = fmaxf(fmax, __shfl_xor_sync(0xffffffffu, fmax, o));
    nempty += __shfl_xor_sync(0xffffffffu, nempty, o);
    fsum += __shfl_xor_sync(0xffffffffu, fsum, o);
  }
  if (lane == 0) { red[0][warp] = fp; red[1][warp] = fmax; red[2][warp] = nempty; red[3][warp] = fsum; }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, m = 0.f, n = 0.f, fs = 0.f;
    for (int w = 0; w < kLbFinalThreads / 32; ++w) {
      a += red[0][w];
      m = fmaxf(m, red[1][w]);
      n += red[2][w];
      fs += red[3][w];
    }
    stats[0] = static_cast<float>(E) * a;
    stats[1] = static_cast<float>(E) * m;
    stats[2] = n;
    stats[3] = fs;
  }
}

// One warp per token: g[t,i] = scale * (E/T) * p_i * (f_i - sum_e f_e p_e).
template <int V>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
load_balance_backward_kernel(const float* __restrict__ logits, const float* __restrict__ frac,
                             int T, int E, float coef, int accumulate,
                             float* __restrict__ dlogits) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + t * E;
  float v[V], f[V];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(row + e) : -INFINITY;
    f[i] = (e < E) ? __ldg(frac + e) : 0.f;
    mx = fmaxf(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    v[i] = (lane + 32 * i < E) ? expf(v[i] - mx) : 0.f;
    s += v[i];
  }
  s = warp_sum(s);
  float fdot = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    v[i] /= s;   // p_i
    fdot += f[i] * v[i];
  }
  fdot = warp_sum(fdot);
  float* out = dlogits + t * E;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float g = coef * v[i] * (f[i] - fdot);
      out[e] = accumulate ? out[e] + g : g;
    }
  }
}

template <int V>
struct LbLauncher {
  static int run(const float* logits, const int32_t* counts, int T, int E, int K, float* frac,
                 float* pmean, float* stats, float* partial, cudaStream_t st) {
    const int nblk = static_cast<int>(
        std::min<long long>(kLbBlocks, (static_cast<long long>(T) + kWarpsPerBlock - 1) / kWarpsPerBlock));
    int rc;
    {
      ProfScope prof("load_balance", st);
      rc = launch_pdl(load_balance_partial_kernel<V>, nblk, kWarpsPerBlock * 32, 0, st, 1, logits,
                      T, E, partial);
    }
    if (rc) return rc;
    ProfScope prof("load_balance_final", st);
    return launch_pdl(load_balance_final_kernel, 1, kLbFinalThreads, 0, st, 1,
                      static_cast<const float*>(partial), nblk, counts, T, E, K, frac, pmean, stats);
  }
};

template <int V>
struct LbBwdLauncher {
  static int run(const float* logits, const float* frac, int T, int E, float coef, int accumulate,
                 float* dl, cudaStream_t st) {
    const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
    ProfScope prof("load_balance_backward", st);
    return launch_pdl(load_balance_backward_kernel<V>, blocks, kWarpsPerBlock * 32, 0, st, 1,
                      logits, frac, T, E, coef, accumulate, dl);
  }
};

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

namespace moe {
namespace {
template <int G, int V>
int launch_route_group(const float* logits, int T, int E, int K, int renorm, int32_t* idx,
                       float* w, cudaStream_t st) {
  const long long per_block = static_cast<long long>(kWarpsPerBlock) * (32 / G);
  const int blocks = static_cast<int>((T + per_block - 1) / per_block);
  ProfScope prof("route_topk", st);
  return launch_pdl(route_topk_group_kernel<G, V>, blocks, kWarpsPerBlock * 32, 0, st, 1, logits,
                    T, E, K, renorm, idx, w);
}
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
  // up to 16 logits per lane: a group of G = 4 .. 16 lanes per token
  if (E <= 32) return launch_route_group<4, 8>(logits, T, E, K, renorm, topk_idx, topk_w, st);
  if (E <= 64) return launch_route_group<4, 16>(logits, T, E, K, renorm, topk_idx, topk_w, st);
  if (E <= 128) return launch_route_group<8, 16>(logits, T, E, K, renorm, topk_idx, topk_w, st);
  if (E <= 256) return launch_route_group<16, 16>(logits, T, E, K, renorm, topk_idx, topk_w, st);
  return dispatch_v<FwdLauncher>(E, logits, T, E, K, renorm, topk_idx, topk_w, st);
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

namespace moe {
size_t load_balance_workspace(int E) {
  if (E < 1 || E > 1024) return 0;
  return kWorkspaceHeader + static_cast<size_t>(kLbBlocks) * E * sizeof(float);
}
}  // namespace moe

extern "C" int moe_load_balance(const float* logits, const int32_t* counts, int T, int E, int K,
                                float* load_frac, float* prob_mean, float* stats, void* ws,
                                size_t ws_bytes, void* stream) {
  using namespace moe;
  if (T < 1 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOE_ERR_INVALID_ARG;
  if (!logits || !counts || !load_frac || !prob_mean || !stats) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(counts) || !aligned16(load_frac) || !aligned16(prob_mean) ||
      !aligned16(stats))
    return MOE_ERR_MISALIGNED;
  if (!ws || !aligned16(ws) || ws_bytes < load_balance_workspace(E)) return MOE_ERR_WORKSPACE;
  float* partial = reinterpret_cast<float*>(static_cast<char*>(ws) + kWorkspaceHeader);
  return dispatch_v<LbLauncher>(E, logits, counts, T, E, K, load_frac, prob_mean, stats, partial,
                                as_stream(stream));
}

extern "C" int moe_load_balance_backward(const float* logits, const float* load_frac, int T, int E,
                                         float scale, int accumulate, float* dlogits,
                                         void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > 1024) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !load_frac || !dlogits) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(load_frac) || !aligned16(dlogits)) return MOE_ERR_MISALIGNED;
  const float coef = scale * static_cast<float>(E) / static_cast<float>(T);
  return dispatch_v<LbBwdLauncher>(E, logits, load_frac, T, E, coef, accumulate ? 1 : 0, dlogits,
                                   as_stream(stream));
}

namespace moe {
MOE_DEBUG_STATUS_READER(route)
}  // namespace moe
