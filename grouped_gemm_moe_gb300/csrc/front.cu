// The forward's front in two launches: router top-k with the per-chunk expert
// histogram, then the offsets, the stable expert-major permutation and the
// layout of an all-to-all over R simulated expert-parallel ranks.
//
// Sources: "Three axes of Parallelism" (nanoTitan blog), section "Expert
// Parallel (EP)" -> "Producing assignments" (top-K experts per token, bincount
// and cumulative offsets, expert-major packing in flat assignment order) and
// "Dispatch, expert computation and combine" (send splits per destination,
// source-major receive buffer, regroup by local expert); modalities PR "expert
// parallelism for the Nemotron-3 Nano MoE layers", section "Design" (indices
// built on the device, one device-to-host copy of the splits).
//
// The outputs are those of moe_route_topk followed by moe_build_permutation_ep,
// bit for bit. That pair is three launches (top-k, chunk histograms, scatter),
// each a short chain of dependent steps; here the histogram comes with the
// top-k:
//   1. route_hist: one CTA per chunk (a contiguous token range inside one sender
//      block; about one chunk per SM) routes its tokens with a group of G lanes
//      per token, writes the top-k outputs and the chunk's expert histogram row;
//   2. place: one CTA per chunk reads its ids back, brings the whole histogram
//      table into shared memory with one bulk copy, forms per expert the sums
//      over all chunks, earlier chunks and this sender's chunks, and places
//      every assignment in closed form (the counting sort's positions).
// The launch boundary, under programmatic dependent launch, is the only
// grid-wide synchronisation: the second kernel's CTAs are scheduled while the
// first finishes and wait (griddepcontrol.wait) for its writes.
#include "common.cuh"
#include "topk.cuh"

namespace moe {

size_t permutation_workspace(long long TK, int E, int R);   // permute.cu

namespace {

constexpr int kFrontWarps = 16;
constexpr int kFrontThreads = kFrontWarps * 32;
constexpr int kFrontMaxIds = 16384;     // assignments of one chunk held in shared memory
constexpr int kFrontMaxChunks = 1024;   // bound of the histogram rows in the workspace
constexpr size_t kFrontSmemMax = 200 * 1024;
constexpr unsigned long long kCopyTimeoutNs = 2000000000ull;

struct FrontArgs {
  const float* logits;
  int T, E, K, renorm, R;
  int Ts;    // tokens per sender block (T / R)
  int cps;   // chunks per sender block
  int ct;    // tokens per chunk
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* splits;          // [R*E] counts per (sender, expert), then [R*R] send splits
  int32_t* send_index;
  int32_t* a2a_index;
  int32_t* regroup_index;
  int32_t* hist;            // [NC][hist_stride(E)] chunk histograms (workspace)
  int* status;              // workspace status word
};

// Histogram rows are padded to a multiple of four experts (16-byte rows, so
// the table is one contiguous bulk copy).
__host__ __device__ constexpr int hist_stride(int E) { return (E + 3) & ~3; }

__device__ __forceinline__ uint64_t front_globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t front_smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// A chunk's token range [t0, t1), its sender s and its index cc within the sender.
struct Chunk {
  int s, cc, t0, t1;
};
__device__ __forceinline__ Chunk chunk_of(const FrontArgs& a, int c) {
  Chunk k;
  k.s = c / a.cps;
  k.cc = c - k.s * a.cps;
  k.t0 = min(k.s * a.Ts + k.cc * a.ct, (k.s + 1) * a.Ts);
  k.t1 = min(k.t0 + a.ct, (k.s + 1) * a.Ts);
  return k;
}

// ---------------------------------------------------------------- 1. route_hist
// Shared memory: the chunk's per-expert counts, ids and weights.
size_t route_hist_smem_bytes(int E, int ids) {
  return (static_cast<size_t>(hist_stride(E)) + 2 * static_cast<size_t>(ids)) * sizeof(int);
}

template <int G, int V>
__global__ void __launch_bounds__(kFrontThreads, 1) route_hist_kernel(const FrontArgs a) {
  constexpr int SLOTS = (32 + G - 1) / G;
  constexpr int TPW = 32 / G;   // tokens per warp and pass
  extern __shared__ __align__(16) int smem[];
  const int E = a.E, K = a.K;
  const int Ep = hist_stride(E);
  int* cnt = smem;                                         // [Ep] this chunk's counts
  int* sid = cnt + Ep;                                     // [ct*K] ids, flat order
  float* swt = reinterpret_cast<float*>(sid + a.ct * K);   // [ct*K] weights

  pdl_enter();   // logits come from an earlier launch; the next launch may be scheduled now
  const Chunk ch = chunk_of(a, blockIdx.x);
  const int n = (ch.t1 - ch.t0) * K;
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < Ep; e += kFrontThreads) cnt[e] = 0;
  __syncthreads();

  const int g = lane & (G - 1);
  for (int tb = ch.t0 + w * TPW; tb < ch.t1; tb += kFrontWarps * TPW) {   // uniform per warp
    const int t = tb + lane / G;
    const bool live = t < ch.t1;
    float sv[SLOTS], top, den;
    int sidv[SLOTS];
    group_topk<G, V>(a.logits + static_cast<size_t>(live ? t : 0) * E, live, g, E, K, a.renorm, sv,
                     sidv, top, den);
    if (live) {
#pragma unroll
      for (int q = 0; q < SLOTS; ++q) {
        const int j = q * G + g;
        if (j < K) {
          sid[(t - ch.t0) * K + j] = sidv[q];
          swt[(t - ch.t0) * K + j] = expf(sv[q] - top) / den;
          atomicAdd(&cnt[sidv[q]], 1);   // counts only: their order does not matter
        }
      }
    }
  }
  __syncthreads();
  // the chunk's outputs are one contiguous range [t0*K, t1*K): coalesced stores
  const size_t a0 = static_cast<size_t>(ch.t0) * K;
  for (int i = threadIdx.x; i < n; i += kFrontThreads) {
    a.topk_idx[a0 + i] = sid[i];
    a.topk_w[a0 + i] = swt[i];
  }
  for (int e = threadIdx.x; e < Ep; e += kFrontThreads)
    a.hist[static_cast<size_t>(blockIdx.x) * Ep + e] = cnt[e];
}

// ---------------------------------------------------------------- 2. place
// Shared memory: the histogram table (NC rows), the per-warp counts, the
// table pass's partial sums, the offset and prefix tables and the chunk's ids.
size_t place_smem_bytes(int E, int ids, int NC) {
  return (static_cast<size_t>(NC) * hist_stride(E) + static_cast<size_t>(kFrontWarps) * E +
          5 * kFrontThreads + 6 * E + 3 + static_cast<size_t>(ids)) * sizeof(int);
}

__global__ void __launch_bounds__(kFrontThreads, 1) place_kernel(const FrontArgs a) {
  extern __shared__ __align__(16) int smem[];
  __shared__ __align__(8) uint64_t tab_bar;
  const int E = a.E, K = a.K;
  const int Ep = hist_stride(E);
  const int NC = gridDim.x;
  int* tab = smem;                                     // [NC][Ep] the histogram table
  int* wh = tab + static_cast<size_t>(NC) * Ep;        // [kFrontWarps][E] warp counts, then prefix
  int* part = wh + kFrontWarps * E;                    // [5][kFrontThreads] table-pass partials
  int* off = part + 5 * kFrontThreads;                 // [E+1] offsets
  int* ball = off + (E + 1);             // [E] sum of the histogram rows before this chunk
  int* bs = ball + E;                    // [E] same, restricted to this sender
  int* cs = bs + E;                      // [E+1] C[s][e] -> exclusive scan (send prefix)
  int* craw = cs + (E + 1);              // [E] C[s][e]
  int* csb = craw + E;                   // [E+1] sum of C[s'][e], s' < s -> exclusive scan
  int* sid = csb + (E + 1);              // [ct*K] the chunk's expert ids, flat order

  const int c = blockIdx.x;
  const Chunk ch = chunk_of(a, c);
  const int s = ch.s;
  const int n = (ch.t1 - ch.t0) * K;
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar = front_smem_u32(&tab_bar);
  for (int i = threadIdx.x; i < kFrontWarps * E; i += kFrontThreads) wh[i] = 0;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();   // the route_hist launch's ids and histogram rows are complete and visible
  pdl_launch_dependents();
  if (threadIdx.x == 0) {   // the whole table: one bulk copy, a few large requests
    const uint32_t bytes = static_cast<uint32_t>(NC) * Ep * sizeof(int);
    asm volatile("fence.proxy.async.global;" ::: "memory");   // the rows, to the async proxy
    asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(front_smem_u32(tab)), "l"(a.hist), "r"(bytes), "r"(bar)
        : "memory");
  }
  const size_t a0 = static_cast<size_t>(ch.t0) * K;
  for (int i = threadIdx.x; i < n; i += kFrontThreads) sid[i] = __ldcg(a.topk_idx + a0 + i);
  __syncthreads();

  // per-warp counts: warp w takes the contiguous range [wa0, wa1)
  const int per_w = ((n + kFrontThreads - 1) / kFrontThreads) * 32;
  const int wa0 = w * per_w;
  const int wa1 = min(wa0 + per_w, n);
  for (int b = wa0; b < wa0 + per_w; b += 32) {   // same trip count on every lane
    const int ai = b + lane;
    const int e = ai < wa1 ? sid[ai] : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(grp) - 1) wh[w * E + e] += __popc(grp);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kFrontThreads) {   // exclusive prefix across warps
    int run = 0;
#pragma unroll 4
    for (int k = 0; k < kFrontWarps; ++k) {
      const int v = wh[k * E + e];
      wh[k * E + e] = run;
      run += v;
    }
  }

  // the table has landed (bounded wait; on a timeout nothing is placed)
  {
    const uint64_t t0 = front_globaltimer();
    uint32_t done = 0;
    while (!done) {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}"
          : "=r"(done) : "r"(bar) : "memory");
      if (!done && front_globaltimer() - t0 > kCopyTimeoutNs) break;
    }
    if (!__syncthreads_and(done != 0)) {
      if (threadIdx.x == 0) report_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
  // per expert: the sums over all chunks, the chunks before this one, this
  // sender's chunks (all, and before this one) and earlier senders' chunks; P
  // threads per expert split the chunks
  int P = 1;
  while (2 * P * E <= kFrontThreads) P *= 2;
  for (int t = threadIdx.x; t < P * E; t += kFrontThreads) {
    const int e = t % E, q = t / E;
    int tot = 0, b_all = 0, b_s = 0, c_s = 0, c_sb = 0;
    const int k0 = q * NC / P, k1 = (q + 1) * NC / P;
    int sk = k0 / a.cps;              // sender of chunk k, advanced without a division
    int next = (sk + 1) * a.cps;
#pragma unroll 8
    for (int k = k0; k < k1; ++k) {
      if (k == next) { ++sk; next += a.cps; }
      const int h = tab[k * Ep + e];
      tot += h;
      if (k < c) b_all += h;
      if (sk == s) { c_s += h; if (k < c) b_s += h; }
      if (sk < s) c_sb += h;
    }
    part[t] = tot;
    part[kFrontThreads + t] = b_all;
    part[2 * kFrontThreads + t] = b_s;
    part[3 * kFrontThreads + t] = c_s;
    part[4 * kFrontThreads + t] = c_sb;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kFrontThreads) {
    int v[5] = {0, 0, 0, 0, 0};
    for (int q = 0; q < P; ++q)
#pragma unroll
      for (int i = 0; i < 5; ++i) v[i] += part[i * kFrontThreads + q * E + e];
    off[e] = v[0];
    ball[e] = v[1];
    bs[e] = v[2];
    cs[e] = v[3];
    craw[e] = v[3];
    csb[e] = v[4];
  }
  if (threadIdx.x == 0) { off[E] = 0; cs[E] = 0; csb[E] = 0; }
  __syncthreads();
  if (w == 0) warp_exscan(off, E + 1);
  if (w == 1) warp_exscan(cs, E + 1);
  if (w == 2) warp_exscan(csb, E + 1);
  __syncthreads();

  const int El = E / a.R;
  if (c == 0) {
    for (int e = threadIdx.x; e <= E; e += kFrontThreads) {
      a.offsets[e] = off[e];
      if (e < E) a.counts[e] = off[e + 1] - off[e];
    }
  }
  if (ch.cc == 0) {   // the sender's first chunk writes its row of the splits
    for (int e = threadIdx.x; e < E; e += kFrontThreads) a.splits[static_cast<size_t>(s) * E + e] = craw[e];
    for (int d = threadIdx.x; d < a.R; d += kFrontThreads)
      a.splits[static_cast<size_t>(a.R) * E + static_cast<size_t>(s) * a.R + d] =
          cs[(d + 1) * El] - cs[d * El];
  }

  // positions: rank among the expert's assignments = earlier chunks + earlier
  // warps of this chunk + earlier steps and lanes of this warp
  int* mine = wh + w * E;
  const int send_base = s * a.Ts * K;
  for (int b = wa0; b < wa0 + per_w; b += 32) {
    const int ai = b + lane;
    const int e = ai < wa1 ? sid[ai] : -1;
    const bool valid = e >= 0;
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const int before = valid ? mine[e] : 0;
    __syncwarp();
    if (valid && lane == __ffs(grp) - 1) mine[e] = before + __popc(grp);
    __syncwarp();
    if (!valid) continue;
    const int rank = before + __popc(grp & lanemask_lt());
    const int p = off[e] + ball[e] + rank;
    const int ag = static_cast<int>(a0 + ai);
    a.perm[p] = ag;
    a.inv_perm[ag] = p;
    const int rank_se = bs[e] + rank;
    const int e0 = (e / El) * El;
    const int q = send_base + cs[e] + rank_se;
    const int r = off[e0] + (csb[e0 + El] - csb[e0]) + (cs[e] - cs[e0]) + rank_se;
    a.send_index[q] = ag;
    a.a2a_index[r] = q;
    a.regroup_index[p] = r;
  }
}

// Shared-memory opt-in once per device and kernel.
template <typename Kern>
int front_smem_optin(Kern kern, int* configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (*configured == dev) return MOE_OK;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kFrontSmemMax));
  if (e != cudaSuccess) { set_last_cuda_error(e); return MOE_ERR_CUDA; }
  *configured = dev;
  return MOE_OK;
}

template <int G, int V>
int launch_front(const FrontArgs& a, int NC, cudaStream_t st) {
  static thread_local int configured_rh = -1, configured_pl = -1;
  const int ids = a.ct * a.K;
  const size_t sm_rh = route_hist_smem_bytes(a.E, ids);
  const size_t sm_pl = place_smem_bytes(a.E, ids, NC);
  if (sm_rh > kFrontSmemMax || sm_pl > kFrontSmemMax) return MOE_ERR_UNSUPPORTED;
  int rc = front_smem_optin(route_hist_kernel<G, V>, &configured_rh);
  if (rc) return rc;
  rc = front_smem_optin(place_kernel, &configured_pl);
  if (rc) return rc;
  {
    ProfScope prof("route_hist", st);
    rc = launch_pdl(route_hist_kernel<G, V>, NC, kFrontThreads, sm_rh, st, 1, a);
  }
  if (rc) return rc;
  ProfScope prof("place_ep", st);
  return launch_pdl(place_kernel, NC, kFrontThreads, sm_pl, st, 1, a);
}

}  // namespace

size_t route_permute_workspace(long long TK, int E, int R) {
  const size_t fused =
      kWorkspaceHeader + static_cast<size_t>(kFrontMaxChunks) * hist_stride(E) * sizeof(int32_t);
  const size_t split = permutation_workspace(TK, E, R);
  return fused > split ? fused : split;
}

}  // namespace moe

extern "C" int moe_route_permute_ep(const float* logits, int T, int E, int K, int renorm, int R,
                                    int32_t* topk_idx, float* topk_w, int32_t* counts,
                                    int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                    int32_t* ep_splits, int32_t* send_index, int32_t* a2a_index,
                                    int32_t* regroup_index, int32_t* host_splits, void* ws,
                                    size_t ws_bytes, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E || R < 1 || R > 64 || E % R || T % R)
    return MOE_ERR_INVALID_ARG;
  const long long TK = static_cast<long long>(T) * K;
  if (TK >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !ep_splits) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (T > 0) {
    if (!logits || !topk_idx || !topk_w || !perm || !inv_perm || !send_index || !a2a_index ||
        !regroup_index)
      return MOE_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(counts) ||
        !aligned16(offsets) || !aligned16(perm) || !aligned16(inv_perm) || !aligned16(ep_splits) ||
        !aligned16(send_index) || !aligned16(a2a_index) || !aligned16(regroup_index))
      return MOE_ERR_MISALIGNED;
    if (!ws || !aligned16(ws) || ws_bytes < route_permute_workspace(TK, E, R)) return MOE_ERR_WORKSPACE;
    // chunk geometry: about one chunk per SM, split evenly over the senders,
    // at least 8 tokens per chunk
    const int Ts = T / R;
    int cps = num_sms() / R;
    if (cps < 1) cps = 1;
    const int min_tokens = 8;
    if (cps > (Ts + min_tokens - 1) / min_tokens) cps = (Ts + min_tokens - 1) / min_tokens;
    const int ct = (Ts + cps - 1) / cps;
    const int NC = R * cps;
    int rc = MOE_ERR_UNSUPPORTED;
    if (E <= 256 && static_cast<long long>(ct) * K <= kFrontMaxIds && NC <= kFrontMaxChunks) {
      FrontArgs a{};
      a.logits = logits;
      a.T = T; a.E = E; a.K = K; a.renorm = renorm; a.R = R;
      a.Ts = Ts; a.cps = cps; a.ct = ct;
      a.topk_idx = topk_idx; a.topk_w = topk_w;
      a.counts = counts; a.offsets = offsets; a.perm = perm; a.inv_perm = inv_perm;
      a.splits = ep_splits; a.send_index = send_index; a.a2a_index = a2a_index;
      a.regroup_index = regroup_index;
      a.hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kWorkspaceHeader);
      a.status = static_cast<int*>(ws);
      if (E <= 32) rc = launch_front<4, 8>(a, NC, st);
      else if (E <= 64) rc = launch_front<4, 16>(a, NC, st);
      else if (E <= 128) rc = launch_front<8, 16>(a, NC, st);
      else rc = launch_front<16, 16>(a, NC, st);
    }
    if (rc == MOE_ERR_UNSUPPORTED) {   // the stand-alone kernels: the same outputs
      rc = moe_route_topk(logits, T, E, K, renorm, topk_idx, topk_w, stream);
      if (rc) return rc;
      return moe_build_permutation_ep(topk_idx, T, E, K, R, counts, offsets, perm, inv_perm,
                                      ep_splits, send_index, a2a_index, regroup_index, host_splits,
                                      ws, ws_bytes, stream);
    }
    if (rc) return rc;
  } else {
    cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st);
    cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    cudaMemsetAsync(ep_splits, 0, sizeof(int32_t) * (static_cast<size_t>(R) * E + R * R), st);
  }
  if (host_splits) {
    const size_t split_bytes = sizeof(int32_t) * (static_cast<size_t>(R) * E + R * R);
    const cudaError_t e = cudaMemcpyAsync(host_splits, ep_splits, split_bytes,
                                          cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) { set_last_cuda_error(e); return MOE_ERR_CUDA; }
  }
  return check_launch();
}
