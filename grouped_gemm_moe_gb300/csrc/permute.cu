// Per-expert histogram, offsets, stable expert-major permutation, and the
// layout of an all-to-all over R simulated expert-parallel ranks.
//
// Sources: "Three axes of Parallelism" (nanoTitan blog), section "Expert
// Parallel (EP)" -> "Producing assignments" (bincount + cumulative offsets,
// expert-major packing) and "Dispatch, expert computation and combine"
// (send matrix per destination, source-major receive buffer, regroup into
// local-expert-major order); modalities PR "expert parallelism for the
// Nemotron-3 Nano MoE layers", section "Design" (indices built on device
// with no per-(sender, expert) host round trips; one device-to-host copy of
// the splits).
//
// Design: a two-kernel stable counting sort, deterministic and free of
// atomics on positions.
//  1. hist:    the assignments are cut into chunks of 1024 that never straddle
//              a sender block. Each warp counts its 128 assignments per expert
//              with __match_any_sync (one leader per equal-id group adds the
//              group's popcount to a warp-private counter), then the CTA sums
//              the 8 warps into hist[chunk][e].
//  2. scatter: every CTA reads the whole (small) hist table and derives, per
//              expert, the counts/offsets and the prefix of earlier chunks;
//              it redoes the warp counts, scans them across warps, and walks
//              its assignments again so each one gets
//              rank = earlier chunks + earlier warps + earlier steps + earlier
//              lanes with the same expert. Positions follow in closed form.
#include <atomic>
#include <mutex>
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSteps = 4;
constexpr int kPerWarp = kSteps * 32;          // 128 assignments per warp
constexpr int kChunk = kWarps * kPerWarp;      // 1024 assignments per CTA

struct ChunkGeom {
  long long seg_len;   // assignments per sender block (T*K/R)
  int cps;             // chunks per sender block
};

__device__ __forceinline__ void chunk_range(const ChunkGeom& g, int c, long long& start,
                                            long long& end, int& s) {
  s = c / g.cps;
  const int cc = c % g.cps;
  start = static_cast<long long>(s) * g.seg_len + static_cast<long long>(cc) * kChunk;
  end = min(start + kChunk, static_cast<long long>(s + 1) * g.seg_len);
}

// This warp's experts of the chunk, one per lane and step (-1 past the chunk),
// loaded up front so that their latency overlaps whatever the block does next.
__device__ __forceinline__ void load_warp_ids(const int32_t* __restrict__ idx, long long wstart,
                                              long long end, int E, int (&ev)[kSteps]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const long long a = wstart + st * 32 + lane;
    int e = (a < end) ? __ldg(idx + a) : -1;
    if (e >= 0 && !index_ok(e < E)) e = -1;   // debug builds: an id past E is dropped
    ev[st] = e;
  }
}

// Counts this warp's assignments of the chunk into wh[e] (warp-private row).
__device__ __forceinline__ void warp_count(const int (&ev)[kSteps], int* wh) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int e = ev[st];
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(grp) - 1) wh[e] += __popc(grp);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kThreads)
hist_kernel(const int32_t* __restrict__ idx, int E, ChunkGeom g, int32_t* __restrict__ hist) {
  pdl_enter();
  extern __shared__ int smem[];
  int* wh = smem;  // [kWarps][E]
  for (int i = threadIdx.x; i < kWarps * E; i += kThreads) wh[i] = 0;
  __syncthreads();
  long long start, end;
  int s;
  chunk_range(g, blockIdx.x, start, end, s);
  const int w = threadIdx.x >> 5;
  int ev[kSteps];
  load_warp_ids(idx, start + static_cast<long long>(w) * kPerWarp, end, E, ev);
  warp_count(ev, wh + w * E);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int sum = 0;
#pragma unroll
    for (int k = 0; k < kWarps; ++k) sum += wh[k * E + e];
    hist[static_cast<size_t>(blockIdx.x) * E + e] = sum;
  }
}

struct PermOut {           // moe_build_permutation outputs
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
};

struct EpOut {             // moe_ep_layout outputs
  int32_t* splits;         // [R*E] counts then [R*R] send splits
  int32_t* send_index;
  int32_t* a2a_index;
  int32_t* regroup_index;
  int R;
  int El;
};

template <bool EP>
__global__ void __launch_bounds__(kThreads)
scatter_kernel(const int32_t* __restrict__ idx, int E, ChunkGeom g, int NC,
               const int32_t* __restrict__ hist, PermOut po, EpOut eo) {
  pdl_enter();
  extern __shared__ int smem[];
  int* wh = smem;                    // [kWarps][E]
  int* off = wh + kWarps * E;        // [E+1] offsets
  int* ball = off + (E + 1);         // [E]   sum of hist over chunks before this one
  int* bs = ball + E;                // [E]   same, restricted to this sender
  int* cs = bs + E;                  // [E+1] C[s][e] -> exclusive scan (send prefix)
  int* craw = cs + (E + 1);          // [E]   C[s][e]
  int* csb = craw + E;               // [E+1] sum of C[s'][e] for s' < s -> exclusive scan
  int* part = csb + (E + 1);         // [5][kThreads] partial sums of the table pass

  const int c = blockIdx.x;
  long long start, end;
  int s;
  chunk_range(g, c, start, end, s);
  const int w = threadIdx.x >> 5;
  const long long wstart = start + static_cast<long long>(w) * kPerWarp;
  int ev[kSteps];
  load_warp_ids(idx, wstart, end, E, ev);

  for (int i = threadIdx.x; i < kWarps * E; i += kThreads) wh[i] = 0;
  // Table pass: per expert, sums of hist over all chunks, the chunks before this
  // one, and (EP) this sender's chunks, those before this chunk, earlier senders'.
  // With E <= 128 the chunks are split over P = 2 or 4 threads per expert.
  const int P = (4 * E <= kThreads) ? 4 : ((2 * E <= kThreads) ? 2 : 1);
  for (int t = threadIdx.x; t < P * E; t += kThreads) {
    const int e = t % E, q = t / E;
    int tot = 0, b_all = 0, b_s = 0, c_s = 0, c_sb = 0;
#pragma unroll 16
    for (int k = q * NC / P; k < (q + 1) * NC / P; ++k) {
      const int h = __ldg(hist + static_cast<size_t>(k) * E + e);
      tot += h;
      if (k < c) b_all += h;
      if (EP) {
        const int sk = k / g.cps;
        if (sk == s) { c_s += h; if (k < c) b_s += h; }
        if (sk < s) c_sb += h;
      }
    }
    if (P == 1) {
      off[e] = tot;
      ball[e] = b_all;
      if (EP) { bs[e] = b_s; cs[e] = c_s; craw[e] = c_s; csb[e] = c_sb; }
    } else {
      part[t] = tot;
      part[kThreads + t] = b_all;
      part[2 * kThreads + t] = b_s;
      part[3 * kThreads + t] = c_s;
      part[4 * kThreads + t] = c_sb;
    }
  }
  if (P > 1) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) {
      int v[5] = {0, 0, 0, 0, 0};
      for (int q = 0; q < P; ++q)
#pragma unroll
        for (int i = 0; i < 5; ++i) v[i] += part[i * kThreads + q * E + e];
      off[e] = v[0];
      ball[e] = v[1];
      if (EP) { bs[e] = v[2]; cs[e] = v[3]; craw[e] = v[3]; csb[e] = v[4]; }
    }
  }
  if (threadIdx.x == 0) { off[E] = 0; if (EP) { cs[E] = 0; csb[E] = 0; } }
  __syncthreads();
  if (w == 0) warp_exscan(off, E + 1);
  if (EP && w == 1) warp_exscan(cs, E + 1);
  if (EP && w == 2) warp_exscan(csb, E + 1);
  // per-warp counts of this chunk
  warp_count(ev, wh + w * E);
  __syncthreads();

  if (c == 0 && (!EP || po.counts)) {   // counts and offsets (the EP pass writes them on request)
    for (int e = threadIdx.x; e <= E; e += kThreads) {
      po.offsets[e] = off[e];
      if (e < E) po.counts[e] = off[e + 1] - off[e];
    }
  }
  if (EP && c % g.cps == 0) {
    for (int e = threadIdx.x; e < E; e += kThreads) eo.splits[static_cast<size_t>(s) * E + e] = craw[e];
    for (int d = threadIdx.x; d < eo.R; d += kThreads)
      eo.splits[static_cast<size_t>(eo.R) * E + static_cast<size_t>(s) * eo.R + d] =
          cs[(d + 1) * eo.El] - cs[d * eo.El];
  }
  // exclusive scan of the warp counts across warps, per expert
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int run = 0;
#pragma unroll
    for (int k = 0; k < kWarps; ++k) {
      const int v = wh[k * E + e];
      wh[k * E + e] = run;
      run += v;
    }
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  int* mine = wh + w * E;
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const long long a = wstart + st * 32 + lane;
    const int e = ev[st];
    const bool valid = e >= 0;   // -1 past the chunk (and, in debug builds, for a dropped id)
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const int before = valid ? mine[e] : 0;
    __syncwarp();
    if (valid && lane == __ffs(grp) - 1) mine[e] = before + __popc(grp);
    __syncwarp();
    if (!valid) continue;
    const int rank = before + __popc(grp & lanemask_lt());
    const int p = off[e] + ball[e] + rank;
    if (!EP) {
      po.perm[p] = static_cast<int32_t>(a);
      po.inv_perm[a] = p;
    } else {
      const int rank_se = bs[e] + rank;
      const int dst = e / eo.El;
      const int e0 = dst * eo.El;
      const int q = static_cast<int>(static_cast<long long>(s) * g.seg_len) + cs[e] + rank_se;
      const int r = off[e0] + (csb[e0 + eo.El] - csb[e0]) + (cs[e] - cs[e0]) + rank_se;
      eo.send_index[q] = static_cast<int32_t>(a);
      eo.a2a_index[r] = q;
      eo.regroup_index[p] = r;
      if (po.perm) {
        po.perm[p] = static_cast<int32_t>(a);
        po.inv_perm[a] = p;
      }
    }
  }
}

// Dynamic shared memory of scatter_kernel: the warp counts, the offset and
// prefix tables (6E + 3 ints) and the table pass's partial sums (5 x kThreads).
size_t scatter_smem_bytes(int E) {
  return (static_cast<size_t>(kWarps) * E + 6 * E + 3 + 5 * kThreads) * sizeof(int);
}

size_t hist_bytes(long long TK, int E, int R) {
  const long long seg = TK / R;
  const long long cps = (seg + kChunk - 1) / kChunk;
  return static_cast<size_t>(cps) * R * E * sizeof(int32_t);
}

int launch_counting_sort(bool ep, const int32_t* idx, long long TK, int E, int R, PermOut po,
                         EpOut eo, void* ws, size_t ws_bytes, cudaStream_t st) {
  ChunkGeom g;
  g.seg_len = TK / R;
  g.cps = static_cast<int>((g.seg_len + kChunk - 1) / kChunk);
  const int NC = g.cps * R;
  int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kWorkspaceHeader);
  const size_t sh_hist = static_cast<size_t>(kWarps) * E * sizeof(int);
  const size_t sh_scatter = scatter_smem_bytes(E);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    cudaFuncSetAttribute(scatter_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         160 * 1024);
    cudaFuncSetAttribute(scatter_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         160 * 1024);
    configured_dev = dev;
  }
  (void)ws_bytes;
  int rc;
  {
    ProfScope prof(ep ? "ep_hist" : "perm_hist", st);
    rc = launch_pdl(hist_kernel, NC, kThreads, sh_hist, st, 1, idx, E, g, hist);
  }
  if (rc) return rc;
  ProfScope prof(ep ? "ep_scatter" : "perm_scatter", st);
  if (ep)
    return launch_pdl(scatter_kernel<true>, NC, kThreads, sh_scatter, st, 1, idx, E, g, NC, hist,
                      po, eo);
  return launch_pdl(scatter_kernel<false>, NC, kThreads, sh_scatter, st, 1, idx, E, g, NC, hist, po,
                    eo);
}

}  // namespace

size_t permutation_workspace(long long TK, int E, int R) {
  return kWorkspaceHeader + hist_bytes(TK, E, R);
}

}  // namespace moe

extern "C" int moe_build_permutation(const int32_t* topk_idx, int T, int E, int K,
                                     int32_t* counts, int32_t* offsets, int32_t* perm,
                                     int32_t* inv_perm, void* ws, size_t ws_bytes,
                                     void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
  const long long TK = static_cast<long long>(T) * K;
  if (TK >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (TK == 0) {
    cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st);
    cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    return check_launch();
  }
  if (!topk_idx || !perm || !inv_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(topk_idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(perm) ||
      !aligned16(inv_perm))
    return MOE_ERR_MISALIGNED;
  if (!ws || ws_bytes < permutation_workspace(TK, E, 1) || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  PermOut po{counts, offsets, perm, inv_perm};
  EpOut eo{};
  return launch_counting_sort(false, topk_idx, TK, E, 1, po, eo, ws, ws_bytes, st);
}

extern "C" int moe_ep_layout(const int32_t* topk_idx, int T, int E, int K, int R,
                             int32_t* ep_splits, int32_t* send_index, int32_t* a2a_index,
                             int32_t* regroup_index, int32_t* host_splits, void* ws,
                             size_t ws_bytes, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > E || R < 1 || R > 64 || E % R || T % R)
    return MOE_ERR_INVALID_ARG;
  const long long TK = static_cast<long long>(T) * K;
  if (TK >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (!ep_splits) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  const size_t split_bytes = sizeof(int32_t) * (static_cast<size_t>(R) * E + R * R);
  if (TK == 0) {
    cudaMemsetAsync(ep_splits, 0, split_bytes, st);
  } else {
    if (!topk_idx || !send_index || !a2a_index || !regroup_index) return MOE_ERR_INVALID_ARG;
    if (!aligned16(topk_idx) || !aligned16(ep_splits) || !aligned16(send_index) ||
        !aligned16(a2a_index) || !aligned16(regroup_index))
      return MOE_ERR_MISALIGNED;
    if (!ws || ws_bytes < permutation_workspace(TK, E, R) || !aligned16(ws))
      return MOE_ERR_WORKSPACE;
    PermOut po{};
    EpOut eo{ep_splits, send_index, a2a_index, regroup_index, R, E / R};
    const int rc = launch_counting_sort(true, topk_idx, TK, E, R, po, eo, ws, ws_bytes, st);
    if (rc) return rc;
  }
  if (host_splits) {
    const cudaError_t e = cudaMemcpyAsync(host_splits, ep_splits, split_bytes,
                                          cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) { set_last_cuda_error(e); return MOE_ERR_CUDA; }
  }
  return check_launch();
}

extern "C" int moe_build_permutation_ep(const int32_t* topk_idx, int T, int E, int K, int R,
                                        int32_t* counts, int32_t* offsets, int32_t* perm,
                                        int32_t* inv_perm, int32_t* ep_splits,
                                        int32_t* send_index, int32_t* a2a_index,
                                        int32_t* regroup_index, int32_t* host_splits, void* ws,
                                        size_t ws_bytes, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > E || R < 1 || R > 64 || E % R || T % R)
    return MOE_ERR_INVALID_ARG;
  const long long TK = static_cast<long long>(T) * K;
  if (TK >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !ep_splits) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  const size_t split_bytes = sizeof(int32_t) * (static_cast<size_t>(R) * E + R * R);
  if (TK == 0) {
    cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st);
    cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    cudaMemsetAsync(ep_splits, 0, split_bytes, st);
  } else {
    if (!topk_idx || !perm || !inv_perm || !send_index || !a2a_index || !regroup_index)
      return MOE_ERR_INVALID_ARG;
    if (!aligned16(topk_idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(perm) ||
        !aligned16(inv_perm) || !aligned16(ep_splits) || !aligned16(send_index) ||
        !aligned16(a2a_index) || !aligned16(regroup_index))
      return MOE_ERR_MISALIGNED;
    if (!ws || ws_bytes < permutation_workspace(TK, E, R) || !aligned16(ws))
      return MOE_ERR_WORKSPACE;
    PermOut po{counts, offsets, perm, inv_perm};
    EpOut eo{ep_splits, send_index, a2a_index, regroup_index, R, E / R};
    const int rc = launch_counting_sort(true, topk_idx, TK, E, R, po, eo, ws, ws_bytes, st);
    if (rc) return rc;
  }
  if (host_splits) {
    const cudaError_t e = cudaMemcpyAsync(host_splits, ep_splits, split_bytes,
                                          cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) { set_last_cuda_error(e); return MOE_ERR_CUDA; }
  }
  return check_launch();
}

// ---------------------------------------------------------------------------
// moe_build_permutation_static: the same two kernels with the chunk histogram
// in a fixed device array instead of a caller workspace, for callers that
// cannot allocate. Host code must not pass g_static_hist itself to a kernel
// (in host code the name is a host-side stand-in, not a device address); it
// passes the address cudaGetSymbolAddress returns for the current device.
namespace moe {

static __device__ __align__(256) int32_t g_static_hist[MOE_STATIC_HIST_INTS];

namespace {

constexpr int kMaxStaticDevices = 64;

// Per-device set-up of the static entry point, done once per device under a
// lock (host threads may make their first call on a device concurrently):
// the device address of g_static_hist and the kernels' shared-memory limits.
// A failed set-up is not recorded, so the next call retries it.
struct StaticDeviceState {
  std::atomic<int32_t*> hist{nullptr};
};
StaticDeviceState g_static_state[kMaxStaticDevices];
std::mutex g_static_mutex;

int static_setup_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { set_last_cuda_error(e); return MOE_ERR_CUDA; }
  if (dev < 0 || dev >= kMaxStaticDevices) return MOE_ERR_UNSUPPORTED;
  StaticDeviceState& s = g_static_state[dev];
  int32_t* p = s.hist.load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_static_mutex);
    p = s.hist.load(std::memory_order_relaxed);
    if (!p) {
      e = cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               160 * 1024);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(scatter_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
      void* ptr = nullptr;
      if (e == cudaSuccess) e = cudaGetSymbolAddress(&ptr, g_static_hist);
      if (e != cudaSuccess || !ptr) {
        set_last_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        return MOE_ERR_CUDA;
      }
      p = static_cast<int32_t*>(ptr);
      s.hist.store(p, std::memory_order_release);
    }
  }
  *out = p;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_build_permutation_static(const int32_t* topk_idx, int T, int E, int K,
                                            int32_t* counts, int32_t* offsets, int32_t* perm,
                                            int32_t* inv_perm, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
  const long long TK = static_cast<long long>(T) * K;
  if (TK >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (TK == 0) {
    cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st);
    cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    return check_launch();
  }
  if (!topk_idx || !perm || !inv_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(topk_idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(perm) ||
      !aligned16(inv_perm))
    return MOE_ERR_MISALIGNED;
  ChunkGeom g;
  g.seg_len = TK;
  g.cps = static_cast<int>((TK + kChunk - 1) / kChunk);
  const int NC = g.cps;
  if (static_cast<long long>(NC) * E > MOE_STATIC_HIST_INTS) return MOE_ERR_WORKSPACE;
  int32_t* hist = nullptr;
  int rc = static_setup_current_device(&hist);
  if (rc) return rc;
  const size_t sh_hist = static_cast<size_t>(kWarps) * E * sizeof(int);
  const size_t sh_scatter = scatter_smem_bytes(E);
  PermOut po{counts, offsets, perm, inv_perm};
  EpOut eo{};
  {
    ProfScope prof("perm_hist", st);
    rc = launch_pdl(hist_kernel, NC, kThreads, sh_hist, st, 1, topk_idx, E, g, hist);
  }
  if (rc) return rc;
  ProfScope prof("perm_scatter", st);
  return launch_pdl(scatter_kernel<false>, NC, kThreads, sh_scatter, st, 1, topk_idx, E, g, NC, hist,
                    po, eo);
}

namespace moe {
MOE_DEBUG_STATUS_READER(permute)
}  // namespace moe
