// Expert parallelism over real ranks: the per-rank pieces on either side of
// the collectives.
//
// 1. All-to-all EP ("Three axes of Parallelism" (nanoTitan blog), section
//    "Expert Parallel (EP)" -> "Dispatch, expert computation and combine":
//    every rank packs its assignments expert-major, exchanges the counts,
//    sends each destination the rows of the experts it owns, and the
//    destination regroups the source-major receive buffer by local expert;
//    modalities PR "expert parallelism for the Nemotron-3 Nano MoE layers",
//    section "Design" items 1-2: that regroup index built on device, one
//    device-to-host copy of both split lists). A rank's send buffer is its
//    local expert-major permutation (moe_dispatch_scatter), so the only new
//    kernel is the receive side's layout: from the exchanged counts
//    C[s][e] (source s, local expert e) it writes the send and receive split
//    lists, the local expert offsets of the regrouped rows and
//    regroup_index[p] = the receive-buffer row of regrouped row p.
//
// 2. All-gather / reduce-scatter EP (SpecForge PR "expert parallelism for MoE
//    drafters on the FSDP2 backend", "What this adds", the MoELayer.forward
//    under EP bullet: all-gather the group's tokens, run the replicated router
//    on them, compute only the locally owned experts, reduce-scatter the
//    partial outputs, add the shared expert on the local tokens). Every rank
//    holds the permutation of all tokens; its experts [e_lo, e_hi) own the
//    packed rows [offsets[e_lo], offsets[e_hi)), read on the device. The slice
//    kernels move only those rows: a token-major gather into the compact local
//    rows, a combine into fp32 partials of every token, the combine's
//    backward on the local assignments (zero dtopk_w elsewhere), the dispatch
//    backward into fp32 partials, and the bf16 finish after the reduction.
//
// The row kernels are HBM-bound: one thread per 16-byte vector of a token's
// row, 16-byte loads and stores, fp32 accumulation in slot order, no atomics.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

int grid_for(long long work, int per_block, int blocks_per_sm = 16) {
  long long b = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(num_sms()) * blocks_per_sm;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

__device__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int s = 0;
  for (int w = 0; w < kThreads / 32; ++w) s += red[w];
  return s;
}

// ----------------------------------------------------------------- 1. A2A
// One CTA per (local expert e, source s), in regrouped order b = e * R + s.
// C = recv_counts as [R][El]. The segment (e, s) holds C[s][e] rows; they sit
// in the receive buffer at src0 = sum of C over flat indices < s*El + e (the
// buffer is source-major, each source's block expert-major) and are
// regrouped to dst0 = sum over (e' < e, all s') + sum over (e, s' < s).
__global__ void __launch_bounds__(kThreads)
ep_recv_layout_kernel(const int32_t* __restrict__ counts_local, const int32_t* __restrict__ recv,
                      int R, int El, int32_t* __restrict__ splits,
                      int32_t* __restrict__ local_offsets, int32_t* __restrict__ regroup,
                      long long capacity, int* status) {
  pdl_enter();
  __shared__ int red[kThreads / 32];
  const int b = blockIdx.x;
  const int e = b / R, s = b - e * R;
  const int n_cells = R * El;
  int a_src = 0, a_dst = 0;
  for (int i = threadIdx.x; i < n_cells; i += kThreads) {
    const int si = i / El, ei = i - si * El;
    const int c = __ldg(recv + i);
    if (i < s * El + e) a_src += c;
    if (ei < e || (ei == e && si < s)) a_dst += c;
  }
  const long long src0 = block_sum(a_src, red);
  const long long dst0 = block_sum(a_dst, red);
  const int n = __ldg(recv + s * El + e);
  if (b == 0) {
    // split lists: what this rank sends to each destination, receives from each source
    for (int q = threadIdx.x; q < 2 * R; q += kThreads) {
      int v = 0;
      if (q < R) {
        for (int j = 0; j < El; ++j) v += __ldg(counts_local + q * El + j);
      } else {
        for (int j = 0; j < El; ++j) v += __ldg(recv + (q - R) * El + j);
      }
      splits[q] = v;
    }
    for (int q = threadIdx.x; q <= El; q += kThreads) {
      int v = 0;
      for (int i = 0; i < R * q; ++i) v += __ldg(recv + (i % R) * El + i / R);
      local_offsets[q] = v;
    }
  }
  if (dst0 + n > capacity || src0 + n > capacity) {
    if (threadIdx.x == 0) report_status(status, MOE_ERR_DEVICE_CHECK);
    return;
  }
  for (int i = threadIdx.x; i < n; i += kThreads)
    regroup[dst0 + i] = static_cast<int32_t>(src0 + i);
}

// ----------------------------------------------------------------- 2. AG/RS
struct Window {
  const int32_t* offsets;
  int e_lo, e_hi;
};

__device__ __forceinline__ void window_rows(const Window& w, int& lo, int& hi) {
  lo = __ldg(w.offsets + w.e_lo);
  hi = __ldg(w.offsets + w.e_hi);
}

// xs[p - lo] = x[t] for every assignment a = t*K + j with p = inv_perm[a] in
// [lo, hi). Block 0 also writes local_offsets[i] = offsets[e_lo + i] - lo.
template <int KMAX>
__global__ void __launch_bounds__(kThreads)
dispatch_slice_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv_perm, int K,
                      int nv, long long total, Window win, uint4* __restrict__ xs,
                      int32_t* __restrict__ local_offsets) {
  pdl_enter();
  int lo, hi;
  window_rows(win, lo, hi);
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i <= win.e_hi - win.e_lo; i += kThreads)
      local_offsets[i] = __ldg(win.offsets + win.e_lo + i) - lo;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += stride) {
    const long long t = i / nv;
    const int c = static_cast<int>(i - t * nv);
    const int32_t* ip = inv_perm + t * K;
    int32_t pos[KMAX];
    bool any = false;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      pos[j] = -1;
      if (j < K) {
        const int p = __ldg(ip + j);
        if (p >= lo && p < hi) { pos[j] = p - lo; any = true; }
      }
    }
    if (!any) continue;
    const uint4 v = ldg_nc_v4(x + i);
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K && pos[j] >= 0) stg_v4(xs + static_cast<long long>(pos[j]) * nv + c, v);
  }
}

// out[t] (fp32) = sum over slots j whose row p = inv_perm[t*K+j] lies in
// [lo, hi) of w[t,j] * rows[p - lo] (w == nullptr means 1), in slot order;
// tokens with no such slot get zeros.
template <int KMAX>
__global__ void __launch_bounds__(kThreads)
gather_sum_slice_kernel(const uint4* __restrict__ rows, const float* __restrict__ w,
                        const int32_t* __restrict__ inv_perm, int K, int nv, long long total,
                        Window win, float4* __restrict__ out) {
  pdl_enter();
  int lo, hi;
  window_rows(win, lo, hi);
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += stride) {
    const long long t = i / nv;
    const int c = static_cast<int>(i - t * nv);
    const int32_t* ip = inv_perm + t * K;
    int32_t pos[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      pos[j] = -1;
      if (j < K) {
        const int p = __ldg(ip + j);
        if (p >= lo && p < hi) pos[j] = p - lo;
      }
    }
    uint4 v[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K && pos[j] >= 0) v[j] = ldg_nc_v4(rows + static_cast<long long>(pos[j]) * nv + c);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < K && pos[j] >= 0) {
        const float wj = w ? __ldg(w + t * K + j) : 1.f;
        float f[8];
        unpack8(v[j], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(wj, f[q], acc[q]);
      }
    }
    out[2 * i] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    out[2 * i + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// One warp per assignment a = t*K + j with p = inv_perm[a]: inside the window,
// dy_s[p - lo] = bf16(w[a] * dout[t]) and dw[a] = <dout[t], y_s[p - lo]>;
// outside it dw[a] = 0 (another rank owns that slot).
constexpr int kCbUnroll = 4;

__global__ void __launch_bounds__(kThreads)
combine_backward_slice_kernel(const uint4* __restrict__ dout, const uint4* __restrict__ y,
                              const float* __restrict__ w, const int32_t* __restrict__ inv_perm,
                              long long TK, int K, int nv, Window win, uint4* __restrict__ dy,
                              float* __restrict__ dw) {
  pdl_enter();
  int lo, hi;
  window_rows(win, lo, hi);
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kThreads / 32);
  for (long long a = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
       a < TK; a += warps) {
    const int p = __ldg(inv_perm + a);
    if (p < lo || p >= hi) {
      if (lane == 0) dw[a] = 0.f;
      continue;
    }
    const long long t = a / K;
    const uint4* drow = dout + t * nv;
    const long long prow = static_cast<long long>(p - lo) * nv;
    const uint4* yrow = y + prow;
    uint4* orow = dy + prow;
    const float wa = __ldg(w + a);
    float dot = 0.f;
    for (int c0 = lane; c0 < nv; c0 += 32 * kCbUnroll) {
      uint4 dv[kCbUnroll], yv[kCbUnroll];
#pragma unroll
      for (int u = 0; u < kCbUnroll; ++u) {
        const int c = c0 + 32 * u;
        if (c < nv) {
          dv[u] = ldg_nc_v4(drow + c);
          yv[u] = ldg_nc_v4(yrow + c);
        }
      }
#pragma unroll
      for (int u = 0; u < kCbUnroll; ++u) {
        const int c = c0 + 32 * u;
        if (c < nv) {
          float fd[8], fy[8], g[8];
          unpack8(dv[u], fd);
          unpack8(yv[u], fy);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            dot = fmaf(fd[q], fy[q], dot);
            g[q] = mul_bf16_exact(wa, fd[q]);
          }
          stg_v4(orow + c, pack8(g));
        }
      }
    }
    const float sum = warp_sum(dot);
    if (lane == 0) dw[a] = sum;
  }
}

// out[i] = bf16(partial[i] + extra[i]) (extra == nullptr: 0), 8 columns per thread.
__global__ void __launch_bounds__(kThreads)
finish_kernel(const float4* __restrict__ partial, const uint4* __restrict__ extra, long long total,
              uint4* __restrict__ out) {
  pdl_enter();
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += stride) {
    const float4 a = partial[2 * i], b = partial[2 * i + 1];
    float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (extra) {
      float g[8];
      unpack8(ldg_nc_v4(extra + i), g);
#pragma unroll
      for (int q = 0; q < 8; ++q) f[q] += g[q];
    }
    stg_v4(out + i, pack8(f));
  }
}

bool slice_ok(int T, int K, int d, int E, int e_lo, int e_hi) {
  return T >= 0 && K >= 1 && K <= 32 && d > 0 && d % 8 == 0 && E >= 1 && e_lo >= 0 &&
         e_lo < e_hi && e_hi <= E;
}

int launch_gather_sum_slice(const char* name, const void* rows, const float* w,
                            const int32_t* inv_perm, int T, int K, int d, const int32_t* offsets,
                            int e_lo, int e_hi, float* out, cudaStream_t st) {
  const int nv = d / 8;
  const long long total = static_cast<long long>(T) * nv;
  const int grid = grid_for(total, kThreads);
  const Window win{offsets, e_lo, e_hi};
  auto r = static_cast<const uint4*>(rows);
  auto o = reinterpret_cast<float4*>(out);
  ProfScope prof(name, st);
  auto go = [&](auto kern) {
    return launch_pdl(kern, grid, kThreads, 0, st, 1, r, w, inv_perm, K, nv, total, win, o);
  };
  if (K <= 2) return go(gather_sum_slice_kernel<2>);
  if (K <= 4) return go(gather_sum_slice_kernel<4>);
  if (K <= 8) return go(gather_sum_slice_kernel<8>);
  if (K <= 16) return go(gather_sum_slice_kernel<16>);
  return go(gather_sum_slice_kernel<32>);
}

}  // namespace
}  // namespace moe

extern "C" int moe_ep_recv_layout(const int32_t* counts_local, const int32_t* recv_counts, int E,
                                  int R, int capacity, int32_t* splits, int32_t* local_offsets,
                                  int32_t* regroup_index, int32_t* host_splits, void* ws,
                                  size_t ws_bytes, void* stream) {
  using namespace moe;
  if (E < 1 || R < 1 || E % R || E > 1024 || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (!counts_local || !recv_counts || !splits || !local_offsets) return MOE_ERR_INVALID_ARG;
  if (capacity > 0 && !regroup_index) return MOE_ERR_INVALID_ARG;
  if (!aligned16(counts_local) || !aligned16(recv_counts) || !aligned16(splits) ||
      !aligned16(local_offsets) || (regroup_index && !aligned16(regroup_index)))
    return MOE_ERR_MISALIGNED;
  if (!ws || !aligned16(ws) || ws_bytes < kWorkspaceHeader) return MOE_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  const int El = E / R;
  {
    ProfScope prof("ep_recv_layout", st);
    const int rc = launch_pdl(ep_recv_layout_kernel, R * El, kThreads, 0, st, 1, counts_local,
                              recv_counts, R, El, splits, local_offsets, regroup_index,
                              static_cast<long long>(capacity), static_cast<int*>(ws));
    if (rc) return rc;
  }
  if (host_splits) {
    const cudaError_t e = cudaMemcpyAsync(host_splits, splits, sizeof(int32_t) * 2 * R,
                                          cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) { set_last_cuda_error(e); return MOE_ERR_CUDA; }
  }
  return check_launch();
}

extern "C" int moe_dispatch_slice(const moe_bf16* x, int T, int d, int K, const int32_t* inv_perm,
                                  const int32_t* offsets, int E, int e_lo, int e_hi, moe_bf16* xs,
                                  int32_t* local_offsets, void* stream) {
  using namespace moe;
  if (!slice_ok(T, K, d, E, e_lo, e_hi)) return MOE_ERR_INVALID_ARG;
  if (!offsets || !local_offsets || (T > 0 && (!x || !inv_perm || !xs))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(local_offsets) || (T > 0 && (!aligned16(x) || !aligned16(inv_perm) || !aligned16(xs))))
    return MOE_ERR_MISALIGNED;
  const int nv = d / 8;
  const long long total = static_cast<long long>(T) * nv;
  const int grid = grid_for(total, kThreads, 32);
  cudaStream_t st = as_stream(stream);
  const Window win{offsets, e_lo, e_hi};
  ProfScope prof("dispatch_slice", st);
  auto xi = reinterpret_cast<const uint4*>(x);
  auto o = reinterpret_cast<uint4*>(xs);
  auto go = [&](auto kern) {
    return launch_pdl(kern, grid, kThreads, 0, st, 1, xi, inv_perm, K, nv, total, win, o,
                      local_offsets);
  };
  if (K <= 2) return go(dispatch_slice_kernel<2>);
  if (K <= 4) return go(dispatch_slice_kernel<4>);
  if (K <= 8) return go(dispatch_slice_kernel<8>);
  if (K <= 16) return go(dispatch_slice_kernel<16>);
  return go(dispatch_slice_kernel<32>);
}


extern "C" int moe_combine_slice(const moe_bf16* y_local, const float* topk_w,
                                 const int32_t* inv_perm, const int32_t* offsets, int E, int e_lo,
                                 int e_hi, int T, int K, int d, float* out_partial, void* stream) {
  using namespace moe;
  if (!slice_ok(T, K, d, E, e_lo, e_hi)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y_local || !topk_w || !inv_perm || !offsets || !out_partial) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_local) || !aligned16(topk_w) || !aligned16(inv_perm) || !aligned16(out_partial))
    return MOE_ERR_MISALIGNED;
  return launch_gather_sum_slice("combine_slice", y_local, topk_w, inv_perm, T, K, d, offsets,
                                 e_lo, e_hi, out_partial, as_stream(stream));
}

extern "C" int moe_dispatch_backward_slice(const moe_bf16* dxs, const int32_t* inv_perm,
                                           const int32_t* offsets, int E, int e_lo, int e_hi,
                                           int T, int K, int d, float* dx_partial, void* stream) {
  using namespace moe;
  if (!slice_ok(T, K, d, E, e_lo, e_hi)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!dxs || !inv_perm || !offsets || !dx_partial) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dxs) || !aligned16(inv_perm) || !aligned16(dx_partial)) return MOE_ERR_MISALIGNED;
  return launch_gather_sum_slice("dispatch_backward_slice", dxs, nullptr, inv_perm, T, K, d,
                                 offsets, e_lo, e_hi, dx_partial, as_stream(stream));
}

extern "C" int moe_combine_backward_slice(const moe_bf16* dout, const moe_bf16* y_local,
                                          const float* topk_w, const int32_t* inv_perm,
                                          const int32_t* offsets, int E, int e_lo, int e_hi,
                                          int T, int K, int d, moe_bf16* dy_local, float* dtopk_w,
                                          void* stream) {
  using namespace moe;
  if (!slice_ok(T, K, d, E, e_lo, e_hi)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!dout || !y_local || !topk_w || !inv_perm || !offsets || !dy_local || !dtopk_w)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(y_local) || !aligned16(topk_w) || !aligned16(inv_perm) ||
      !aligned16(dy_local) || !aligned16(dtopk_w))
    return MOE_ERR_MISALIGNED;
  const long long TK = static_cast<long long>(T) * K;
  const int per_block = kThreads / 32;
  long long blocks = (TK + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(num_sms()) * 48;
  if (blocks > cap) blocks = cap;
  cudaStream_t st = as_stream(stream);
  const Window win{offsets, e_lo, e_hi};
  ProfScope prof("combine_backward_slice", st);
  return launch_pdl(combine_backward_slice_kernel, static_cast<unsigned>(blocks), kThreads, 0, st,
                    1, reinterpret_cast<const uint4*>(dout),
                    reinterpret_cast<const uint4*>(y_local), topk_w, inv_perm, TK, K, d / 8, win,
                    reinterpret_cast<uint4*>(dy_local), dtopk_w);
}

extern "C" int moe_reduce_finish(const float* partial, const moe_bf16* extra, int T, int d,
                                 moe_bf16* out, void* stream) {
  using namespace moe;
  if (T < 0 || d <= 0 || d % 8) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!partial || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(partial) || !aligned16(out) || (extra && !aligned16(extra)))
    return MOE_ERR_MISALIGNED;
  const long long total = static_cast<long long>(T) * (d / 8);
  cudaStream_t st = as_stream(stream);
  ProfScope prof("reduce_finish", st);
  return launch_pdl(finish_kernel, grid_for(total, kThreads), kThreads, 0, st, 1,
                    reinterpret_cast<const float4*>(partial),
                    reinterpret_cast<const uint4*>(extra), total, reinterpret_cast<uint4*>(out));
}

namespace moe {
MOE_DEBUG_STATUS_READER(ep)
}  // namespace moe
