// Dispatch gather, weighted combine, and their transposes.
//
// Sources: "Three axes of Parallelism" (nanoTitan blog), section "Expert
// Parallel (EP)" -> "Producing assignments" (the [T*K, D] assignment buffer
// packed expert-major) and "Dispatch, expert computation and combine" (undo
// the packing with the saved indices, multiply each expert output by its
// router weight and sum the K outputs); modalities PR "expert parallelism for
// the Nemotron-3 Nano MoE layers", section "Design" (the index_select /
// index_copy permutation pair); SpecForge PR "expert parallelism for MoE
// drafters on the FSDP2 backend", "What this adds" (shared expert added on
// the local tokens).
//
// All kernels are HBM-bound row moves: 16-byte vector loads and stores, rows
// of d bf16 = d/8 vectors. The token-major kernels (dispatch by inv_perm, the
// two reductions) map one thread to one 16-byte vector of a token's row, so a
// warp touches 512 contiguous bytes; each thread of the reductions issues its
// K independent gathered loads before it accumulates (fp32, slot order, no
// atomics). Dispatch by perm moves whole packed rows on the bulk-copy engine.
#include <algorithm>

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

// xp[p] = x[perm[p] / K]. One warp per packed row (rows strided over the
// grid's warps); a lane issues all of its 16-byte loads of a 4 KB slice of the
// row before its stores, so each warp keeps a whole row in flight.
constexpr int kRowVecs = 8;   // 16-byte vectors per lane per pass (4 KB per warp)

__global__ void __launch_bounds__(kThreads)
dispatch_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm, int K, int nv,
                long long rows, uint4* __restrict__ xp) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (kThreads / 32);
  for (long long p = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
       p < rows; p += nwarps) {
    long long a = __ldg(perm + p);
    if (!index_ok(a >= 0 && a < rows)) a = 0;
    const long long t = a / K;
    const uint4* src = x + t * nv;
    uint4* dst = xp + p * nv;
    for (int c0 = 0; c0 < nv; c0 += 32 * kRowVecs) {
      uint4 v[kRowVecs];
#pragma unroll
      for (int u = 0; u < kRowVecs; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nv) v[u] = ldg_nc_v4(src + c);
      }
#pragma unroll
      for (int u = 0; u < kRowVecs; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nv) stg_v4(dst + c, v[u]);
      }
    }
  }
}

// xp[p] = x[perm[p] / K] on the bulk-copy engine: one thread per CTA moves
// whole rows (contiguous, 16-byte multiples) global -> shared -> global through
// a ring of kBulkSlots row buffers, loads running kBulkLag rows ahead of the
// stores. Every wait is bounded; a wait that runs out ends the CTA's loop.
constexpr int kBulkSlots = 8;
constexpr int kBulkLag = 4;

__device__ __forceinline__ bool bulk_bar_wait(uint32_t bar, uint32_t parity) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 1000000000ull) return false;
  }
}

__global__ void __launch_bounds__(32)
dispatch_bulk_kernel(const uint8_t* __restrict__ x, const int32_t* __restrict__ perm, int K,
                     int row_bytes, long long rows, uint8_t* __restrict__ xp) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t bars[kBulkSlots];
  if (threadIdx.x != 0) return;
  const uint32_t ring_addr = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const uint32_t bar_addr = static_cast<uint32_t>(__cvta_generic_to_shared(bars));
  for (int s = 0; s < kBulkSlots; ++s)
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_addr + 8 * s) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const long long first = blockIdx.x, step = gridDim.x;
  const long long n = (rows > first) ? (rows - first + step - 1) / step : 0;
  long long loaded = 0, stored = 0;   // rows whose load was issued / whose store was issued
  for (long long i = 0; i < n + kBulkLag; ++i) {
    if (i < n) {   // load row i into slot i % kBulkSlots
      const int slot = static_cast<int>(i % kBulkSlots);
      if (i >= kBulkSlots)   // the store of row i - kBulkSlots has read this slot
        asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kBulkSlots - kBulkLag - 1) : "memory");
      const long long p = first + i * step;
      long long a = __ldg(perm + p);
      if (!index_ok(a >= 0 && a < rows)) a = 0;
      const long long t = a / K;
      const uint32_t bar = bar_addr + 8 * slot;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                   "r"(row_bytes)
                   : "memory");
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
              "r"(ring_addr + slot * row_bytes),
          "l"(x + t * row_bytes), "r"(row_bytes), "r"(bar)
          : "memory");
      loaded = i + 1;
    }
    const long long j = i - kBulkLag;
    if (j >= 0 && j < n) {   // store row j once it has landed
      const int slot = static_cast<int>(j % kBulkSlots);
      if (!bulk_bar_wait(bar_addr + 8 * slot, static_cast<uint32_t>((j / kBulkSlots) & 1))) break;
      const long long p = first + j * step;
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                       xp + p * row_bytes),
                   "r"(ring_addr + slot * row_bytes), "r"(row_bytes)
                   : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      stored = j + 1;
    }
  }
  // loads that were issued but never stored (only after a wait ran out) must land first
  for (long long r = stored; r < loaded; ++r)
    bulk_bar_wait(bar_addr + 8 * static_cast<int>(r % kBulkSlots),
                  static_cast<uint32_t>((r / kBulkSlots) & 1));
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// xp[inv_perm[a]] = x[a / K] for every assignment a = t*K + j: the rows of the
// gather above, moved token-major. One thread per 16-byte vector of a token's
// row loads it once (a warp reads 512 contiguous bytes of x) and stores it into
// the token's K packed rows; the K positions are loaded first so the K stores
// issue back to back. x is read from HBM once instead of once per assignment,
// and within each expert's segment the stores advance row by row (a segment
// lists its tokens in ascending order).
template <int KMAX>
__global__ void __launch_bounds__(kThreads)
dispatch_scatter_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv_perm, int K,
                        int nv, long long total, uint4* __restrict__ xp) {
  pdl_enter();
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += stride) {
    const long long t = i / nv;
    const int c = static_cast<int>(i - t * nv);
    const int32_t* ip = inv_perm + t * K;
    int32_t pos[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K) pos[j] = __ldg(ip + j);
    const uint4 v = ldg_nc_v4(x + i);
    const long long rows = (total / nv) * K;
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < K && index_ok(pos[j] >= 0 && pos[j] < rows))
        stg_v4(xp + static_cast<long long>(pos[j]) * nv + c, v);
  }
}

// out[t] = bf16( sum_j w[t,j] * rows[inv_perm[t*K+j]] + extra[t] ); w == nullptr means 1.
template <int KMAX>
__global__ void __launch_bounds__(kThreads)
gather_sum_kernel(const uint4* __restrict__ rows, const float* __restrict__ w,
                  const int32_t* __restrict__ inv_perm, int K, int nv, long long total,
                  const uint4* __restrict__ extra, uint4* __restrict__ out) {
  pdl_enter();
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += stride) {
    const long long t = i / nv;
    const int c = static_cast<int>(i - t * nv);
    const int32_t* ip = inv_perm + t * K;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    uint4 v[KMAX];
    const long long nrows = (total / nv) * K;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < K) {
        long long pj = __ldg(ip + j);
        if (!index_ok(pj >= 0 && pj < nrows)) pj = 0;
        v[j] = ldg_nc_v4(rows + pj * nv + c);
      }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < K) {
        const float wj = w ? __ldg(w + t * K + j) : 1.f;
        float f[8];
        unpack8(v[j], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(wj, f[q], acc[q]);
      }
    }
    if (extra) {
      float f[8];
      unpack8(ldg_nc_v4(extra + i), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += f[q];
    }
    stg_v4(out + i, pack8(acc));
  }
}

// One warp per assignment a = t*K + j (p = inv_perm[a]): dy[p] = bf16(w[a] *
// dout[t]) and dw[a] = <dout[t], y[p]>. Each lane walks its 16-byte columns
// c = lane, lane+32, ... in order, with kUnroll columns' loads in flight before
// it computes, so the dot product sums in a fixed order; the K warps of a
// token run next to each other and share dout[t] through the caches. dy is
// the exact product rounded once, so it is bit-identical to any correctly
// rounded evaluation. 64 registers per thread: four 256-thread blocks (32
// warps) per SM, each warp with 4 KB of loads in flight.
constexpr int kCbUnroll = 4;

__global__ void __launch_bounds__(kThreads)
combine_backward_kernel(const uint4* __restrict__ dout, const uint4* __restrict__ y,
                        const float* __restrict__ w, const int32_t* __restrict__ inv_perm,
                        long long TK, int K, int nv, uint4* __restrict__ dy,
                        float* __restrict__ dw) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kThreads / 32);
  for (long long a = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
       a < TK; a += warps) {
    const long long t = a / K;
    const uint4* drow = dout + t * nv;
    const int pa = __ldg(inv_perm + a);
    if (!index_ok(pa >= 0 && pa < TK)) {   // debug builds: nothing is read or written for it
      if (lane == 0) dw[a] = 0.f;
      continue;
    }
    const long long prow = static_cast<long long>(pa) * nv;
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

int launch_gather_sum(const void* rows, const float* w, const int32_t* inv_perm, int T, int K,
                      int d, const void* extra, void* out, cudaStream_t st) {
  const int nv = d / 8;
  const long long total = static_cast<long long>(T) * nv;
  const int grid = grid_for(total, kThreads);
  auto r = static_cast<const uint4*>(rows);
  auto x = static_cast<const uint4*>(extra);
  auto o = static_cast<uint4*>(out);
  ProfScope prof(w ? "combine" : "dispatch_backward", st);
  auto go = [&](auto kern) {
    return launch_pdl(kern, grid, kThreads, 0, st, 1, r, w, inv_perm, K, nv, total, x, o);
  };
  if (K <= 2) return go(gather_sum_kernel<2>);
  if (K <= 4) return go(gather_sum_kernel<4>);
  if (K <= 8) return go(gather_sum_kernel<8>);
  if (K <= 16) return go(gather_sum_kernel<16>);
  return go(gather_sum_kernel<32>);
}

int launch_dispatch_scatter(const void* x, const int32_t* inv_perm, int T, int K, int d, void* xp,
                            cudaStream_t st) {
  const int nv = d / 8;
  const long long total = static_cast<long long>(T) * nv;
  // 32 blocks per SM of grid-stride work: measured ~5% faster than 8 or 16 on
  // the qwen3 shape (more stores in flight per SM)
  const int grid = grid_for(total, kThreads, 32);
  auto xi = static_cast<const uint4*>(x);
  auto o = static_cast<uint4*>(xp);
  ProfScope prof("dispatch", st);
  auto go = [&](auto kern) {
    return launch_pdl(kern, grid, kThreads, 0, st, 1, xi, inv_perm, K, nv, total, o);
  };
  if (K <= 2) return go(dispatch_scatter_kernel<2>);
  if (K <= 4) return go(dispatch_scatter_kernel<4>);
  if (K <= 8) return go(dispatch_scatter_kernel<8>);
  if (K <= 16) return go(dispatch_scatter_kernel<16>);
  return go(dispatch_scatter_kernel<32>);
}

bool shape_ok(int T, int K, int d) { return T >= 0 && K >= 1 && K <= 32 && d > 0 && d % 8 == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_dispatch(const moe_bf16* x, int T, int d, int K, const int32_t* perm,
                            moe_bf16* xp, void* stream) {
  using namespace moe;
  if (!shape_ok(T, K, d)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !perm || !xp) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(perm) || !aligned16(xp)) return MOE_ERR_MISALIGNED;
  const long long rows = static_cast<long long>(T) * K;
  const int row_bytes = d * 2;
  const size_t ring = static_cast<size_t>(kBulkSlots) * row_bytes;
  cudaStream_t st = as_stream(stream);
  if (ring <= 96 * 1024) {
    static thread_local int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured != dev) {
      cudaFuncSetAttribute(dispatch_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           96 * 1024);
      configured = dev;
    }
    // enough CTAs that each SM keeps several rings busy
    const int per_sm = static_cast<int>(std::min<size_t>(8, (200 * 1024) / (ring + 1024)));
    long long grid = static_cast<long long>(num_sms()) * (per_sm > 0 ? per_sm : 1);
    if (grid > rows) grid = rows;
    ProfScope prof("dispatch", st);
    return launch_pdl(dispatch_bulk_kernel, static_cast<unsigned>(grid), 32, ring, st, 1,
                      reinterpret_cast<const uint8_t*>(x), perm, K, row_bytes, rows,
                      reinterpret_cast<uint8_t*>(xp));
  }
  const int nv = d / 8;
  const int grid = grid_for(rows, kThreads / 32);
  ProfScope prof("dispatch", st);
  return launch_pdl(dispatch_kernel, grid, kThreads, 0, st, 1, reinterpret_cast<const uint4*>(x),
                    perm, K, nv, rows, reinterpret_cast<uint4*>(xp));
}

extern "C" int moe_dispatch_scatter(const moe_bf16* x, int T, int d, int K,
                                    const int32_t* inv_perm, moe_bf16* xp, void* stream) {
  using namespace moe;
  if (!shape_ok(T, K, d)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !inv_perm || !xp) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(inv_perm) || !aligned16(xp)) return MOE_ERR_MISALIGNED;
  return launch_dispatch_scatter(x, inv_perm, T, K, d, xp, as_stream(stream));
}

extern "C" int moe_combine(const moe_bf16* y, const float* topk_w, const int32_t* inv_perm, int T,
                           int K, int d, const moe_bf16* shared_y, moe_bf16* out, void* stream) {
  using namespace moe;
  if (!shape_ok(T, K, d)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !topk_w || !inv_perm || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(topk_w) || !aligned16(inv_perm) || !aligned16(out) ||
      (shared_y && !aligned16(shared_y)))
    return MOE_ERR_MISALIGNED;
  return launch_gather_sum(y, topk_w, inv_perm, T, K, d, shared_y, out, as_stream(stream));
}

extern "C" int moe_dispatch_backward(const moe_bf16* dxp, const int32_t* inv_perm, int T, int K,
                                     int d, const moe_bf16* dx_shared, moe_bf16* dx,
                                     void* stream) {
  using namespace moe;
  if (!shape_ok(T, K, d)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!dxp || !inv_perm || !dx) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dxp) || !aligned16(inv_perm) || !aligned16(dx) ||
      (dx_shared && !aligned16(dx_shared)))
    return MOE_ERR_MISALIGNED;
  return launch_gather_sum(dxp, nullptr, inv_perm, T, K, d, dx_shared, dx, as_stream(stream));
}

extern "C" int moe_combine_backward(const moe_bf16* dout, const moe_bf16* y, const float* topk_w,
                                    const int32_t* inv_perm, int T, int K, int d, moe_bf16* dy,
                                    float* dtopk_w, void* stream) {
  using namespace moe;
  if (!shape_ok(T, K, d)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!dout || !y || !topk_w || !inv_perm || !dy || !dtopk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(y) || !aligned16(topk_w) || !aligned16(inv_perm) ||
      !aligned16(dy) || !aligned16(dtopk_w))
    return MOE_ERR_MISALIGNED;
  const long long TK = static_cast<long long>(T) * K;
  const int per_block = kThreads / 32;
  long long blocks = (TK + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(num_sms()) * 48;
  if (blocks > cap) blocks = cap;
  ProfScope prof("combine_backward", as_stream(stream));
  return launch_pdl(combine_backward_kernel, static_cast<unsigned>(blocks), kThreads, 0,
                    as_stream(stream), 1, reinterpret_cast<const uint4*>(dout),
                    reinterpret_cast<const uint4*>(y), topk_w, inv_perm, TK, K, d / 8,
                    reinterpret_cast<uint4*>(dy), dtopk_w);
}

namespace moe {
MOE_DEBUG_STATUS_READER(gather)
}  // namespace moe
