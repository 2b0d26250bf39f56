// Grouped SwiGLU expert GEMMs on the 5th-generation tensor cores (tcgen05,
// accumulators in TMEM, operands staged by TMA), forward and backward.
//
// Source: "Three axes of Parallelism" (nanoTitan blog), section "Expert
// Parallel (EP)": the stacked expert weights W_gate [E,d,I], W_val [E,d,I],
// W_out [E,I,d] ("Mapping experts to EP ranks"); with each expert's rows
// contiguous, expert computation is E independent MLPs ("Dispatch, expert
// computation and combine"); expert gradients stay with their expert
// ("EP backward pass"). SpecForge PR "expert parallelism for MoE drafters on
// the FSDP2 backend" names a grouped_mm backend over expert-sorted rows; that
// is prior art, this is an independent kernel.
//
// Kernel shape (two templates, six problem kinds, all on CTA pairs):
//   * every GEMM runs on clusters of two CTAs sharing one tcgen05 MMA of
//     M = 256 (cta_group::2): each CTA stages its 128 rows of A and half of
//     B's N, the leader issues the MMA, and each CTA's TMEM holds its own 128
//     rows of the accumulator;
//   * persistent: one cluster per SM pair, static round-robin over a tile list
//     that every CTA derives on device from the expert offsets (no host sync);
//   * 192 threads, warp-specialised: warp 0 issues TMA loads into a ring of
//     shared-memory stages (completing on the leader's barrier), warp 1 owns
//     TMEM and, in the leader, issues tcgen05.mma (one thread), warps 2-5 drain
//     the accumulator with tcgen05.ld and run the fused epilogue (SwiGLU,
//     SwiGLU backward, bf16 or fp32 stores through TMA bulk tensor stores);
//   * 256 x BN x 64 pair tiles (BN = 256 or 128 for the forward and
//     input-gradient kinds, 256 for the weight gradients), fp32 accumulators
//     double-buffered in TMEM so the epilogue of tile i overlaps the MMAs of
//     tile i+1; the ring depth grows when the expert count leaves shared
//     memory for it;
//   * d and I are any multiples of 8: the weights are 3-D tensor maps
//     [E][rows][cols] and [G | U], [dG | dU] are read and written through maps
//     of their halves, so K and N tails read zeros and bulk stores clip at the
//     edges (no padding, no copies);
//   * operands use the 128-byte swizzle. K-major tiles come from row-major
//     activations and from the weights in the backward; MN-major tiles from
//     the weights in the forward and from both operands of the weight
//     gradients, so no operand is ever transposed in memory;
//   * ragged segments: forward / input-gradient tiles start at an expert's
//     first row and mask stores past its last row; the weight gradients run a
//     ragged K loop over the expert's rows, issue only the K16 steps that hold
//     valid rows and take the one step that straddles the expert's end from a
//     zero-padded copy (written by the dH launch), so rows of the next expert
//     never enter the product;
//   * each GEMM waits on its producer through programmatic dependent launch
//     before it reads the expert offsets;
//   * every mbarrier wait is bounded (a few seconds of %globaltimer); on
//     timeout the CTA records MOE_ERR_DEVICE_TIMEOUT in the workspace status
//     word, drains its own TMA loads and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <type_traits>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "mxfp8.cuh"

namespace moe {
namespace gemm {

enum Kind : int {
  FWD_GATEUP = 0,  // [G|U] = X [Wg|Wu]; epilogue H = silu(G)*U (+ save GU)
  FWD_DOWN = 1,    // Y = H Wd
  BWD_DH = 2,      // dH = dY Wd^T; epilogue dG, dU from saved GU
  BWD_DX = 3,      // dX = [dG|dU] [Wg|Wu]^T
  WGRAD_GU = 4,    // [dWg|dWu] = X^T [dG|dU]   (ragged K)
  WGRAD_D = 5      // dWd = H^T dY              (ragged K)
};

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
constexpr unsigned long long kTimeoutNs = 4000000000ull;

// One zero-padded straddling step to prepare for the weight gradients: for each
// expert whose row count is not a multiple of 16, the 16-row step that holds its
// last rows, rows past the expert set to zero (a [M, C] bf16 -> pad [E, 16, C]).
struct PadJob {
  const __nv_bfloat16* a;
  __nv_bfloat16* pad;
  int C;
};

// The backward's data part leaves [dG | dU] and the padded straddling steps in
// the workspace for the weight part. It records what they were computed for in
// the workspace header (words kTagFirst.. after the status word); the weight
// part's kernels compare that record with their own arguments and, on a
// mismatch (no data part on this workspace, other sizes or other offsets),
// report MOE_ERR_DEVICE_CHECK and compute nothing.
constexpr int kTagNone = 0, kTagWrite = 1, kTagCheck = 2;
constexpr int kTagWords = 6;
constexpr int kTagFirst = 4;                  // int32 index in the workspace header
constexpr uint32_t kTagMagic = 0x4D6F4542u;

struct Params {
  const int32_t* offsets;  // [E+1] expert row offsets (device)
  int E;
  int M;                   // rows of the packed activations
  int d;
  int I;
  int n_tiles;             // tiles along N
  int m_tiles;             // weight gradients: 256-row tile pairs along M (dW rows d or I)
  int k_blocks;            // forward / input gradients: k-blocks of K (64 bf16 or 128 E4M3)
  int nt_half;             // gate/up weight gradients: n-tiles of each of dWg and dWu
  __nv_bfloat16* out;      // h, y, dgu or dxp
  __nv_bfloat16* out2;     // gu (forward, may be null)
  const __nv_bfloat16* aux;  // gu (BWD_DH)
  float* outf0;            // dWg / dWd
  float* outf1;            // dWu
  int ld_out;              // row length of `out` in elements
  int* status;             // workspace status word
  PadJob pad[2];           // BWD_DH: the weight gradients' pads of X and H (a == null: none)
  int kb_half;             // BWD_DX: k-blocks of the dG half of K (then as many of the dU half)
  int tag_mode;            // kTagNone, kTagWrite (data part's dH) or kTagCheck (weight part)
  uint32_t tag[kTagWords]; // the backward's scratch tag: magic, M, E, d, I, offsets (low 32 bits)
  uint8_t* hq;             // MXFP8 gate/up: E4M3 of H for the down projection (null: not fused)
  uint8_t* hsf;            //   and H's scale atoms (row tiles in the tile list's m-tile order)
};

// ----------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `bar` with the given parity to complete.
// Returns false if this CTA is aborting (another role timed out) or the wait
// itself ran past kTimeoutNs (then it raises the abort flag and the status).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            volatile int* abort_flag, int* status,
                                            uint64_t timeout_ns = kTimeoutNs) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > timeout_ns) {
        *abort_flag = 1;
        report_status(status, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// Fast path inline (the phase is usually complete already), slow path out of line.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
  if (mbar_try(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, status);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i gets row (lane base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Bulk tensor store shared -> global (2-D tile), tracked by this thread's bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// At most one of this thread's committed bulk store groups is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// This thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory accesses with later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- CTA-pair (cluster of two, tcgen05 cta_group::2) helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t n_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}
// The same over a 3-D map [E][rows][cols] (x = column, y = row, z = expert):
// rows and columns past the expert's extent read the fill value (zero).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
      : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]^T, M = 256.
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at this offset in both CTAs when this thread's MMAs complete.
__device__ __forceinline__ void tc_commit_pair_both(uint32_t bar) {
  const uint16_t mask = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16: fp32 D, bf16 A and B, M rows (128, or 256 for a pair).
template <int N, bool A_MN, bool B_MN, int M = BM>
__host__ __device__ constexpr uint32_t make_idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((A_MN ? 1u : 0u) << 15) |
         ((B_MN ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor for kind::mxf8f6f4 with block scaling: fp32 D, E4M3 A and
// B (both K-major), UE8M0 scale factors, M rows (256 for a pair). The scale
// factor ids (which byte of each 32-bit scale column a K32 step uses) are
// or-ed in per step: bits 4-5 for B, 29-30 for A.
template <int N, int M>
__host__ __device__ constexpr uint32_t make_idesc_mxf8() {
  return (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t mx_sf_ids(uint32_t a_id, uint32_t b_id) {
  return (b_id << 4) | (a_id << 29);
}

// D[tmem of both CTAs] (+)= (A * 2^SFA) (B * 2^SFB)^T with E4M3 operands and one
// UE8M0 scale per 32 K for every row of A and of B, M = 256 over the pair.
__device__ __forceinline__ void tc_mma_pair_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t sfa_tmem,
                                               uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4],"
      " [%5], p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared memory -> TMEM of both CTAs of the pair (each from its own shared
// memory): a 32 x 128-bit block (512 B, rows 16 B apart) to lanes 0-31 of four
// consecutive columns, repeated in the other three lane quarters.
__device__ __forceinline__ void tc_cp_pair_32x128(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Shared-memory descriptor of an unswizzled block of 16-byte rows (8-row core
// matrices 128 B apart), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_rows16(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// silu(g) = g * sigmoid(g) with the fast exponential and reciprocal: a few
// ulp of fp32, far below the bf16 rounding of H. For g < -87 the denominator
// overflows and the quotient is 0, the limit of silu.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// nvalid: the row's columns left from dst (a multiple of 8); 8-column chunks
// past it are not written.
__device__ __forceinline__ void store16_bf16(__nv_bfloat16* dst, const float (&v)[16], int nvalid) {
  uint4 a, b;
  a.x = pack_bf16(v[0], v[1]);   a.y = pack_bf16(v[2], v[3]);
  a.z = pack_bf16(v[4], v[5]);   a.w = pack_bf16(v[6], v[7]);
  b.x = pack_bf16(v[8], v[9]);   b.y = pack_bf16(v[10], v[11]);
  b.z = pack_bf16(v[12], v[13]); b.w = pack_bf16(v[14], v[15]);
  uint4* p = reinterpret_cast<uint4*>(dst);
  if (nvalid > 0) p[0] = a;
  if (nvalid > 8) p[1] = b;
}

// Debug builds: the expert offsets the tile scheduler decodes must start at 0,
// never decrease and end within the M rows; otherwise the kernel records
// MOE_ERR_DEVICE_CHECK in the workspace status word and takes no tile. Every
// thread of the block calls it (it ends with a block-wide vote). Release builds:
// always true.
__device__ __forceinline__ bool offsets_ok(const int* s_off, const Params& p) {
#ifdef MOE_DEBUG_CHECKS
  bool ok = true;
  for (int e = threadIdx.x; e < p.E; e += kThreads) ok = ok && s_off[e] <= s_off[e + 1];
  if (threadIdx.x == 0) ok = ok && s_off[0] == 0 && s_off[p.E] <= p.M;
  ok = __syncthreads_and(ok) != 0;
  if (!ok && threadIdx.x == 0) report_status(p.status, MOE_ERR_DEVICE_CHECK);
  index_ok(ok);
  return ok;
#else
  (void)s_off;
  (void)p;
  return true;
#endif
}

// ----------------------------------------------------------------- CTA-pair kernel
// Forward and input-gradient kinds on a cluster of two CTAs that share one
// tcgen05 MMA of M = 256 (cta_group::2): each CTA holds 128 rows of A and half
// of B's N in its own shared memory, the leader (cluster rank 0) issues the
// MMA, and each CTA's TMEM receives its own 128 rows of the 256 x BN
// accumulator. Per CTA a k-block stage is 32 KB for 276 ns of MMA work (half
// the bytes of a single-CTA 128 x 256 tile), so six stages hide 1.4 us of
// load latency.
//
// Tiles pair two 128-row m-tiles of the same expert (the second may be past
// the expert's end and then stores nothing), times BN-wide n-tiles.
struct PTile {
  int e;
  int row0;   // this CTA's first packed row
  int rows;   // this CTA's valid rows (<= 0: none)
  int n0;
  int mg;     // the tile's pair index in the expert-ordered list of m-tile pairs
};

template <int KIND, int BN>
__device__ __forceinline__ PTile decode_pair(int t, int rank, const Params& p, const int* s_off,
                                             const int* s_mp) {
  PTile tl;
  const int mg = t / p.n_tiles;
  const int nt = t - mg * p.n_tiles;
  int lo = 0, hi = p.E - 1;   // largest e with s_mp[e] <= mg
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_mp[mid] <= mg) lo = mid; else hi = mid - 1;
  }
  tl.e = lo;
  tl.mg = mg;
  tl.row0 = s_off[lo] + (2 * (mg - s_mp[lo]) + rank) * BM;
  tl.rows = min(BM, s_off[lo + 1] - tl.row0);
  tl.n0 = nt * (KIND == FWD_GATEUP ? BN / 2 : BN);
  return tl;
}

// This CTA's boxes of one k-block: its 128 A rows and its half of B (gate or up
// for the gate/up GEMM), counted on the leader's full barrier.
template <int KIND, int BN>
__device__ __forceinline__ void issue_pair(const PTile& tl, int kb, uint32_t rank, const Params& p,
                                           const CUtensorMap* tmA, const CUtensorMap* tmA2,
                                           const CUtensorMap* tmB0, const CUtensorMap* tmB1,
                                           uint32_t sa, uint32_t sb, uint32_t fb) {
  constexpr uint32_t MN_ATOM = 64 * 128;
  constexpr int HB = BN / 2;
  // The weights are 3-D maps [E][rows][cols]: a box past the expert's rows or
  // columns reads zeros, so K and N tails need no masking.
  if constexpr (KIND == BWD_DX) {
    // K = [dG | dU]: the dG half's k-blocks, then the dU half's, each from its
    // own half map (so no k-block mixes the two halves) with Wg or Wu
    const bool up = kb >= p.kb_half;
    const int kx = (up ? kb - p.kb_half : kb) * BK;
    tma_load_2d_pair(sa, up ? tmA2 : tmA, fb, kx, tl.row0);
    tma_load_3d_pair(sb, up ? tmB1 : tmB0, fb, kx, tl.n0 + static_cast<int>(rank) * HB, tl.e);
    return;
  }
  tma_load_2d_pair(sa, tmA, fb, kb * BK, tl.row0);
  if constexpr (KIND == FWD_GATEUP) {
    const CUtensorMap* m = rank ? tmB1 : tmB0;
#pragma unroll
    for (int i = 0; i < HB / 64; ++i)
      tma_load_3d_pair(sb + i * MN_ATOM, m, fb, tl.n0 + 64 * i, kb * BK, tl.e);
  } else if constexpr (KIND == FWD_DOWN) {
#pragma unroll
    for (int i = 0; i < HB / 64; ++i)
      tma_load_3d_pair(sb + i * MN_ATOM, tmB0, fb, tl.n0 + static_cast<int>(rank) * HB + 64 * i,
                       kb * BK, tl.e);
  } else {  // BWD_DH
    tma_load_3d_pair(sb, tmB0, fb, kb * BK, tl.n0 + static_cast<int>(rank) * HB, tl.e);
  }
}

// Fills pad[e] of one PadJob (see PadJob) with nthreads threads numbered tid,
// each with up to kPadVec 16-byte loads in flight. s_off: the expert offsets.
constexpr int kPadVec = 8;

__device__ __forceinline__ void pad_straddle_step(const int* s_off, const PadJob& j, int e, int tid,
                                                  int nthreads) {
  const int r0 = s_off[e];
  const int rows = s_off[e + 1] - r0;
  const int v = rows & 15;
  if (v == 0) return;
  const int nv = j.C / 8;          // 16-byte vectors per row
  const int total = 16 * nv;       // vectors of the 16-row step
  const uint4* src = reinterpret_cast<const uint4*>(j.a + static_cast<size_t>(r0 + (rows & ~15)) * j.C);
  uint4* dst = reinterpret_cast<uint4*>(j.pad + static_cast<size_t>(e) * 16 * j.C);
  for (int base = tid; base < total; base += nthreads * kPadVec) {
    uint4 x[kPadVec];
#pragma unroll
    for (int u = 0; u < kPadVec; ++u) {
      const int i = base + u * nthreads;
      x[u] = (i < total && i / nv < v) ? ldg_nc_v4(src + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kPadVec; ++u) {
      const int i = base + u * nthreads;
      if (i < total) dst[i] = x[u];
    }
  }
}

// Pair-kernel epilogue shared memory: per epilogue warp two [32 rows x 64
// columns] 128-byte-swizzled bf16 boxes: alternating bulk-store staging
// (gate/up streams H, G and U through them in turn), and for dh the G and U
// prefetch boxes, which the dG/dU results overwrite before their store.
template <int KIND>
__host__ __device__ constexpr uint32_t pair_epi_bytes() {
  return 4u * 2u * 4096u;
}

// Writes 32 consecutive columns (values v) of this lane's row into a
// [32 rows x 64 bf16] box with 128-byte swizzle, at 16-byte chunk j0 .. j0+3.
__device__ __forceinline__ void stage_row32(uint8_t* box, int lane, int j0, const float (&v)[32]) {
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int off = lane * 128 + (((j0 + jj) ^ (lane & 7)) << 4);
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = v[8 * jj + i];
    *reinterpret_cast<uint4*>(box + off) = pack8(f);
  }
}

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const float (&v)[32], int nvalid) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = v[8 * jj + i];
    if (8 * jj < nvalid) p[jj] = pack8(f);
  }
}

// One K32 block of H for the MXFP8 down projection: the values rounded to bf16
// (as H is stored), their amax and power-of-two scale, and the 32 E4M3 bytes
// (the row quantizer's arithmetic, element for element). Returns X (the byte
// stored is X + 127).
__device__ __forceinline__ int quantize_row32(const float (&h)[32], uint4 (&q)[2]) {
  float hb[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    hb[i] = __bfloat162float(__float2bfloat16_rn(h[i]));
    amax = fmaxf(amax, fabsf(hb[i]));
  }
  const int X = mx_exponent(amax);
  const float sc = inv_pow2(X);
  uint32_t* w = reinterpret_cast<uint32_t*>(q);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = to_e4m3x4(hb[4 * i] * sc, hb[4 * i + 1] * sc, hb[4 * i + 2] * sc, hb[4 * i + 3] * sc);
  return X;
}

// FP8 = true: the forward kinds on MXFP8 operands (E4M3 elements, one UE8M0
// scale per 32 K; tcgen05.mma kind::mxf8f6f4 with block scaling). A k-block is
// then 128 K (the same 128-byte rows), B is K-major (the weights are quantized
// into a transposed layout, gate and up interleaved in 128-row blocks), and each
// stage also carries one 512-byte scale atom for the CTA's 128 A rows (tmB1)
// and one per 128 of the pair's B columns (tmS): 128 rows x 4 K32 scales, row r
// at byte (r % 32) * 16 + (r / 32) * 4 + k. The MMA thread copies both atoms
// into TMEM (tcgen05.cp, 32 x 128 bit repeated over the four lane quarters,
// four columns each, a column ring per stage beside the accumulators) before
// the stage's four K32 MMAs, which pick the scale byte by the descriptor's
// scale ids. The A atoms follow the m-tiles of the tile list (pair index mg:
// m-tiles 2 mg and 2 mg + 1), so the quantizer lays them out per expert.
template <int KIND, int BN, int STAGES, bool FP8 = false>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB0,
                         const __grid_constant__ CUtensorMap tmB1,
                         const __grid_constant__ CUtensorMap tmC0,
                         const __grid_constant__ CUtensorMap tmC1,
                         const __grid_constant__ CUtensorMap tmC2,
                         const __grid_constant__ CUtensorMap tmS, const Params p) {
  static_assert(KIND == FWD_GATEUP || KIND == FWD_DOWN || KIND == BWD_DH || KIND == BWD_DX,
                "pair kernel: forward and input-gradient kinds");
  static_assert(!FP8 || ((KIND == FWD_GATEUP || KIND == FWD_DOWN) && (BN == 128 || BN == 256)),
                "MXFP8: forward kinds on 256 x 128 or 256 x 256 pair tiles");
  constexpr bool B_MN = !FP8 && (KIND == FWD_GATEUP || KIND == FWD_DOWN);
  constexpr uint32_t A_BYTES = BM * BK * 2;          // 128 rows x 128 bytes (bf16 or fp8)
  constexpr uint32_t B_BYTES = (BN / 2) * BK * 2;
  constexpr uint32_t SFB_ATOMS = BN / 128;           // scale atoms of the pair's B columns
  // scale atoms per stage: the A rows' atom, then the B columns' atoms, padded to 1 KB
  constexpr uint32_t SF_BYTES = FP8 ? ((512u * (1u + SFB_ATOMS) + 1023u) & ~1023u) : 0u;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
  // Two accumulator buffers: the epilogue of tile i overlaps the MMAs of tile
  // i + 1. MXFP8 keeps its per-stage scale ring in TMEM too: beside the two
  // buffers for 256 x 128 tiles; for 256 x 256 tiles (the two buffers fill all
  // 512 columns) in the first 64 columns of the buffer the previous tile
  // accumulated into (RING_SWAP): tile i's MMAs start once tile i - 1's
  // epilogue has read those columns (its first 64-column step, which signals
  // ring_free), and tile i's own accumulator region held tile i - 1's ring,
  // whose MMAs completed before that epilogue began.
  constexpr int NACC = 2;
  constexpr bool RING_SWAP = FP8 && BN == 256;
  constexpr uint32_t TMEM_COLS = FP8 ? 512u : 2u * BN;
  constexpr uint32_t SF_COLS = 4u * (1u + SFB_ATOMS);   // TMEM columns of one stage's scales
  constexpr uint32_t SF_COL0 = static_cast<uint32_t>(NACC) * BN;
  static_assert(!FP8 || RING_SWAP || SF_COL0 + SF_COLS * STAGES <= TMEM_COLS,
                "MXFP8 scale ring in TMEM");
  static_assert(!RING_SWAP || SF_COLS * STAGES <= 64, "MXFP8 scale ring in a drained step");
  constexpr uint32_t IDESC = FP8 ? make_idesc_mxf8<BN, 2 * BM>() : make_idesc<BN, false, B_MN, 2 * BM>();
  constexpr uint32_t MN_ATOM = 64 * 128;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* epi = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + pair_epi_bytes<KIND>());
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, aux[4], ring_free[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_mp = s_off + (p.E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = (rank == 0);
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 4);
  auto aux_bar = [&](int w) { return bar_base + 8u * (2 * STAGES + 5 + w); };
  auto ring_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 9 + a); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    // the leader's accumulator-empty (and ring-free) barriers collect the four
    // epilogue warps of both CTAs
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);
      mbar_init(ring_bar(a), 8);
    }
    mbar_init(drain_bar, 1);
    for (int w = 0; w < 4; ++w) mbar_init(aux_bar(w), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB1)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmC0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmC1)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmC2)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmS)) : "memory");
  }
  if (warp == 1) {   // one warp in each CTA of the pair allocates collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  pdl_wait();   // offsets and operands come from earlier launches
  pdl_launch_dependents();
  if (p.tag_mode == kTagWrite && blockIdx.x == 0 && threadIdx.x < kTagWords)
    reinterpret_cast<uint32_t*>(p.status)[kTagFirst + threadIdx.x] = p.tag[threadIdx.x];
  for (int e = threadIdx.x; e <= p.E; e += kThreads) s_off[e] = __ldg(p.offsets + e);
  __syncthreads();
  const bool offs_ok = offsets_ok(s_off, p);
  if (warp == 0) {   // exclusive prefix of per-expert m-tile pairs
    int carry = 0;
    for (int base = 0; base <= p.E; base += 32) {
      const int i = base + lane;
      const int v = (i < p.E) ? ((s_off[i + 1] - s_off[i] + BM - 1) / BM + 1) / 2 : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (i <= p.E) s_mp[i] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers exist before any remote arrive or TMA
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // both CTAs must hold the same TMEM columns for the pair's MMAs; otherwise do nothing
  uint32_t peer_base;
  asm volatile("ld.shared::cluster.u32 %0, [%1];"
               : "=r"(peer_base)
               : "r"(map_to_rank(smem_u32(tmem_slot), rank ^ 1u))
               : "memory");
  const bool tmem_ok = (peer_base == tmem_base);
  if (!tmem_ok && threadIdx.x == 0) report_status(p.status, MOE_ERR_DEVICE_CHECK);
  const int total = (tmem_ok && offs_ok) ? s_mp[p.E] * p.n_tiles : 0;
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(n_clusters_x());

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) issued[s] = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        const PTile tl = decode_pair<KIND, BN>(t, static_cast<int>(rank), p, s_off, s_mp);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          const uint32_t fb_local = full_bar(stage);
          // both CTAs' boxes (the scale area's padding is not loaded)
          if (leader)
            mbar_expect_tx(fb_local, 2 * (FP8 ? A_BYTES + B_BYTES + 512u * (1u + SFB_ATOMS)
                                              : STAGE_BYTES));
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          if constexpr (FP8) {
            // A rows, the CTA's BN / 2 B rows (gate or up for gate/up: interleaved
            // blocks), then the A rows' scale atom and the pair's B scale atoms
            const uint32_t fb = map_to_rank(fb_local, 0);
            const int nq = (KIND == FWD_GATEUP) ? 2 * p.I : p.d;    // B rows per expert
            const int nrow = (KIND == FWD_GATEUP) ? 2 * tl.n0 : tl.n0;
            tma_load_2d_pair(sa, &tmA, fb, kb * 128, tl.row0);
            tma_load_2d_pair(sa + A_BYTES, &tmB0, fb, kb * 128,
                             tl.e * nq + nrow + static_cast<int>(rank) * (BN / 2));
            tma_load_2d_pair(sa + A_BYTES + B_BYTES, &tmB1, fb, 0,
                             (2 * tl.mg + static_cast<int>(rank)) * p.k_blocks + kb);
#pragma unroll
            for (uint32_t j = 0; j < SFB_ATOMS; ++j)
              tma_load_2d_pair(sa + A_BYTES + B_BYTES + 512 * (1 + j), &tmS, fb, 0,
                               (tl.e * (nq / 128) + nrow / 128 + static_cast<int>(j)) * p.k_blocks +
                                   kb);
          } else {
            issue_pair<KIND, BN>(tl, kb, rank, p, &tmA, &tmC2, &tmB0, &tmB1, sa, sa + A_BYTES,
                                 map_to_rank(fb_local, 0));
          }
          issued[stage] += 1;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (leader) {
        // the leader's full barriers count both CTAs' loads: wait for the last phases
        for (int s = 0; s < STAGES; ++s) {
          if (!issued[s]) continue;
          const uint32_t par = (issued[s] - 1u) & 1u;
          const uint64_t t0 = globaltimer();
          while (!mbar_try(full_bar(s), par) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
      } else if (!ok) {
        // loads of this CTA may still be landing after a timeout: give them a moment
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 1000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int j = 0;   // this cluster's tile count
      for (int t = cid; t < total && ok; t += ncl, ++j) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
        if (RING_SWAP && j > 0) {
          // the previous tile's epilogue has read the columns this tile's scale ring takes
          if (!mbar_wait(ring_bar(acc ^ 1), static_cast<uint32_t>((j - 1) >> 1) & 1u, abort_flag,
                         p.status)) { ok = false; break; }
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const uint32_t ring0 = RING_SWAP ? static_cast<uint32_t>((acc ^ 1) * BN) : SF_COL0;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status)) { ok = false; break; }
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          if (lane == 0) {
            if constexpr (FP8) {
              const uint32_t t_sfa = tmem_base + ring0 + SF_COLS * static_cast<uint32_t>(stage);
              const uint32_t t_sfb = t_sfa + 4u;
              const uint32_t sf = sb + B_BYTES;
              tc_cp_pair_32x128(t_sfa, smem_desc_rows16(sf));
#pragma unroll
              for (uint32_t j = 0; j < SFB_ATOMS; ++j)
                tc_cp_pair_32x128(t_sfb + 4u * j, smem_desc_rows16(sf + 512 * (1 + j)));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {   // K32 steps of 32 bytes
                const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
                const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024);
                tc_mma_pair_mx(d_tmem, ad, bd, IDESC | mx_sf_ids(kk, kk), t_sfa, t_sfb,
                               (kb | kk) != 0 ? 1u : 0u);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
                uint64_t bd;
                if constexpr (B_MN) bd = smem_desc(sb + kk * 2048, MN_ATOM, 1024);
                else bd = smem_desc(sb + kk * 32, 16, 1024);
                tc_mma_pair(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
              }
            }
            tc_commit_pair_both(empty_bar(stage));
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) tc_commit_pair_both(tfull_bar(acc));
        __syncwarp();
        if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
      }
      if (lane == 0) {
        tc_commit_pair_local(drain_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try(drain_bar, 0) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // Each warp drains 32 accumulator rows. A slice whose 32 rows all belong to
    // the tile's expert goes out through shared-memory staging and bulk tensor
    // stores; a slice that crosses the expert's end is stored row by row, so no
    // write reaches the next expert's rows.
    const int q = warp & 3;
    const int ew = warp - 2;
    const int r = q * 32 + lane;
    if constexpr (KIND == BWD_DH) {
      // Until the first accumulator is ready these warps are idle: they prepare the
      // weight gradients' zero-padded straddling steps of X and H meanwhile.
      if (p.pad[0].a) {
        for (int job = static_cast<int>(blockIdx.x); job < 2 * p.E; job += static_cast<int>(gridDim.x))
          pad_straddle_step(s_off, p.pad[job & 1], job >> 1, threadIdx.x - 64, 128);
      }
    }
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t aux_phase = 0;
    bool aux_pending = false;
    int buf = 0;
    for (int t = cid; t < total; t += ncl) {
      const PTile tl = decode_pair<KIND, BN>(t, static_cast<int>(rank), p, s_off, s_mp);
      const bool valid = r < tl.rows;
      const size_t grow = static_cast<size_t>(tl.row0 + r);
      const int growq = tl.row0 + q * 32;          // first row of this warp's slice
      const bool full = (tl.rows - q * 32) >= 32;  // every row of the slice is valid
      if constexpr (KIND == BWD_DH) {
        // The warp's 32 rows go 64 columns at a time: G[c0,+64) and U[c0,+64) are
        // TMA-loaded into two boxes, dG and dU overwrite them in place and leave
        // through bulk stores. Four such steps per tile take well under the next
        // tile's MMA time, and the 8 KB per warp leaves room for a sixth stage.
        uint8_t* aux = epi + ew * 8192;   // boxes: G[c0,+64) then U[c0,+64)
        const uint32_t aux_addr = smem_u32(aux);
        const uint32_t ab = aux_bar(ew);
        auto request = [&](int c0) {
          if (lane == 0) {
            bulk_wait_read_all();          // earlier dG/dU stores from these boxes are done
            mbar_expect_tx(ab, 8192);
            tma_load_2d(aux_addr, &tmC0, ab, tl.n0 + c0, growq);          // G half of gu
            tma_load_2d(aux_addr + 4096, &tmS, ab, tl.n0 + c0, growq);    // U half of gu
          }
          aux_pending = true;
        };
        request(0);
        if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tacc = tmem_base + lane_addr + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        // when I % 256 != 0 the last n-tile's columns past I are neither read nor stored
        const int cend = min(BN, p.I - tl.n0);
        for (int c0 = 0; c0 < cend; c0 += 64) {
          if (c0) request(c0);
          if (!mbar_wait(ab, aux_phase, abort_flag, p.status)) { ok = false; break; }
          aux_phase ^= 1u;
          aux_pending = false;
          for (int c = 0; c < 64; c += 16) {
            float dh[16];
            tmem_ld16(tacc + c0 + c, dh);
            tmem_wait_ld();
            const int j0 = c >> 3;
            float g[16], u[16];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int off = lane * 128 + (((j0 + hh) ^ (lane & 7)) << 4);
              float f[8];
              unpack8(*reinterpret_cast<const uint4*>(aux + off), f);
#pragma unroll
              for (int i = 0; i < 8; ++i) g[8 * hh + i] = f[i];
              unpack8(*reinterpret_cast<const uint4*>(aux + 4096 + off), f);
#pragma unroll
              for (int i = 0; i < 8; ++i) u[8 * hh + i] = f[i];
            }
            float dg[16], du[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float sg = __fdividef(1.f, 1.f + __expf(-g[i]));
              dg[i] = dh[i] * u[i] * sg * (1.f + g[i] * (1.f - sg));
              du[i] = dh[i] * g[i] * sg;
            }
            if (full) {   // in place over G and U: this lane's own row chunks
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int off = lane * 128 + (((j0 + hh) ^ (lane & 7)) << 4);
                *reinterpret_cast<uint4*>(aux + off) = pack8(&dg[8 * hh]);
                *reinterpret_cast<uint4*>(aux + 4096 + off) = pack8(&du[8 * hh]);
              }
            } else if (valid) {
              __nv_bfloat16* orow = p.out + grow * (2 * p.I);
              const int left = p.I - (tl.n0 + c0 + c);
              store16_bf16(orow + tl.n0 + c0 + c, dg, left);
              store16_bf16(orow + p.I + tl.n0 + c0 + c, du, left);
            }
          }
          fence_proxy_async();
          __syncwarp();
          if (full && lane == 0) {
            tma_store_2d(&tmC1, aux_addr, tl.n0 + c0, growq);          // dG half of dgu
            tma_store_2d(&tmC2, aux_addr + 4096, tl.n0 + c0, growq);   // dU half of dgu
            bulk_commit();
          }
        }
        if (!ok) break;
      } else {
        if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tacc = tmem_base + lane_addr + static_cast<uint32_t>(acc * BN);
        // MXFP8 256 x 256: once this tile's columns [0, 64) have been read for the
        // last time (in its first 64-column step), the next tile's scale ring may
        // take them
        auto ring_free = [&]() {
          if constexpr (RING_SWAP) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(ring_bar(acc), 0));
          }
        };
        if constexpr (KIND == FWD_GATEUP) {
          // H, then (when saved) G and U leave one stream at a time through the
          // warp's two alternating [32 x 64] boxes; the accumulator is read again for
          // each stream rather than holding all three in registers, which keeps the
          // staging at 8 KB per warp and leaves shared memory for a deeper ring.
          constexpr int HALF = BN / 2;
          const int nstreams = p.out2 ? 3 : 1;
          // MXFP8: H's E4M3 copy for the down projection is written with the H
          // stream, from the same registers (fused quantization: the bf16-rounded
          // H of each K32 block, its amax, scale and elements, as the row
          // quantizer computes them; each lane stores its row's 32 bytes)
          const bool fuse_q = FP8 && p.hq != nullptr;
          const int nst = nstreams;
          const int rr = q * 32 + lane;                                // row in the CTA's m-tile
          const long long qtile = 2LL * tl.mg + static_cast<long long>(rank);
          const int cend = min(HALF, p.I - tl.n0);   // columns of the tile within I
          for (int c64 = 0; c64 < cend; c64 += 64) {
            if (!full) {   // a slice that crosses the expert's end: row-wise stores
              for (int sub = 0; sub < 64; sub += 32) {
                float g[32], u[32], h[32];
                tmem_ld32(tacc + c64 + sub, g);   // warp-wide: every lane loads
                tmem_ld32(tacc + HALF + c64 + sub, u);
                tmem_wait_ld();
                if (c64 == 0 && sub == 32) ring_free();
                if (valid) {
#pragma unroll
                  for (int i = 0; i < 32; ++i) h[i] = silu_f(g[i]) * u[i];
                  const int left = p.I - (tl.n0 + c64 + sub);
                  store32_bf16(p.out + grow * p.I + tl.n0 + c64 + sub, h, left);
                  if (p.out2) {
                    store32_bf16(p.out2 + grow * (2 * p.I) + tl.n0 + c64 + sub, g, left);
                    store32_bf16(p.out2 + grow * (2 * p.I) + p.I + tl.n0 + c64 + sub, u, left);
                  }
                  if (fuse_q) {
                    uint4 qb[2];
                    const int X = quantize_row32(h, qb);
                    uint4* dst = reinterpret_cast<uint4*>(p.hq + grow * p.I + tl.n0 + c64 + sub);
                    dst[0] = qb[0];
                    dst[1] = qb[1];
                    const int col = tl.n0 + c64 + sub;
                    p.hsf[atom_byte(qtile * (p.I / 128) + col / 128, rr, (col & 127) >> 5)] =
                        static_cast<uint8_t>(X + 127);
                  }
                }
              }
              continue;
            }
            // MXFP8 256 x 256, first step with G and U saved: H and G are staged
            // together from the same registers (both boxes), so columns [0, 64)
            // are read once and the next tile's scale ring can take them sooner
            const bool hg = RING_SWAP && c64 == 0 && nst == 3;
            if (hg) {
              uint8_t* sth = epi + ew * 8192 + buf * 4096;
              uint8_t* stg = epi + ew * 8192 + (buf ^ 1) * 4096;
              if (lane == 0) bulk_wait_read_all();   // both boxes' stores are done
              __syncwarp();
              for (int sub = 0; sub < 64; sub += 32) {
                float g[32], u[32], v[32];
                tmem_ld32(tacc + sub, g);
                tmem_ld32(tacc + HALF + sub, u);
                tmem_wait_ld();
                if (sub == 32) ring_free();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = silu_f(g[i]) * u[i];
                if (fuse_q) {
                  uint4 qb[2];
                  const int X = quantize_row32(v, qb);
                  uint4* dst = reinterpret_cast<uint4*>(p.hq + grow * p.I + tl.n0 + sub);
                  dst[0] = qb[0];
                  dst[1] = qb[1];
                  const int col = tl.n0 + sub;
                  p.hsf[atom_byte(qtile * (p.I / 128) + col / 128, rr, (col & 127) >> 5)] =
                      static_cast<uint8_t>(X + 127);
                }
                stage_row32(sth, lane, sub >> 3, v);
                stage_row32(stg, lane, sub >> 3, g);
              }
              fence_proxy_async();
              __syncwarp();
              if (lane == 0) {   // two bulk groups: H's box is the older one
                tma_store_2d(&tmC0, smem_u32(sth), tl.n0, growq);
                bulk_commit();
                tma_store_2d(&tmC1, smem_u32(stg), tl.n0, growq);
                bulk_commit();
              }
            }
            for (int sidx = hg ? 2 : 0; sidx < nst; ++sidx) {
              uint8_t* st = epi + ew * 8192 + buf * 4096;
              if (lane == 0) bulk_wait_read_1();   // the store that used this box is done
              __syncwarp();
              for (int sub = 0; sub < 64; sub += 32) {
                float v[32];
                if (sidx == 0) {
                  float g[32], u[32];
                  tmem_ld32(tacc + c64 + sub, g);
                  tmem_ld32(tacc + HALF + c64 + sub, u);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 32; ++i) v[i] = silu_f(g[i]) * u[i];
                  if (fuse_q) {
                    uint4 qb[2];
                    const int X = quantize_row32(v, qb);
                    uint4* dst = reinterpret_cast<uint4*>(p.hq + grow * p.I + tl.n0 + c64 + sub);
                    dst[0] = qb[0];
                    dst[1] = qb[1];
                    const int col = tl.n0 + c64 + sub;
                    p.hsf[atom_byte(qtile * (p.I / 128) + col / 128, rr, (col & 127) >> 5)] =
                        static_cast<uint8_t>(X + 127);
                  }
                } else {
                  tmem_ld32(tacc + (sidx == 1 ? 0 : HALF) + c64 + sub, v);
                  tmem_wait_ld();
                }
                // columns [0, 64) are last read by the G stream (H alone: the H stream)
                if (!hg && c64 == 0 && sub == 32 && sidx == (nst > 1 ? 1 : 0)) ring_free();
                stage_row32(st, lane, sub >> 3, v);
              }
              fence_proxy_async();
              __syncwarp();
              if (lane == 0) {
                // H, then the G and U halves of gu (each its own half map)
                tma_store_2d(sidx == 0 ? &tmC0 : (sidx == 1 ? &tmC1 : &tmC2), smem_u32(st),
                             tl.n0 + c64, growq);
                bulk_commit();
              }
              buf ^= 1;
            }
          }
        } else {  // FWD_DOWN, BWD_DX: one bf16 output, two staging boxes in turn
          const int cend = min(BN, p.ld_out - tl.n0);   // columns of the tile within the output
          for (int c64 = 0; c64 < cend; c64 += 64) {
            uint8_t* st = epi + ew * 8192 + buf * 4096;
            if (full) {
              if (lane == 0) bulk_wait_read_1();   // the store that used this box is done
              __syncwarp();
            }
            for (int sub = 0; sub < 64; sub += 32) {
              float v[32];
              tmem_ld32(tacc + c64 + sub, v);
              tmem_wait_ld();
              if (c64 == 0 && sub == 32) ring_free();
              if (full) stage_row32(st, lane, sub >> 3, v);
              else if (valid)
                store32_bf16(p.out + grow * p.ld_out + tl.n0 + c64 + sub, v,
                             p.ld_out - (tl.n0 + c64 + sub));
            }
            if (full) {
              fence_proxy_async();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmC0, smem_u32(st), tl.n0 + c64, growq);
                bulk_commit();
              }
              buf ^= 1;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
      if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
    }
    if constexpr (KIND == BWD_DH) {
      if (lane == 0 && aux_pending) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try(aux_bar(ew), aux_phase) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
    if (lane == 0) bulk_wait_all();   // bulk stores complete before shared memory is released
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the leader's MMAs into both TMEMs and all remote arrivals are done
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ----------------------------------------------------------------- CTA-pair weight gradients
// dW[e] = A_e^T B_e with K = expert e's rows (ragged): A = X (or H) and
// B = [dG|dU] (or dY), both MN-major boxes of the row-major activations. A pair
// tile is 256 rows of dW (128 per CTA: the M split of the pair MMA) by 256
// columns (each CTA loads 128 of them as its half of B), so a CTA moves 32 KB
// per k-block instead of the 48 KB of a single-CTA 128 x 256 tile.
//
// Both CTAs' boxes complete on the leader's full barrier, as in the forward
// pair kernel. In the ragged last k-block of an expert the MMA issues only the
// K16 steps that hold a valid row. The one step that straddles the expert's
// end would bring in rows of the next expert, so that k-block's A comes in
// 16-row boxes: its full steps from the activations (tmA16) and the straddling
// step from a zero-padded copy of it (tmP, filled by the dH launch's epilogue
// warps before their first tile); B's rows past the expert then meet zero rows
// of A. Nothing
// is zeroed in shared memory: zeroing the rows there from the MMA thread (both
// CTAs' A, the follower's through distributed shared memory, then a
// cluster-scope proxy fence) cost this kernel ~8%.
//
// Accumulator buffers: the leader's epilogue warps arrive on its
// accumulator-empty barrier locally, the follower's remotely with a relaxed
// arrive. The barrier orders only TMEM reads before the leader's next MMA into
// the same columns: tcgen05.wait::ld has completed those reads before the
// arrive is issued, and no memory written by the epilogue is published through
// it. (A cluster-scope release from warps with bulk stores in flight costs this
// kernel about a third of its time.)
//
// The epilogue streams fp32 rows out through two alternating [32 x 32] staging
// blocks per warp and bulk tensor stores into 3-D maps of dW ([E][rows][cols]).
// Rows past the M extent (d or I) and columns past the N extent read the fill
// value in A and B; a 32 x 32 block that starts past either is not stored and
// one that ends past it is clipped by the store.
struct WTile {
  int e;
  int row0;   // expert's first packed row (the K start)
  int rows;   // expert's rows (K)
  int m0;     // this CTA's first dW row
  int n0;     // the tile's first dW column (this CTA loads n0 + 128*rank ..)
  int part;   // gate/up: 0 for dWg, 1 for dWu (each its own n-tiles and half of [dG | dU])
  int nkb;
};

template <int KIND>
__device__ __forceinline__ WTile decode_wgrad_pair(int t, int rank, const Params& p,
                                                   const int* s_off) {
  WTile tl;
  const int per_e = p.m_tiles * p.n_tiles;
  tl.e = t / per_e;
  const int rem = t - tl.e * per_e;
  const int mt = rem / p.n_tiles;
  const int nt = rem - mt * p.n_tiles;
  tl.m0 = mt * 2 * BM + rank * BM;
  tl.part = (KIND == WGRAD_GU && nt >= p.nt_half) ? 1 : 0;
  tl.n0 = (nt - tl.part * p.nt_half) * 256;
  tl.row0 = s_off[tl.e];
  tl.rows = s_off[tl.e + 1] - tl.row0;
  tl.nkb = (tl.rows + BK - 1) / BK;
  return tl;
}

__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

constexpr uint32_t kWgradPairEpiBytes = 4u * 2u * 4096u;
constexpr int kWgradPairBars(int stages) { return 2 * stages + 5; }

template <int KIND, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_pair_wgrad_kernel(const __grid_constant__ CUtensorMap tmA,
                               const __grid_constant__ CUtensorMap tmB,
                               const __grid_constant__ CUtensorMap tmB2,
                               const __grid_constant__ CUtensorMap tmC0,
                               const __grid_constant__ CUtensorMap tmC1,
                               const __grid_constant__ CUtensorMap tmA16,
                               const __grid_constant__ CUtensorMap tmP, const Params p) {
  static_assert(KIND == WGRAD_GU || KIND == WGRAD_D, "pair weight-gradient kernel");
  constexpr int BN = 256;
  constexpr uint32_t MN_ATOM = 64 * 128;
  constexpr uint32_t A_BYTES = BM * BK * 2;
  constexpr uint32_t B_BYTES = (BN / 2) * BK * 2;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = 2 * BN;
  constexpr uint32_t IDESC = make_idesc<BN, true, true, 2 * BM>();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* epi = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + kWgradPairEpiBytes);
  // bars: full[STAGES] (leader), empty[STAGES], tfull[2], tempty[2] (leader), drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kWgradPairBars(STAGES));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = (rank == 0);
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 4);
  const int mdim = (KIND == WGRAD_GU) ? p.d : p.I;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    // the leader's accumulator-empty barriers collect the four epilogue warps of both CTAs
    for (int a = 0; a < 2; ++a) { mbar_init(tfull_bar(a), 1); mbar_init(tempty_bar(a), 8); }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB2)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmC0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmC1)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA16)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmP)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  pdl_wait();   // offsets and operands come from earlier launches
  pdl_launch_dependents();
  for (int e = threadIdx.x; e <= p.E; e += kThreads) s_off[e] = __ldg(p.offsets + e);
  tc_fence_before();
  __syncthreads();
  const bool offs_ok = offsets_ok(s_off, p);
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  uint32_t peer_base;
  asm volatile("ld.shared::cluster.u32 %0, [%1];"
               : "=r"(peer_base)
               : "r"(map_to_rank(smem_u32(tmem_slot), rank ^ 1u))
               : "memory");
  const bool tmem_ok = (peer_base == tmem_base);
  if (!tmem_ok && threadIdx.x == 0) report_status(p.status, MOE_ERR_DEVICE_CHECK);
  // the data part's record of the scratch this launch reads (every CTA reads it)
  bool tag_ok = true;
  if (p.tag_mode == kTagCheck) {
    const volatile uint32_t* rec = reinterpret_cast<const volatile uint32_t*>(p.status) + kTagFirst;
#pragma unroll
    for (int i = 0; i < kTagWords; ++i) tag_ok = tag_ok && rec[i] == p.tag[i];
    if (!tag_ok && blockIdx.x == 0 && threadIdx.x == 0) report_status(p.status, MOE_ERR_DEVICE_CHECK);
  }
  const int total = (tmem_ok && tag_ok && offs_ok) ? p.E * p.m_tiles * p.n_tiles : 0;
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(n_clusters_x());

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t fpar = 0, fused = 0;   // per stage: parity of the next phase, used at all
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        const WTile tl = decode_wgrad_pair<KIND>(t, static_cast<int>(rank), p, s_off);
        const int nb = tl.n0 + static_cast<int>(rank) * (BN / 2);
        for (int kb = 0; kb < tl.nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const int ky = tl.row0 + kb * BK;
          const uint32_t fb = full_bar(stage);
          const uint32_t fr = map_to_rank(fb, 0);
          const int kvalid = min(BK, tl.rows - kb * BK);
          if ((kvalid & 15) == 0) {
            if (leader) mbar_expect_tx(fb, 2 * STAGE_BYTES);   // both CTAs' boxes
            tma_load_2d_pair(sa, &tmA, fr, tl.m0, ky);
            tma_load_2d_pair(sa + MN_ATOM, &tmA, fr, tl.m0 + 64, ky);
          } else {
            // straddling k-block: A in 16-row boxes, the last one zero-padded; the
            // K16 steps past it are neither loaded nor read
            const int nfull = kvalid >> 4;
            if (leader) mbar_expect_tx(fb, 2 * (static_cast<uint32_t>(nfull + 1) * 2 * 2048u + B_BYTES));
#pragma unroll
            for (int atom = 0; atom < 2; ++atom) {
              const uint32_t da = sa + atom * MN_ATOM;
              const int x = tl.m0 + 64 * atom;
              for (int kk = 0; kk < nfull; ++kk) tma_load_2d_pair(da + kk * 2048, &tmA16, fr, x, ky + 16 * kk);
              tma_load_2d_pair(da + nfull * 2048, &tmP, fr, x, tl.e * 16);
            }
          }
          const CUtensorMap* mb = tl.part ? &tmB2 : &tmB;   // dG or dU half (gate/up)
          tma_load_2d_pair(sa + A_BYTES, mb, fr, nb, ky);
          tma_load_2d_pair(sa + A_BYTES + MN_ATOM, mb, fr, nb + 64, ky);
          fpar ^= 1u << stage;
          fused |= 1u << stage;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (leader) {
        // the leader's full barriers count both CTAs' loads: wait for the last phases
        for (int s = 0; s < STAGES; ++s) {
          if (!(fused & (1u << s))) continue;
          const uint32_t par = ((fpar >> s) & 1u) ^ 1u;
          const uint64_t t0 = globaltimer();
          while (!mbar_try(full_bar(s), par) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
      } else if (!ok) {
        const uint64_t t0 = globaltimer();   // loads may still land after a timeout
        while (globaltimer() - t0 < 1000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        const WTile tl = decode_wgrad_pair<KIND>(t, 0, p, s_off);
        if (tl.nkb == 0) continue;
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        // One k-block: FULL, the four K16 steps of 64 rows (unrolled: the issuing
        // thread keeps the tensor pipe fed; a loop with a run-time trip count cost
        // the weight gradients ~9% of their cycles); otherwise the ragged last
        // k-block, only the K16 steps that hold a valid row.
        auto kblock = [&](int kb, auto full) -> bool {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status)) return false;
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          if (lane == 0) {
            if constexpr (decltype(full)::value) {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad = smem_desc(sa + kk * 2048, MN_ATOM, 1024);
                const uint64_t bd = smem_desc(sb + kk * 2048, MN_ATOM, 1024);
                tc_mma_pair(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
              }
            } else {
              const int nsteps = (tl.rows - kb * BK + 15) >> 4;   // K16 steps with a valid row
              for (int kk = 0; kk < nsteps; ++kk) {
                const uint64_t ad = smem_desc(sa + kk * 2048, MN_ATOM, 1024);
                const uint64_t bd = smem_desc(sb + kk * 2048, MN_ATOM, 1024);
                tc_mma_pair(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
              }
            }
            tc_commit_pair_both(empty_bar(stage));
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          return true;
        };
        const int nfull = tl.rows / BK;
        for (int kb = 0; kb < nfull && ok; ++kb) ok = kblock(kb, std::true_type{});
        if (ok && tl.nkb > nfull) ok = kblock(nfull, std::false_type{});
        if (!ok) break;
        if (lane == 0) tc_commit_pair_both(tfull_bar(acc));
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (lane == 0) {
        tc_commit_pair_local(drain_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try(drain_bar, 0) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int ew = warp - 2;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    int buf = 0;
    for (int t = cid; t < total; t += ncl) {
      const WTile tl = decode_wgrad_pair<KIND>(t, static_cast<int>(rank), p, s_off);
      const bool empty = (tl.nkb == 0);   // expert without rows: its gradient is zero
      if (!empty) {
        if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.status)) break;
        tc_fence_after();
      }
      const bool in_range = tl.m0 < mdim;   // false only for the follower past the M extent
      const int ncols = (KIND == WGRAD_GU) ? p.I : p.d;   // columns of this tile's dW
      const uint32_t tacc = tmem_base + lane_addr + static_cast<uint32_t>(acc * BN);
      const int mrow = tl.m0 + q * 32;
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        if (!empty) {
          tmem_ld32(tacc + c, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        // past the M or N extent: not stored (a slice that ends past it is clipped by the store)
        if (!in_range || mrow >= mdim || tl.n0 + c >= ncols) continue;
        uint8_t* stg = epi + ew * 8192 + buf * 4096;
        if (lane == 0) bulk_wait_read_1();   // the store that last used this block has read it
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float4* dst = reinterpret_cast<float4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4));
          *dst = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          // 3-D maps [E][rows][cols] of dW: rows and columns past the expert's are clipped
          tma_store_3d(tl.part ? &tmC1 : &tmC0, smem_u32(stg), tl.n0 + c, mrow, tl.e);
          bulk_commit();
        }
        // Spread the tile's stores over ~40% of the next tile's MMA time (~0.3 us of
        // MMA per k-block): a burst of 32 stores per CTA at the start of a tile
        // delays that tile's operand loads and takes issue slots from the MMA warp
        // (the drafter-shaped weight gradient spends 5% fewer cycles paced)
        if (c + 32 < BN) __nanosleep(15u * static_cast<unsigned>(tl.nkb));
        buf ^= 1;
      }
      if (empty) continue;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(acc));
        else mbar_arrive_cluster_relaxed(map_to_rank(tempty_bar(acc), 0));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ----------------------------------------------------------------- diagnostics
// One thread waits, through the GEMMs' bounded wait, on an mbarrier that nothing
// arrives on; the wait runs out after timeout_ns and records the timeout.
__global__ void wait_timeout_kernel(int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_slow(b, 0, &abort_flag, status, timeout_ns);
}

// ----------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D tensor map over a row-major [outer, inner] array of bf16 (or fp32), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer, bool fp32 = false, uint64_t row_elems = 0) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(row_elems ? row_elems : inner) * (fp32 ? 4 : 2)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One half of a row-major [rows, 2 * half] bf16 array ([G | U] and [dG | dU]):
// columns [col0, col0 + half) of every row as a [rows, half] tensor, so a box
// past column half reads zeros and a store past it is clipped (the other half
// is never touched).
bool make_half_map(CUtensorMap* m, const void* base, uint64_t half, uint64_t rows, uint64_t col0,
                   uint32_t box_inner, uint32_t box_outer) {
  return make_map(m, static_cast<const uint16_t*>(base) + col0, half, rows, box_inner, box_outer,
                  false, 2 * half);
}

// 3-D tensor map over a row-major [E, rows, cols] array of bf16 (or fp32), 128-byte
// swizzle: boxes of box_cols x box_rows x 1 at (column, row, expert); rows and
// columns past an expert's extent read zeros and are clipped on stores.
bool make_map3(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t E,
               uint32_t box_cols, uint32_t box_rows, bool fp32 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t es_b = fp32 ? 4 : 2;
  cuuint64_t dims[3] = {cols, rows, E};
  cuuint64_t strides[2] = {cols * es_b, cols * rows * es_b};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map over a row-major [outer, inner] array of bytes (E4M3), 128-byte
// swizzle unless another is given.
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over n_atoms 512-byte scale atoms (as [n_atoms, 128] uint32), one atom per box.
bool make_map_atoms(CUtensorMap* m, const void* base, uint64_t n_atoms) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, n_atoms};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifndef MOE_PAIR_BN_MAX
#define MOE_PAIR_BN_MAX 256
#endif

template <int KIND, int BN, int STAGES, bool FP8 = false>
constexpr size_t pair_smem_bytes(int E) {
  return 1024 + STAGES * (BM * BK * 2 + (BN / 2) * BK * 2 +
                          (FP8 ? ((512 * (1 + BN / 128) + 1023) & ~1023) : 0)) +
         pair_epi_bytes<KIND>() + 8 * (2 * STAGES + 11) + 16 + sizeof(int) * 2 * (E + 1) + 16;
}

// Launches a cluster-of-two kernel on as many clusters as can be resident
// (at most tiles_upper). The shared-memory opt-in and the occupancy query run
// once per kernel instantiation and device (the caller owns those two slots).
template <typename... KArgs, typename... Args>
int launch_cluster2(void (*kern)(KArgs...), size_t sm, size_t sm_max, int* configured,
                    int* max_clusters, long long tiles_upper, const char* name, cudaStream_t st,
                    const Args&... args) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (*configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sm_max));
    if (e != cudaSuccess) { set_last_cuda_error(e); return MOE_ERR_CUDA; }
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2 * num_sms(), 1, 1);
    q.dynamicSmemBytes = sm_max;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &q);
    if (e != cudaSuccess || n < 1) {
      set_last_cuda_error(e == cudaSuccess ? cudaErrorInvalidConfiguration : e);
      return MOE_ERR_CUDA;
    }
    *max_clusters = n;
    *configured = dev;
  }
  long long ncl = *max_clusters;
  if (tiles_upper < ncl) ncl = tiles_upper;
  if (ncl < 1) return MOE_OK;
  ProfScope prof(name, st);
  return launch_pdl(kern, static_cast<unsigned>(2 * ncl), kThreads, sm, st, 2, args...);
}

// Launches the CTA-pair kernel of a forward or input-gradient kind with the
// shared-memory opt-in sized for the largest expert count it is used with.
template <int KIND, int BN, int STAGES, bool FP8 = false>
int launch_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                const CUtensorMap& c0, const CUtensorMap& c1, const CUtensorMap& c2,
                const CUtensorMap& s, const Params& p, long long tiles_upper, int e_max,
                cudaStream_t st) {
  static thread_local int configured = -1;
  static thread_local int max_clusters = 0;
  static const char* kNames[] = {"gemm_gate_up", "gemm_down", "gemm_dh", "gemm_dx", "", ""};
  static const char* kNamesFp8[] = {"gemm_gate_up_fp8", "gemm_down_fp8", "", "", "", ""};
  return launch_cluster2(grouped_gemm_pair_kernel<KIND, BN, STAGES, FP8>,
                         pair_smem_bytes<KIND, BN, STAGES, FP8>(p.E),
                         pair_smem_bytes<KIND, BN, STAGES, FP8>(e_max), &configured,
                         &max_clusters, tiles_upper, FP8 ? kNamesFp8[KIND] : kNames[KIND], st, a,
                         b0, b1, c0, c1, c2, s, p);
}

// Weight gradients on CTA pairs: six 32 KB stages while the expert table fits
// beside them (E <= 448), five otherwise.
template <int STAGES>
constexpr size_t pair_wgrad_smem_bytes(int E) {
  return 1024 + STAGES * (BM * BK * 2 + 128 * BK * 2) + kWgradPairEpiBytes +
         8 * kWgradPairBars(STAGES) + 16 + sizeof(int) * (E + 1) + 16;
}
constexpr int kWgradPair6MaxE = 448;
static_assert(pair_wgrad_smem_bytes<6>(kWgradPair6MaxE) <= 232448, "pair wgrad smem (6 stages)");
static_assert(pair_wgrad_smem_bytes<5>(1024) <= 232448, "pair wgrad smem (5 stages)");

template <int KIND, int STAGES>
int launch_pair_wgrad_stages(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                             const CUtensorMap& c0, const CUtensorMap& c1, const CUtensorMap& a16,
                             const CUtensorMap& pad, const Params& p, long long tiles,
                             cudaStream_t st) {
  static thread_local int configured = -1;
  static thread_local int max_clusters = 0;
  return launch_cluster2(grouped_gemm_pair_wgrad_kernel<KIND, STAGES>,
                         pair_wgrad_smem_bytes<STAGES>(p.E),
                         pair_wgrad_smem_bytes<STAGES>(STAGES == 6 ? kWgradPair6MaxE : 1024),
                         &configured, &max_clusters, tiles,
                         KIND == WGRAD_GU ? "gemm_wgrad_gate_up" : "gemm_wgrad_down", st, a, b,
                         b2, c0, c1, a16, pad, p);
}

// b, b2: B (gate/up: the dG and dU halves); c0, c1: the dW maps (gate/up: dWg
// and dWu); a16: A again with 16-row boxes; pad: the zero-padded straddling
// steps of A.
template <int KIND>
int launch_pair_wgrad(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                      const CUtensorMap& c0, const CUtensorMap& c1, const CUtensorMap& a16,
                      const CUtensorMap& pad, const Params& p, long long tiles, cudaStream_t st) {
  if (p.E <= kWgradPair6MaxE)
    return launch_pair_wgrad_stages<KIND, 6>(a, b, b2, c0, c1, a16, pad, p, tiles, st);
  return launch_pair_wgrad_stages<KIND, 5>(a, b, b2, c0, c1, a16, pad, p, tiles, st);
}

constexpr long long kSmemOptIn = 232448;   // shared memory a CTA may opt into

// Largest expert count whose offset tables fit beside STAGES pair stages (-1: none).
template <int KIND, int BN, int STAGES, bool FP8 = false>
constexpr int pair_max_e() {
  return static_cast<int>(
      (kSmemOptIn - static_cast<long long>(pair_smem_bytes<KIND, BN, STAGES, FP8>(0))) /
      (2 * static_cast<long long>(sizeof(int))));
}

// Pair pipeline depth. The shallow ring fits beside the expert tables of up to
// 1024 experts; the deep ring (one or two more stages) is used when the expert
// count leaves room for it. Measured on E=128 x 512 rows, the deep rings take
// gate/up 309 -> 289 us, dH 219 -> 206, dX 264 -> 254, down 149 -> 141: a
// stage is 32 KB for ~0.3 us of MMA work, so the ring covers more of a load's
// latency.
template <int KIND, int BN>
constexpr int pair_stages() {
  return BN == 256 ? 5 : 7;
}
template <int KIND, int BN>
constexpr int pair_stages_deep() {
  return BN == 256 ? 6 : 8;
}

template <int KIND, int BN, bool FP8 = false>
int launch_pair_depth(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                      const CUtensorMap& c0, const CUtensorMap& c1, const CUtensorMap& c2,
                      const CUtensorMap& s, const Params& p, long long tiles_upper,
                      cudaStream_t st) {
  constexpr int kDeep = pair_stages_deep<KIND, BN>();
  constexpr int kShallow = pair_stages<KIND, BN>();
  constexpr int kDeepMaxE = pair_max_e<KIND, BN, kDeep, FP8>();
  static_assert(pair_max_e<KIND, BN, kShallow, FP8>() >= 1024,
                "shallow pair ring must fit 1024 experts");
  if constexpr (kDeepMaxE >= 1) {
    if (p.E <= kDeepMaxE)
      return launch_pair<KIND, BN, kDeep, FP8>(a, b0, b1, c0, c1, c2, s, p, tiles_upper,
                                               kDeepMaxE < 1024 ? kDeepMaxE : 1024, st);
  }
  return launch_pair<KIND, BN, kShallow, FP8>(a, b0, b1, c0, c1, c2, s, p, tiles_upper, 1024, st);
}

// The bf16 kinds: c0..c2 the epilogue's maps (gate/up: H and the G, U halves of
// [G | U]; dH: the G half of [G | U], then the dG and dU halves of [dG | dU]),
// s the U half of [G | U] for dH (another map otherwise, not read).
template <int KIND>
int launch_pair_bn(int bn, const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                   const CUtensorMap& c0, const CUtensorMap& c1, const CUtensorMap& c2,
                   const CUtensorMap& s, const Params& p, long long tiles_upper, cudaStream_t st) {
#if MOE_PAIR_BN_MAX >= 256
  if (bn == 256) return launch_pair_depth<KIND, 256>(a, b0, b1, c0, c1, c2, s, p, tiles_upper, st);
#endif
  return launch_pair_depth<KIND, 128>(a, b0, b1, c0, c1, c2, s, p, tiles_upper, st);
}

// The N width a pair tile uses for an output of n columns: 256 unless 128-wide
// tiles leave fewer columns idle (n % 256 in 1 .. 128).
inline int pair_bn(int n) {
  const int r = n % 256;
  return ((r == 0 || r > 128) && MOE_PAIR_BN_MAX >= 256) ? 256 : 128;
}


}  // namespace gemm

// [dG | dU] as bf16 [M, 2I], then the zero-padded straddling steps of X and H
// for the weight gradients: bf16 [E, 16, d] and [E, 16, I].
size_t ffn_backward_scratch(long long M, int E, int d, int I) {
  return (static_cast<size_t>(M) * 2 * I + static_cast<size_t>(E) * 16 * (d + I)) * sizeof(uint16_t);
}

long long mxfp8_row_tiles(long long M, int E);                                     // fp8.cu
int launch_quantize_rows(const void* x, const int32_t* offsets, int E, int M, int K, void* q,
                         void* sf, cudaStream_t st);                               // fp8.cu

// The MXFP8 forward's scratch: X and H quantized (E4M3 [M, d], [M, I]) with
// their scale atoms, each region 1024-byte aligned.
struct Fp8Scratch {
  size_t xq, xsf, hq, hsf, total;
};
Fp8Scratch ffn_fp8_layout(long long M, int E, int d, int I) {
  auto up = [](size_t b) { return (b + 1023) & ~static_cast<size_t>(1023); };
  const long long tiles = mxfp8_row_tiles(M, E);
  Fp8Scratch s;
  s.xq = 0;
  s.xsf = up(static_cast<size_t>(M) * d);
  s.hq = s.xsf + up(static_cast<size_t>(tiles) * (d / 128) * 512);
  s.hsf = s.hq + up(static_cast<size_t>(M) * I);
  s.total = s.hsf + up(static_cast<size_t>(tiles) * (I / 128) * 512);
  return s;
}
size_t ffn_fp8_scratch(long long M, int E, int d, int I) { return ffn_fp8_layout(M, E, d, I).total; }

}  // namespace moe

namespace {

bool ffn_shape_ok(int E, int M, int d, int I) {
  return E >= 1 && E <= 1024 && M >= 0 && d > 0 && I > 0 && d % 8 == 0 && I % 8 == 0;
}

}  // namespace

extern "C" int moe_grouped_ffn(const moe_bf16* xp, const int32_t* offsets, int E, int M, int d,
                               int I, const moe_bf16* w_gate, const moe_bf16* w_up,
                               const moe_bf16* w_down, moe_bf16* y, moe_bf16* h, moe_bf16* gu,
                               void* ws, size_t ws_bytes, void* stream) {
  using namespace moe;
  using namespace moe::gemm;
  if (!ffn_shape_ok(E, M, d, I)) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!xp || !offsets || !w_gate || !w_up || !w_down || !y || !h) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(offsets) || !aligned16(w_gate) || !aligned16(w_up) ||
      !aligned16(w_down) || !aligned16(y) || !aligned16(h) || (gu && !aligned16(gu)))
    return MOE_ERR_MISALIGNED;
  if (!ws || ws_bytes < kWorkspaceHeader || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  if (cc_major() < 10) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  Params p{};
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.d = d;
  p.I = I;
  p.status = static_cast<int*>(ws);
  p.tag[0] = kTagMagic;
  p.tag[1] = static_cast<uint32_t>(M);
  p.tag[2] = static_cast<uint32_t>(E);
  p.tag[3] = static_cast<uint32_t>(d);
  p.tag[4] = static_cast<uint32_t>(I);
  p.tag[5] = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(offsets));
  const long long mt_upper = (M + BM - 1) / BM + E;
  CUtensorMap ta, tb0, tb1, tc0, tc1, tc2;
  // gate/up projection with the SwiGLU epilogue (H and [G|U] leave through bulk
  // stores). The weights are 3-D maps [E][d][I]: a K or N tail past d or I reads
  // zeros, and the stores clip at column I of H and of each half of [G|U].
  if (!make_map(&ta, xp, d, M, 64, BM) || !make_map3(&tb0, w_gate, I, d, E, 64, 64) ||
      !make_map3(&tb1, w_up, I, d, E, 64, 64) || !make_map(&tc0, h, I, M, 64, 32))
    return MOE_ERR_CUDA;
  if (gu) {
    if (!make_half_map(&tc1, gu, I, M, 0, 64, 32) || !make_half_map(&tc2, gu, I, M, I, 64, 32))
      return MOE_ERR_CUDA;
  } else {
    tc1 = tc2 = tc0;   // not stored through
  }
  // 128 gate + 128 up columns per tile, or 64 + 64 when that leaves fewer idle
  const int bn_gu = (I % 128 == 0 || I % 128 > 64) && MOE_PAIR_BN_MAX >= 256 ? 256 : 128;
  p.n_tiles = (I + bn_gu / 2 - 1) / (bn_gu / 2);
  p.k_blocks = (d + BK - 1) / BK;
  p.out = reinterpret_cast<__nv_bfloat16*>(h);
  p.out2 = reinterpret_cast<__nv_bfloat16*>(gu);
  p.ld_out = I;
  int rc = launch_pair_bn<FWD_GATEUP>(bn_gu, ta, tb0, tb1, tc0, tc1, tc2, tc0, p,
                                      mt_upper * p.n_tiles, st);
  if (rc) return rc;
  // down projection (Wd as [E][I][d])
  const int bn = pair_bn(d);
  if (!make_map(&ta, h, I, M, 64, BM) || !make_map3(&tb0, w_down, d, I, E, 64, 64) ||
      !make_map(&tc0, y, d, M, 64, 32))
    return MOE_ERR_CUDA;
  p.n_tiles = (d + bn - 1) / bn;
  p.k_blocks = (I + BK - 1) / BK;
  p.out = reinterpret_cast<__nv_bfloat16*>(y);
  p.out2 = nullptr;
  p.ld_out = d;
  return launch_pair_bn<FWD_DOWN>(bn, ta, tb0, tb0, tc0, tc0, tc0, tc0, p, mt_upper * p.n_tiles, st);
}

namespace {

constexpr int kBwdData = 1;      // dH (with the weight gradients' padded steps) and dX
constexpr int kBwdWeights = 2;   // the weight gradients

// The backward GEMMs, in two parts that share the workspace: the data part
// writes [dG | dU] and the padded straddling steps into it, the weight part
// reads them. Arguments a part does not use may be null.
int ffn_backward_parts(int parts, const moe_bf16* dy, const moe_bf16* xp, const moe_bf16* gu,
                       const moe_bf16* h, const int32_t* offsets, int E, int M, int d, int I,
                       const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                       moe_bf16* dxp, float* dw_gate, float* dw_up, float* dw_down, void* ws,
                       size_t ws_bytes, void* stream) {
  using namespace moe;
  using namespace moe::gemm;
  const bool data = parts & kBwdData, weights = parts & kBwdWeights;
  if (!ffn_shape_ok(E, M, d, I)) return MOE_ERR_INVALID_ARG;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (data && (!w_gate || !w_up || !w_down)) return MOE_ERR_INVALID_ARG;
  if (weights && (!dw_gate || !dw_up || !dw_down)) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!dy || !xp || !h || (data && (!gu || !dxp)))) return MOE_ERR_INVALID_ARG;
  if ((M > 0 && (!aligned16(dy) || !aligned16(xp) || !aligned16(h) ||
                 (data && (!aligned16(gu) || !aligned16(dxp))))) ||
      !aligned16(offsets) ||
      (data && (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down))) ||
      (weights && (!aligned16(dw_gate) || !aligned16(dw_up) || !aligned16(dw_down))))
    return MOE_ERR_MISALIGNED;
  if (!ws || !aligned16(ws) || ws_bytes < kWorkspaceHeader + ffn_backward_scratch(M, E, d, I))
    return MOE_ERR_WORKSPACE;
  if (cc_major() < 10) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  const size_t wbytes = static_cast<size_t>(E) * d * I * sizeof(float);
  if (M == 0) {
    if (weights) {
      cudaMemsetAsync(dw_gate, 0, wbytes, st);
      cudaMemsetAsync(dw_up, 0, wbytes, st);
      cudaMemsetAsync(dw_down, 0, wbytes, st);
    }
    return check_launch();
  }
  auto dgu = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + kWorkspaceHeader);
  auto pad_x = dgu + static_cast<size_t>(M) * 2 * I;          // [E, 16, d]
  auto pad_h = pad_x + static_cast<size_t>(E) * 16 * d;       // [E, 16, I]

  Params p{};
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.d = d;
  p.I = I;
  p.status = static_cast<int*>(ws);
  p.tag[0] = kTagMagic;
  p.tag[1] = static_cast<uint32_t>(M);
  p.tag[2] = static_cast<uint32_t>(E);
  p.tag[3] = static_cast<uint32_t>(d);
  p.tag[4] = static_cast<uint32_t>(I);
  p.tag[5] = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(offsets));
  const long long mt_upper = (M + BM - 1) / BM + E;
  CUtensorMap ta, tb0, tb1, tc0, tc1, tc2, ts;
  int rc = MOE_OK;
  if (data) {
    // dH = dY Wd^T with the SwiGLU backward epilogue -> [dG | dU], on 256-wide
    // tiles also when I % 256 != 0 (the last tile's columns past I read zeros
    // from the 3-D map of Wd and store nothing): 128-wide tiles fetch 1.5x the
    // operand bytes per MMA flop. G and U come in, and dG and dU leave, through
    // half maps of [G | U] and [dG | dU].
    const int bn_h = MOE_PAIR_BN_MAX >= 256 ? 256 : 128;
    if (!make_map(&ta, dy, d, M, 64, BM) || !make_map3(&tb0, w_down, d, I, E, 64, bn_h / 2) ||
        !make_half_map(&tc0, gu, I, M, 0, 64, 32) || !make_half_map(&ts, gu, I, M, I, 64, 32) ||
        !make_half_map(&tc1, dgu, I, M, 0, 64, 32) || !make_half_map(&tc2, dgu, I, M, I, 64, 32))
      return MOE_ERR_CUDA;
    p.n_tiles = (I + bn_h - 1) / bn_h;
    p.k_blocks = (d + BK - 1) / BK;
    p.out = dgu;
    p.aux = reinterpret_cast<const __nv_bfloat16*>(gu);
    p.ld_out = 2 * I;
    // the dH launch also fills the weight gradients' padded straddling steps
    p.pad[0] = PadJob{reinterpret_cast<const __nv_bfloat16*>(xp), pad_x, d};
    p.pad[1] = PadJob{reinterpret_cast<const __nv_bfloat16*>(h), pad_h, I};
    p.tag_mode = kTagWrite;
    rc = launch_pair_bn<BWD_DH>(bn_h, ta, tb0, tb0, tc0, tc1, tc2, ts, p, mt_upper * p.n_tiles, st);
    p.tag_mode = kTagNone;
    if (rc) return rc;
    // dX = dG Wg^T + dU Wu^T: K runs over the dG half's k-blocks (with Wg), then
    // the dU half's (with Wu), each A from its own half map (tc2: the dU half) so
    // that a K tail reads zeros instead of the other half
    const int bn_x = pair_bn(d);
    if (!make_half_map(&ta, dgu, I, M, 0, 64, BM) || !make_half_map(&tc2, dgu, I, M, I, 64, BM) ||
        !make_map3(&tb0, w_gate, I, d, E, 64, bn_x / 2) ||
        !make_map3(&tb1, w_up, I, d, E, 64, bn_x / 2) || !make_map(&tc0, dxp, d, M, 64, 32))
      return MOE_ERR_CUDA;
    p.n_tiles = (d + bn_x - 1) / bn_x;
    p.kb_half = (I + BK - 1) / BK;
    p.k_blocks = 2 * p.kb_half;
    p.out = reinterpret_cast<__nv_bfloat16*>(dxp);
    p.aux = nullptr;
    p.ld_out = d;
    p.pad[0] = p.pad[1] = PadJob{nullptr, nullptr, 0};
    rc = launch_pair_bn<BWD_DX>(bn_x, ta, tb0, tb1, tc0, tc0, tc2, tc0, p, mt_upper * p.n_tiles, st);
    if (rc) return rc;
  }
  if (!weights) return MOE_OK;
  // dWg = X^T dG and dWu = X^T dU on CTA pairs over 256 dW rows x 256 columns:
  // the n-tiles of dWg, then those of dWu, B from the matching half map of
  // [dG | dU]; the dW maps are 3-D [E][d][I], so rows past d and columns past I
  // (the TMA fill value in the operands) are clipped from the stores.
  CUtensorMap ta16, tpad, tb2;
  if (!make_map(&ta, xp, d, M, 64, 64) || !make_half_map(&tb0, dgu, I, M, 0, 64, 64) ||
      !make_half_map(&tb2, dgu, I, M, I, 64, 64) || !make_map(&ta16, xp, d, M, 64, 16) ||
      !make_map(&tpad, pad_x, d, static_cast<uint64_t>(E) * 16, 64, 16) ||
      !make_map3(&tc0, dw_gate, I, d, E, 32, 32, true) ||
      !make_map3(&tc1, dw_up, I, d, E, 32, 32, true))
    return MOE_ERR_CUDA;
  p.m_tiles = (d + 2 * BM - 1) / (2 * BM);
  p.nt_half = (I + 255) / 256;
  p.n_tiles = 2 * p.nt_half;
  p.outf0 = dw_gate;
  p.outf1 = dw_up;
  p.out = nullptr;
  p.tag_mode = kTagCheck;
  rc = launch_pair_wgrad<WGRAD_GU>(ta, tb0, tb2, tc0, tc1, ta16, tpad, p,
                                   static_cast<long long>(E) * p.m_tiles * p.n_tiles, st);
  if (rc) return rc;
  // dWd = H^T dY on CTA pairs, dWd as [E][I][d]
  if (!make_map(&ta, h, I, M, 64, 64) || !make_map(&tb0, dy, d, M, 64, 64) ||
      !make_map3(&tc0, dw_down, d, I, E, 32, 32, true) || !make_map(&ta16, h, I, M, 64, 16) ||
      !make_map(&tpad, pad_h, I, static_cast<uint64_t>(E) * 16, 64, 16))
    return MOE_ERR_CUDA;
  p.outf0 = dw_down;
  p.outf1 = nullptr;
  p.m_tiles = (I + 2 * BM - 1) / (2 * BM);
  p.nt_half = 0;
  p.n_tiles = (d + 255) / 256;
  return launch_pair_wgrad<WGRAD_D>(ta, tb0, tb0, tc0, tc0, ta16, tpad, p,
                                    static_cast<long long>(E) * p.m_tiles * p.n_tiles, st);
}

}  // namespace

extern "C" int moe_grouped_ffn_backward(const moe_bf16* dy, const moe_bf16* xp, const moe_bf16* gu,
                                        const moe_bf16* h, const int32_t* offsets, int E, int M,
                                        int d, int I, const moe_bf16* w_gate, const moe_bf16* w_up,
                                        const moe_bf16* w_down, moe_bf16* dxp, float* dw_gate,
                                        float* dw_up, float* dw_down, void* ws, size_t ws_bytes,
                                        void* stream) {
  if (!w_gate || !w_up || !w_down || !dw_gate || !dw_up || !dw_down) return MOE_ERR_INVALID_ARG;
  if (M > 0 && !gu) return MOE_ERR_INVALID_ARG;
  return ffn_backward_parts(kBwdData | kBwdWeights, dy, xp, gu, h, offsets, E, M, d, I, w_gate,
                            w_up, w_down, dxp, dw_gate, dw_up, dw_down, ws, ws_bytes, stream);
}

extern "C" int moe_grouped_ffn_backward_data(const moe_bf16* dy, const moe_bf16* xp,
                                             const moe_bf16* gu, const moe_bf16* h,
                                             const int32_t* offsets, int E, int M, int d, int I,
                                             const moe_bf16* w_gate, const moe_bf16* w_up,
                                             const moe_bf16* w_down, moe_bf16* dxp, void* ws,
                                             size_t ws_bytes, void* stream) {
  return ffn_backward_parts(kBwdData, dy, xp, gu, h, offsets, E, M, d, I, w_gate, w_up, w_down,
                            dxp, nullptr, nullptr, nullptr, ws, ws_bytes, stream);
}

extern "C" int moe_grouped_ffn_backward_weights(const moe_bf16* dy, const moe_bf16* xp,
                                                const moe_bf16* h, const int32_t* offsets, int E,
                                                int M, int d, int I, float* dw_gate, float* dw_up,
                                                float* dw_down, void* ws, size_t ws_bytes,
                                                void* stream) {
  return ffn_backward_parts(kBwdWeights, dy, xp, nullptr, h, offsets, E, M, d, I, nullptr,
                            nullptr, nullptr, nullptr, dw_gate, dw_up, dw_down, ws, ws_bytes,
                            stream);
}

extern "C" int moe_debug_wait_timeout(void* ws, int timeout_us, void* stream) {
  using namespace moe;
  if (!ws || !aligned16(ws) || timeout_us < 1 || timeout_us > 10000000) return MOE_ERR_INVALID_ARG;
  gemm::wait_timeout_kernel<<<1, 32, 0, as_stream(stream)>>>(
      static_cast<int*>(ws), static_cast<uint64_t>(timeout_us) * 1000ull);
  return check_launch();
}

extern "C" int moe_grouped_ffn_fp8(const moe_bf16* xp, const int32_t* offsets, int E, int M, int d,
                                   int I, const uint8_t* wgu_q, const uint8_t* wgu_sf,
                                   const uint8_t* wd_q, const uint8_t* wd_sf, moe_bf16* y,
                                   moe_bf16* h, moe_bf16* gu, void* ws, size_t ws_bytes,
                                   void* stream) {
  using namespace moe;
  using namespace moe::gemm;
  if (!ffn_shape_ok(E, M, d, I)) return MOE_ERR_INVALID_ARG;
  if (d % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;   // whole scale blocks and tiles
  if (M == 0) return MOE_OK;
  if (!xp || !offsets || !wgu_q || !wgu_sf || !wd_q || !wd_sf || !y || !h) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(offsets) || !aligned16(wgu_q) || !aligned16(wgu_sf) ||
      !aligned16(wd_q) || !aligned16(wd_sf) || !aligned16(y) || !aligned16(h) ||
      (gu && !aligned16(gu)))
    return MOE_ERR_MISALIGNED;
  const Fp8Scratch lay = ffn_fp8_layout(M, E, d, I);
  if (!ws || !aligned16(ws) || ws_bytes < kWorkspaceHeader + lay.total) return MOE_ERR_WORKSPACE;
  if (cc_major() < 10) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  uint8_t* scratch = static_cast<uint8_t*>(ws) + kWorkspaceHeader;
  uint8_t* xq = scratch + lay.xq;
  uint8_t* xsf = scratch + lay.xsf;
  uint8_t* hq = scratch + lay.hq;
  uint8_t* hsf = scratch + lay.hsf;
  const long long tiles = mxfp8_row_tiles(M, E);
  Params p{};
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.d = d;
  p.I = I;
  p.status = static_cast<int*>(ws);
  const long long mt_upper = (M + BM - 1) / BM + E;
  int rc = launch_quantize_rows(xp, offsets, E, M, d, xq, xsf, st);
  if (rc) return rc;
  CUtensorMap ta, tb0, tb1, tc0, tc1, tc2, ts;
  // gate/up on 256 x 256 pair tiles (128 gate + 128 up columns), SwiGLU epilogue;
  // the epilogue also writes H's E4M3 copy and its scale atoms for the down
  // projection (the quantization fused: no second pass over H)
  if (!make_map_u8(&ta, xq, d, M, 128, BM) ||
      !make_map_u8(&tb0, wgu_q, d, static_cast<uint64_t>(E) * 2 * I, 128, 128) ||
      !make_map_atoms(&tb1, xsf, static_cast<uint64_t>(tiles) * (d / 128)) ||
      !make_map_atoms(&ts, wgu_sf, static_cast<uint64_t>(E) * (2 * I / 128) * (d / 128)) ||
      !make_map(&tc0, h, I, M, 64, 32))
    return MOE_ERR_CUDA;
  if (gu) {
    if (!make_half_map(&tc1, gu, I, M, 0, 64, 32) || !make_half_map(&tc2, gu, I, M, I, 64, 32))
      return MOE_ERR_CUDA;
  } else {
    tc1 = tc2 = tc0;   // not stored through
  }
  p.n_tiles = I / 128;
  p.k_blocks = d / 128;
  p.out = reinterpret_cast<__nv_bfloat16*>(h);
  p.out2 = reinterpret_cast<__nv_bfloat16*>(gu);
  p.ld_out = I;
  p.hq = hq;
  p.hsf = hsf;
  rc = launch_pair_depth<FWD_GATEUP, 256, true>(ta, tb0, tb1, tc0, tc1, tc2, ts, p,
                                                 mt_upper * p.n_tiles, st);
  if (rc) return rc;
  p.hq = nullptr;
  p.hsf = nullptr;
  // down on 256 x 256 pair tiles (256 x 128 when d is an odd multiple of 128)
  const int bn = pair_bn(d);
  if (!make_map_u8(&ta, hq, I, M, 128, BM) ||
      !make_map_u8(&tb0, wd_q, I, static_cast<uint64_t>(E) * d, 128, bn / 2) ||
      !make_map_atoms(&tb1, hsf, static_cast<uint64_t>(tiles) * (I / 128)) ||
      !make_map_atoms(&ts, wd_sf, static_cast<uint64_t>(E) * (d / 128) * (I / 128)) ||
      !make_map(&tc0, y, d, M, 64, 32))
    return MOE_ERR_CUDA;
  p.n_tiles = d / bn;
  p.k_blocks = I / 128;
  p.out = reinterpret_cast<__nv_bfloat16*>(y);
  p.out2 = nullptr;
  p.ld_out = d;
  if (bn == 256)
    return launch_pair_depth<FWD_DOWN, 256, true>(ta, tb0, tb1, tc0, tc0, tc0, ts, p,
                                                   mt_upper * p.n_tiles, st);
  return launch_pair_depth<FWD_DOWN, 128, true>(ta, tb0, tb1, tc0, tc0, tc0, ts, p,
                                                 mt_upper * p.n_tiles, st);
}

namespace moe {
MOE_DEBUG_STATUS_READER(gemm)
}  // namespace moe
