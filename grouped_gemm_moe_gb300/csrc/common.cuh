// Shared helpers of the MoE-layer kernels: status handling, argument checks,
// bf16 packing, warp reductions and per-device attributes.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

// Host side ------------------------------------------------------------------

void set_last_cuda_error(cudaError_t e);

inline int check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of SMs of the current device (cached per device).
int num_sms();
// Current device's compute capability major version (cached per device).
int cc_major();

constexpr size_t kWorkspaceHeader = 256;   // bytes; int32 status word at offset 0

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Per-launch timing hook (moe_profile_*): brackets one kernel launch with
// events on its stream while recording is on; a no-op otherwise.
void prof_begin(const char* name, cudaStream_t st);
void prof_end(cudaStream_t st);
struct ProfScope {
  cudaStream_t st;
  ProfScope(const char* name, cudaStream_t s) : st(s) { prof_begin(name, s); }
  ~ProfScope() { prof_end(st); }
};

// Launches a kernel with programmatic dependent launch: it may be scheduled
// while the previous kernel of the stream is still finishing, so it must run
// pdl_wait() before it reads anything an earlier launch wrote (every kernel of
// this library does so first thing). cluster_x > 1 adds a cluster dimension.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      unsigned cluster_x, const Args&... args) {
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return check_launch();
}

// Device side ----------------------------------------------------------------

// Programmatic dependent launch: wait until the grids this one depends on have
// completed and their memory is visible, then let the next launch of the
// stream be scheduled (its own pdl_wait() still waits for this grid to end).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Both, as the first statement of a kernel.
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_launch_dependents();
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Round two floats to bf16 (round to nearest even) and pack (lo in low half).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The exact product a*b prepared for one rounding to bf16 (to nearest, ties to
// even, by the caller's pack): rounded to odd at fp32 first (truncated toward
// zero, then the last bit set when the truncation was inexact, which the FMA
// residual a*b - trunc tells exactly). Rounding to odd at a precision at least
// two bits above the target's makes the second rounding (to nearest) correct:
// Boldo and Melquiond, "Emulation of FMA and correctly rounded sums: proved
// algorithms using rounding to odd" (IEEE Trans. Computers, 2008). The residual
// is exact while it is representable, i.e. for |a*b| above about 2^-103; below
// that a nonzero residual can round to zero and the odd bit be missed.
__device__ __forceinline__ float mul_bf16_exact(float a, float b) {
  const float pz = __fmul_rz(a, b);
  const float r = fmaf(a, b, -pz);
  return __uint_as_float(__float_as_uint(pz) | (r != 0.f ? 1u : 0u));
}

__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
  uint4 v;
  v.x = pack_bf16(f[0], f[1]);
  v.y = pack_bf16(f[2], f[3]);
  v.z = pack_bf16(f[4], f[5]);
  v.w = pack_bf16(f[6], f[7]);
  return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void stg_v4(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan of a[0..n) in shared memory by one warp (called by that warp
// only): each lane sums a run of ceil(n / 32) consecutive entries, one warp
// scan offsets the runs, and each lane rewrites its run (integer sums: exact in
// any order).
__device__ __forceinline__ void warp_exscan(int* a, int n) {
  const int lane = threadIdx.x & 31;
  const int per = (n + 31) >> 5;
  const int b = min(lane * per, n), e = min(b + per, n);
  int sum = 0;
  for (int i = b; i < e; ++i) sum += a[i];
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  int run = x - sum;
  for (int i = b; i < e; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
}

// Records a device-side error code in the workspace status word (first one wins).
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Debug builds (-DMOE_DEBUG_CHECKS): every gathered or scattered index is
// range-checked before its access and the GEMM tile scheduler checks the
// expert offsets. A failed check skips or redirects the access to a valid row
// and records MOE_ERR_DEVICE_CHECK in the translation unit's debug status word
// (read and cleared by moe_debug_check_status). Release builds compile the
// checks away.
#ifdef MOE_DEBUG_CHECKS
static __device__ int g_debug_status;   // one per translation unit
__device__ __forceinline__ bool index_ok(bool ok) {
  if (!ok) atomicCAS(&g_debug_status, 0, static_cast<int>(MOE_ERR_DEVICE_CHECK));
  return ok;
}
// Host side: this translation unit's debug status word, read and cleared.
#define MOE_DEBUG_STATUS_READER(name)                                                   \
  int debug_status_##name() {                                                           \
    int v = 0, z = 0;                                                                   \
    if (cudaMemcpyFromSymbol(&v, g_debug_status, sizeof(int)) != cudaSuccess ||         \
        cudaMemcpyToSymbol(g_debug_status, &z, sizeof(int)) != cudaSuccess)            \
      return MOE_ERR_CUDA;                                                              \
    return v;                                                                           \
  }
#else
__device__ __forceinline__ bool index_ok(bool) { return true; }
#define MOE_DEBUG_STATUS_READER(name)
#endif

}  // namespace moe
