// Library-wide entry points: workspace sizes, device status word, status
// strings, error bookkeeping and cached device attributes.
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"

namespace moe {

size_t permutation_workspace(long long TK, int E, int R);   // permute.cu
size_t ffn_backward_scratch(long long M, int E, int d, int I);   // grouped_gemm.cu
size_t load_balance_workspace(int E);                       // route.cu
size_t ffn_fp8_scratch(long long M, int E, int d, int I);   // grouped_gemm.cu
size_t route_permute_workspace(long long TK, int E, int R);   // front.cu

namespace {
thread_local int g_last_cuda_error = 0;
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};
int g_major[kMaxDevices] = {0};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}
}  // namespace

void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

namespace {
struct ProfRec {
  const char* name;
  cudaEvent_t a;
  cudaEvent_t b;
};
ProfRec* g_prof = nullptr;
int g_prof_cap = 0;       // events allocated
int g_prof_limit = 0;     // records allowed in this session
int g_prof_n = 0;         // records taken
bool g_prof_on = false;
bool g_prof_open = false; // a begin without its end
}  // namespace

void prof_begin(const char* name, cudaStream_t st) {
  if (!g_prof_on || g_prof_n >= g_prof_limit) return;
  g_prof[g_prof_n].name = name;
  cudaEventRecord(g_prof[g_prof_n].a, st);
  g_prof_open = true;
}

void prof_end(cudaStream_t st) {
  if (!g_prof_on || !g_prof_open) return;
  cudaEventRecord(g_prof[g_prof_n].b, st);
  g_prof_open = false;
  ++g_prof_n;
}

int num_sms() {
  const int dev = current_device();
  if (!g_sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = v > 0 ? v : 1;
  }
  return g_sms[dev];
}

int cc_major() {
  const int dev = current_device();
  if (!g_major[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev);
    g_major[dev] = v > 0 ? v : -1;
  }
  return g_major[dev];
}

}  // namespace moe

extern "C" size_t moe_workspace_size(int op, int T, int E, int K, int R, int d, int I) {
  using namespace moe;
  if (T < 0 || E < 1 || K < 1) return 0;
  const long long TK = static_cast<long long>(T) * K;
  switch (op) {
    case MOE_OP_BUILD_PERMUTATION:
      return permutation_workspace(TK, E, 1);
    case MOE_OP_EP_LAYOUT:
      if (R < 1 || E % R || T % R) return 0;
      return permutation_workspace(TK, E, R);
    case MOE_OP_GROUPED_FFN:
      return kWorkspaceHeader;
    case MOE_OP_GROUPED_FFN_BACKWARD:
      if (I < 1 || d < 1) return 0;
      return kWorkspaceHeader + ffn_backward_scratch(TK, E, d, I);
    case MOE_OP_LOAD_BALANCE:
      return load_balance_workspace(E);
    case MOE_OP_EP_RECV_LAYOUT:
      return kWorkspaceHeader;
    case MOE_OP_ROUTE_PERMUTE_EP:
      if (R < 1 || E % R || T % R) return 0;
      return route_permute_workspace(TK, E, R);
    case MOE_OP_GROUPED_FFN_FP8:
      if (I < 128 || d < 128 || d % 128 || I % 128) return 0;
      return kWorkspaceHeader + ffn_fp8_scratch(TK, E, d, I);
    default:
      return 0;
  }
}

#ifdef MOE_DEBUG_CHECKS
namespace moe {
int debug_status_route();
int debug_status_permute();
int debug_status_gather();
int debug_status_ep();
int debug_status_fp8();
int debug_status_gemm();
}  // namespace moe
#endif

extern "C" int moe_debug_check_status(int* host_status) {
  if (!host_status) return MOE_ERR_INVALID_ARG;
#ifdef MOE_DEBUG_CHECKS
  using namespace moe;
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  int first = 0;
  for (int v : {debug_status_route(), debug_status_permute(), debug_status_gather(),
                debug_status_ep(), debug_status_fp8(), debug_status_gemm()}) {
    if (v == MOE_ERR_CUDA) return MOE_ERR_CUDA;
    if (!first) first = v;
  }
  *host_status = first;
  return MOE_OK;
#else
  *host_status = 0;
  return MOE_ERR_UNSUPPORTED;
#endif
}

extern "C" int moe_read_device_status(void* ws, void* stream, int* host_status) {
  using namespace moe;
  if (!ws || !host_status) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int), st);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  *host_status = v;
  return MOE_OK;
}

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

extern "C" int moe_profile_start(int capacity) {
  using namespace moe;
  if (capacity < 1) return MOE_ERR_INVALID_ARG;
  if (capacity > g_prof_cap) {
    ProfRec* n = static_cast<ProfRec*>(realloc(g_prof, sizeof(ProfRec) * capacity));
    if (!n) return MOE_ERR_INVALID_ARG;
    g_prof = n;
    for (int i = g_prof_cap; i < capacity; ++i) {
      g_prof[i].name = "";
      cudaError_t e = cudaEventCreate(&g_prof[i].a);
      if (e == cudaSuccess) e = cudaEventCreate(&g_prof[i].b);
      if (e != cudaSuccess) {
        g_prof_cap = i;
        set_last_cuda_error(e);
        return MOE_ERR_CUDA;
      }
    }
    g_prof_cap = capacity;
  }
  g_prof_limit = capacity;
  g_prof_n = 0;
  g_prof_open = false;
  g_prof_on = true;
  return MOE_OK;
}

extern "C" int moe_profile_stop(void) {
  moe::g_prof_on = false;
  return moe::g_prof_n;
}

extern "C" int moe_profile_record(int i, const char** name, float* ms) {
  using namespace moe;
  if (i < 0 || i >= g_prof_n || !name || !ms) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaEventSynchronize(g_prof[i].b);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, g_prof[i].a, g_prof[i].b);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  *name = g_prof[i].name;
  return MOE_OK;
}

extern "C" int moe_last_cuda_error(void) { return moe::g_last_cuda_error; }

extern "C" int moe_version(void) { return 200; }
