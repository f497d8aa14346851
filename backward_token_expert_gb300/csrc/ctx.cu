// Context lifetime, status word, workspace queries and the bounded-wait
// self test of the library.
#include <stdlib.h>

#include "lrm_internal.cuh"

using namespace lrm;

namespace lrm {
size_t route_stats_workspace_bytes(const lrm_dims& d);
size_t select_workspace_bytes(const lrm_dims& d);
size_t zero_dropped_workspace_bytes(const lrm_dims& d);
size_t combine_workspace_bytes(const lrm_dims& d);
}  // namespace lrm

namespace {

__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    // Nothing ever arrives on `bar`, so phase 0 never completes.
    if (!mbar_wait(&bar, 0, budget_ns, nullptr)) raise_flag(status, LRM_ERR_TIMEOUT);
  }
}

}  // namespace

extern "C" {

const char* lrm_status_string(lrm_status s) {
  switch (s) {
    case LRM_OK: return "LRM_OK";
    case LRM_ERR_INVALID_ARG: return "LRM_ERR_INVALID_ARG";
    case LRM_ERR_SHAPE: return "LRM_ERR_SHAPE";
    case LRM_ERR_ALIGN: return "LRM_ERR_ALIGN";
    case LRM_ERR_WORKSPACE: return "LRM_ERR_WORKSPACE";
    case LRM_ERR_INDEX: return "LRM_ERR_INDEX";
    case LRM_ERR_QUOTA: return "LRM_ERR_QUOTA";
    case LRM_ERR_TIMEOUT: return "LRM_ERR_TIMEOUT";
    case LRM_ERR_ARCH: return "LRM_ERR_ARCH";
    case LRM_ERR_CUDA: return "LRM_ERR_CUDA";
  }
  return "LRM_ERR_UNKNOWN";
}

int32_t lrm_abi_version(void) { return LRM_ABI_VERSION; }

lrm_status lrm_create(int device, lrm_ctx** out) {
  if (out == nullptr) return LRM_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return LRM_ERR_CUDA;
  if (device < 0 || device >= ndev) return LRM_ERR_INVALID_ARG;
  DeviceGuard guard(device);
  if (!guard.ok) return LRM_ERR_CUDA;
  cudaDeviceProp prop;
  LRM_CHECK_CUDA(cudaGetDeviceProperties(&prop, device));
  if (prop.major != 10 || prop.minor != 3) return LRM_ERR_ARCH;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, selftest_wait_kernel) != cudaSuccess) {
    cudaGetLastError();
    return LRM_ERR_ARCH;
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return LRM_ERR_CUDA;
  lrm_ctx* c = static_cast<lrm_ctx*>(calloc(1, sizeof(lrm_ctx)));
  if (c == nullptr) return LRM_ERR_CUDA;
  c->device = device;
  c->sm_count = prop.multiProcessorCount;
  c->smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
  c->wait_budget_ns = 2000000000ull;
  c->encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  if (cudaMalloc(&c->d_status, sizeof(unsigned int)) != cudaSuccess ||
      cudaMemset(c->d_status, 0, sizeof(unsigned int)) != cudaSuccess) {
    if (c->d_status) cudaFree(c->d_status);
    free(c);
    return LRM_ERR_CUDA;
  }
  *out = c;
  return LRM_OK;
}

lrm_status lrm_destroy(lrm_ctx* ctx) {
  if (ctx == nullptr) return LRM_OK;
  DeviceGuard guard(ctx->device);
  if (ctx->d_status) cudaFree(ctx->d_status);
  free(ctx);
  return LRM_OK;
}

lrm_status lrm_sm_count(const lrm_ctx* ctx, int32_t* out) {
  if (ctx == nullptr || out == nullptr) return LRM_ERR_INVALID_ARG;
  *out = ctx->sm_count;
  return LRM_OK;
}

lrm_status lrm_workspace_size(const lrm_ctx* ctx, lrm_op op, lrm_dims dims, size_t* bytes) {
  if (ctx == nullptr || bytes == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  switch (op) {
    case LRM_OP_ROUTE_STATS: *bytes = route_stats_workspace_bytes(dims); return LRM_OK;
    case LRM_OP_SELECT: *bytes = select_workspace_bytes(dims); return LRM_OK;
    case LRM_OP_ZERO_DROPPED: *bytes = zero_dropped_workspace_bytes(dims); return LRM_OK;
    case LRM_OP_COMBINE: *bytes = combine_workspace_bytes(dims); return LRM_OK;
  }
  return LRM_ERR_INVALID_ARG;
}

lrm_status lrm_get_device_status(lrm_ctx* ctx, void* stream, uint32_t* flags) {
  if (ctx == nullptr || flags == nullptr) return LRM_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  LRM_CHECK_CUDA(cudaMemcpyAsync(&host, ctx->d_status, sizeof(unsigned int), cudaMemcpyDeviceToHost, s));
  LRM_CHECK_CUDA(cudaStreamSynchronize(s));
  LRM_CHECK_CUDA(cudaMemsetAsync(ctx->d_status, 0, sizeof(unsigned int), s));
  LRM_CHECK_CUDA(cudaStreamSynchronize(s));
  *flags = host;
  return LRM_OK;
}

lrm_status lrm_set_wait_budget(lrm_ctx* ctx, uint64_t ns) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  ctx->wait_budget_ns = ns;
  return LRM_OK;
}

lrm_status lrm_selftest_wait_timeout(lrm_ctx* ctx, uint64_t budget_ns, void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  if (budget_ns > 10000000000ull) return LRM_ERR_INVALID_ARG;  // at most 10 s
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ctx->d_status, budget_ns);
  return launch_status();
}

}  // extern "C"
