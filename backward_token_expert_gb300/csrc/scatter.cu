// The inverse mapping of LRMoE (sec. 1 and 3.3; Alg. 1, ScatterWithZeros;
// sec. 3.4): every kept row returns to the slot its pair had before
// compaction, and the slots of dropped pairs are filled with zeros so that
// the next dense layer sees the layout it expects.
// lrm_grouped_dgrad_scatter writes every retained row of the input gradient
// to its pair's row; this file zeroes the rows of the pairs that were not
// retained.  Two launches:
//   mark_kernel   one thread per retained row sets bit sel_ids[r] of an
//                 N-bit map (the map is cleared on the stream first);
//   zero_kernel   one warp per pair row: rows whose bit is clear are written
//                 with zeros (16-byte stores; HBM-bound, no reads but the map).
#include "lrm_internal.cuh"

namespace lrm {
namespace {

constexpr int ZR_THREADS = 256;
constexpr int ZR_WARPS = ZR_THREADS / 32;

__global__ void __launch_bounds__(ZR_THREADS) mark_kernel(const int32_t* __restrict__ sel_offsets, int E,
                                                          const int32_t* __restrict__ sel_ids, int max_rows, int N,
                                                          uint32_t* __restrict__ bits, unsigned int* status) {
  const int total = min(max(__ldg(sel_offsets + E), 0), max_rows);
  for (int r = blockIdx.x * ZR_THREADS + threadIdx.x; r < total; r += gridDim.x * ZR_THREADS) {
    const int u = __ldg(sel_ids + r);
    if (u < 0 || u >= N) {
      raise_flag(status, LRM_ERR_INDEX);
      continue;
    }
    atomicOr(bits + (u >> 5), 1u << (u & 31));
  }
}

__global__ void __launch_bounds__(ZR_THREADS) zero_kernel(const uint32_t* __restrict__ bits, int N, int iv,
                                                          uint4* __restrict__ rows) {
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * ZR_WARPS;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int u = blockIdx.x * ZR_WARPS + (threadIdx.x >> 5); u < N; u += warps_total) {
    if ((__ldg(bits + (u >> 5)) >> (u & 31)) & 1u) continue;  // retained: dgrad wrote it
    uint4* row = rows + static_cast<size_t>(u) * iv;
    for (int v = lane; v < iv; v += 32) row[v] = z;
  }
}

}  // namespace

size_t zero_dropped_workspace_bytes(const lrm_dims& d) {
  const size_t N = static_cast<size_t>(d.T) * d.k;
  return ((N + 31) / 32) * sizeof(uint32_t);
}

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_zero_dropped_rows(lrm_ctx* ctx, const int32_t* sel_offsets, const int32_t* sel_ids,
                                            lrm_dims dims, int32_t max_rows, uint16_t* rows, void* ws,
                                            size_t ws_bytes, void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0 || sel_offsets == nullptr) return LRM_ERR_INVALID_ARG;
  const int N = dims.T * dims.k;
  if (N == 0) return LRM_OK;
  if (rows == nullptr || ws == nullptr || (max_rows > 0 && sel_ids == nullptr)) return LRM_ERR_INVALID_ARG;
  if (ws_bytes < zero_dropped_workspace_bytes(dims)) return LRM_ERR_WORKSPACE;
  if (!aligned(rows, 16) || !aligned(ws, 4) || !aligned(sel_offsets, 4) || (sel_ids && !aligned(sel_ids, 4)))
    return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* bits = static_cast<uint32_t*>(ws);
  LRM_CHECK_CUDA(cudaMemsetAsync(bits, 0, zero_dropped_workspace_bytes(dims), s));
  if (max_rows > 0) {
    const int need = (max_rows + ZR_THREADS - 1) / ZR_THREADS;
    const int cap = ctx->sm_count * 4;
    mark_kernel<<<need < cap ? need : cap, ZR_THREADS, 0, s>>>(sel_offsets, dims.E, sel_ids, max_rows, N, bits,
                                                               ctx->d_status);
    if ((st = launch_status()) != LRM_OK) return st;
  }
  static thread_local int cap_device = -1, cap = 0;
  if (cap_device != ctx->device) {
    cap = resident_grid(ctx, zero_kernel, ZR_THREADS, 0);
    cap_device = ctx->device;
  }
  const int need = (N + ZR_WARPS - 1) / ZR_WARPS;
  zero_kernel<<<need < cap ? need : cap, ZR_THREADS, 0, s>>>(bits, N, dims.I / 8, reinterpret_cast<uint4*>(rows));
  return launch_status();
}
