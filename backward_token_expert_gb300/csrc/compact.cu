// Step 4 of the path: physical compaction (LRMoE sec. 3.1, 3.3 and 3.4,
// Fig. 4; weighted cotangent of appendix eq. (5)).  The retained gradient
// rows and their saved FC2 inputs are gathered into contiguous expert-major
// segments, in the order selection emitted them:
//   delta_c[r] = bf16_rne(alpha_u * g_t)   (one fp32 multiply per element)
//   phi_c[r]   = phi_u                     (bit copy)
//   alpha_c[r] = alpha_u
// for u = sel_ids[r], t = u / k, r < sel_offsets[E].  HBM-bound: per retained
// row it reads 2h + 2I bytes and writes the same.
//
// Also the zero-masked, capacity-padded layout of sec. 3.4 used as the
// measurement comparator.
#include "lrm_internal.cuh"
#include "vec.cuh"

namespace lrm {
namespace {

constexpr int CP_THREADS = 256;
constexpr int CP_WARPS = CP_THREADS / 32;

__device__ __forceinline__ void copy_scaled_row(const uint4* __restrict__ src, uint4* __restrict__ dst, int nv,
                                                float a, int lane) {
  int v = lane;
  for (; v + 96 < nv; v += 128) {
    const uint4 x0 = ld_stream(src + v);
    const uint4 x1 = ld_stream(src + v + 32);
    const uint4 x2 = ld_stream(src + v + 64);
    const uint4 x3 = ld_stream(src + v + 96);
    st_v4(dst + v, scale_bf16x8(x0, a));
    st_v4(dst + v + 32, scale_bf16x8(x1, a));
    st_v4(dst + v + 64, scale_bf16x8(x2, a));
    st_v4(dst + v + 96, scale_bf16x8(x3, a));
  }
  for (; v < nv; v += 32) st_v4(dst + v, scale_bf16x8(ld_stream(src + v), a));
}

__device__ __forceinline__ void copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst, int nv,
                                         int lane) {
  int v = lane;
  for (; v + 96 < nv; v += 128) {
    const uint4 x0 = ld_stream(src + v);
    const uint4 x1 = ld_stream(src + v + 32);
    const uint4 x2 = ld_stream(src + v + 64);
    const uint4 x3 = ld_stream(src + v + 96);
    st_v4(dst + v, x0);
    st_v4(dst + v + 32, x1);
    st_v4(dst + v + 64, x2);
    st_v4(dst + v + 96, x3);
  }
  for (; v < nv; v += 32) st_v4(dst + v, ld_stream(src + v));
}

__device__ __forceinline__ void zero_row(uint4* __restrict__ dst, int nv, int lane) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int v = lane; v < nv; v += 32) st_v4(dst + v, z);
}

__global__ void __launch_bounds__(CP_THREADS) compact_kernel(
    const uint4* __restrict__ g, const uint4* __restrict__ phi, const float* __restrict__ alpha,
    const int32_t* __restrict__ sel_offsets, const int32_t* __restrict__ sel_ids, int E, int N, int k, int hv,
    int iv, int max_rows, uint4* __restrict__ delta_c, uint4* __restrict__ phi_c, float* __restrict__ alpha_c,
    unsigned int* status) {
  const int lane = threadIdx.x & 31;
  int total = __ldg(sel_offsets + E);
  if (total > max_rows) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_flag(status, LRM_ERR_SHAPE);
    total = max_rows;
  }
  const int warps_total = gridDim.x * CP_WARPS;
  for (int r = blockIdx.x * CP_WARPS + (threadIdx.x >> 5); r < total; r += warps_total) {
    const int u = __ldg(sel_ids + r);
    if (u < 0 || u >= N) {
      if (lane == 0) raise_flag(status, LRM_ERR_INDEX);
      continue;
    }
    const float a = __ldg(alpha + u);
    const int t = u / k;
    copy_scaled_row(g + static_cast<size_t>(t) * hv, delta_c + static_cast<size_t>(r) * hv, hv, a, lane);
    copy_row(phi + static_cast<size_t>(u) * iv, phi_c + static_cast<size_t>(r) * iv, iv, lane);
    if (alpha_c != nullptr && lane == 0) alpha_c[r] = a;
  }
}

__global__ void __launch_bounds__(CP_THREADS) compact_padded_kernel(
    const uint4* __restrict__ delta_c, const uint4* __restrict__ phi_c, const int32_t* __restrict__ sel_offsets,
    int E, int C, int hv, int iv, uint4* __restrict__ delta_pad, uint4* __restrict__ phi_pad,
    int32_t* __restrict__ pad_offsets, unsigned int* status) {
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += CP_THREADS) pad_offsets[e] = e * C;
  const long long slots = static_cast<long long>(E) * C;
  const int warps_total = gridDim.x * CP_WARPS;
  for (long long i = blockIdx.x * CP_WARPS + (threadIdx.x >> 5); i < slots; i += warps_total) {
    const int e = static_cast<int>(i / C);
    const int s = static_cast<int>(i % C);
    const int start = __ldg(sel_offsets + e);
    int q = __ldg(sel_offsets + e + 1) - start;
    if (q > C) {
      if (s == 0 && lane == 0) raise_flag(status, LRM_ERR_SHAPE);
      q = C;
    }
    uint4* dd = delta_pad + static_cast<size_t>(i) * hv;
    uint4* pd = phi_pad + static_cast<size_t>(i) * iv;
    if (s < q) {
      copy_row(delta_c + static_cast<size_t>(start + s) * hv, dd, hv, lane);
      copy_row(phi_c + static_cast<size_t>(start + s) * iv, pd, iv, lane);
    } else {
      zero_row(dd, hv, lane);
      zero_row(pd, iv, lane);
    }
  }
}

}  // namespace
}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_compact(lrm_ctx* ctx, const uint16_t* g, const uint16_t* phi, const float* alpha,
                                  const int32_t* sel_offsets, const int32_t* sel_ids, lrm_dims dims,
                                  int32_t max_rows, uint16_t* delta_c, uint16_t* phi_c, float* alpha_c,
                                  void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0) return LRM_ERR_INVALID_ARG;
  if (sel_offsets == nullptr) return LRM_ERR_INVALID_ARG;
  if (max_rows == 0) return LRM_OK;
  if (g == nullptr || phi == nullptr || alpha == nullptr || sel_ids == nullptr || delta_c == nullptr ||
      phi_c == nullptr)
    return LRM_ERR_INVALID_ARG;
  if (!aligned(g, 16) || !aligned(phi, 16) || !aligned(delta_c, 16) || !aligned(phi_c, 16) ||
      !aligned(alpha, 4) || !aligned(sel_offsets, 4) || !aligned(sel_ids, 4) ||
      (alpha_c != nullptr && !aligned(alpha_c, 4)))
    return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  static thread_local int cap_device = -1, cap = 0;
  if (cap_device != ctx->device) {
    cap = resident_grid(ctx, compact_kernel, CP_THREADS, 0);
    cap_device = ctx->device;
  }
  const int need = (max_rows + CP_WARPS - 1) / CP_WARPS;
  const int grid = need < cap ? need : cap;
  compact_kernel<<<grid, CP_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(g), reinterpret_cast<const uint4*>(phi), alpha, sel_offsets, sel_ids,
      dims.E, dims.T * dims.k, dims.k, dims.h / 8, dims.I / 8, max_rows, reinterpret_cast<uint4*>(delta_c),
      reinterpret_cast<uint4*>(phi_c), alpha_c, ctx->d_status);
  return launch_status();
}

extern "C" lrm_status lrm_compact_padded(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* phi_c,
                                         const int32_t* sel_offsets, lrm_dims dims, int32_t C,
                                         uint16_t* delta_pad, uint16_t* phi_pad, int32_t* pad_offsets,
                                         void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (C < 0 || (long long)C * dims.E >= (1ll << 31)) return LRM_ERR_SHAPE;
  if (sel_offsets == nullptr || pad_offsets == nullptr) return LRM_ERR_INVALID_ARG;
  if (C > 0 && (delta_c == nullptr || phi_c == nullptr || delta_pad == nullptr || phi_pad == nullptr))
    return LRM_ERR_INVALID_ARG;
  if (!aligned(delta_c, 16) || !aligned(phi_c, 16) || !aligned(delta_pad, 16) || !aligned(phi_pad, 16) ||
      !aligned(sel_offsets, 4) || !aligned(pad_offsets, 4))
    return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  const long long slots = static_cast<long long>(dims.E) * C;
  long long need = (slots + CP_WARPS - 1) / CP_WARPS;
  if (need < 1) need = 1;
  static thread_local int cap_device = -1, cap = 0;
  if (cap_device != ctx->device) {
    cap = resident_grid(ctx, compact_padded_kernel, CP_THREADS, 0);
    cap_device = ctx->device;
  }
  const int grid = static_cast<int>(need < cap ? need : cap);
  compact_padded_kernel<<<grid, CP_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(delta_c), reinterpret_cast<const uint4*>(phi_c), sel_offsets, dims.E, C,
      dims.h / 8, dims.I / 8, reinterpret_cast<uint4*>(delta_pad), reinterpret_cast<uint4*>(phi_pad),
      pad_offsets, ctx->d_status);
  return launch_status();
}
