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

// TMA-staged gather (the default when a row pair fits the ring): each warp
// owns a ring of `depth` slots in shared memory, one retained row per slot.
// Lane 0 fetches the row's g_t and phi_u with two bulk copies that complete
// on the slot's mbarrier; the warp scales g_t by alpha_u in place (fp32
// multiply, round to nearest even); lane 0 then writes the slot out to
// delta_c[r] and phi_c[r] with two bulk stores and, once the previous row's
// stores have read their slot, refills that slot with the row `depth` ahead.
// The copies run in the async proxy, so each warp keeps up to `depth` rows
// of loads and stores in flight with one thread issuing them.
constexpr int CT_WARPS = 4;
constexpr int CT_THREADS = 32 * CT_WARPS;
constexpr int CT_MAX_DEPTH = 4;

__global__ void __launch_bounds__(CT_THREADS) compact_tma_kernel(
    const uint8_t* __restrict__ g, const uint8_t* __restrict__ phi, const float* __restrict__ alpha,
    const int32_t* __restrict__ sel_offsets, const int32_t* __restrict__ sel_ids, int E, int N, int k,
    uint32_t gbytes, uint32_t pbytes, uint32_t slot_bytes, int depth, int max_rows, uint8_t* __restrict__ delta_c,
    uint8_t* __restrict__ phi_c, float* __restrict__ alpha_c, unsigned int* status, unsigned long long budget_ns) {
  extern __shared__ __align__(128) uint8_t ct_smem[];
  __shared__ __align__(8) uint64_t bars[CT_WARPS][CT_MAX_DEPTH];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int total = __ldg(sel_offsets + E);
  if (total > max_rows) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_flag(status, LRM_ERR_SHAPE);
    total = max_rows;
  }
  if (lane == 0) {
    for (int s = 0; s < depth; ++s) mbar_init(&bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  uint8_t* ring = ct_smem + static_cast<size_t>(warp) * depth * slot_bytes;
  const uint32_t g_off = (gbytes + 127u) & ~127u;  // phi part of a slot
  const int gw = blockIdx.x * CT_WARPS + warp;
  const int W = gridDim.x * CT_WARPS;
  // rows gw, gw + W, ... of this warp
  const int n_rows = gw < total ? static_cast<int>((static_cast<long long>(total) - gw + W - 1) / W) : 0;

  // lane 0: fetch the i-th row of this warp into slot i % depth
  auto issue = [&](int i) {
    uint64_t* bar = &bars[warp][i % depth];
    uint8_t* slot = ring + static_cast<size_t>(i % depth) * slot_bytes;
    const int u = __ldg(sel_ids + gw + static_cast<size_t>(i) * W);
    if (u < 0 || u >= N) {
      raise_flag(status, LRM_ERR_INDEX);
      mbar_arrive(bar);  // completes the phase with nothing loaded; the row is skipped
      return;
    }
    mbar_arrive_expect_tx(bar, gbytes + pbytes);
    bulk_load(slot, g + static_cast<size_t>(u / k) * gbytes, gbytes, bar);
    bulk_load(slot + g_off, phi + static_cast<size_t>(u) * pbytes, pbytes, bar);
  };
  if (lane == 0)
    for (int i = 0; i < depth && i < n_rows; ++i) issue(i);
  int issued = depth < n_rows ? depth : n_rows;

  int i = 0;
  for (; i < n_rows; ++i) {
    const int s = i % depth;
    const bool got = mbar_wait(&bars[warp][s], static_cast<uint32_t>(i / depth) & 1u, budget_ns, nullptr);
    if (!__all_sync(0xffffffffu, got)) {  // the whole warp leaves together
      if (lane == 0) raise_flag(status, LRM_ERR_TIMEOUT);
      break;
    }
    const size_t r = gw + static_cast<size_t>(i) * W;
    const int u = __ldg(sel_ids + r);
    uint8_t* slot = ring + static_cast<size_t>(s) * slot_bytes;
    if (u >= 0 && u < N) {
      const float a = __ldg(alpha + u);
      uint4* gv = reinterpret_cast<uint4*>(slot);
      for (uint32_t v = lane; v < gbytes / 16; v += 32) gv[v] = scale_bf16x8(gv[v], a);
      fence_proxy_async_smem();  // the scaled row, written by the warp, is read by the bulk store
      __syncwarp();
      if (lane == 0) {
        bulk_store(delta_c + r * gbytes, slot, gbytes);
        bulk_store(phi_c + r * pbytes, slot + g_off, pbytes);
        if (alpha_c != nullptr) alpha_c[r] = a;
      }
    }
    if (lane == 0) {
      bulk_commit();  // one group per row (empty for a skipped row)
      // the previous row's stores have read their slot: refill it `depth` rows ahead
      if (i >= 1 && issued < n_rows) {
        bulk_wait_read<1>();
        issue(issued);
        ++issued;
      }
    }
    __syncwarp();
  }
  if (lane == 0) {
    // after a timeout, let the fetches already issued land before the block exits
    for (int j = i; j < issued; ++j)
      if (!mbar_wait(&bars[warp][j % depth], static_cast<uint32_t>(j / depth) & 1u, budget_ns, nullptr)) break;
    bulk_wait<0>();
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // TMA-staged gather when a ring of at least two row slots per warp fits in
  // shared memory (every shape up to h + I of about 13k)
  const uint32_t gbytes = static_cast<uint32_t>(dims.h) * 2, pbytes = static_cast<uint32_t>(dims.I) * 2;
  const uint32_t slot = ((gbytes + 127u) & ~127u) + ((pbytes + 127u) & ~127u);
  const size_t smem_cap = static_cast<size_t>(ctx->smem_optin) - 1024;  // static barriers and slack
  int depth = CT_MAX_DEPTH;
  while (depth >= 2 && static_cast<size_t>(CT_WARPS) * depth * slot > smem_cap) --depth;
  if (depth >= 2) {
    static thread_local int tma_device = -1;
    if (tma_device != ctx->device) {
      LRM_CHECK_CUDA(cudaFuncSetAttribute(compact_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem_cap)));
      tma_device = ctx->device;
    }
    const size_t smem = static_cast<size_t>(CT_WARPS) * depth * slot;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compact_tma_kernel, CT_THREADS, smem) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    const long long need = (static_cast<long long>(max_rows) + CT_WARPS - 1) / CT_WARPS;
    const long long cap = static_cast<long long>(per_sm) * ctx->sm_count;
    const int grid = static_cast<int>(need < cap ? need : cap);
    compact_tma_kernel<<<grid, CT_THREADS, smem, s>>>(
        reinterpret_cast<const uint8_t*>(g), reinterpret_cast<const uint8_t*>(phi), alpha, sel_offsets, sel_ids,
        dims.E, dims.T * dims.k, dims.k, gbytes, pbytes, slot, depth, max_rows, reinterpret_cast<uint8_t*>(delta_c),
        reinterpret_cast<uint8_t*>(phi_c), alpha_c, ctx->d_status, ctx->wait_budget_ns);
    return launch_status();
  }
  static thread_local int cap_device = -1, cap = 0;
  if (cap_device != ctx->device) {
    cap = resident_grid(ctx, compact_kernel, CP_THREADS, 0);
    cap_device = ctx->device;
  }
  const int need = (max_rows + CP_WARPS - 1) / CP_WARPS;
  const int grid = need < cap ? need : cap;
  compact_kernel<<<grid, CP_THREADS, 0, s>>>(
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
