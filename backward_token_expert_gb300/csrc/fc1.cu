// FC1 side of the expert backward on the retained pairs (LRMoE sec. 3.4:
// the compacted row count is the M or K of every expert-backward GEMM, the
// input- and weight-gradient products of both FC1 and FC2).  The activation is read as SwiGLU:
// FC1 gives [a | b] (gate, up; width 2I) and the FC2 input is
// phi = silu(a) * b.  The two FC1 GEMMs are the grouped dgrad / wgrad kernels
// with the dimensions relabelled (K = 2I); this file holds the two pieces
// around them:
//   swiglu_bwd_kernel   dh1 = [dphi * b * silu'(a) | dphi * silu(a)] for every
//                       compacted row, fp32 math, bf16 round-to-nearest-even;
//                       one warp per row, 16-byte vectors (HBM-bound);
//   map_kernel /        the FC1 input gradient of every token: the sum of the
//   combine_kernel      rows of its retained pairs (the inverse mapping and the
//                       MoE combine over its k experts), fp32 sums, bf16 out;
//                       a pair -> row map first, then one warp per token.
#include "lrm_internal.cuh"
#include "vec.cuh"

namespace lrm {
namespace {

constexpr int F1_THREADS = 256;
constexpr int F1_WARPS = F1_THREADS / 32;

__device__ __forceinline__ float silu_grad(float a, float& silu) {
  const float s = 1.0f / (1.0f + expf(-a));
  silu = a * s;
  return s * (1.0f + a * (1.0f - s));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// one bf16 pair (2 columns) of a row: dphi word d, gate word a, up word b
__device__ __forceinline__ void swiglu_pair(uint32_t d, uint32_t a, uint32_t b, uint32_t& da, uint32_t& db) {
  float s0, s1;
  const float g0 = silu_grad(bf16_lo(a), s0), g1 = silu_grad(bf16_hi(a), s1);
  const float d0 = bf16_lo(d), d1 = bf16_hi(d);
  da = pack_bf16x2(d0 * bf16_lo(b) * g0, d1 * bf16_hi(b) * g1);
  db = pack_bf16x2(d0 * s0, d1 * s1);
}

__global__ void __launch_bounds__(F1_THREADS) swiglu_bwd_kernel(const uint4* __restrict__ dphi,
                                                                const uint4* __restrict__ ab,
                                                                const int32_t* __restrict__ sel_offsets, int E,
                                                                int max_rows, int iv, uint4* __restrict__ dh1) {
  const int lane = threadIdx.x & 31;
  const int rows = min(max(__ldg(sel_offsets + E), 0), max_rows);
  const int warps_total = gridDim.x * F1_WARPS;
  for (int r = blockIdx.x * F1_WARPS + (threadIdx.x >> 5); r < rows; r += warps_total) {
    const uint4* drow = dphi + static_cast<size_t>(r) * iv;
    const uint4* arow = ab + static_cast<size_t>(r) * 2 * iv;
    uint4* orow = dh1 + static_cast<size_t>(r) * 2 * iv;
    for (int v = lane; v < iv; v += 32) {
      const uint4 d = ld_stream(drow + v), a = ld_stream(arow + v), b = ld_stream(arow + iv + v);
      uint4 da, db;
      swiglu_pair(d.x, a.x, b.x, da.x, db.x);
      swiglu_pair(d.y, a.y, b.y, da.y, db.y);
      swiglu_pair(d.z, a.z, b.z, da.z, db.z);
      swiglu_pair(d.w, a.w, b.w, da.w, db.w);
      orow[v] = da;
      orow[iv + v] = db;
    }
  }
}

// pos[sel_ids[r]] = r (pos was set to -1 on the stream first)
__global__ void __launch_bounds__(F1_THREADS) map_kernel(const int32_t* __restrict__ sel_offsets, int E,
                                                         const int32_t* __restrict__ sel_ids, int max_rows, int N,
                                                         int32_t* __restrict__ pos, unsigned int* status) {
  const int rows = min(max(__ldg(sel_offsets + E), 0), max_rows);
  for (int r = blockIdx.x * F1_THREADS + threadIdx.x; r < rows; r += gridDim.x * F1_THREADS) {
    const int u = __ldg(sel_ids + r);
    if (u < 0 || u >= N) {
      raise_flag(status, LRM_ERR_INDEX);
      continue;
    }
    pos[u] = r;
  }
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4& x) {
  acc[0] += bf16_lo(x.x);
  acc[1] += bf16_hi(x.x);
  acc[2] += bf16_lo(x.y);
  acc[3] += bf16_hi(x.y);
  acc[4] += bf16_lo(x.z);
  acc[5] += bf16_hi(x.z);
  acc[6] += bf16_lo(x.w);
  acc[7] += bf16_hi(x.w);
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  return make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                    pack_bf16x2(acc[6], acc[7]));
}

// out[t] = bf16(sum over the retained pairs u of t, in slot order, of
// rows[pos[u]]); one warp per token.  The warp first moves the row indices of
// its retained pairs to its low lanes (n of them), then each lane sums two
// 16-byte chunks of the row at a time with up to eight loads in flight.
__global__ void __launch_bounds__(F1_THREADS) combine_kernel(const uint4* __restrict__ rows,
                                                             const int32_t* __restrict__ pos, int T, int k, int wv,
                                                             uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * F1_WARPS;
  for (int t = blockIdx.x * F1_WARPS + (threadIdx.x >> 5); t < T; t += warps_total) {
    const int my = lane < k ? __ldg(pos + static_cast<size_t>(t) * k + lane) : -1;
    const unsigned kept = __ballot_sync(0xffffffffu, my >= 0);
    const int n = __popc(kept);
    const unsigned src = __fns(kept, 0, lane + 1);  // slot of the (lane+1)-th kept pair
    const int row = __shfl_sync(0xffffffffu, my, static_cast<int>(src & 31u));
    uint4* orow = out + static_cast<size_t>(t) * wv;
    for (int v0 = 0; v0 < wv; v0 += 64) {  // uniform trip count: the shuffles below need every lane
      const int va = v0 + lane, vb = va + 32;
      const bool ia = va < wv, ib = vb < wv;
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      int j = 0;
      for (; j + 4 <= n; j += 4) {
        const int r0 = __shfl_sync(0xffffffffu, row, j), r1 = __shfl_sync(0xffffffffu, row, j + 1);
        const int r2 = __shfl_sync(0xffffffffu, row, j + 2), r3 = __shfl_sync(0xffffffffu, row, j + 3);
        const uint4* p0 = rows + static_cast<size_t>(r0) * wv;
        const uint4* p1 = rows + static_cast<size_t>(r1) * wv;
        const uint4* p2 = rows + static_cast<size_t>(r2) * wv;
        const uint4* p3 = rows + static_cast<size_t>(r3) * wv;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint4 xa0 = ia ? ld_stream(p0 + va) : z, xa1 = ia ? ld_stream(p1 + va) : z;
        const uint4 xa2 = ia ? ld_stream(p2 + va) : z, xa3 = ia ? ld_stream(p3 + va) : z;
        const uint4 xb0 = ib ? ld_stream(p0 + vb) : z, xb1 = ib ? ld_stream(p1 + vb) : z;
        const uint4 xb2 = ib ? ld_stream(p2 + vb) : z, xb3 = ib ? ld_stream(p3 + vb) : z;
        add8(a, xa0);
        add8(a, xa1);
        add8(a, xa2);
        add8(a, xa3);
        add8(b, xb0);
        add8(b, xb1);
        add8(b, xb2);
        add8(b, xb3);
      }
      for (; j < n; ++j) {
        const int r = __shfl_sync(0xffffffffu, row, j);
        const uint4* pr = rows + static_cast<size_t>(r) * wv;
        if (ia) add8(a, ld_stream(pr + va));
        if (ib) add8(b, ld_stream(pr + vb));
      }
      if (ia) orow[va] = pack8(a);
      if (ib) orow[vb] = pack8(b);
    }
  }
}

template <typename Kern>
int grid_for(const lrm_ctx* ctx, Kern kern, long long need) {
  const int cap = resident_grid(ctx, kern, F1_THREADS, 0);
  return static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace

size_t combine_workspace_bytes(const lrm_dims& d) { return static_cast<size_t>(d.T) * d.k * sizeof(int32_t); }

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_swiglu_backward(lrm_ctx* ctx, const uint16_t* dphi_c, const uint16_t* ab_c,
                                          const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows,
                                          uint16_t* dh1, void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0 || sel_offsets == nullptr) return LRM_ERR_INVALID_ARG;
  if (max_rows == 0) return LRM_OK;
  if (dphi_c == nullptr || ab_c == nullptr || dh1 == nullptr) return LRM_ERR_INVALID_ARG;
  if (!aligned(dphi_c, 16) || !aligned(ab_c, 16) || !aligned(dh1, 16) || !aligned(sel_offsets, 4))
    return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static thread_local int dev = -1, grid = 0;
  if (dev != ctx->device) {
    grid = grid_for(ctx, swiglu_bwd_kernel, 1ll << 30);
    dev = ctx->device;
  }
  const long long need = (static_cast<long long>(max_rows) + F1_WARPS - 1) / F1_WARPS;
  swiglu_bwd_kernel<<<static_cast<int>(need < grid ? need : grid), F1_THREADS, 0, s>>>(
      reinterpret_cast<const uint4*>(dphi_c), reinterpret_cast<const uint4*>(ab_c), sel_offsets, dims.E, max_rows,
      dims.I / 8, reinterpret_cast<uint4*>(dh1));
  return launch_status();
}

extern "C" lrm_status lrm_combine_rows(lrm_ctx* ctx, const uint16_t* rows, const int32_t* sel_offsets,
                                       const int32_t* sel_ids, lrm_dims dims, int32_t max_rows, int32_t width,
                                       uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0 || sel_offsets == nullptr || width < 8 || width % 8 != 0 || width > 65536)
    return LRM_ERR_INVALID_ARG;
  if (dims.T == 0) return LRM_OK;
  if (out == nullptr || ws == nullptr || (max_rows > 0 && (rows == nullptr || sel_ids == nullptr)))
    return LRM_ERR_INVALID_ARG;
  if (ws_bytes < combine_workspace_bytes(dims)) return LRM_ERR_WORKSPACE;
  if (!aligned(out, 16) || !aligned(ws, 4) || !aligned(sel_offsets, 4) || (rows && !aligned(rows, 16)) ||
      (sel_ids && !aligned(sel_ids, 4)))
    return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int N = dims.T * dims.k;
  int32_t* pos = static_cast<int32_t*>(ws);
  LRM_CHECK_CUDA(cudaMemsetAsync(pos, 0xFF, static_cast<size_t>(N) * sizeof(int32_t), s));
  if (max_rows > 0) {
    map_kernel<<<min((max_rows + F1_THREADS - 1) / F1_THREADS, ctx->sm_count * 4), F1_THREADS, 0, s>>>(
        sel_offsets, dims.E, sel_ids, max_rows, N, pos, ctx->d_status);
    if ((st = launch_status()) != LRM_OK) return st;
  }
  static thread_local int dev = -1, grid = 0;
  if (dev != ctx->device) {
    grid = grid_for(ctx, combine_kernel, 1ll << 30);
    dev = ctx->device;
  }
  const int need = (dims.T + F1_WARPS - 1) / F1_WARPS;
  combine_kernel<<<need < grid ? need : grid, F1_THREADS, 0, s>>>(reinterpret_cast<const uint4*>(rows), pos, dims.T,
                                                                  dims.k, width / 8, reinterpret_cast<uint4*>(out));
  return launch_status();
}
