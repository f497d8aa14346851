// Step 2 of the path: the Load Recalibration Metric of LRMoE (sec. 3.2,
// Prop. 3.1 eq. (3); Alg. 1 line 13; appendix 7.1 eq. (11)-(12)):
//   R_u = alpha_u^2 * ||g_t||^2 * ||phi_u||^2 for every routed pair u = t*k + j.
// The squared norm of g_t is computed once per token and shared by its k
// pairs.  HBM-bound: every byte of g and phi is read exactly once.
//
// One warp per token: 128-bit streaming loads, 8 independent fp32 chains per
// lane (one per bf16 lane of a 16-byte vector), a butterfly shuffle
// reduction, and one coalesced store of the token's k scores.
#include "lrm_internal.cuh"
#include "vec.cuh"

namespace lrm {
namespace {

constexpr int SC_THREADS = 256;
constexpr int SC_WARPS = SC_THREADS / 32;

// Sum of squares of a row of nv 16-byte vectors, reduced over the warp
// (every lane returns the total).
__device__ __forceinline__ float row_sumsq(const uint4* __restrict__ row, int nv, int lane) {
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int v = lane;
  for (; v + 96 < nv; v += 128) {
    const uint4 x0 = ld_stream(row + v);
    const uint4 x1 = ld_stream(row + v + 32);
    const uint4 x2 = ld_stream(row + v + 64);
    const uint4 x3 = ld_stream(row + v + 96);
    acc_sq8(x0, a);
    acc_sq8(x1, a);
    acc_sq8(x2, a);
    acc_sq8(x3, a);
  }
  for (; v < nv; v += 32) acc_sq8(ld_stream(row + v), a);
  float s = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

__global__ void __launch_bounds__(SC_THREADS) score_kernel(const uint4* __restrict__ g,
                                                           const uint4* __restrict__ phi,
                                                           const float* __restrict__ alpha, int T, int k,
                                                           int hv, int iv, float* __restrict__ R) {
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * SC_WARPS;
  for (int t = blockIdx.x * SC_WARPS + (threadIdx.x >> 5); t < T; t += warps_total) {
    const size_t u0 = static_cast<size_t>(t) * k;
    const float a = lane < k ? __ldg(alpha + u0 + lane) : 0.f;
    const float gs = row_sumsq(g + static_cast<size_t>(t) * hv, hv, lane);
    float mine = 0.f;
    for (int j = 0; j < k; ++j) {
      const float ps = row_sumsq(phi + (u0 + j) * iv, iv, lane);
      if (lane == j) mine = ps;
    }
    if (lane < k) R[u0 + lane] = __fmul_rn(__fmul_rn(__fmul_rn(a, a), gs), mine);
  }
}

}  // namespace
}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_score(lrm_ctx* ctx, const uint16_t* g, const uint16_t* phi, const float* alpha,
                                lrm_dims dims, float* score, void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (dims.T == 0) return LRM_OK;
  if (g == nullptr || phi == nullptr || alpha == nullptr || score == nullptr) return LRM_ERR_INVALID_ARG;
  if (!aligned(g, 16) || !aligned(phi, 16) || !aligned(alpha, 4) || !aligned(score, 4)) return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  static thread_local int cap_device = -1, cap = 0;
  if (cap_device != ctx->device) {
    cap = resident_grid(ctx, score_kernel, SC_THREADS, 0);
    cap_device = ctx->device;
  }
  const int need = (dims.T + SC_WARPS - 1) / SC_WARPS;
  const int grid = need < cap ? need : cap;
  score_kernel<<<grid, SC_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(g), reinterpret_cast<const uint4*>(phi), alpha, dims.T, dims.k,
      dims.h / 8, dims.I / 8, score);
  return launch_status();
}
