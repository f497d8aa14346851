// Step 2 of the path: the Load Recalibration Metric of LRMoE (sec. 3.2,
// Prop. 3.1 eq. (3); Alg. 1; appendix 7.1 eq. (11)-(12)):
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

// Row reduction of the gradient-only metrics of LRMoE's ablation (sec. 4.7,
// Table 2): the sum of squares (L1 = false) or of magnitudes (L1 = true) of a
// row of nv 16-byte vectors, reduced over the warp.
template <bool L1>
__device__ __forceinline__ float row_metric(const uint4* __restrict__ row, int nv, int lane) {
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int v = lane;
  for (; v + 96 < nv; v += 128) {
    const uint4 x0 = ld_stream(row + v);
    const uint4 x1 = ld_stream(row + v + 32);
    const uint4 x2 = ld_stream(row + v + 64);
    const uint4 x3 = ld_stream(row + v + 96);
    if (L1) {
      acc_abs8(x0, a);
      acc_abs8(x1, a);
      acc_abs8(x2, a);
      acc_abs8(x3, a);
    } else {
      acc_sq8(x0, a);
      acc_sq8(x1, a);
      acc_sq8(x2, a);
      acc_sq8(x3, a);
    }
  }
  for (; v < nv; v += 32) {
    if (L1)
      acc_abs8(ld_stream(row + v), a);
    else
      acc_sq8(ld_stream(row + v), a);
  }
  float s = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Gradient-only scores: every pair of token t gets the token's ||g_t||^2
// (L1 = false) or sum_i |g_t,i| (L1 = true).  One warp per token.
template <bool L1>
__global__ void __launch_bounds__(SC_THREADS) grad_metric_kernel(const uint4* __restrict__ g, int T, int k, int hv,
                                                                 float* __restrict__ R) {
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * SC_WARPS;
  for (int t = blockIdx.x * SC_WARPS + (threadIdx.x >> 5); t < T; t += warps_total) {
    const float m = row_metric<L1>(g + static_cast<size_t>(t) * hv, hv, lane);
    if (lane < k) R[static_cast<size_t>(t) * k + lane] = m;
  }
}

// Random-drop scores: pair u gets the (u+1)-th output of the SplitMix64
// generator (Steele, Lea and Flood, OOPSLA 2014) started from state `seed`,
// whose top 24 bits become a uniform value in [0, 1), exact in fp32.
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t u) {
  uint64_t z = seed + (u + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void __launch_bounds__(SC_THREADS) random_score_kernel(uint64_t seed, long long N, float* __restrict__ R) {
  const long long stride = static_cast<long long>(gridDim.x) * SC_THREADS;
  for (long long u = static_cast<long long>(blockIdx.x) * SC_THREADS + threadIdx.x; u < N; u += stride)
    R[u] = static_cast<float>(static_cast<uint32_t>(splitmix64_at(seed, static_cast<uint64_t>(u)) >> 40)) *
           (1.0f / 16777216.0f);
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
  // one warp per token, no persistent grid: the block scheduler evens out
  // the tail (3-4 % faster than one resident wave walking the tokens)
  const int grid = (dims.T + SC_WARPS - 1) / SC_WARPS;
  score_kernel<<<grid, SC_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(g), reinterpret_cast<const uint4*>(phi), alpha, dims.T, dims.k,
      dims.h / 8, dims.I / 8, score);
  return launch_status();
}

extern "C" lrm_status lrm_score_metric(lrm_ctx* ctx, int32_t metric, const uint16_t* g, const uint16_t* phi,
                                       const float* alpha, lrm_dims dims, uint64_t seed, float* score,
                                       void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  if (metric == LRM_METRIC_LRM) return lrm_score(ctx, g, phi, alpha, dims, score, stream);
  if (metric != LRM_METRIC_GRAD_L2SQ && metric != LRM_METRIC_GRAD_L1 && metric != LRM_METRIC_RANDOM)
    return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (dims.T == 0) return LRM_OK;
  if (score == nullptr || (metric != LRM_METRIC_RANDOM && g == nullptr)) return LRM_ERR_INVALID_ARG;
  if (!aligned(score, 4) || (g != nullptr && !aligned(g, 16))) return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long N = static_cast<long long>(dims.T) * dims.k;
  if (metric == LRM_METRIC_RANDOM) {
    static thread_local int cap_device = -1, cap = 0;
    if (cap_device != ctx->device) {
      cap = resident_grid(ctx, random_score_kernel, SC_THREADS, 0);
      cap_device = ctx->device;
    }
    const long long need = (N + SC_THREADS - 1) / SC_THREADS;
    random_score_kernel<<<static_cast<int>(need < cap ? need : cap), SC_THREADS, 0, s>>>(seed, N, score);
    return launch_status();
  }
  const int need = (dims.T + SC_WARPS - 1) / SC_WARPS;
  if (metric == LRM_METRIC_GRAD_L2SQ) {
    static thread_local int cap_device = -1, cap = 0;
    if (cap_device != ctx->device) {
      cap = resident_grid(ctx, grad_metric_kernel<false>, SC_THREADS, 0);
      cap_device = ctx->device;
    }
    grad_metric_kernel<false><<<need < cap ? need : cap, SC_THREADS, 0, s>>>(reinterpret_cast<const uint4*>(g),
                                                                             dims.T, dims.k, dims.h / 8, score);
  } else {
    static thread_local int cap_device = -1, cap = 0;
    if (cap_device != ctx->device) {
      cap = resident_grid(ctx, grad_metric_kernel<true>, SC_THREADS, 0);
      cap_device = ctx->device;
    }
    grad_metric_kernel<true><<<need < cap ? need : cap, SC_THREADS, 0, s>>>(reinterpret_cast<const uint4*>(g),
                                                                            dims.T, dims.k, dims.h / 8, score);
  }
  return launch_status();
}
