// Step 1 of the path: routing statistics, capacity, drop rate and retention
// quotas ("Expert Parallel Math Deep": importance P_e, load f_e, the
// auxiliary loss E * sum f_e P_e, capacity C = CF * T k / E and the drop
// rate; LRMoE sec. 3.1 and Alg. 1: routed counts n_e and quotas
// 0 <= Q_e <= n_e), plus the stable expert bucket and prefix offsets that
// selection and compaction consume (LRMoE sec. 3.3).
//
// Three launches:
//   rs_count    one block per contiguous chunk of tokens: the chunk's expert
//               ids are staged in shared memory (validated there), counted
//               with shared-memory atomics, and the softmax of each token
//               (a warp takes up to four tokens at a time, their logits
//               loaded together) is summed per warp in registers, then per
//               block in a fixed order;
//   rs_rows     one warp per expert row of the expert-major workspace: n_e,
//               P_e, f_e, the quota, and per-(expert, block) bucket bases
//               relative to the expert's start (loads issued eight at a time);
//   rs_scatter  every block scans the E counts for the expert offsets (block
//               0 also writes offsets[] and the summary), then, with the same
//               chunking as rs_count, scatters its pair ids stably into the
//               bucket (each warp owns a contiguous sub-range, ranks inside a
//               warp come from __match_any_sync).
#include <limits.h>
#include <math.h>

#include <mutex>

#include "block_scan.cuh"
#include "lrm_internal.cuh"

namespace lrm {

namespace {

constexpr int RS_THREADS = 512;
constexpr int RS_WARPS = RS_THREADS / 32;
constexpr int RS_PAIRS_PER_BLOCK = 1024;
constexpr int RS_MAX_PER_THREAD = (RS_PAIRS_PER_BLOCK + RS_THREADS - 1) / RS_THREADS;
constexpr int RR_WARPS = 8;  // rs_rows: experts per block, one warp each
constexpr int RR_THREADS = 32 * RR_WARPS;
constexpr int FIN_UNROLL = 8;

struct RsLayout {
  int tpb;   // tokens per block
  int nblk;  // blocks of rs_count / rs_scatter
  size_t hist_off, p_off, bytes;
};

RsLayout rs_layout(const lrm_dims& d) {
  RsLayout L;
  L.tpb = RS_PAIRS_PER_BLOCK / d.k;
  if (L.tpb < 1) L.tpb = 1;
  L.nblk = (d.T + L.tpb - 1) / L.tpb;
  const size_t cells = static_cast<size_t>(L.nblk) * d.E;
  L.hist_off = 0;
  L.p_off = ((cells * sizeof(int32_t) + 255) / 256) * 256;
  L.bytes = L.p_off + cells * sizeof(float);
  return L;
}

// Stages the block's pair ids [p0, p1) in shared memory (p0 is the first
// pair of a token) and replaces every invalid id (outside [0,E) or equal to
// an earlier slot of the same token) by -1.  Returns true if one was found.
__device__ __forceinline__ bool stage_ids(const int32_t* __restrict__ idx, int p0, int p1, int k, int E,
                                          int* s_ids) {
  for (int p = p0 + static_cast<int>(threadIdx.x); p < p1; p += RS_THREADS) s_ids[p - p0] = __ldg(idx + p);
  __syncthreads();
  int fix[RS_MAX_PER_THREAD];
  int nf = 0;
  for (int i = threadIdx.x; i < p1 - p0; i += RS_THREADS) {
    const int e = s_ids[i];
    bool ok = e >= 0 && e < E;
    for (int q = i - (i % k); ok && q < i; ++q) ok = s_ids[q] != e;
    if (!ok) fix[nf++] = i;
  }
  __syncthreads();
  for (int j = 0; j < nf; ++j) s_ids[fix[j]] = -1;
  __syncthreads();
  return nf > 0;
}

template <int VPL>
__device__ __forceinline__ void load_logits(const float* __restrict__ row, int E, int lane, float (&v)[VPL]) {
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(row + e) : -INFINITY;
  }
}

template <int VPL>
__global__ void __launch_bounds__(RS_THREADS) rs_count(const float* __restrict__ logits,
                                                       const int32_t* __restrict__ idx, int T, int E, int k,
                                                       int tpb, int nblk, int32_t* __restrict__ ws_hist,
                                                       float* __restrict__ ws_p, unsigned int* status) {
  extern __shared__ float rs_smem[];
  float* pw = rs_smem;                                         // [RS_WARPS][E]
  int* hist = reinterpret_cast<int*>(rs_smem + RS_WARPS * E);  // [E]
  int* s_ids = hist + E;                                       // [RS_PAIRS_PER_BLOCK]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < E; i += RS_THREADS) hist[i] = 0;

  const int tok0 = blockIdx.x * tpb;
  const int tok1 = min(T, tok0 + tpb);
  if (stage_ids(idx, tok0 * k, tok1 * k, k, E, s_ids)) raise_flag(status, LRM_ERR_INDEX);
  for (int i = tid; i < (tok1 - tok0) * k; i += RS_THREADS) {
    const int e = s_ids[i];
    if (e >= 0) atomicAdd(&hist[e], 1);
  }

  // softmax over all E experts, one warp per token; lane owns experts lane + 32 i.
  // DEPTH tokens of a warp are loaded together (a warp walks several tokens,
  // and one load in flight left it waiting on DRAM once per token)
  constexpr int DEPTH = VPL <= 4 ? 4 : (VPL <= 8 ? 2 : 1);
  float acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
  for (int t0 = tok0 + warp; t0 < tok1; t0 += DEPTH * RS_WARPS) {
    float cur[DEPTH][VPL];
#pragma unroll
    for (int d = 0; d < DEPTH; ++d) {
      const int t = t0 + d * RS_WARPS;
      if (t < tok1) {
        load_logits<VPL>(logits + static_cast<size_t>(t) * E, E, lane, cur[d]);
      } else {
#pragma unroll
        for (int i = 0; i < VPL; ++i) cur[d][i] = -INFINITY;
      }
    }
#pragma unroll
    for (int d = 0; d < DEPTH; ++d) {
      if (t0 + d * RS_WARPS >= tok1) break;
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < VPL; ++i) mx = fmaxf(mx, cur[d][i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      // the CUDA fast exponential (cur - mx <= 0, where its error is a few ulp
      // of each term) and one reciprocal per token: P_e is a mean over tokens,
      // held to 1e-5 relative against the fp64 oracle
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        cur[d][i] = (lane + 32 * i < E) ? __expf(cur[d][i] - mx) : 0.f;
        s += cur[d][i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const float inv = 1.f / s;
#pragma unroll
      for (int i = 0; i < VPL; ++i) acc[i] += cur[d][i] * inv;
    }
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) pw[warp * E + e] = acc[i];
  }
  __syncthreads();
  for (int e = tid; e < E; e += RS_THREADS) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < RS_WARPS; ++w) a += pw[w * E + e];
    ws_p[static_cast<size_t>(e) * nblk + blockIdx.x] = a;
    ws_hist[static_cast<size_t>(e) * nblk + blockIdx.x] = hist[e];
  }
}

// One warp per expert row of the expert-major workspace: the routed count,
// the summed importance, and, in place, the stable-scatter base of every count
// block relative to the expert's first bucket slot (an exclusive scan along
// the row).  Writes the per-expert outputs: n_e, P_e, f_e and the quota
// Q_e = ceil(rho min(n_e, C)) in exact integer arithmetic.
__global__ void __launch_bounds__(RR_THREADS) rs_rows(int T, int E, int k, int nblk, int32_t cf_num, int32_t cf_den,
                                                      int32_t rho_num, int32_t rho_den,
                                                      int32_t* __restrict__ ws_hist, const float* __restrict__ ws_p,
                                                      int32_t* __restrict__ counts, float* __restrict__ P,
                                                      float* __restrict__ f, int32_t* __restrict__ quota) {
  const int lane = threadIdx.x & 31;
  const int x = blockIdx.x * RR_WARPS + (threadIdx.x >> 5);
  if (x >= E) return;
  const long long N = static_cast<long long>(T) * k;
  const size_t row = static_cast<size_t>(x) * nblk;
  int run = 0;
  float ps = 0.f;
  for (int b0 = 0; b0 < nblk; b0 += 32 * FIN_UNROLL) {
    int hv[FIN_UNROLL];
    float pv[FIN_UNROLL];
#pragma unroll
    for (int j = 0; j < FIN_UNROLL; ++j) {
      const int b = b0 + lane + 32 * j;
      hv[j] = b < nblk ? ws_hist[row + b] : 0;
      pv[j] = b < nblk ? ws_p[row + b] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < FIN_UNROLL; ++j) ps += pv[j];
#pragma unroll
    for (int j = 0; j < FIN_UNROLL; ++j) {
      const int b = b0 + lane + 32 * j;
      int incl = hv[j];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (b < nblk) ws_hist[row + b] = run + incl - hv[j];
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
  if (lane == 0) {
    const int cnt = run;
    const long long C = capacity_of(N, E, cf_num, cf_den);
    counts[x] = cnt;
    // fp32 throughout: fp64 runs at a small fraction of the fp32 rate on this part
    P[x] = T > 0 ? ps / static_cast<float>(T) : 0.f;
    f[x] = N > 0 ? static_cast<float>(cnt) / static_cast<float>(N) : 0.f;
    quota[x] = static_cast<int32_t>(quota_of(cnt, C, rho_num, rho_den));
  }
}

// The summary of the step from the per-expert outputs (one warp, a fixed
// reduction order, so the floats are the same on every run).
__device__ void write_summary(int T, int E, int k, int32_t cf_num, int32_t cf_den, const int32_t* __restrict__ counts,
                              const float* __restrict__ P, const float* __restrict__ f,
                              const int32_t* __restrict__ quota, lrm_route_summary* __restrict__ summary) {
  const int lane = threadIdx.x & 31;
  const long long N = static_cast<long long>(T) * k;
  const long long C = capacity_of(N, E, cf_num, cf_den);
  long long drop = 0, ret = 0, mx = LLONG_MIN, mn = LLONG_MAX, nonempty = 0;
  float fp = 0.f, sp = 0.f;
  for (int e = lane; e < E; e += 32) {
    const long long cnt = counts[e];
    drop += cnt > C ? cnt - C : 0;
    ret += quota[e];
    mx = max(mx, cnt);
    mn = min(mn, cnt);
    nonempty += cnt > 0 ? 1 : 0;
    fp += f[e] * P[e];
    sp += P[e];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    drop += __shfl_xor_sync(0xffffffffu, drop, o);
    ret += __shfl_xor_sync(0xffffffffu, ret, o);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    nonempty += __shfl_xor_sync(0xffffffffu, nonempty, o);
    fp += __shfl_xor_sync(0xffffffffu, fp, o);
    sp += __shfl_xor_sync(0xffffffffu, sp, o);
  }
  if (lane == 0) {
    lrm_route_summary s;
    s.N = static_cast<int32_t>(N);
    s.C = static_cast<int32_t>(C);
    s.slots = static_cast<int32_t>(C * E);
    s.dropped = static_cast<int32_t>(drop);
    s.retained = static_cast<int32_t>(ret);
    s.max_count = static_cast<int32_t>(mx);
    s.min_count = static_cast<int32_t>(mn);
    s.nonempty = static_cast<int32_t>(nonempty);
    s.aux_unscaled = static_cast<float>(E) * fp;
    s.drop_rate = N > 0 ? static_cast<float>(drop) / static_cast<float>(N) : 0.f;
    s.util = C > 0 ? static_cast<float>(N - drop) / static_cast<float>(C * E) : 0.f;
    s.rho_real = N > 0 ? static_cast<float>(ret) / static_cast<float>(N) : 0.f;
    s.max_over_mean = N > 0 ? static_cast<float>(mx) * static_cast<float>(E) / static_cast<float>(N) : 0.f;
    s.sum_P = sp;
    *summary = s;
  }
}

// Expert offsets (exclusive scan of the counts) in every block; block 0 also
// writes offsets[] and the summary.  Then the stable scatter of the block's
// pairs (none when the layer has no token: one block is launched for the
// offsets and the summary).
__global__ void __launch_bounds__(RS_THREADS) rs_scatter(const int32_t* __restrict__ idx, int T, int E, int k,
                                                         int tpb, int nblk, int32_t cf_num, int32_t cf_den,
                                                         const int32_t* __restrict__ ws_base,
                                                         const int32_t* __restrict__ counts,
                                                         const float* __restrict__ P, const float* __restrict__ f,
                                                         const int32_t* __restrict__ quota,
                                                         int32_t* __restrict__ offsets,
                                                         lrm_route_summary* __restrict__ summary,
                                                         int32_t* __restrict__ bucket) {
  extern __shared__ int rs_cnt[];  // [RS_WARPS][E], then the staged ids
  __shared__ int s_off[1024];      // first bucket slot of every expert (E <= 1024)
  int* s_ids = rs_cnt + RS_WARPS * E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    // a run of experts per lane, then a warp scan
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int local = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) local += counts[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - local;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      s_off[e] = run;
      if (blockIdx.x == 0) offsets[e] = run;
      run += counts[e];
    }
    if (blockIdx.x == 0 && lane == 31) offsets[E] = incl;
  } else if (warp == 1 && blockIdx.x == 0) {
    write_summary(T, E, k, cf_num, cf_den, counts, P, f, quota, summary);
  }
  if (nblk == 0) return;
  for (int i = tid; i < RS_WARPS * E; i += RS_THREADS) rs_cnt[i] = 0;
  const int p0 = blockIdx.x * tpb * k;
  const int p1 = min(T, (blockIdx.x + 1) * tpb) * k;
  stage_ids(idx, p0, p1, k, E, s_ids);
  const int span = (p1 - p0 + RS_WARPS - 1) / RS_WARPS;
  const int w0 = min(p1, p0 + warp * span);
  const int w1 = min(p1, w0 + span);
  int* mine = rs_cnt + warp * E;
  const unsigned lt_mask = (1u << lane) - 1u;

  // pass A: per-warp histogram of its contiguous sub-range
  for (int base = w0; base < w1; base += 32) {
    const int p = base + lane;
    const int e = p < w1 ? s_ids[p - p0] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (peers & lt_mask) == 0) mine[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // per expert: the block's base offset, then exclusive prefix over the warps
  for (int e = tid; e < E; e += RS_THREADS) {
    int run = s_off[e] + ws_base[static_cast<size_t>(e) * nblk + blockIdx.x];
#pragma unroll
    for (int w = 0; w < RS_WARPS; ++w) {
      const int c = rs_cnt[w * E + e];
      rs_cnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass B: stable placement, ascending pair index within every expert
  for (int base = w0; base < w1; base += 32) {
    const int p = base + lane;
    const int e = p < w1 ? s_ids[p - p0] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int pos = 0;
    if (e >= 0) pos = mine[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (e >= 0) {
      bucket[pos] = p;
      if ((peers & lt_mask) == 0) mine[e] += __popc(peers);
    }
    __syncwarp();
  }
}

template <int VPL>
cudaError_t launch_count(int nblk, size_t smem, cudaStream_t s, const float* logits, const int32_t* idx,
                         const lrm_dims& d, int tpb, int32_t* ws_hist, float* ws_p, unsigned int* status) {
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(rs_count<VPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  rs_count<VPL><<<nblk, RS_THREADS, smem, s>>>(logits, idx, d.T, d.E, d.k, tpb, nblk, ws_hist, ws_p, status);
  return cudaGetLastError();
}

// The three launches of the step on `s` (shared by both entry points).
lrm_status launch_route_stats(lrm_ctx* ctx, const RsLayout& L, const lrm_dims& dims, const float* logits,
                              const int32_t* expert_idx, int32_t cf_num, int32_t cf_den, int32_t rho_num,
                              int32_t rho_den, int32_t* counts, int32_t* offsets, int32_t* bucket, float* P, float* f,
                              int32_t* quota, lrm_route_summary* summary, int32_t* ws_hist, float* ws_p,
                              cudaStream_t s) {
  if (L.nblk > 0) {
    const size_t smem1 = (RS_WARPS * dims.E + dims.E + RS_PAIRS_PER_BLOCK) * sizeof(float);
    const int vpl = (dims.E + 31) / 32;
    cudaError_t e;
    if (vpl <= 1)
      e = launch_count<1>(L.nblk, smem1, s, logits, expert_idx, dims, L.tpb, ws_hist, ws_p, ctx->d_status);
    else if (vpl <= 2)
      e = launch_count<2>(L.nblk, smem1, s, logits, expert_idx, dims, L.tpb, ws_hist, ws_p, ctx->d_status);
    else if (vpl <= 4)
      e = launch_count<4>(L.nblk, smem1, s, logits, expert_idx, dims, L.tpb, ws_hist, ws_p, ctx->d_status);
    else if (vpl <= 8)
      e = launch_count<8>(L.nblk, smem1, s, logits, expert_idx, dims, L.tpb, ws_hist, ws_p, ctx->d_status);
    else if (vpl <= 16)
      e = launch_count<16>(L.nblk, smem1, s, logits, expert_idx, dims, L.tpb, ws_hist, ws_p, ctx->d_status);
    else
      e = launch_count<32>(L.nblk, smem1, s, logits, expert_idx, dims, L.tpb, ws_hist, ws_p, ctx->d_status);
    if (e != cudaSuccess) return LRM_ERR_CUDA;
  }
  rs_rows<<<(dims.E + RR_WARPS - 1) / RR_WARPS, RR_THREADS, 0, s>>>(dims.T, dims.E, dims.k, L.nblk, cf_num, cf_den,
                                                                     rho_num, rho_den, ws_hist, ws_p, counts, P, f,
                                                                     quota);
  lrm_status st = launch_status();
  if (st != LRM_OK) return st;
  const size_t smem3 = (RS_WARPS * dims.E + RS_PAIRS_PER_BLOCK) * sizeof(int);
  if (smem3 > 48 * 1024 &&
      cudaFuncSetAttribute(rs_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem3)) !=
          cudaSuccess)
    return LRM_ERR_CUDA;
  rs_scatter<<<L.nblk > 0 ? L.nblk : 1, RS_THREADS, smem3, s>>>(expert_idx, dims.T, dims.E, dims.k, L.tpb, L.nblk,
                                                                 cf_num, cf_den, ws_hist, counts, P, f, quota,
                                                                 offsets, summary, bucket);
  return launch_status();
}

}  // namespace

size_t route_stats_workspace_bytes(const lrm_dims& d) { return rs_layout(d).bytes; }

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_route_stats(lrm_ctx* ctx, const float* logits, const int32_t* expert_idx, lrm_dims dims,
                                      int32_t cf_num, int32_t cf_den, int32_t rho_num, int32_t rho_den,
                                      int32_t* counts, int32_t* offsets, int32_t* bucket, float* P, float* f,
                                      int32_t* quota, lrm_route_summary* summary, void* ws, size_t ws_bytes,
                                      void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (cf_num <= 0 || cf_den <= 0 || rho_den <= 0 || rho_num < 0 || rho_num > rho_den)
    return LRM_ERR_INVALID_ARG;
  if (counts == nullptr || offsets == nullptr || P == nullptr || f == nullptr || quota == nullptr ||
      summary == nullptr)
    return LRM_ERR_INVALID_ARG;
  if (dims.T > 0 && (logits == nullptr || expert_idx == nullptr || bucket == nullptr))
    return LRM_ERR_INVALID_ARG;
  const void* ptrs[] = {logits, expert_idx, counts, offsets, bucket, P, f, quota, summary, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned(p, 4)) return LRM_ERR_ALIGN;
  const RsLayout L = rs_layout(dims);
  if (L.nblk > 0 && (ws == nullptr || ws_bytes < L.bytes)) return LRM_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* ws_hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.hist_off);
  float* ws_p = reinterpret_cast<float*>(static_cast<char*>(ws) + L.p_off);
  return launch_route_stats(ctx, L, dims, logits, expert_idx, cf_num, cf_den, rho_num, rho_den, counts, offsets,
                            bucket, P, f, quota, summary, ws_hist, ws_p, s);
}

// Host queries of the capacity and quota rule, with the kernels' own helpers.
namespace {
lrm_status check_rationals(const lrm_dims& dims, int32_t cf_num, int32_t cf_den, int32_t rho_num, int32_t rho_den) {
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (cf_num <= 0 || cf_den <= 0 || rho_den <= 0 || rho_num < 0 || rho_num > rho_den) return LRM_ERR_INVALID_ARG;
  return LRM_OK;
}
}  // namespace

extern "C" lrm_status lrm_capacity(lrm_dims dims, int32_t cf_num, int32_t cf_den, int32_t* C) {
  if (C == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_rationals(dims, cf_num, cf_den, 0, 1);
  if (st != LRM_OK) return st;
  const long long N = static_cast<long long>(dims.T) * dims.k;
  const long long c = capacity_of(N, dims.E, cf_num, cf_den);
  if (c > INT32_MAX / dims.E) return LRM_ERR_SHAPE;  // E * C slots must fit the summary's int32
  *C = static_cast<int32_t>(c);
  return LRM_OK;
}

extern "C" lrm_status lrm_max_rows(lrm_dims dims, int32_t cf_num, int32_t cf_den, int32_t rho_num, int32_t rho_den,
                                   int32_t* max_rows) {
  if (max_rows == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_rationals(dims, cf_num, cf_den, rho_num, rho_den);
  if (st != LRM_OK) return st;
  const long long N = static_cast<long long>(dims.T) * dims.k;
  const long long c = capacity_of(N, dims.E, cf_num, cf_den);
  if (c > INT32_MAX / dims.E) return LRM_ERR_SHAPE;
  // every quota is at most quota_of(C, C) and at most n_e (sum N); and
  // ceil(rho m) <= (rho_num m + rho_den - 1) / rho_den summed over E experts
  long long bound = N;
  const long long per_expert = quota_of(c, c, rho_num, rho_den) * dims.E;
  if (per_expert < bound) bound = per_expert;
  const long long by_rate = (static_cast<long long>(rho_num) * N + static_cast<long long>(dims.E) * (rho_den - 1)) /
                            rho_den;
  if (by_rate < bound) bound = by_rate;
  *max_rows = static_cast<int32_t>(bound);
  return LRM_OK;
}

// ---------------------------------------------------------------------------
// Variant without a caller workspace, for callers that cannot allocate device
// memory: the scratch of the three kernels is this fixed array.  Host code
// only sees a stand-in symbol for it, so its device address is looked up
// with the device current and passed to the kernels.

namespace lrm {
namespace {

static __device__ __align__(256) unsigned char g_route_stats_scratch[LRM_ROUTE_STATS_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_stats_scratch on the current device.  Outside a
// stream capture it is looked up on every call (a reset of the device's
// context unloads the module, and the address found before it would be
// stale); while `stream` is capturing, the address of the last uncaptured
// call on this device is used, so that the capture records no lookup.
lrm_status scratch_address(int device, cudaStream_t stream, void** out) {
  if (device < 0 || device >= kMaxDevices) return LRM_ERR_INVALID_ARG;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone;
  if (capturing) cudaGetLastError();
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!capturing) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_stats_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LRM_ERR_CUDA;
    }
    g_scratch_addr[device] = p;
  }
  if (g_scratch_addr[device] == nullptr) return LRM_ERR_CUDA;  // first call inside a capture
  *out = g_scratch_addr[device];
  return LRM_OK;
}

}  // namespace
}  // namespace lrm

extern "C" lrm_status lrm_route_stats_noalloc(lrm_ctx* ctx, const float* logits, const int32_t* expert_idx,
                                              lrm_dims dims, int32_t cf_num, int32_t cf_den, int32_t rho_num,
                                              int32_t rho_den, int32_t* counts, int32_t* offsets, int32_t* bucket,
                                              float* P, float* f, int32_t* quota, lrm_route_summary* summary,
                                              void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (cf_num <= 0 || cf_den <= 0 || rho_den <= 0 || rho_num < 0 || rho_num > rho_den)
    return LRM_ERR_INVALID_ARG;
  if (counts == nullptr || offsets == nullptr || P == nullptr || f == nullptr || quota == nullptr ||
      summary == nullptr)
    return LRM_ERR_INVALID_ARG;
  if (dims.T > 0 && (logits == nullptr || expert_idx == nullptr || bucket == nullptr))
    return LRM_ERR_INVALID_ARG;
  const void* ptrs[] = {logits, expert_idx, counts, offsets, bucket, P, f, quota, summary};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned(p, 4)) return LRM_ERR_ALIGN;
  const RsLayout L = rs_layout(dims);
  if (L.bytes > LRM_ROUTE_STATS_SCRATCH_BYTES) return LRM_ERR_SHAPE;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if ((st = scratch_address(ctx->device, s, &ws)) != LRM_OK) return st;
  int32_t* ws_hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.hist_off);
  float* ws_p = reinterpret_cast<float*>(static_cast<char*>(ws) + L.p_off);
  return launch_route_stats(ctx, L, dims, logits, expert_idx, cf_num, cf_den, rho_num, rho_den, counts, offsets,
                            bucket, P, f, quota, summary, ws_hist, ws_p, s);
}
