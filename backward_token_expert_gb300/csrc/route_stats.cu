// Step 1 of the path: routing statistics, capacity, drop rate and retention
// quotas ("Expert Parallel Math Deep": importance P_e, load f_e, the
// auxiliary loss E * sum f_e P_e, capacity C = CF * T k / E and the drop
// rate; LRMoE sec. 3.1 and Alg. 1 line 1: routed counts n_e and quotas
// 0 <= Q_e <= n_e), plus the stable expert bucket and prefix offsets that
// selection and compaction consume (LRMoE sec. 3.3).
//
// Three launches:
//   rs_count    one block per contiguous chunk of tokens: the chunk's expert
//               ids are staged in shared memory (validated there), counted
//               with shared-memory atomics, and the softmax of each token
//               (one warp per token, the next token's logits prefetched) is
//               summed per warp in registers, then per block in a fixed order;
//   rs_finalize one block: counts, offsets, per-(expert, block) bucket bases,
//               P, f, quotas and the summary (one warp per expert row of the
//               expert-major workspace, loads issued eight at a time);
//   rs_scatter  same chunking as rs_count: stable scatter of pair ids into
//               the bucket (each warp owns a contiguous sub-range, ranks
//               inside a warp come from __match_any_sync).
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
constexpr int RS_FIN_THREADS = 1024;
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

  // softmax over all E experts, one warp per token; lane owns experts lane + 32 i
  float acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
  int t = tok0 + warp;
  float cur[VPL];
  if (t < tok1) load_logits<VPL>(logits + static_cast<size_t>(t) * E, E, lane, cur);
  for (; t < tok1; t += RS_WARPS) {
    float nxt[VPL];
    const int tn = t + RS_WARPS;
    if (tn < tok1) load_logits<VPL>(logits + static_cast<size_t>(tn) * E, E, lane, nxt);
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) mx = fmaxf(mx, cur[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      cur[i] = (lane + 32 * i < E) ? expf(cur[i] - mx) : 0.f;
      s += cur[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[i] += cur[i] / s;
#pragma unroll
    for (int i = 0; i < VPL; ++i) cur[i] = nxt[i];
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

__global__ void __launch_bounds__(RS_FIN_THREADS) rs_finalize(
    int T, int E, int k, int nblk, int32_t cf_num, int32_t cf_den, int32_t rho_num, int32_t rho_den,
    int32_t* __restrict__ ws_hist, const float* __restrict__ ws_p, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, float* __restrict__ P, float* __restrict__ f, int32_t* __restrict__ quota,
    lrm_route_summary* __restrict__ summary) {
  __shared__ int s_warp[32];
  __shared__ int s_total;
  __shared__ int s_cnt[1024];
  __shared__ int s_off[1024];
  __shared__ float s_P[1024];
  __shared__ long long s_red_i[6][32];
  __shared__ float s_red_d[2][32];
  const int e = threadIdx.x;
  const int lane = e & 31, warp = e >> 5;
  const bool live = e < E;
  const long long N = static_cast<long long>(T) * k;

  // phase 1: one warp per expert row (expert-major workspace, coalesced)
  for (int x = warp; x < E; x += RS_FIN_THREADS / 32) {
    const size_t row = static_cast<size_t>(x) * nblk;
    int c = 0;
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
      for (int j = 0; j < FIN_UNROLL; ++j) {
        c += hv[j];
        ps += pv[j];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      c += __shfl_xor_sync(0xffffffffu, c, o);
      ps += __shfl_xor_sync(0xffffffffu, ps, o);
    }
    if (lane == 0) {
      s_cnt[x] = c;
      s_P[x] = ps;
    }
  }
  __syncthreads();
  const int cnt = live ? s_cnt[e] : 0;
  const int off = block_exclusive_scan_1024(cnt, s_warp, &s_total);
  if (live) {
    counts[e] = cnt;
    offsets[e] = off;
    s_off[e] = off;
  }
  if (e == 0) offsets[E] = s_total;
  __syncthreads();
  // phase 2: per-(expert, block) base offsets of the stable scatter, in place
  for (int x = warp; x < E; x += RS_FIN_THREADS / 32) {
    const size_t row = static_cast<size_t>(x) * nblk;
    int run = s_off[x];
    for (int b0 = 0; b0 < nblk; b0 += 32 * FIN_UNROLL) {
      int hv[FIN_UNROLL];
#pragma unroll
      for (int j = 0; j < FIN_UNROLL; ++j) {
        const int b = b0 + lane + 32 * j;
        hv[j] = b < nblk ? ws_hist[row + b] : 0;
      }
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
  }

  // capacity and quota in exact integer arithmetic
  const long long C = (static_cast<long long>(cf_num) * N) / (static_cast<long long>(cf_den) * E);
  // fp32 throughout: fp64 runs at a small fraction of the fp32 rate on this part
  float Pe = 0.f;
  long long q = 0, drop = 0;
  if (live) {
    Pe = (T > 0) ? s_P[e] / static_cast<float>(T) : 0.f;
    const long long m = cnt < C ? cnt : C;
    q = (static_cast<long long>(rho_num) * m + rho_den - 1) / rho_den;
    drop = cnt > C ? cnt - C : 0;
    P[e] = Pe;
    f[e] = N > 0 ? static_cast<float>(cnt) / static_cast<float>(N) : 0.f;
    quota[e] = static_cast<int32_t>(q);
  }
  const float fe = (live && N > 0) ? static_cast<float>(cnt) / static_cast<float>(N) : 0.f;

  // deterministic block reductions
  long long vi[5] = {drop, q, live ? cnt : LLONG_MIN, live ? cnt : LLONG_MAX, (live && cnt > 0) ? 1 : 0};
  float vd[2] = {fe * Pe, Pe};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    vi[0] += __shfl_xor_sync(0xffffffffu, vi[0], o);
    vi[1] += __shfl_xor_sync(0xffffffffu, vi[1], o);
    vi[2] = max(vi[2], __shfl_xor_sync(0xffffffffu, vi[2], o));
    vi[3] = min(vi[3], __shfl_xor_sync(0xffffffffu, vi[3], o));
    vi[4] += __shfl_xor_sync(0xffffffffu, vi[4], o);
    vd[0] += __shfl_xor_sync(0xffffffffu, vd[0], o);
    vd[1] += __shfl_xor_sync(0xffffffffu, vd[1], o);
  }
  if (lane == 0) {
    for (int i = 0; i < 5; ++i) s_red_i[i][warp] = vi[i];
    s_red_d[0][warp] = vd[0];
    s_red_d[1][warp] = vd[1];
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    long long a0 = lane < nw ? s_red_i[0][lane] : 0, a1 = lane < nw ? s_red_i[1][lane] : 0;
    long long a2 = lane < nw ? s_red_i[2][lane] : LLONG_MIN, a3 = lane < nw ? s_red_i[3][lane] : LLONG_MAX;
    long long a4 = lane < nw ? s_red_i[4][lane] : 0;
    float d0 = lane < nw ? s_red_d[0][lane] : 0.f, d1 = lane < nw ? s_red_d[1][lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a0 += __shfl_xor_sync(0xffffffffu, a0, o);
      a1 += __shfl_xor_sync(0xffffffffu, a1, o);
      a2 = max(a2, __shfl_xor_sync(0xffffffffu, a2, o));
      a3 = min(a3, __shfl_xor_sync(0xffffffffu, a3, o));
      a4 += __shfl_xor_sync(0xffffffffu, a4, o);
      d0 += __shfl_xor_sync(0xffffffffu, d0, o);
      d1 += __shfl_xor_sync(0xffffffffu, d1, o);
    }
    if (lane == 0) {
      lrm_route_summary s;
      s.N = static_cast<int32_t>(N);
      s.C = static_cast<int32_t>(C);
      s.slots = static_cast<int32_t>(C * E);
      s.dropped = static_cast<int32_t>(a0);
      s.retained = static_cast<int32_t>(a1);
      s.max_count = static_cast<int32_t>(a2);
      s.min_count = static_cast<int32_t>(a3);
      s.nonempty = static_cast<int32_t>(a4);
      s.aux_unscaled = static_cast<float>(E) * d0;
      s.drop_rate = N > 0 ? static_cast<float>(a0) / static_cast<float>(N) : 0.f;
      s.util = C > 0 ? static_cast<float>(N - a0) / static_cast<float>(C * E) : 0.f;
      s.rho_real = N > 0 ? static_cast<float>(a1) / static_cast<float>(N) : 0.f;
      s.max_over_mean = N > 0 ? static_cast<float>(a2) * static_cast<float>(E) / static_cast<float>(N) : 0.f;
      s.sum_P = d1;
      *summary = s;
    }
  }
}

__global__ void __launch_bounds__(RS_THREADS) rs_scatter(const int32_t* __restrict__ idx, int T, int E, int k,
                                                         int tpb, int nblk, const int32_t* __restrict__ ws_base,
                                                         int32_t* __restrict__ bucket) {
  extern __shared__ int rs_cnt[];  // [RS_WARPS][E], then the staged ids
  int* s_ids = rs_cnt + RS_WARPS * E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    int run = ws_base[static_cast<size_t>(e) * nblk + blockIdx.x];
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
  rs_finalize<<<1, RS_FIN_THREADS, 0, s>>>(dims.T, dims.E, dims.k, L.nblk, cf_num, cf_den, rho_num, rho_den,
                                           ws_hist, ws_p, counts, offsets, P, f, quota, summary);
  if ((st = launch_status()) != LRM_OK) return st;
  if (L.nblk > 0) {
    const size_t smem3 = (RS_WARPS * dims.E + RS_PAIRS_PER_BLOCK) * sizeof(int);
    if (smem3 > 48 * 1024 &&
        cudaFuncSetAttribute(rs_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem3)) !=
            cudaSuccess)
      return LRM_ERR_CUDA;
    rs_scatter<<<L.nblk, RS_THREADS, smem3, s>>>(expert_idx, dims.T, dims.E, dims.k, L.tpb, L.nblk, ws_hist,
                                                 bucket);
    if ((st = launch_status()) != LRM_OK) return st;
  }
  return LRM_OK;
}

// ---------------------------------------------------------------------------
// Variant without a caller workspace, for callers that cannot allocate device
// memory: the scratch of the three kernels is this fixed array.  Host code
// only sees a stand-in symbol for it, so its device address is looked up
// once per device (with that device current) and passed to the kernels.

namespace lrm {
namespace {

static __device__ __align__(256) unsigned char g_route_stats_scratch[LRM_ROUTE_STATS_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_stats_scratch on the current device (cached).
lrm_status scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return LRM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_stats_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LRM_ERR_CUDA;
    }
    g_scratch_addr[device] = p;
  }
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
  void* ws = nullptr;
  if ((st = scratch_address(ctx->device, &ws)) != LRM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* ws_hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.hist_off);
  float* ws_p = reinterpret_cast<float*>(static_cast<char*>(ws) + L.p_off);
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
  rs_finalize<<<1, RS_FIN_THREADS, 0, s>>>(dims.T, dims.E, dims.k, L.nblk, cf_num, cf_den, rho_num, rho_den,
                                           ws_hist, ws_p, counts, offsets, P, f, quota, summary);
  if ((st = launch_status()) != LRM_OK) return st;
  if (L.nblk > 0) {
    const size_t smem3 = (RS_WARPS * dims.E + RS_PAIRS_PER_BLOCK) * sizeof(int);
    if (smem3 > 48 * 1024 &&
        cudaFuncSetAttribute(rs_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem3)) !=
            cudaSuccess)
      return LRM_ERR_CUDA;
    rs_scatter<<<L.nblk, RS_THREADS, smem3, s>>>(expert_idx, dims.T, dims.E, dims.k, L.tpb, L.nblk, ws_hist,
                                                 bucket);
    if ((st = launch_status()) != LRM_OK) return st;
  }
  return LRM_OK;
}
