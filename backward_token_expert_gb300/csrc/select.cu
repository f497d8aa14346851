// Step 3 of the path: per-expert TopK within the quota (LRMoE sec. 3.2 and
// 3.3, Alg. 1 line 14; appendix 7.2 Prop. 7.1: for fixed per-expert quotas,
// keeping the largest scores of every expert is optimal, and ties only
// change which of the equal boundary scores are kept).
//
// Two launches.  select_gather_kernel reads the scores in bucket order over
// the whole GPU (four independent bucket reads and score gathers in flight
// per thread) and writes them as sortable keys into a contiguous
// expert-major workspace: scores are non-negative fp32, so their bit
// patterns order like the values.  select_kernel then runs one 1024-thread
// block per expert on its contiguous key slice (cached in shared memory when
// it holds at most SEL_SMEM_KEYS keys): a most-significant-digit radix select
// with 11/11/10-bit digits and warp-aggregated shared-memory histograms finds
// the boundary key tau and how many keys equal to tau are still needed; as
// soon as a whole histogram bin is taken the search stops and the rule
// becomes "key >= prefix".  The output pass walks the candidates in
// ascending pair index, eight consecutive per thread, keeps every key above
// tau plus the first needed keys equal to tau (ties go to the lower pair
// index), and places them with one packed block scan per 8192 candidates, so
// the retained ids come out in ascending u.
#include "block_scan.cuh"
#include "lrm_internal.cuh"

namespace lrm {
namespace {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_SMEM_KEYS = 40960;
constexpr int SEL_GATHER = 4;  // independent loads in flight per thread
constexpr int SEL_MAX_BINS = 2048;
constexpr int GATHER_THREADS = 256;
constexpr int SEL_ITEMS = 8;   // consecutive candidates per thread in the output pass

__device__ __forceinline__ uint32_t score_key(float r) { return __float_as_uint(r) & 0x7FFFFFFFu; }

__global__ void __launch_bounds__(GATHER_THREADS) select_gather_kernel(const float* __restrict__ R,
                                                                       const int32_t* __restrict__ bucket, int N,
                                                                       uint32_t* __restrict__ keys) {
  const int stride = gridDim.x * GATHER_THREADS * SEL_GATHER;
  for (int i0 = blockIdx.x * GATHER_THREADS * SEL_GATHER + threadIdx.x; i0 < N; i0 += stride) {
    int id[SEL_GATHER];
#pragma unroll
    for (int j = 0; j < SEL_GATHER; ++j) {
      const int i = i0 + j * GATHER_THREADS;
      id[j] = i < N ? __ldg(bucket + i) : -1;
    }
    float r[SEL_GATHER];
#pragma unroll
    for (int j = 0; j < SEL_GATHER; ++j) r[j] = (id[j] >= 0 && id[j] < N) ? __ldg(R + id[j]) : 0.f;
#pragma unroll
    for (int j = 0; j < SEL_GATHER; ++j) {
      const int i = i0 + j * GATHER_THREADS;
      if (i < N) keys[i] = score_key(r[j]);
    }
  }
}

__global__ void __launch_bounds__(SEL_THREADS, 1)
    select_kernel(const float* __restrict__ R, const int32_t* __restrict__ offsets,
                  const int32_t* __restrict__ bucket, const int32_t* __restrict__ quota, int E, int max_rows,
                  int32_t* __restrict__ sel_offsets, int32_t* __restrict__ sel_ids,
                  const uint32_t* __restrict__ keys_ws, unsigned int* status) {
  extern __shared__ uint32_t s_keys[];
  __shared__ int s_hist[SEL_MAX_BINS];
  __shared__ int s_warp[SEL_WARPS];
  __shared__ int s_total;
  __shared__ int s_digit, s_above, s_bincnt;

  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;

  // exclusive prefix of the clamped quotas of the experts before e
  int part = 0;
  for (int x = tid; x < e; x += SEL_THREADS) {
    const int nx = max(0, __ldg(offsets + x + 1) - __ldg(offsets + x));
    part += min(max(__ldg(quota + x), 0), nx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) s_warp[warp] = part;
  __syncthreads();
  int base = 0;
#pragma unroll 8
  for (int w = 0; w < SEL_WARPS; ++w) base += s_warp[w];

  const int off = __ldg(offsets + e);
  const int n = max(0, __ldg(offsets + e + 1) - off);
  const int q_raw = __ldg(quota + e);
  const int q = min(max(q_raw, 0), n);
  if (tid == 0) {
    if (q != q_raw) raise_flag(status, LRM_ERR_QUOTA);
    sel_offsets[e] = base;
    if (e == E - 1) sel_offsets[E] = base + q;
  }
  int q_out = q;  // rows that fit below max_rows
  if (base + q > max_rows) {
    if (tid == 0) raise_flag(status, LRM_ERR_SHAPE);
    q_out = max(0, max_rows - base);
  }
  if (q == 0 || q_out == 0) return;
  const int32_t* src = bucket + off;
  int32_t* out = sel_ids + base;
  if (q == n) {
    for (int i = tid; i < q_out; i += SEL_THREADS) out[i] = __ldg(src + i);
    return;
  }

  const uint32_t* K = keys_ws + off;
  if (n <= SEL_SMEM_KEYS) {
    for (int i0 = 0; i0 < n; i0 += SEL_THREADS * SEL_GATHER) {
      uint32_t v[SEL_GATHER];
#pragma unroll
      for (int j = 0; j < SEL_GATHER; ++j) {
        const int i = i0 + j * SEL_THREADS + tid;
        v[j] = i < n ? __ldg(K + i) : 0u;
      }
#pragma unroll
      for (int j = 0; j < SEL_GATHER; ++j) {
        const int i = i0 + j * SEL_THREADS + tid;
        if (i < n) s_keys[i] = v[j];
      }
    }
    K = s_keys;
  }
  __syncthreads();

  uint32_t prefix = 0, mask = 0;
  int want = q;
  bool ge_mode = false;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int bits = pass == 2 ? 10 : 11;
    const int nbins = 1 << bits;
    const uint32_t dmask = static_cast<uint32_t>(nbins - 1);
    for (int b = tid; b < nbins; b += SEL_THREADS) s_hist[b] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += SEL_THREADS * SEL_GATHER) {
      uint32_t kk[SEL_GATHER];
#pragma unroll
      for (int j = 0; j < SEL_GATHER; ++j) {
        const int i = i0 + j * SEL_THREADS + tid;
        kk[j] = i < n ? K[i] : 0u;
      }
#pragma unroll
      for (int j = 0; j < SEL_GATHER; ++j) {
        const int i = i0 + j * SEL_THREADS + tid;
        int bin = SEL_MAX_BINS;
        if (i < n && (kk[j] & mask) == prefix) bin = static_cast<int>((kk[j] >> shift) & dmask);
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (bin < SEL_MAX_BINS && (peers & lt_mask) == 0) atomicAdd(&s_hist[bin], __popc(peers));
      }
    }
    __syncthreads();
    // thread t owns bins hi = nbins-1-2t and hi-1 (descending); "above" counts
    // every key of the current prefix in a higher bin
    const int hi = nbins - 1 - 2 * tid;
    const int c_hi = hi >= 0 ? s_hist[hi] : 0;
    const int c_lo = hi >= 1 ? s_hist[hi - 1] : 0;
    const int above = block_exclusive_scan_1024(c_hi + c_lo, s_warp, &s_total);
    if (hi >= 0 && above < want && want <= above + c_hi) {
      s_digit = hi;
      s_above = above;
      s_bincnt = c_hi;
    } else if (hi >= 1 && above + c_hi < want && want <= above + c_hi + c_lo) {
      s_digit = hi - 1;
      s_above = above + c_hi;
      s_bincnt = c_lo;
    }
    __syncthreads();
    want -= s_above;
    prefix |= static_cast<uint32_t>(s_digit) << shift;
    mask |= dmask << shift;
    const bool all_taken = (s_bincnt == want);
    __syncthreads();
    if (all_taken) {
      ge_mode = true;
      break;
    }
  }
  const uint32_t tau = prefix;

  int run_out = 0, run_eq = 0;
  for (int i0 = 0; i0 < n; i0 += SEL_THREADS * SEL_ITEMS) {
    const int ib = i0 + tid * SEL_ITEMS;
    uint32_t kk[SEL_ITEMS];
    int id[SEL_ITEMS];
#pragma unroll
    for (int j = 0; j < SEL_ITEMS; ++j) {
      const int i = ib + j;
      kk[j] = i < n ? K[i] : 0u;
      id[j] = i < n ? __ldg(src + i) : -1;
    }
    int cg = 0, ce = 0;
    unsigned gt_bits = 0, eq_bits = 0;
#pragma unroll
    for (int j = 0; j < SEL_ITEMS; ++j) {
      const bool live = ib + j < n;
      const bool gt = live && (ge_mode ? (kk[j] >= tau) : (kk[j] > tau));
      const bool eq = live && !ge_mode && kk[j] == tau;
      gt_bits |= static_cast<unsigned>(gt) << j;
      eq_bits |= static_cast<unsigned>(eq) << j;
      cg += gt;
      ce += eq;
    }
    const int excl = block_exclusive_scan_1024(cg | (ce << 16), s_warp, &s_total);
    const int tot = s_total;
    const int eq_left = max(0, want - run_eq);
    int gtb = excl & 0xFFFF, eqb = excl >> 16;
#pragma unroll
    for (int j = 0; j < SEL_ITEMS; ++j) {
      const bool gt = (gt_bits >> j) & 1u, eq = (eq_bits >> j) & 1u;
      const bool sel = gt || (eq && eqb < eq_left);
      const int pos = run_out + gtb + min(eqb, eq_left);
      if (sel && pos < q_out) out[pos] = id[j];
      gtb += gt;
      eqb += eq;
    }
    run_out += (tot & 0xFFFF) + min(tot >> 16, eq_left);
    run_eq += tot >> 16;
  }
}

}  // namespace

size_t select_workspace_bytes(const lrm_dims& d) { return static_cast<size_t>(d.T) * d.k * sizeof(uint32_t); }

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_select(lrm_ctx* ctx, const float* score, const int32_t* offsets, const int32_t* bucket,
                                 const int32_t* quota, lrm_dims dims, int32_t max_rows, int32_t* sel_offsets,
                                 int32_t* sel_ids, void* ws, size_t ws_bytes, void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0) return LRM_ERR_INVALID_ARG;
  if (offsets == nullptr || quota == nullptr || sel_offsets == nullptr) return LRM_ERR_INVALID_ARG;
  if (dims.T > 0 && (score == nullptr || bucket == nullptr)) return LRM_ERR_INVALID_ARG;
  if (max_rows > 0 && sel_ids == nullptr) return LRM_ERR_INVALID_ARG;
  const size_t need = select_workspace_bytes(dims);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return LRM_ERR_WORKSPACE;
  const void* ptrs[] = {score, offsets, bucket, quota, sel_offsets, sel_ids, ws};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned(p, 4)) return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  const size_t smem = SEL_SMEM_KEYS * sizeof(uint32_t);
  static thread_local int configured_device = -1;
  if (configured_device != ctx->device) {
    LRM_CHECK_CUDA(
        cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
    configured_device = ctx->device;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int N = dims.T * dims.k;
  if (N > 0) {
    const int per_block = GATHER_THREADS * SEL_GATHER;
    const int need_blocks = (N + per_block - 1) / per_block;
    const int cap = ctx->sm_count * 8;
    select_gather_kernel<<<need_blocks < cap ? need_blocks : cap, GATHER_THREADS, 0, s>>>(
        score, bucket, N, static_cast<uint32_t*>(ws));
    if ((st = launch_status()) != LRM_OK) return st;
  }
  select_kernel<<<dims.E, SEL_THREADS, smem, s>>>(score, offsets, bucket, quota, dims.E, max_rows, sel_offsets,
                                                  sel_ids, static_cast<const uint32_t*>(ws), ctx->d_status);
  return launch_status();
}
