// Step 3 of the path: per-expert TopK within the quota (LRMoE sec. 3.2 and
// 3.3, Alg. 1 line 14; appendix 7.2 Prop. 7.1: for fixed per-expert quotas,
// keeping the largest scores of every expert is optimal, and ties only
// change which of the equal boundary scores are kept).
//
// One 1024-thread block per expert.  Scores are non-negative fp32, so their
// bit patterns order like the values; a most-significant-digit radix select
// (four 8-bit digits, warp-aggregated shared-memory histograms) finds the
// boundary key tau and how many keys equal to tau are still needed.  As soon
// as a whole histogram bin is taken the search stops and the rule becomes
// "key >= prefix".  A final pass walks the expert's bucket in ascending pair
// index and keeps every key above tau plus the first needed keys equal to tau
// (ties go to the lower pair index), writing them in ascending u with
// ballot-based block scans.  Keys of experts with at most SEL_SMEM_KEYS
// candidates stay in shared memory; larger experts re-gather from the score
// array (which is L2-resident at these sizes) on every pass.
#include "lrm_internal.cuh"

namespace lrm {
namespace {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_SMEM_KEYS = 40960;

__device__ __forceinline__ uint32_t score_key(float r) { return __float_as_uint(r) & 0x7FFFFFFFu; }

__global__ void __launch_bounds__(SEL_THREADS, 1)
    select_kernel(const float* __restrict__ R, const int32_t* __restrict__ offsets,
                  const int32_t* __restrict__ bucket, const int32_t* __restrict__ quota, int E, int max_rows,
                  int32_t* __restrict__ sel_offsets, int32_t* __restrict__ sel_ids, unsigned int* status) {
  extern __shared__ uint32_t s_keys[];
  __shared__ int s_hist[256];
  __shared__ int s_warp[SEL_WARPS];
  __shared__ int s_wgt[SEL_WARPS], s_weq[SEL_WARPS];
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

  const int n = max(0, __ldg(offsets + e + 1) - __ldg(offsets + e));
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
  const int32_t* src = bucket + __ldg(offsets + e);
  int32_t* out = sel_ids + base;
  if (q == n) {
    for (int i = tid; i < q_out; i += SEL_THREADS) out[i] = __ldg(src + i);
    return;
  }

  const bool in_smem = n <= SEL_SMEM_KEYS;
  if (in_smem) {
    for (int i = tid; i < n; i += SEL_THREADS) s_keys[i] = score_key(__ldg(R + __ldg(src + i)));
    __syncthreads();
  }
  auto key_at = [&](int i) -> uint32_t { return in_smem ? s_keys[i] : score_key(__ldg(R + __ldg(src + i))); };

  uint32_t prefix = 0, mask = 0;
  int want = q;
  bool ge_mode = false;
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) s_hist[tid] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += SEL_THREADS) {
      const int i = i0 + tid;
      int bin = 256;
      if (i < n) {
        const uint32_t kk = key_at(i);
        if ((kk & mask) == prefix) bin = static_cast<int>((kk >> shift) & 0xFFu);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin < 256 && (peers & lt_mask) == 0) atomicAdd(&s_hist[bin], __popc(peers));
    }
    __syncthreads();
    // counts of the bins above each bin, from the top bin down
    const int c = tid < 256 ? s_hist[255 - tid] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int above = incl - c;
    for (int w = 0; w < warp; ++w) above += s_warp[w];
    if (tid < 256 && above < want && want <= above + c) {
      s_digit = 255 - tid;
      s_above = above;
      s_bincnt = c;
    }
    __syncthreads();
    want -= s_above;
    prefix |= static_cast<uint32_t>(s_digit) << shift;
    mask |= 0xFFu << shift;
    const bool all_taken = (s_bincnt == want);
    __syncthreads();
    if (all_taken) {
      ge_mode = true;
      break;
    }
  }
  const uint32_t tau = prefix;

  int run_out = 0, run_eq = 0;
  for (int i0 = 0; i0 < n; i0 += SEL_THREADS) {
    const int i = i0 + tid;
    const uint32_t kk = i < n ? key_at(i) : 0u;
    const bool gt = i < n && (ge_mode ? (kk >= tau) : (kk > tau));
    const bool eq = i < n && !ge_mode && kk == tau;
    const unsigned bg = __ballot_sync(0xffffffffu, gt);
    const unsigned be = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) {
      s_wgt[warp] = __popc(bg);
      s_weq[warp] = __popc(be);
    }
    __syncthreads();
    int gt_before = __popc(bg & lt_mask), eq_before = __popc(be & lt_mask);
    int tot_gt = 0, tot_eq = 0;
    for (int w = 0; w < SEL_WARPS; ++w) {
      const int a = s_wgt[w], b = s_weq[w];
      if (w < warp) {
        gt_before += a;
        eq_before += b;
      }
      tot_gt += a;
      tot_eq += b;
    }
    const int eq_left = max(0, want - run_eq);
    const bool sel = gt || (eq && eq_before < eq_left);
    const int pos = run_out + gt_before + min(eq_before, eq_left);
    if (sel && pos < q_out) out[pos] = __ldg(src + i);
    run_out += tot_gt + min(tot_eq, eq_left);
    run_eq += tot_eq;
    __syncthreads();
  }
}

}  // namespace

size_t select_workspace_bytes(const lrm_dims&) { return 0; }

}  // namespace lrm

using namespace lrm;

extern "C" lrm_status lrm_select(lrm_ctx* ctx, const float* score, const int32_t* offsets, const int32_t* bucket,
                                 const int32_t* quota, lrm_dims dims, int32_t max_rows, int32_t* sel_offsets,
                                 int32_t* sel_ids, void* ws, size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0) return LRM_ERR_INVALID_ARG;
  if (offsets == nullptr || quota == nullptr || sel_offsets == nullptr) return LRM_ERR_INVALID_ARG;
  if (dims.T > 0 && (score == nullptr || bucket == nullptr)) return LRM_ERR_INVALID_ARG;
  if (max_rows > 0 && sel_ids == nullptr) return LRM_ERR_INVALID_ARG;
  const void* ptrs[] = {score, offsets, bucket, quota, sel_offsets, sel_ids};
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
  select_kernel<<<dims.E, SEL_THREADS, smem, static_cast<cudaStream_t>(stream)>>>(
      score, offsets, bucket, quota, dims.E, max_rows, sel_offsets, sel_ids, ctx->d_status);
  return launch_status();
}
