// Step 3 of the path: per-expert TopK within the quota (LRMoE sec. 3.2 and
// 3.3, Alg. 1 line 14; appendix 7.2 Prop. 7.1: for fixed per-expert quotas,
// keeping the largest scores of every expert is optimal, and ties only
// change which of the equal boundary scores are kept).
//
// One 1024-thread block per expert.  Scores are non-negative fp32, so their
// bit patterns order like the values.  The block first gathers its
// candidates' keys (four independent bucket reads and score gathers per
// thread in flight) into shared memory, or, for an expert with more than
// SEL_SMEM_KEYS candidates, into its contiguous slice of a workspace.  A
// most-significant-digit radix select (four 8-bit digits, warp-aggregated
// shared-memory histograms) then finds the boundary key tau and how many
// keys equal to tau are still needed; as soon as a whole histogram bin is
// taken the search stops and the rule becomes "key >= prefix".  The output
// pass walks the candidates in ascending pair index, eight consecutive per
// thread, keeps every key above tau plus the first needed keys equal to tau
// (ties go to the lower pair index), and places them with one packed block
// scan per 8192 candidates, so the retained ids come out in ascending u.
#include "block_scan.cuh"
#include "lrm_internal.cuh"

namespace lrm {
namespace {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_SMEM_KEYS = 40960;
constexpr int SEL_GATHER = 4;  // independent gathers in flight per thread
constexpr int SEL_ITEMS = 8;   // consecutive candidates per thread in the output pass

__device__ __forceinline__ uint32_t score_key(float r) { return __float_as_uint(r) & 0x7FFFFFFFu; }

__global__ void __launch_bounds__(SEL_THREADS, 1)
    select_kernel(const float* __restrict__ R, const int32_t* __restrict__ offsets,
                  const int32_t* __restrict__ bucket, const int32_t* __restrict__ quota, int E, int max_rows,
                  int32_t* __restrict__ sel_offsets, int32_t* __restrict__ sel_ids, uint32_t* __restrict__ keys_ws,
                  unsigned int* status) {
  extern __shared__ uint32_t s_keys[];
  __shared__ int s_hist[256];
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

  uint32_t* K = (n <= SEL_SMEM_KEYS) ? s_keys : keys_ws + off;
  for (int i0 = 0; i0 < n; i0 += SEL_THREADS * SEL_GATHER) {
    int id[SEL_GATHER];
    float r[SEL_GATHER];
#pragma unroll
    for (int j = 0; j < SEL_GATHER; ++j) {
      const int i = i0 + j * SEL_THREADS + tid;
      id[j] = i < n ? __ldg(src + i) : -1;
    }
#pragma unroll
    for (int j = 0; j < SEL_GATHER; ++j) r[j] = id[j] >= 0 ? __ldg(R + id[j]) : 0.f;
#pragma unroll
    for (int j = 0; j < SEL_GATHER; ++j) {
      const int i = i0 + j * SEL_THREADS + tid;
      if (i < n) K[i] = score_key(r[j]);
    }
  }
  __syncthreads();

  uint32_t prefix = 0, mask = 0;
  int want = q;
  bool ge_mode = false;
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) s_hist[tid] = 0;
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
        int bin = 256;
        if (i < n && (kk[j] & mask) == prefix) bin = static_cast<int>((kk[j] >> shift) & 0xFFu);
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (bin < 256 && (peers & lt_mask) == 0) atomicAdd(&s_hist[bin], __popc(peers));
      }
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

size_t select_workspace_bytes(const lrm_dims& d) {
  const size_t N = static_cast<size_t>(d.T) * d.k;
  return N > static_cast<size_t>(SEL_SMEM_KEYS) ? N * sizeof(uint32_t) : 0;
}

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
  select_kernel<<<dims.E, SEL_THREADS, smem, static_cast<cudaStream_t>(stream)>>>(
      score, offsets, bucket, quota, dims.E, max_rows, sel_offsets, sel_ids, static_cast<uint32_t*>(ws),
      ctx->d_status);
  return launch_status();
}
