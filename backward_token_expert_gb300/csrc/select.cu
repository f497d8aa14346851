// Step 3 of the path: per-expert TopK within the quota (LRMoE sec. 3.2 and
// 3.3, Alg. 1; appendix 7.2 Prop. 7.1: for fixed per-expert quotas,
// keeping the largest scores of every expert is optimal, and ties only
// change which of the equal boundary scores are kept).
//
// Two launches.  select_gather_kernel reads the scores in bucket order over
// the whole GPU (four independent bucket reads and score gathers in flight
// per thread) and writes them as sortable keys into a contiguous
// expert-major workspace: scores are non-negative fp32, so their bit
// patterns order like the values.  select_kernel then runs one 1024-thread
// block per expert on its contiguous key slice (cached in shared memory when
// it holds at most SEL_SMEM_KEYS keys):
//  - experts with more than SEL_SAMPLE_MIN candidates first sort a sample of
//    1024 keys, bracket the boundary between two sample keys, count the keys
//    above and inside the bracket with ballots and keep only the bracket's
//    keys when the boundary lies inside (else they fall back to all keys);
//  - a most-significant-digit radix select (11/11/10-bit digits,
//    warp-aggregated shared-memory histograms) finds the boundary key; once
//    the boundary bin fits in SEL_CAND_KEYS its keys are compacted and later
//    passes scan only them; as soon as a whole bin is taken the rule becomes
//    "key >= prefix";
//  - the output pass gives each warp a contiguous range of candidates in
//    ascending pair index, counts its kept keys with ballots, scans the 32
//    warp totals and places every kept id, keeping the first needed keys
//    equal to the boundary (ties go to the lower pair index), so the
//    retained ids come out in ascending u.
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
constexpr int SEL_REGION = 192;                         // candidate keys (and positions) a warp may keep
constexpr int SEL_CAND_KEYS = SEL_REGION * SEL_WARPS;
// regions of an expert whose keys are not cached: they take the key cache's
// shared memory (keys, then positions), 4.4 times the room
constexpr int SEL_BIG_REGION = 848;
static_assert(SEL_BIG_REGION * SEL_WARPS * 6 <= SEL_SMEM_KEYS * 4, "big regions fit the key cache");
constexpr int SEL_LOAD = 8;                             // keys per thread in flight while loading an expert
constexpr int SEL_OUT_UNROLL = 4;    // 32-candidate steps whose loads are issued together (more than 4
                                     // leaves too few of the 64 registers for the loads to overlap)
constexpr int SEL_SAMPLE_MIN = 4096; // experts with more candidates bracket the boundary by sampling

__device__ __forceinline__ uint32_t score_key(float r) { return __float_as_uint(r) & 0x7FFFFFFFu; }

// Exclusive prefix of per-warp totals (vals[w] for w < SEL_WARPS) at this
// thread's warp, and their sum; every warp scans the 32 totals itself.
__device__ __forceinline__ int warp_totals_prefix(const int* vals, int warp, int lane, int* total) {
  const int v = vals[lane];
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return __shfl_sync(0xffffffffu, incl - v, warp);
}

// Contiguous candidate range [w0, w1) of warp `warp` over n keys, a multiple
// of 32 wide, so that compaction keeps ascending order within a warp.
__device__ __forceinline__ void warp_range(int n, int warp, int& w0, int& w1) {
  const int span = ((n + SEL_WARPS - 1) / SEL_WARPS + 31) & ~31;
  w0 = min(n, warp * span);
  w1 = min(n, w0 + span);
}

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
    select_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ bucket,
                  const int32_t* __restrict__ quota, int E, int max_rows, int32_t* __restrict__ sel_offsets,
                  int32_t* __restrict__ sel_ids, const uint32_t* __restrict__ keys_ws, unsigned int* status) {
  extern __shared__ uint32_t s_keys[];
  uint32_t* s_cand = s_keys + SEL_SMEM_KEYS;                           // SEL_WARPS regions of keys
  uint16_t* s_cpos = reinterpret_cast<uint16_t*>(s_cand + SEL_CAND_KEYS);  // their positions in the warp's range
  __shared__ int s_hist[SEL_MAX_BINS];
  __shared__ int s_warp[SEL_WARPS];
  __shared__ int s_wgt[SEL_WARPS], s_weq[SEL_WARPS];
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
#pragma unroll
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
    for (int i0 = 0; i0 < n; i0 += SEL_THREADS * SEL_LOAD) {
      uint32_t v[SEL_LOAD];
#pragma unroll
      for (int j = 0; j < SEL_LOAD; ++j) {
        const int i = i0 + j * SEL_THREADS + tid;
        v[j] = i < n ? __ldg(K + i) : 0u;
      }
#pragma unroll
      for (int j = 0; j < SEL_LOAD; ++j) {
        const int i = i0 + j * SEL_THREADS + tid;
        if (i < n) s_keys[i] = v[j];
      }
    }
    K = s_keys;
  }
  __syncthreads();

  // Every pass below works on this warp's contiguous range [w0, w1) of the
  // candidates (ascending u), and candidate keys it keeps go to its own
  // region of s_cand, so no pass needs atomics or a block-wide compaction.
  int w0, w1;
  warp_range(n, warp, w0, w1);
  uint32_t* region = s_cand + warp * SEL_REGION;
  uint16_t* region_pos = s_cpos + warp * SEL_REGION;
  int reg_cap = SEL_REGION;
  if (n > SEL_SMEM_KEYS) {  // the keys stay in global memory: the cache's space holds the regions
    reg_cap = SEL_BIG_REGION;
    region = s_keys + warp * SEL_BIG_REGION;
    region_pos = reinterpret_cast<uint16_t*>(s_keys + SEL_WARPS * SEL_BIG_REGION) + warp * SEL_BIG_REGION;
  }

  uint32_t prefix = 0, mask = 0;
  int want = q;  // keys still to take among the radix candidates
  bool ge_mode = false;
  uint32_t ge_floor = 0;    // in "key >= prefix" mode, keys below ge_floor are not candidates
  bool bracketed = false;   // the radix candidates are the sample bracket's keys
  uint32_t cand_hi = 0xFFFFFFFFu;  // keys above this are kept without being radix candidates
  int w_cap = 0;            // this warp's captured keys (at or above the bracket's low key)
  if (n > SEL_SAMPLE_MIN && (n + SEL_WARPS - 1) / SEL_WARPS <= 65535) {  // positions fit 16 bits
    // Sample select: sort 1024 evenly spaced keys (descending, bitonic), take
    // the sample keys a few standard deviations either side of the expected
    // rank of the boundary as a bracket [lo, hi].  One pass counts the keys
    // above and inside it and captures every key >= lo with its position, in
    // order, into the warp's region; when the boundary lies inside the
    // bracket, the bracket's keys go on to the radix select and the output
    // reads only the regions.
    uint32_t mine = K[static_cast<int>((static_cast<long long>(tid) * n) / SEL_THREADS)];
    int sm_stage = 0;  // exchanges through shared memory alternate between two buffers
    for (int kk = 2; kk <= SEL_THREADS; kk <<= 1) {
      for (int j = kk >> 1; j > 0; j >>= 1) {
        uint32_t other;
        if (j >= 32) {
          uint32_t* buf = reinterpret_cast<uint32_t*>(s_hist) + (sm_stage & 1) * SEL_THREADS;
          ++sm_stage;
          buf[tid] = mine;
          __syncthreads();
          other = buf[tid ^ j];
        } else {
          other = __shfl_xor_sync(0xffffffffu, mine, j);
        }
        // descending overall: the lower index of a pair keeps the larger key
        // in blocks with (tid & kk) == 0, the smaller one otherwise
        const bool lower = (tid & j) == 0;
        const bool desc = (tid & kk) == 0;
        mine = (lower == desc) ? max(mine, other) : min(mine, other);
      }
    }
    uint32_t* samp = reinterpret_cast<uint32_t*>(s_hist) + (sm_stage & 1) * SEL_THREADS;
    samp[tid] = mine;
    __syncthreads();
    const float pr = static_cast<float>(q) / static_cast<float>(n);
    const int r = min(SEL_THREADS - 1, static_cast<int>((static_cast<long long>(q) * SEL_THREADS) / n));
    const int d = static_cast<int>(3.f * sqrtf(SEL_THREADS * pr * (1.f - pr))) + 8;
    const uint32_t hi = samp[max(0, r - d)];
    const uint32_t lo = samp[min(SEL_THREADS - 1, r + d)];
    int w_gt = 0;
#pragma unroll 4
    for (int i = w0 + lane; i - lane < w1; i += 32) {
      const bool live = i < w1;
      const uint32_t kk = live ? K[i] : 0u;
      w_gt += __popc(__ballot_sync(0xffffffffu, live && kk > hi));
      const bool cap = live && kk >= lo;
      const unsigned bc = __ballot_sync(0xffffffffu, cap);
      const int pos = w_cap + __popc(bc & lt_mask);
      if (cap && pos < reg_cap) {
        region[pos] = kk;
        region_pos[pos] = static_cast<uint16_t>(i - w0);
      }
      w_cap += __popc(bc);
    }
    if (lane == 0) {
      s_wgt[warp] = w_gt;
      s_weq[warp] = w_cap;
    }
    __syncthreads();
    int c_gt, c_cap;
    warp_totals_prefix(s_wgt, warp, lane, &c_gt);
    warp_totals_prefix(s_weq, warp, lane, &c_cap);
    const int max_cap = __reduce_max_sync(0xffffffffu, s_weq[lane]);
    if (c_gt < q && q <= c_cap && max_cap <= reg_cap) {
      bracketed = true;
      want = q - c_gt;
      ge_floor = lo;
      cand_hi = hi;
    }
    __syncthreads();  // the sample buffers are the histogram below
  }

  // radix select of the want-th largest candidate: digits of at most 11 bits
  // from the top; the first one (bits 21-31) sees the sign-free exponent and
  // the leading mantissa bits.  Each warp histograms its own candidates: its
  // region, or its whole range until the boundary bin fits in the regions.
  const uint32_t* cand = bracketed ? region : K + w0;
  int ncand = bracketed ? w_cap : w1 - w0;
  bool in_regions = bracketed;
  {
    int lo_bit = 32;  // bits [lo_bit, 32) of the boundary key are known
    while (lo_bit > 0) {
      const int bits = min(11, lo_bit);
      const int shift = lo_bit - bits;
      const int nbins = 1 << bits;
      const uint32_t dmask = static_cast<uint32_t>(nbins - 1);
      for (int b = tid; b < nbins; b += SEL_THREADS) s_hist[b] = 0;
      __syncthreads();
#pragma unroll 4
      for (int i = lane; i - lane < ncand; i += 32) {
        const uint32_t kk = i < ncand ? cand[i] : 0u;
        int bin = SEL_MAX_BINS;
        if (i < ncand && kk <= cand_hi && (kk & mask) == prefix) bin = static_cast<int>((kk >> shift) & dmask);
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (bin < SEL_MAX_BINS && (peers & lt_mask) == 0) atomicAdd(&s_hist[bin], __popc(peers));
      }
      __syncthreads();
      // thread t owns bins hi = nbins-1-2t and hi-1 (descending); "above" counts
      // every key of the current prefix in a higher bin
      const int hb = nbins - 1 - 2 * tid;
      const int c_hi = hb >= 0 ? s_hist[hb] : 0;
      const int c_lo = hb >= 1 ? s_hist[hb - 1] : 0;
      const int above = block_exclusive_scan_1024(c_hi + c_lo, s_warp, &s_total);
      if (hb >= 0 && above < want && want <= above + c_hi) {
        s_digit = hb;
        s_above = above;
        s_bincnt = c_hi;
      } else if (hb >= 1 && above + c_hi < want && want <= above + c_hi + c_lo) {
        s_digit = hb - 1;
        s_above = above + c_hi;
        s_bincnt = c_lo;
      }
      __syncthreads();
      want -= s_above;
      prefix |= static_cast<uint32_t>(s_digit) << shift;
      mask |= dmask << shift;
      const int bincnt = s_bincnt;
      __syncthreads();
      lo_bit = shift;
      if (bincnt == want) {  // the whole bin is kept: "key >= prefix"
        ge_mode = true;
        break;
      }
      if (lo_bit == 0) break;
      // once the boundary bin is small, each warp keeps only its keys of it
      if (!in_regions && bincnt <= reg_cap * SEL_WARPS) {
        int c = 0;
#pragma unroll 4
        for (int i = lane; i - lane < ncand; i += 32) {
          const uint32_t kk = i < ncand ? cand[i] : 0u;
          const bool m = i < ncand && (kk & mask) == prefix;
          const unsigned bm = __ballot_sync(0xffffffffu, m);
          const int pos = c + __popc(bm & lt_mask);
          if (m && pos < reg_cap) region[pos] = kk;
          c += __popc(bm);
        }
        if (!__syncthreads_or(c > reg_cap)) {
          cand = region;
          ncand = c;
          in_regions = true;
        }
      }
    }
  }
  const uint32_t tau = ge_mode ? max(prefix, ge_floor) : prefix;

  // Output: count this warp's kept keys, scan the 32 warp totals, then place
  // the kept ids in ascending u: key x goes to (#keys above tau before x) +
  // min(#keys equal to tau before x, want), keeping the first `want` keys
  // equal to tau.  With a bracket every kept key is in the warp's region
  // (in range order, with its position); otherwise the whole range is read.
  const uint32_t* ksrc = bracketed ? region : K + w0;
  const int kn = bracketed ? w_cap : w1 - w0;
  int cg = 0, ce = 0;
#pragma unroll 4
  for (int i = lane; i - lane < kn; i += 32) {
    const bool live = i < kn;
    const uint32_t kk = live ? ksrc[i] : 0u;
    cg += __popc(__ballot_sync(0xffffffffu, live && (ge_mode ? (kk >= tau) : (kk > tau))));
    ce += __popc(__ballot_sync(0xffffffffu, live && !ge_mode && kk == tau));
  }
  if (lane == 0) {
    s_wgt[warp] = cg;
    s_weq[warp] = ce;
  }
  __syncthreads();
  int tot_unused;
  int gtb = warp_totals_prefix(s_wgt, warp, lane, &tot_unused);
  int eqb = warp_totals_prefix(s_weq, warp, lane, &tot_unused);
  const int32_t* wsrc = src + w0;
  for (int i0 = 0; i0 < kn; i0 += 32 * SEL_OUT_UNROLL) {
    uint32_t kk[SEL_OUT_UNROLL];
    int at[SEL_OUT_UNROLL];
#pragma unroll
    for (int j = 0; j < SEL_OUT_UNROLL; ++j) {
      const int i = i0 + 32 * j + lane;
      kk[j] = i < kn ? ksrc[i] : 0u;
      at[j] = i < kn ? (bracketed ? static_cast<int>(region_pos[i]) : i) : 0;
    }
    // kept keys and their output rows first, then the id loads of the kept ones
    int pos[SEL_OUT_UNROLL];
#pragma unroll
    for (int j = 0; j < SEL_OUT_UNROLL; ++j) {
      const bool live = i0 + 32 * j + lane < kn;
      const bool gt = live && (ge_mode ? (kk[j] >= tau) : (kk[j] > tau));
      const bool eq = live && !ge_mode && kk[j] == tau;
      const unsigned bg = __ballot_sync(0xffffffffu, gt);
      const unsigned be = __ballot_sync(0xffffffffu, eq);
      const int my_gt = gtb + __popc(bg & lt_mask);
      const int my_eq = eqb + __popc(be & lt_mask);
      pos[j] = (gt || (eq && my_eq < want)) ? my_gt + min(my_eq, want) : -1;
      if (pos[j] >= q_out) pos[j] = -1;
      gtb += __popc(bg);
      eqb += __popc(be);
    }
    int id[SEL_OUT_UNROLL];
#pragma unroll
    for (int j = 0; j < SEL_OUT_UNROLL; ++j) id[j] = pos[j] >= 0 ? __ldg(wsrc + at[j]) : 0;
#pragma unroll
    for (int j = 0; j < SEL_OUT_UNROLL; ++j)
      if (pos[j] >= 0) out[pos[j]] = id[j];
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
  const size_t smem = (SEL_SMEM_KEYS + SEL_CAND_KEYS) * sizeof(uint32_t) + SEL_CAND_KEYS * sizeof(uint16_t);
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
  select_kernel<<<dims.E, SEL_THREADS, smem, s>>>(offsets, bucket, quota, dims.E, max_rows, sel_offsets, sel_ids,
                                                  static_cast<const uint32_t*>(ws), ctx->d_status);
  return launch_status();
}
