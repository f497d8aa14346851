// Step 3 of the path: per-expert TopK within the quota (LRMoE sec. 3.2 and
// 3.3, Alg. 1; appendix 7.2 Prop. 7.1: for fixed per-expert quotas,
// keeping the largest scores of every expert is optimal, and ties only
// change which of the equal boundary scores are kept).
//
// One launch.  Every expert gets a cluster of SEL_CL CTAs (thread-block
// clusters; the CTAs of a cluster read each other's shared memory through
// DSMEM and meet at hardware cluster barriers), so the heaviest expert, the
// critical path of the step, is spread over SEL_CL SMs.  CTA r takes the
// r-th contiguous slice of the expert's bucket segment (ascending u), and
// each of its warps a contiguous part of that slice.  Scores are finite and
// non-negative, so the bit patterns of their fp32 values (the keys) order
// like the values.
// Every CTA takes the cluster's decisions itself, from data it reads out of
// the other CTAs' shared memory (a DSMEM load costs a fraction of a cluster
// barrier, so the CTAs pull what they need and meet at three barriers):
//  1. gather: the slice's bucket ids and then their scores are copied into
//     shared memory with cp.async (every copy of a thread in flight at once;
//     slices above SEL_KCAP keys go through the workspace instead), with a
//     histogram of the keys' top 11 bits and a 64-bin summary of it;
//  2. barrier; the boundary bin b1 of the q-th largest key: warp 0 sums the
//     64-bin summaries of all CTAs, finds the group of 32 bins holding the
//     rank, then sums those 32 bins over the CTAs;
//  3. classify: per warp, the keys above bin b1 are counted and the keys
//     inside it kept as candidates (with their slice positions);
//  4. barrier; every CTA copies all candidates of the cluster and one warp
//     finds the exact boundary key tau with up to three radix passes (7, 7
//     and 6 bits) and how many keys equal to tau are kept (the first ones in
//     pair order, so ties go to the lower pair index).  A bin kept whole ends
//     the search early ("key >= bin start").  When a CTA has more candidates
//     than it can hold, the cluster sums two more histogram levels (bits 19-9,
//     8-0);
//  5. barrier; per-warp counts of kept keys, a prefix over the cluster's
//     CTAs and then the warps; each warp lists its kept keys (slice position,
//     output row), loads their pair ids in one round and writes them in
//     ascending u.
// No global atomics and no zeroed workspace.
#include "lrm_internal.cuh"

namespace lrm {
namespace {

constexpr int SEL_CL = 8;                  // CTAs per expert (one cluster)
constexpr int SEL_T = 128;                 // threads per CTA
constexpr int SEL_W = SEL_T / 32;          // warps per CTA
constexpr int SEL_NB = 2048;               // bins of an 11-bit digit
constexpr int SEL_KCAP = 4096;             // keys of a CTA's slice cached in shared memory
constexpr int SEL_CCAP = 256;              // candidates a CTA keeps
constexpr int SEL_WCAP = SEL_CCAP / SEL_W; // in one region per warp
constexpr int SEL_RB = 128;                // bins of the candidates' 7-bit radix digits
constexpr int SEL_GRP = 32;                // bins per group of the 64-bin summary
constexpr int SEL_BATCH = 16;              // independent loads in flight per thread (gather)
constexpr int SEL_UNR = 8;                 // keys per lane loaded together in the passes over a slice
constexpr int SEL_LCAP = SEL_NB / (2 * SEL_W);  // kept (position, row) pairs a warp lists for the id loads
static_assert(SEL_NB / SEL_CL <= 2 * SEL_T, "each thread scans at most two bins of its CTA's share");
static_assert(SEL_CL * SEL_CCAP <= SEL_NB, "the histogram's space holds every CTA's candidates");
static_assert(SEL_WCAP == 64, "a warp moves its candidate region two per lane");
static_assert(SEL_NB == 2 * 32 * SEL_GRP, "warp 0 scans the 64-bin summary two groups per lane");
static_assert(SEL_T % 32 == 0 && (2 * (SEL_NB / SEL_GRP)) % 32 == 0, "the summary loop runs whole warps");

__device__ __forceinline__ uint32_t score_key(float r) { return __float_as_uint(r) & 0x7FFFFFFFu; }

__device__ __forceinline__ int ld_cluster_s32(const int* p, uint32_t rank) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(mapa_shared(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_s32(int* p, uint32_t rank, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(mapa_shared(p, rank)), "r"(v) : "memory");
}
// the two halves of a cluster barrier, so that work can run between them
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// 4-byte asynchronous copy global -> shared (completes at cp_async_wait_all
// for the issuing thread)
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

// Exclusive prefix over a warp's lanes; *total gets the warp's sum.
__device__ __forceinline__ int warp_exclusive_scan(int v, int lane, int* total) {
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

// Exclusive prefix of one int per thread over the SEL_T threads; *total gets
// the sum.  Every thread calls it.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < SEL_W; ++w) {
    const int t = s_warp[w];
    before += w < warp ? t : 0;
    all += t;
  }
  __syncthreads();
  *total = all;
  return before + x - v;
}

struct Shared {
  uint32_t keys[SEL_KCAP];      // the slice's bucket ids, then keys, then output rows
  int hist[SEL_NB];             // this CTA's histogram; after the second barrier the cluster's candidates
  int group[SEL_NB / SEL_GRP];  // the histogram summed over groups of 32 bins
  uint32_t cand_key[SEL_CCAP];  // this CTA's candidates
  int cand_pos[SEL_CCAP];       // and their positions in the slice
  int scratch[SEL_NB / SEL_CL]; // summed bins of a distributed level, or the candidates' radix bins
  int res[4];                   // a level's result: bin, count above it, its count
  int cpre[SEL_CL + 1];         // prefix of the CTAs' candidate counts
  int tab[2];                   // kept keys of this CTA: above tau, equal to tau
  int slice_sum;
  int warp_tmp[SEL_W];
  int w_gt[SEL_W], w_in[SEL_W], w_eq[SEL_W];
  int n_cand;
};

// One distributed radix level (used when candidates overflow): every CTA has
// filled sh.hist[0, nb); returns the bin b of the want-th largest key
// (1 <= want <= the cluster's total count), the count of keys in bins above
// b, and the count in b.  CTA r sums the r-th slice of the bins over the
// cluster, the CTA whose slice holds the boundary rank scans it.
__device__ void cluster_level(Shared& sh, int nb, int want, uint32_t rank, int& bin, int& above, int& cnt) {
  const int tid = threadIdx.x;
  const int slice = nb / SEL_CL;
  const int b0 = static_cast<int>(rank) * slice;
  cluster_sync_all();  // every CTA's histogram is complete
  int mine = 0;
  for (int j = tid; j < slice; j += SEL_T) {
    int acc = 0;
#pragma unroll
    for (uint32_t c = 0; c < SEL_CL; ++c) acc += ld_cluster_s32(&sh.hist[b0 + j], c);
    sh.scratch[j] = acc;
    mine += acc;
  }
  int total;
  cta_exclusive_scan(mine, sh.warp_tmp, &total);
  if (tid == 0) sh.slice_sum = total;
  cluster_sync_all();  // slice totals are visible; nobody reads a histogram any more
  // bins ascend with the CTA rank: the keys above this CTA's bins are those
  // of the higher ranks
  int above_r = 0;
#pragma unroll
  for (uint32_t c = 0; c < SEL_CL; ++c)
    if (c > rank) above_r += ld_cluster_s32(&sh.slice_sum, c);
  if (above_r < want && want <= above_r + total) {
    // thread t holds bins hb = slice-1-2t and hb-1 (descending)
    const int hb = slice - 1 - 2 * tid;
    const int c_hi = hb >= 0 ? sh.scratch[hb] : 0;
    const int c_lo = hb >= 1 ? sh.scratch[hb - 1] : 0;
    int unused;
    const int a = above_r + cta_exclusive_scan(c_hi + c_lo, sh.warp_tmp, &unused);
    int found = -1, f_above = 0, f_cnt = 0;
    if (hb >= 0 && a < want && want <= a + c_hi) {
      found = b0 + hb;
      f_above = a;
      f_cnt = c_hi;
    } else if (hb >= 1 && a + c_hi < want && want <= a + c_hi + c_lo) {
      found = b0 + hb - 1;
      f_above = a + c_hi;
      f_cnt = c_lo;
    }
    if (found >= 0) {
#pragma unroll
      for (uint32_t c = 0; c < SEL_CL; ++c) {
        st_cluster_s32(&sh.res[0], c, found);
        st_cluster_s32(&sh.res[1], c, f_above);
        st_cluster_s32(&sh.res[2], c, f_cnt);
      }
    }
  }
  cluster_sync_all();  // the result is in every CTA
  bin = sh.res[0];
  above = sh.res[1];
  cnt = sh.res[2];
}

// The exact boundary key among the m candidates in sh.hist[0, m) (all in
// bin b1 of the top 11 bits), by radix passes over 7, 7 and 6 bits, run by
// one warp (the candidates are few, so the warp's own synchronisation is
// cheaper than the block's).  want: keys to keep among them (1 <= want <= m).
__device__ void resolve_candidates_warp(Shared& sh, int m, int b1, int want, uint32_t& tau, int& want_eq,
                                        bool& ge) {
  const int lane = threadIdx.x & 31;
  const uint32_t* ck = reinterpret_cast<const uint32_t*>(sh.hist);
  uint32_t pre = static_cast<uint32_t>(b1);
  constexpr int kShift[3] = {13, 6, 0};
  constexpr int kBits[3] = {7, 7, 6};
#pragma unroll
  for (int lv = 0; lv < 3; ++lv) {
    const int shift = kShift[lv], bits = kBits[lv], nb = 1 << bits;
    for (int b = lane; b < SEL_RB; b += 32) sh.scratch[b] = 0;
    __syncwarp();
    for (int i = lane; i < m; i += 32) {
      const uint32_t k = ck[i];
      if ((k >> (shift + bits)) == pre) atomicAdd(&sh.scratch[(k >> shift) & static_cast<uint32_t>(nb - 1)], 1);
    }
    __syncwarp();
    // lane l holds bins nb-1-4l .. nb-4-4l (descending)
    int c[4], sum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int bb = nb - 1 - 4 * lane - j;
      c[j] = bb >= 0 ? sh.scratch[bb] : 0;
      sum += c[j];
    }
    int unused;
    int a = warp_exclusive_scan(sum, lane, &unused);
    int f_bin = -1, f_above = 0, f_cnt = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (a < want && want <= a + c[j]) {
        f_bin = nb - 1 - 4 * lane - j;
        f_above = a;
        f_cnt = c[j];
      }
      a += c[j];
    }
    // exactly one lane holds the rank; max() only keeps a broken invariant
    // from turning into a lane or bin index out of range
    const int src = max(__ffs(__ballot_sync(0xffffffffu, f_bin >= 0)) - 1, 0);
    const int bin = __shfl_sync(0xffffffffu, f_bin, src);
    const int above = __shfl_sync(0xffffffffu, f_above, src);
    const int cnt = __shfl_sync(0xffffffffu, f_cnt, src);
    __syncwarp();  // every lane has read the bins before the next pass clears them
    pre = (pre << bits) | static_cast<uint32_t>(bin);
    want -= above;
    if (cnt == want) {  // the bin is kept whole
      ge = true;
      tau = pre << shift;
      want_eq = 0;
      return;
    }
  }
  ge = false;
  tau = pre;
  want_eq = want;
}

__global__ void __cluster_dims__(SEL_CL, 1, 1) __launch_bounds__(SEL_T, 8)
    select_cluster_kernel(const float* __restrict__ R, const int32_t* __restrict__ offsets,
                          const int32_t* __restrict__ bucket, const int32_t* __restrict__ quota, int N, int E,
                          int max_rows, int32_t* __restrict__ sel_offsets, int32_t* __restrict__ sel_ids,
                          uint32_t* __restrict__ keys_ws, unsigned int* status) {
  __shared__ Shared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const uint32_t rank = cluster_ctarank();
  const int e = blockIdx.x / SEL_CL;

  const int off = __ldg(offsets + e);
  const int n = max(0, __ldg(offsets + e + 1) - off);
  const int q_raw = __ldg(quota + e);
  const int q = min(max(q_raw, 0), n);
  // this CTA's slice [lo, lo + len) of the segment (32-key aligned), and each
  // warp's part [w0, w1) of it
  const int span = ((n + SEL_CL - 1) / SEL_CL + 31) & ~31;
  const int lo = min(n, static_cast<int>(rank) * span);
  const int len = min(n, lo + span) - lo;
  const int wspan = ((len + SEL_W - 1) / SEL_W + 31) & ~31;
  const int w0 = min(len, warp * wspan), w1 = min(len, w0 + wspan);
  const int32_t* ids = bucket + off + lo;
  // every branch below on q, n and the cluster's decisions is taken by the
  // whole cluster, so no CTA skips a cluster barrier
  const bool partial = q > 0 && q < n;
  const bool in_smem = len <= SEL_KCAP;
  uint32_t* K = in_smem ? sh.keys : keys_ws + off + lo;

  for (int b = tid; b < SEL_NB; b += SEL_T) sh.hist[b] = 0;
  if (tid == 0) sh.n_cand = 0;
  __syncthreads();

  // 1. gather: bucket ids, then scores, into the key array
  if (partial && in_smem) {
    for (int i = tid; i < len; i += SEL_T) cp_async4(&K[i], ids + i);
  }
  // meanwhile: the clamped quotas of the experts before e, whose sum is this
  // expert's first output row
  int part = 0;
  for (int x = tid; x < e; x += SEL_T) {
    const int nx = max(0, __ldg(offsets + x + 1) - __ldg(offsets + x));
    part += min(max(__ldg(quota + x), 0), nx);
  }
  if (partial) {
    if (in_smem) {
      cp_async_wait_all();
      for (int i = tid; i < len; i += SEL_T) {
        const int id = static_cast<int>(K[i]);
        if (id >= 0 && id < N)
          cp_async4(&K[i], R + id);
        else
          K[i] = 0u;
      }
      cp_async_wait_all();
      for (int i = tid; i < len; i += SEL_T) {
        const uint32_t k = score_key(__uint_as_float(K[i]));
        K[i] = k;
        atomicAdd(&sh.hist[k >> 20], 1);
      }
    } else {
      for (int i0 = 0; i0 < len; i0 += SEL_T * SEL_BATCH) {
        int id[SEL_BATCH];
#pragma unroll
        for (int j = 0; j < SEL_BATCH; ++j) {
          const int i = i0 + j * SEL_T + tid;
          id[j] = i < len ? __ldg(ids + i) : -1;
        }
        float r[SEL_BATCH];
#pragma unroll
        for (int j = 0; j < SEL_BATCH; ++j) r[j] = (id[j] >= 0 && id[j] < N) ? __ldg(R + id[j]) : 0.f;
#pragma unroll
        for (int j = 0; j < SEL_BATCH; ++j) {
          const int i = i0 + j * SEL_T + tid;
          if (i < len) {
            const uint32_t k = score_key(r[j]);
            K[i] = k;
            atomicAdd(&sh.hist[k >> 20], 1);
          }
        }
      }
    }
  }
  int base;
  cta_exclusive_scan(part, sh.warp_tmp, &base);  // also: the histogram is complete
  if (rank == 0 && tid == 0) {
    if (q != q_raw) raise_flag(status, LRM_ERR_QUOTA);
    sel_offsets[e] = base;
    if (e == E - 1) sel_offsets[E] = base + q;
  }
  int q_out = q;  // rows that fit below max_rows
  if (base + q > max_rows) {
    if (rank == 0 && tid == 0) raise_flag(status, LRM_ERR_SHAPE);
    q_out = max(0, max_rows - base);
  }
  int32_t* out = sel_ids + base;
  if (q_out == 0) return;
  if (q == n) {
    for (int i = tid; i < len; i += SEL_T)
      if (lo + i < q_out) out[lo + i] = __ldg(ids + i);
    return;
  }
  // 64 groups of 32 bins: index t of the loop sums half of group t / 2 (whole
  // warps take part in every iteration, as the shuffle needs)
  for (int t2 = tid; t2 < 2 * (SEL_NB / SEL_GRP); t2 += SEL_T) {
    int g = 0;
    const int b0 = (t2 >> 1) * SEL_GRP + (t2 & 1) * (SEL_GRP / 2);
#pragma unroll
    for (int j = 0; j < SEL_GRP / 2; ++j) g += sh.hist[b0 + j];
    g += __shfl_xor_sync(0xffffffffu, g, 1);
    if ((t2 & 1) == 0) sh.group[t2 >> 1] = g;
  }

  // 2. barrier; bin b1 of the q-th largest key, found by warp 0 of every CTA
  cluster_sync_all();
  if (warp == 0) {
    // lane l holds groups 63-2l and 62-2l (descending), summed over the CTAs
    int ch = 0, cl = 0;
#pragma unroll
    for (uint32_t c = 0; c < SEL_CL; ++c) {
      ch += ld_cluster_s32(&sh.group[63 - 2 * lane], c);
      cl += ld_cluster_s32(&sh.group[62 - 2 * lane], c);
    }
    int unused;
    const int a = warp_exclusive_scan(ch + cl, lane, &unused);
    int grp = -1, ga = 0;
    if (a < q && q <= a + ch) {
      grp = 63 - 2 * lane;
      ga = a;
    } else if (a + ch < q && q <= a + ch + cl) {
      grp = 62 - 2 * lane;
      ga = a + ch;
    }
    const unsigned who = __ballot_sync(0xffffffffu, grp >= 0);
    const int src = max(__ffs(who) - 1, 0);  // exactly one lane holds the rank
    grp = max(__shfl_sync(0xffffffffu, grp, src), 0);  // in [0, 63]: the bins read below stay in range
    ga = __shfl_sync(0xffffffffu, ga, src);
    // lane l holds bin (grp + 1) * 32 - 1 - l of the group (descending)
    const int bin = (grp + 1) * SEL_GRP - 1 - lane;
    int c = 0;
#pragma unroll
    for (uint32_t r = 0; r < SEL_CL; ++r) c += ld_cluster_s32(&sh.hist[bin], r);
    const int a2 = ga + warp_exclusive_scan(c, lane, &unused);
    if (a2 < q && q <= a2 + c) {
      sh.res[0] = bin;
      sh.res[1] = a2;
      sh.res[2] = c;
    }
  }
  __syncthreads();
  const int b1 = sh.res[0], above1 = sh.res[1], cnt1 = sh.res[2];
  const int want1 = q - above1;      // keys to keep from bin b1, 1 <= want1 <= cnt1
  const bool whole = cnt1 == want1;  // bin b1 is kept whole

  // 3. classify this warp's part: count the keys above bin b1 and inside it;
  // keep the ones inside as candidates while there is room
  {
    int gt = 0, in = 0;
    for (int i0 = w0; i0 < w1; i0 += 32 * SEL_UNR) {
      uint32_t kv[SEL_UNR];
#pragma unroll
      for (int j = 0; j < SEL_UNR; ++j) {
        const int i = i0 + 32 * j + lane;
        kv[j] = i < w1 ? K[i] : 0u;
      }
#pragma unroll
      for (int j = 0; j < SEL_UNR; ++j) {
        const int i = i0 + 32 * j + lane;
        const bool live = i < w1;
        const int bin = static_cast<int>(kv[j] >> 20);
        gt += __popc(__ballot_sync(0xffffffffu, live && bin > b1));
        const bool c = live && bin == b1;
        const unsigned bc = __ballot_sync(0xffffffffu, c);
        in += __popc(bc);
        // candidates go to this warp's region of the list, in order
        const int slot = in - __popc(bc) + __popc(bc & lt_mask);
        if (c && !whole && slot < SEL_WCAP) {
          sh.cand_key[warp * SEL_WCAP + slot] = kv[j];
          sh.cand_pos[warp * SEL_WCAP + slot] = i;
        }
      }
    }
    if (lane == 0) {
      sh.w_gt[warp] = gt;
      sh.w_in[warp] = in;
      sh.w_eq[warp] = 0;
    }
  }
  __syncthreads();
  // the list: warp w's candidates at [w SEL_WCAP, w SEL_WCAP + w_in[w]);
  // complete when no warp had more than SEL_WCAP
  bool cand_ok = true;
  int n_cand = 0;
#pragma unroll
  for (int w = 0; w < SEL_W; ++w) {
    cand_ok &= sh.w_in[w] <= SEL_WCAP;
    n_cand += sh.w_in[w];
  }
  if (tid == 0) sh.n_cand = cand_ok ? n_cand : SEL_CCAP + 1;

  // make the list dense (warp regions in order) for the other CTAs to copy
  if (!whole && cand_ok) {
    int before = 0;
#pragma unroll
    for (int w = 0; w < SEL_W; ++w) before += w < warp ? sh.w_in[w] : 0;
    const int mine = sh.w_in[warp];
    uint32_t k0 = 0u, k1 = 0u;
    int p0 = 0, p1 = 0;
    if (lane < mine) { k0 = sh.cand_key[warp * SEL_WCAP + lane]; p0 = sh.cand_pos[warp * SEL_WCAP + lane]; }
    if (lane + 32 < mine) { k1 = sh.cand_key[warp * SEL_WCAP + lane + 32]; p1 = sh.cand_pos[warp * SEL_WCAP + lane + 32]; }
    __syncthreads();
    if (lane < mine) { sh.cand_key[before + lane] = k0; sh.cand_pos[before + lane] = p0; }
    if (lane + 32 < mine) { sh.cand_key[before + lane + 32] = k1; sh.cand_pos[before + lane + 32] = p1; }
  }
  __syncthreads();

  bool ge = true;  // keep every key >= tau (else: > tau, plus want_eq keys equal to tau)
  uint32_t tau = static_cast<uint32_t>(b1) << 20;
  int want_eq = 0;
  if (!whole) {
    // 4. barrier; every CTA takes all candidates of the cluster
    cluster_sync_all();
    if (warp == 0) {
      const int c = lane < SEL_CL ? ld_cluster_s32(&sh.n_cand, static_cast<uint32_t>(lane)) : 0;
      int total;
      const int a = warp_exclusive_scan(min(c, SEL_CCAP + 1), lane, &total);
      if (lane < SEL_CL) sh.cpre[lane] = a;
      // a CTA holding more than SEL_CCAP makes the whole cluster split
      const bool split = __any_sync(0xffffffffu, c > SEL_CCAP);
      if (lane == 0) sh.cpre[SEL_CL] = split ? -1 : total;
    }
    __syncthreads();
    const int m = sh.cpre[SEL_CL];
    if (m >= 0) {
      for (int f = tid; f < m; f += SEL_T) {
        int r = 0;
#pragma unroll
        for (int c = 1; c < SEL_CL; ++c) r += f >= sh.cpre[c] ? 1 : 0;
        sh.hist[f] = ld_cluster_s32(reinterpret_cast<const int*>(&sh.cand_key[f - sh.cpre[r]]),
                                    static_cast<uint32_t>(r));
      }
      __syncthreads();
      if (warp == 0) {
        resolve_candidates_warp(sh, m, b1, want1, tau, want_eq, ge);
        if (lane == 0) {
          sh.res[0] = static_cast<int>(tau);
          sh.res[1] = want_eq;
          sh.res[2] = ge ? 1 : 0;
        }
      }
      __syncthreads();
      tau = static_cast<uint32_t>(sh.res[0]);
      want_eq = sh.res[1];
      ge = sh.res[2] != 0;
    } else {
      // too many candidates somewhere: two histogram levels over the cluster
      const int nc = cand_ok ? n_cand : len;
      for (int b = tid; b < SEL_NB; b += SEL_T) sh.hist[b] = 0;
      __syncthreads();
      for (int i = tid; i < nc; i += SEL_T) {
        const uint32_t k = cand_ok ? sh.cand_key[i] : K[i];
        if (static_cast<int>(k >> 20) == b1) atomicAdd(&sh.hist[(k >> 9) & 2047u], 1);
      }
      int b2, above2, cnt2;
      cluster_level(sh, SEL_NB, want1, rank, b2, above2, cnt2);
      const int want2 = want1 - above2;
      const uint32_t pre2 = (static_cast<uint32_t>(b1) << 11) | static_cast<uint32_t>(b2);  // key >> 9
      tau = pre2 << 9;
      ge = cnt2 == want2;
      want_eq = 0;
      if (!ge) {
        for (int b = tid; b < 512; b += SEL_T) sh.hist[b] = 0;
        __syncthreads();
        for (int i = tid; i < nc; i += SEL_T) {
          const uint32_t k = cand_ok ? sh.cand_key[i] : K[i];
          if ((k >> 9) == pre2) atomicAdd(&sh.hist[k & 511u], 1);
        }
        int b3, above3, cnt3;
        cluster_level(sh, 512, want2, rank, b3, above3, cnt3);
        tau |= static_cast<uint32_t>(b3);
        want_eq = want2 - above3;  // 1 <= want_eq <= cnt3
      }
    }
  }

  // 5. kept keys per warp: above tau (>= tau when ge) and equal to tau
  if (whole) {
    if (tid < SEL_W) sh.w_gt[tid] += sh.w_in[tid];
  } else if (cand_ok) {
    // the keys above bin b1 are all kept; the candidates decide the rest
    for (int i = tid; i < n_cand; i += SEL_T) {
      const uint32_t k = sh.cand_key[i];
      const int w = sh.cand_pos[i] / wspan;
      if (ge ? k >= tau : k > tau)
        atomicAdd(&sh.w_gt[w], 1);
      else if (!ge && k == tau)
        atomicAdd(&sh.w_eq[w], 1);
    }
  } else {
    int gt = 0, eq = 0;
    for (int i0 = w0; i0 < w1; i0 += 32 * SEL_UNR) {
      uint32_t kv[SEL_UNR];
#pragma unroll
      for (int j = 0; j < SEL_UNR; ++j) {
        const int i = i0 + 32 * j + lane;
        kv[j] = i < w1 ? K[i] : 0u;
      }
#pragma unroll
      for (int j = 0; j < SEL_UNR; ++j) {
        const bool live = i0 + 32 * j + lane < w1;
        const uint32_t k = kv[j];
        gt += __popc(__ballot_sync(0xffffffffu, live && (ge ? k >= tau : k > tau)));
        eq += __popc(__ballot_sync(0xffffffffu, live && !ge && k == tau));
      }
    }
    if (lane == 0) {
      sh.w_gt[warp] = gt;
      sh.w_eq[warp] = eq;
    }
  }
  __syncthreads();
  int gtb = 0, eqb = 0;
  if (tid == 0) {
    int cg = 0, ce = 0;
#pragma unroll
    for (int w = 0; w < SEL_W; ++w) {
      cg += sh.w_gt[w];
      ce += sh.w_eq[w];
    }
    sh.tab[0] = cg;
    sh.tab[1] = ce;
  }
#pragma unroll
  for (int w = 0; w < SEL_W; ++w) {
    gtb += w < warp ? sh.w_gt[w] : 0;
    eqb += w < warp ? sh.w_eq[w] : 0;
  }
  // 5. barrier; the counts of the CTAs before this one; the second half of
  // the last barrier is awaited only before leaving, so that no CTA leaves
  // while another may still read its counts
  cluster_sync_all();
#pragma unroll
  for (int c = 0; c < SEL_CL; ++c) {
    if (c < static_cast<int>(rank)) {
      gtb += ld_cluster_s32(&sh.tab[0], static_cast<uint32_t>(c));
      eqb += ld_cluster_s32(&sh.tab[1], static_cast<uint32_t>(c));
    }
  }
  cluster_arrive();

  // place the kept ids of this warp's part in ascending u: a kept key goes to
  // (#kept above tau before it) + min(#equal to tau before it, want_eq).
  // First the output row of every key replaces the key (-1 when dropped) and
  // the kept ones are listed (slice position, output row) in the warp's
  // region of the histogram space, which no CTA reads any more; then the
  // pair ids of the listed keys are loaded all at once and stored (a warp
  // that keeps more than the region holds loads them in batches instead).
  int* kept = sh.hist + warp * 2 * SEL_LCAP;
  int n_kept = 0;
  for (int i0 = w0; i0 < w1; i0 += 32 * SEL_UNR) {
    uint32_t kv[SEL_UNR];
#pragma unroll
    for (int j = 0; j < SEL_UNR; ++j) {
      const int i = i0 + 32 * j + lane;
      kv[j] = i < w1 ? K[i] : 0u;
    }
#pragma unroll
    for (int j = 0; j < SEL_UNR; ++j) {
      const int i = i0 + 32 * j + lane;
      const bool live = i < w1;
      const uint32_t k = kv[j];
      const bool gt = live && (ge ? k >= tau : k > tau);
      const bool eq = live && !ge && k == tau;
      const unsigned bg = __ballot_sync(0xffffffffu, gt);
      const unsigned be = __ballot_sync(0xffffffffu, eq);
      const int my_eq = eqb + __popc(be & lt_mask);
      int pos = (gt || (eq && my_eq < want_eq)) ? gtb + __popc(bg & lt_mask) + min(my_eq, want_eq) : -1;
      if (pos >= q_out) pos = -1;
      if (live) K[i] = static_cast<uint32_t>(pos);
      const unsigned bk = __ballot_sync(0xffffffffu, pos >= 0);
      const int slot = n_kept + __popc(bk & lt_mask);
      if (pos >= 0 && slot < SEL_LCAP) {
        kept[2 * slot] = i;
        kept[2 * slot + 1] = pos;
      }
      n_kept += __popc(bk);
      gtb += __popc(bg);
      eqb += __popc(be);
    }
  }
  __syncwarp();
  if (n_kept <= SEL_LCAP) {
    int id[SEL_LCAP / 32], row[SEL_LCAP / 32];
#pragma unroll
    for (int j = 0; j < SEL_LCAP / 32; ++j) {
      const int x = 32 * j + lane;
      row[j] = x < n_kept ? kept[2 * x + 1] : -1;
      id[j] = x < n_kept ? __ldg(ids + kept[2 * x]) : 0;
    }
#pragma unroll
    for (int j = 0; j < SEL_LCAP / 32; ++j)
      if (row[j] >= 0) out[row[j]] = id[j];
    cluster_wait();
    return;
  }
  for (int i0 = w0; i0 < w1; i0 += 32 * SEL_BATCH) {
    int pos[SEL_BATCH], id[SEL_BATCH];
#pragma unroll
    for (int j = 0; j < SEL_BATCH; ++j) {
      const int i = i0 + 32 * j + lane;
      pos[j] = i < w1 ? static_cast<int>(K[i]) : -1;
    }
#pragma unroll
    for (int j = 0; j < SEL_BATCH; ++j) id[j] = pos[j] >= 0 ? __ldg(ids + i0 + 32 * j + lane) : 0;
#pragma unroll
    for (int j = 0; j < SEL_BATCH; ++j)
      if (pos[j] >= 0) out[pos[j]] = id[j];
  }
  cluster_wait();
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  select_cluster_kernel<<<dims.E * SEL_CL, SEL_T, 0, s>>>(score, offsets, bucket, quota, dims.T * dims.k, dims.E,
                                                           max_rows, sel_offsets, sel_ids,
                                                           static_cast<uint32_t*>(ws), ctx->d_status);
  return launch_status();
}
