// Step 5 of the path: the packed expert backward of FC2 as variable-size
// grouped GEMMs without padding (LRMoE sec. 3.3: the number of kept rows of
// an expert is the M of its input-gradient product and the K of its
// weight-gradient product, and the weight shapes do not change; sec. 3.4 and
// Fig. 4: variable M, no padding rows; appendix 7.1 eq. (6), (8), (9)).  With the compacted, expert-major rows of step 4:
//   dgrad  dphi_c[seg e] = delta_c[seg e] . W_e      M = Q_e (ragged), N = I, K = h
//   wgrad  dW_e          = delta_c[seg e]^T . phi_c  M = h, N = I, K = Q_e (ragged)
//
// Blackwell design: persistent clusters of two CTAs (one per SM of a pair,
// as many pairs as fit at once), each pair owning whole 256-wide output
// tiles.  The even CTA issues tcgen05.mma.cta_group::2 with M = 256 (128
// rows of A from each CTA's shared memory, half of B from each), bf16 in and
// fp32 accumulated in TMEM, double-buffered so the epilogue of one tile
// overlaps the main loop of the next.  Per CTA:
//   warp 0      TMA producer: 128-byte-swizzled tiles into a shared-memory
//               ring (full/empty mbarriers; the pair's loads count their
//               bytes on the even CTA's barrier)
//   warp 1      TMEM owner; in the even CTA, the MMA issuer
//   warps 2..9  epilogue: tcgen05.ld of their 32-lane TMEM quarter, convert
//               and store, then release the accumulator on the even CTA
// The tile schedule is static and computed on the device from sel_offsets:
// every role walks the same list of (expert, tile) pairs, so the ragged sizes
// never travel to the host.  The wgrad zero-fills the rows of an expert's
// last K block that lie past its segment before the MMA reads them, and
// writes exact zeros for experts with no retained row.
// Every wait is bounded (lrm_set_wait_budget); a wait that runs out raises
// LRM_ERR_TIMEOUT, the block winds down, drains its tensor-core work and
// frees its TMEM before returning.
#include <cuda_bf16.h>

#include "lrm_internal.cuh"

namespace lrm {
namespace {

constexpr int MAX_E = 1024;

// ---------------------------------------------------------------------------
// wgrad on CTA pairs: dW_e [h, I] in 256 x BN output tiles, one per cluster of
// two CTAs.  CTA r of a pair loads rows [128r, 128r + 128) of the tile's M
// (= h) range of delta_c^T and columns [r BN/2, (r+1) BN/2) of phi_c into its
// own 4-stage ring (96 K rows, 48 KiB per stage); the even CTA issues the M = 256
// tcgen05.mma.cta_group::2, which reads both CTAs' shared memory, so each B
// byte crosses L2 once per pair.  Each CTA's TMEM holds its 128 rows x BN.
//   warp 0   TMA producer of the CTA's halves.  Full K blocks: both CTAs'
//            loads count their bytes on the even CTA's full barrier
//            (cta_group::2 TMA) and the even CTA gives the phase's two
//            arrivals.  The ragged last K block of an expert: each CTA loads
//            into its own "tail" barrier instead.
//   warp 1   even CTA: waits for the stage, issues the pair MMAs and
//            multicasts the commits to both CTAs' empty / accumulator-full
//            barriers (idle in the odd CTA)
//   warps 2-9 epilogue of the CTA's own 128 rows, two warps per TMEM lane
//            quarter (each takes half of the BN columns; TMEM chunks are
//            prefetched one ahead), a shuffle transpose of 16-byte quads so
//            that each store instruction writes 8 rows x 64 bytes, then
//            release the accumulator on the even CTA's barrier (16 arrivals)
//   warp 10  tail fixer: waits for the CTA's own tail load, zeroes the rows
//            of its halves that lie past the expert's segment (the MMA reads
//            whole 16-row K steps) and arrives on the even CTA's full barrier
//            (release at cluster scope), off the MMA warp's path

template <int BN>
struct CfgPair {
  static constexpr int BKS = 96;                       // K rows per stage: 6 MMAs per barrier round
  static constexpr int ATOM = 64 * BKS * 2;             // one [BKS][64] bf16 swizzle atom
  static constexpr int A_BYTES = 2 * ATOM;              // this CTA's 128 rows of M
  static constexpr int B_BYTES = (BN / 128) * ATOM;     // this CTA's BN/2 columns of N
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 4;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int EPI_WARPS = 8;                       // two per TMEM lane quarter
  static constexpr int THREADS = 64 + 32 * EPI_WARPS + 32;  // + the tail fixer warp
  static constexpr int FIXER_WARP = 2 + EPI_WARPS;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
};

// In-register transpose for the wgrad epilogue.  r holds one accumulator row
// (lane = row within the warp's 32) as eight 16-byte quads, slot 4 beta + s =
// columns 16 beta + 4 s.  Within each group of four lanes the 4 x 4 matrix of
// quads (row i, slot s) is transposed for each beta by two butterfly stages
// (stage b swaps bit b of the lane and of the slot), so that afterwards lane i
// holds, in slot 4 beta + rho, quad s = i of row rho of its group.
__device__ __forceinline__ void quad_transpose_4x4(uint32_t (&r)[32], int lane) {
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const bool hi = (lane >> b) & 1;
#pragma unroll
    for (int beta = 0; beta < 2; ++beta) {
#pragma unroll
      for (int other = 0; other < 2; ++other) {
        // the slot pair that differs in bit b; the other bit is `other`
        const int s0 = 4 * beta + (b == 0 ? 2 * other : other);
        const int s1 = s0 + (1 << b);
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const uint32_t send = hi ? r[4 * s0 + f] : r[4 * s1 + f];
          const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 1 << b);
          if (hi)
            r[4 * s0 + f] = got;
          else
            r[4 * s1 + f] = got;
        }
      }
    }
  }
}

// Start row and length of expert e's segment, clamped to the buffers.
__device__ __forceinline__ void segment(const int32_t* __restrict__ sel_offsets, int e, int max_rows, int& start,
                                        int& len) {
  int st = __ldg(sel_offsets + e), en = __ldg(sel_offsets + e + 1);
  st = min(max(st, 0), max_rows);
  en = min(max(en, st), max_rows);
  start = st;
  len = en - st;
}

// dW element type: fp32, or bf16 (round to nearest even) when OutT is uint16_t
template <typename OutT>
struct DwStore;
template <>
struct DwStore<float> {
  __device__ static __forceinline__ void put(float* o, float4 v, int accumulate) {
    if (accumulate) {
      const float4 old = *reinterpret_cast<const float4*>(o);
      v.x += old.x;
      v.y += old.y;
      v.z += old.z;
      v.w += old.w;
    }
    *reinterpret_cast<float4*>(o) = v;
  }
};
template <>
struct DwStore<uint16_t> {
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&r);
  }
  __device__ static __forceinline__ void put(uint16_t* o, float4 v, int accumulate) {
    if (accumulate) {
      const uint2 old = *reinterpret_cast<const uint2*>(o);
      v.x += __uint_as_float(old.x << 16);
      v.y += __uint_as_float(old.x & 0xFFFF0000u);
      v.z += __uint_as_float(old.y << 16);
      v.w += __uint_as_float(old.y & 0xFFFF0000u);
    }
    *reinterpret_cast<uint2*>(o) = make_uint2(pack(v.x, v.y), pack(v.z, v.w));
  }
};

template <int BN, typename OutT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(CfgPair<BN>::THREADS, 1)
    wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const int32_t* __restrict__ sel_offsets, int E,
                      int h, int I, int max_rows, int accumulate, OutT* __restrict__ out, unsigned int* status,
                      unsigned long long budget_ns) {
  using C = CfgPair<BN>;
  extern __shared__ uint8_t dsmem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tail_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_len[MAX_E];
  __shared__ int s_start[MAX_E];  // segment bounds, so no role reads sel_offsets per tile
  __shared__ uint16_t s_order[MAX_E];  // experts by descending retained rows (ties: lower id)
  static_assert(C::STAGES <= 32, "tail parities are kept in one 32-bit mask");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int tiles_n = (I + BN - 1) / BN;
  const int tiles_m = (h + 255) / 256;
  const int per_expert = tiles_m * tiles_n;
  const int total_tiles = E * per_expert;

  // Schedule: the pair tiles of all experts, heaviest expert first, cut into
  // rounds of one tile per pair, dealt as a snake (forward in even rounds,
  // backward in odd ones), which balances the ragged K loops; the tiles of
  // one expert run side by side (their operands are shared through L2).
  // Measured against rounds that alternate between the heavy front and the
  // light back of the list: equal on the Qwen3-shaped layer, 2-3.5 % faster
  // on the GLM-4.5-, DeepSeek-V2-shaped and 131k-token layers (back-to-back
  // light tiles let the ring run several tiles ahead).
  for (int e = tid; e < E; e += C::THREADS) {
    int st, ln;
    segment(sel_offsets, e, max_rows, st, ln);
    s_len[e] = ln;
    s_start[e] = st;
  }
  __syncthreads();
  for (int e = tid; e < E; e += C::THREADS) {
    const int le = s_len[e];
    int rank = 0;
    for (int x = 0; x < E; ++x) {
      const int lx = s_len[x];
      rank += (lx > le) || (lx == le && x < e);
    }
    s_order[rank] = static_cast<uint16_t>(e);
  }
  if (tid == 0) {
    s_abort = 0;
    if (blockIdx.x == 0 && __ldg(sel_offsets + E) > max_rows) raise_flag(status, LRM_ERR_SHAPE);
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full_bar[i], 2);  // full block: the even CTA twice; tail block: each fixer once
      mbar_init(&tail_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 2 * C::EPI_WARPS);
    }
    mbar_init(&drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem_base, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort_flag = &s_abort;
  auto fail = [&]() {
    *abort_flag = 1;
    raise_flag(status, LRM_ERR_TIMEOUT);
  };
  const int nblocks = (total_tiles + npairs - 1) / npairs;
  auto tile_of = [&](int round) { return round * npairs + ((round & 1) ? npairs - 1 - pair : pair); };
  auto decode = [&](int tile, int& e, int& mt, int& nt) {
    const int slot = tile / per_expert;
    e = s_order[slot];
    const int rem = tile - slot * per_expert;
    mt = rem / tiles_n;
    nt = rem - mt * tiles_n;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      const uint32_t full0 = mapa_shared(&full_bar[0], 0);  // the even CTA's full barriers
      uint32_t it = 0, tail_par = 0;
      bool ok = true;
      for (int round = 0; round < nblocks && ok; ++round) {
        const int tile = tile_of(round);
        if (tile >= total_tiles) continue;
        int e, mt, nt;
        decode(tile, e, mt, nt);
        const int start = s_start[e], len = s_len[e];
        const int nkb = (len + C::BKS - 1) / C::BKS;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty_bar[s], ph ^ 1u, budget_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          uint8_t* a_dst = smem + s * C::STAGE_BYTES;
          uint8_t* b_dst = a_dst + C::A_BYTES;
          const int xa = mt * 256 + static_cast<int>(rank) * 128;
          const int xb = nt * BN + static_cast<int>(rank) * (BN / 2);
          const int y = start + kb * C::BKS;
          if (len - kb * C::BKS >= C::BKS) {
            if (leader) {
              // both arrivals of a full block come from here; the odd CTA's
              // loads only add their bytes
              mbar_arrive_expect_tx(&full_bar[s], 2 * C::STAGE_BYTES);
              mbar_arrive(&full_bar[s]);
            }
            const uint32_t bar = full0 + s * 8;
#pragma unroll
            for (int c = 0; c < 2; ++c) tma_load_2d_pair(a_dst + c * C::ATOM, &tmA, bar, xa + c * 64, y);
#pragma unroll
            for (int c = 0; c < BN / 128; ++c) tma_load_2d_pair(b_dst + c * C::ATOM, &tmB, bar, xb + c * 64, y);
          } else {
            mbar_arrive_expect_tx(&tail_bar[s], C::STAGE_BYTES);
#pragma unroll
            for (int c = 0; c < 2; ++c) tma_load_2d(a_dst + c * C::ATOM, &tmA, &tail_bar[s], xa + c * 64, y);
#pragma unroll
            for (int c = 0; c < BN / 128; ++c)
              tma_load_2d(b_dst + c * C::ATOM, &tmB, &tail_bar[s], xb + c * 64, y);
            tail_par ^= 1u << s;
          }
        }
      }
      // the even CTA's commits arrive on these barriers asynchronously: wait
      // for the release of the last STAGES stages so none is still in flight
      // when the block exits (also lets issued copies land after a timeout)
      for (uint32_t j = it; j < it + C::STAGES; ++j)
        if (!mbar_wait(&empty_bar[j % C::STAGES], ((j / C::STAGES) & 1u) ^ 1u, budget_ns, ok ? abort_flag : nullptr))
          break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16_f32(256, BN, 1u, 1u);
    uint32_t it = 0, acc_it = 0;
    bool ok = leader;
    for (int round = 0; round < nblocks && ok; ++round) {
      const int tile = tile_of(round);
      if (tile >= total_tiles) continue;
      int e, mt, nt;
      decode(tile, e, mt, nt);
      const int len = s_len[e];
      const int nkb = (len + C::BKS - 1) / C::BKS;
      if (nkb == 0) continue;
      const uint32_t acc = acc_it & 1u;
      const uint32_t aph = (acc_it >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(&tempty_bar[acc], aph ^ 1u, budget_ns, abort_flag))) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const uint32_t s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1u;
        const int valid = len - kb * C::BKS;
        const bool tail = valid < C::BKS;
        const int nk = tail ? (valid + 15) / 16 : C::BKS / 16;
        // a tail stage was zero-filled by the fixer warps of both CTAs
        const bool got = tail ? mbar_wait_cluster(&full_bar[s], ph, budget_ns, abort_flag)
                              : mbar_wait(&full_bar[s], ph, budget_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = smem_u32(smem + s * C::STAGE_BYTES);
          const uint64_t adesc = smem_desc_sw128(a_addr, C::ATOM, 1024);
          const uint64_t bdesc = smem_desc_sw128(a_addr + C::A_BYTES, C::ATOM, 1024);
          // a K step of 16 rows is 2048 bytes, 128 in the descriptor's address field; the
          // MMAs of a full stage are issued back to back (the tensor pipe queues few)
          if (!tail) {
#pragma unroll
            for (int kk = 0; kk < C::BKS / 16; ++kk)
              mma_bf16_ss_pair(d_tmem, adesc + kk * 128, bdesc + kk * 128, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          } else {
            for (int kk = 0; kk < nk; ++kk)
              mma_bf16_ss_pair(d_tmem, adesc + kk * 128, bdesc + kk * 128, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_pair_multicast(&empty_bar[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit_pair_multicast(&tfull_bar[acc]);
      __syncwarp();
      ++acc_it;
    }
    if (leader) {
      if (lane == 0) {
        mma_commit_pair_local(&drain_bar);
        if (!mbar_wait(&drain_bar, 0, budget_ns, nullptr)) raise_flag(status, LRM_ERR_TIMEOUT);
      }
      __syncwarp();
    }
  } else if (warp == C::FIXER_WARP) {
    // ------------------------------------------------------------ tail fixer
    const uint32_t full0 = mapa_shared(&full_bar[0], 0);
    uint32_t it = 0, tail_par = 0;
    bool ok = true;
    for (int round = 0; round < nblocks && ok; ++round) {
      const int tile = tile_of(round);
      if (tile >= total_tiles) continue;
      int e, mt, nt;
      decode(tile, e, mt, nt);
      const int len = s_len[e];
      const int nkb = (len + C::BKS - 1) / C::BKS;
      if (nkb == 0) continue;
      it += nkb - 1;  // full blocks need no fixing
      const int valid = len - (nkb - 1) * C::BKS;
      if (valid < C::BKS) {
        const uint32_t s = it % C::STAGES;
        const uint32_t tph = (tail_par >> s) & 1u;
        tail_par ^= 1u << s;
        if (!__all_sync(0xffffffffu, mbar_wait(&tail_bar[s], tph, budget_ns, abort_flag))) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        uint8_t* a_stage = smem + s * C::STAGE_BYTES;
        uint8_t* b_stage = a_stage + C::A_BYTES;
        // rows [valid, 16 ceil(valid/16)) of this CTA's halves lie past the segment
        const int nz = ((valid + 15) / 16) * 16 - valid;
        constexpr int atoms = 2 + BN / 128;
        const int units = nz * 8 * atoms;
        for (int i = lane; i < units; i += 32) {
          const int atom = i / (nz * 8);
          const int rem = i - atom * nz * 8;
          uint8_t* base = atom < 2 ? a_stage + atom * C::ATOM : b_stage + (atom - 2) * C::ATOM;
          *reinterpret_cast<uint4*>(base + (valid + rem / 8) * 128 + (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(&full_bar[s]);
          else
            mbar_arrive_cluster(full0 + s * 8);
        }
        __syncwarp();
      }
      ++it;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int c_begin = ((warp - 2) >> 2) * (BN / 2);  // this warp's half of the columns
    // store layout: a warp instruction covers 8 rows x 16 columns (64 bytes
    // of each row); lane = (row within the 8) * 4 + column quad
    const int sub_row = lane >> 2, quad = (lane & 3) * 4;
    const uint32_t tempty0 = mapa_shared(&tempty_bar[0], 0);
    uint32_t acc_it = 0;
    for (int round = 0; round < nblocks; ++round) {
      const int tile = tile_of(round);
      if (tile >= total_tiles) continue;
      int e, mt, nt;
      decode(tile, e, mt, nt);
      const int row_w = mt * 256 + static_cast<int>(rank) * 128 + q * 32;  // first dW row of this warp
      OutT* obase = out + (static_cast<size_t>(e) * h + row_w) * I;
      const int len = s_len[e];
      if (len == 0) {
        if (!accumulate) {
          for (int c = 0; c < BN / 2; c += 16) {
            const int col = nt * BN + c_begin + c + quad;
            if (col >= I) break;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int rr = 8 * v + sub_row;
              if (row_w + rr < h)
                DwStore<OutT>::put(obase + static_cast<size_t>(rr) * I + col, make_float4(0.f, 0.f, 0.f, 0.f), 0);
            }
          }
        }
        continue;
      }
      const uint32_t acc = acc_it & 1u;
      const uint32_t aph = (acc_it >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull_bar[acc], aph, budget_ns, abort_flag))) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c_begin;
      uint32_t r[32], nx[32];
      tmem_ld_32x32b_x32(taddr, r);
      tmem_ld_wait();
      for (int c = 0; c < BN / 2; c += 32) {
        const bool more = c + 32 < BN / 2;
        if (more) tmem_ld_32x32b_x32(taddr + c + 32, nx);  // next chunk in flight while this one is stored
        // 4 x 4 transpose of 16-byte quads inside each group of four lanes (two
        // butterfly stages): lane 4g + i then holds, for each row 4g + rho and
        // 16-column half beta, the quad of columns 16 beta + 4i.
        quad_transpose_4x4(r, lane);
        const int col = nt * BN + c_begin + c + 4 * (lane & 3);
#pragma unroll
        for (int beta = 0; beta < 2; ++beta) {
          if (col + 16 * beta < I) {
#pragma unroll
            for (int rho = 0; rho < 4; ++rho) {
              const int rr = 4 * (lane >> 2) + rho;
              if (row_w + rr < h) {
                float4 val = make_float4(__uint_as_float(r[16 * beta + 4 * rho]), __uint_as_float(r[16 * beta + 4 * rho + 1]),
                                         __uint_as_float(r[16 * beta + 4 * rho + 2]),
                                         __uint_as_float(r[16 * beta + 4 * rho + 3]));
                DwStore<OutT>::put(obase + static_cast<size_t>(rr) * I + col + 16 * beta, val, accumulate);
              }
            }
          }
        }
        if (more) {
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = nx[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty_bar[acc]);
        else
          mbar_arrive_cluster(tempty0 + acc * 8);
      }
      ++acc_it;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its partner may still read its shared memory or TMEM
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// dgrad on CTA pairs, computed transposed: dphi_c[seg e]^T = W_e^T .
// delta_c[seg e]^T, so M runs over the expert width I (256 per pair tile) and
// N over the segment's rows (256 per tile; the last tile of a segment rounds
// its remainder up to 32 only, so few rows are computed for nothing).
//   A = W_e^T   MN-major: CTA r loads I columns [256 mt + 128 r, +128) of W_e
//   B = rows    K-major:  CTA r loads segment rows [256 nt + r N/2, +N/2)
// K = h has no ragged tail, so both CTAs' loads count their bytes on the
// even CTA's full barrier (cta_group::2 TMA) and the even CTA issues the
// M = 256, N = 16..256 tcgen05.mma.cta_group::2.  The MMAs release each stage
// in two K halves (a commit after the first four of its eight), and the
// producer refills each half as soon as it is free.  CTA r's TMEM then holds its
// 128 I columns (lanes) x N rows (columns) of the tile.
//   warp 0    TMA producer; warp 1 MMA issuer (even CTA);
//   warps 2-9 epilogue: two warps per TMEM lane quarter, each half of the N
//             columns; a TMEM load gives every lane one I column of 32 output
//             rows, so the warp transposes the 32 x 32 block through padded
//             shared memory and each lane then writes its own row's 64
//             contiguous bytes (16-byte stores); rows past the segment are
//             skipped.

template <int BNR>
struct CfgDgradPair {
  static constexpr int BKS = 128;                    // K (= h) per stage: 8 MMAs per barrier round
  static constexpr int A_ATOM = 64 * BKS * 2;         // [BKS][64] bf16: 64 I columns of W_e, MN-major
  static constexpr int B_ATOM = (BNR / 2) * 64 * 2;   // [BNR/2][64] bf16: 64 K of this CTA's rows, K-major
  static constexpr int A_BYTES = 2 * A_ATOM;          // this CTA's 128 I columns
  static constexpr int B_BYTES = (BKS / 64) * B_ATOM;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 3;
  static_assert(BKS == 128, "a stage is released in two K halves of one B atom each");
  static constexpr int TMEM_COLS = 2 * BNR;
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int T_PITCH = 32;  // bf16 per row of a warp's transpose buffer (64 B; 16-byte chunks XOR-swizzled)
  static constexpr int STAGING_BYTES = EPI_WARPS * 32 * T_PITCH * 2;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024;
};

template <int BNR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(CfgDgradPair<BNR>::THREADS, 1)
    dgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const int32_t* __restrict__ sel_offsets, int E, int h, int I, int max_rows,
                      uint16_t* __restrict__ out, const int32_t* __restrict__ row_map, int out_rows,
                      unsigned int* status, unsigned long long budget_ns) {
  using C = CfgDgradPair<BNR>;
  extern __shared__ uint8_t dsmem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_lo[C::STAGES];  // the stage's first K half has been read
  __shared__ __align__(8) uint64_t empty_hi[C::STAGES];  // its second K half has been read
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_len[MAX_E];
  __shared__ int s_start[MAX_E];  // segment bounds, so no role reads sel_offsets per tile
  __shared__ uint16_t s_order[MAX_E];  // experts in schedule order (descending index)
  __shared__ int s_prefix[MAX_E + 1];  // first pair tile of the expert at each position of s_order

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int tiles_m = (I + 255) / 256;  // pair tiles over the expert width

  // Schedule: experts in descending index order, the tiles of one expert
  // side by side (they share W_e through L2), dealt round robin to the pairs.
  // Compaction writes the segments in ascending expert order, so the ones it
  // wrote last are still in L2 when dgrad starts (4-6 % faster than a
  // heaviest-first order, measured); the tiles cost nearly the same whatever
  // the expert, so the order does not unbalance the pairs.
  for (int e = tid; e < E; e += C::THREADS) {
    int st, ln;
    segment(sel_offsets, e, max_rows, st, ln);
    s_len[e] = ln;
    s_start[e] = st;
    s_order[E - 1 - e] = static_cast<uint16_t>(e);
  }
  __syncthreads();
  if (warp == 0) {
    // pair tiles per expert: ceil(len / BNR) x tiles_m (a run of positions per lane, then a warp scan)
    const int per = (E + 31) / 32;
    const int i0 = lane * per;
    int local = 0;
    for (int i = i0; i < min(E, i0 + per); ++i) local += ((s_len[s_order[i]] + BNR - 1) / BNR) * tiles_m;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - local;
    for (int i = i0; i < min(E, i0 + per); ++i) {
      s_prefix[i] = run;
      run += ((s_len[s_order[i]] + BNR - 1) / BNR) * tiles_m;
    }
    if (lane == 31) s_prefix[E] = incl;
  }
  if (tid == 0) {
    s_abort = 0;
    if (blockIdx.x == 0 && __ldg(sel_offsets + E) > max_rows) raise_flag(status, LRM_ERR_SHAPE);
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full_bar[i], 2);  // both arrivals come from the even CTA's producer
      mbar_init(&empty_lo[i], 1);
      mbar_init(&empty_hi[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 2 * C::EPI_WARPS);
    }
    mbar_init(&drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem_base, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total_tiles = s_prefix[E];
  volatile int* abort_flag = &s_abort;
  auto fail = [&]() {
    *abort_flag = 1;
    raise_flag(status, LRM_ERR_TIMEOUT);
  };
  // tile -> expert, row tile nt (over the segment), width tile mt (over I);
  // within an expert the row tiles run fastest, so pairs dealt neighbouring
  // tiles share the same W_e columns (1-4 % faster than width tiles fastest
  // on the Qwen3-, GLM-4.5- and DeepSeek-V2-shaped layers, measured)
  auto decode = [&](int tile, int& e, int& nt, int& mt) {
    int lo = 0, hi = E - 1;  // last position with s_prefix <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_prefix[mid] <= tile)
        lo = mid;
      else
        hi = mid - 1;
    }
    e = s_order[lo];
    const int rem = tile - s_prefix[lo];
    const int n_nt = (s_len[e] + BNR - 1) / BNR;
    mt = rem / n_nt;
    nt = rem - mt * n_nt;
  };
  // rows of row tile nt that the MMA computes: the remainder rounded up to 32
  // (N of a pair MMA with M = 256 is a multiple of 32)
  auto tile_rows = [&](int len, int nt) { return min(BNR, ((len - nt * BNR + 31) / 32) * 32); };
  const int nkb = (h + C::BKS - 1) / C::BKS;  // K past h reads as zeros (tensor bounds)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      const uint32_t full0 = mapa_shared(&full_bar[0], 0);  // the even CTA's full barriers
      uint32_t it = 0;
      bool ok = true;
      for (int tile = pair; tile < total_tiles && ok; tile += npairs) {
        int e, nt, mt;
        decode(tile, e, nt, mt);
        const int start = s_start[e], len = s_len[e];
        const int half = tile_rows(len, nt) / 2;
        const int xa = mt * 256 + static_cast<int>(rank) * 128;
        const int yb = start + nt * BNR + static_cast<int>(rank) * half;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty_lo[s], ph ^ 1u, budget_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          uint8_t* a_dst = smem + s * C::STAGE_BYTES;
          uint8_t* b_dst = a_dst + C::A_BYTES;
          if (leader) {
            mbar_arrive_expect_tx(&full_bar[s], 2 * C::STAGE_BYTES);
            mbar_arrive(&full_bar[s]);
          }
          const uint32_t bar = full0 + s * 8;
          // The first K half (64 rows of each A atom, the first B atom) as soon
          // as its MMAs have read the slot, the second half once theirs have:
          // the MMAs hold a stage while the ones before it run, so refilling
          // by halves keeps more of the ring loading (dgrad 2-6 % faster).
          constexpr int HK = C::BKS / 2;
          constexpr int HOFF = HK * 128;  // bytes of the first half in an A atom
#pragma unroll
          for (int c = 0; c < 2; ++c) tma_load_3d_pair(a_dst + c * C::A_ATOM, &tmA, bar, xa + c * 64, kb * C::BKS, e);
          tma_load_2d_pair(b_dst, &tmB, bar, kb * C::BKS, yb);
          if (!mbar_wait(&empty_hi[s], ph ^ 1u, budget_ns, abort_flag)) {
            fail();
            ok = false;
            ++it;  // this stage's first half is in flight
            break;
          }
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_3d_pair(a_dst + c * C::A_ATOM + HOFF, &tmA, bar, xa + c * 64, kb * C::BKS + HK, e);
          tma_load_2d_pair(b_dst + C::B_ATOM, &tmB, bar, kb * C::BKS + HK, yb);
        }
      }
      // the even CTA's commits arrive on these barriers asynchronously: wait
      // for the release of the last STAGES stages before the block can exit
      // (a stage's second half is released last)
      for (uint32_t j = it; j < it + C::STAGES; ++j)
        if (!mbar_wait(&empty_hi[j % C::STAGES], ((j / C::STAGES) & 1u) ^ 1u, budget_ns, ok ? abort_flag : nullptr))
          break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    uint32_t it = 0, acc_it = 0;
    bool ok = leader;
    for (int tile = pair; tile < total_tiles && ok; tile += npairs) {
      int e, nt, mt;
      decode(tile, e, nt, mt);
      const int len = s_len[e];
      const uint32_t idesc = idesc_bf16_f32(256, static_cast<uint32_t>(tile_rows(len, nt)), 1u, 0u);
      const uint32_t acc = acc_it & 1u;
      const uint32_t aph = (acc_it >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(&tempty_bar[acc], aph ^ 1u, budget_ns, abort_flag))) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BNR;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const uint32_t s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], ph, budget_ns, abort_flag))) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = smem_u32(smem + s * C::STAGE_BYTES);
          const uint64_t adesc = smem_desc_sw128(a_addr, C::A_ATOM, 1024);
          const uint64_t bdesc = smem_desc_sw128(a_addr + C::A_BYTES, 16, 1024);
          // descriptor address field in 16-byte units: A (MN-major) advances 2048 B per
          // 16 K rows; B (K-major) 32 B per 16 K inside an atom, then the next atom
#pragma unroll
          for (int kk = 0; kk < C::BKS / 16; ++kk) {
            mma_bf16_ss_pair(d_tmem, adesc + kk * 128, bdesc + (kk >> 2) * (C::B_ATOM >> 4) + (kk & 3) * 2, idesc,
                             (kb > 0 || kk > 0) ? 1u : 0u);
            if (kk == C::BKS / 32 - 1) mma_commit_pair_multicast(&empty_lo[s]);  // first K half read
          }
          mma_commit_pair_multicast(&empty_hi[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit_pair_multicast(&tfull_bar[acc]);
      __syncwarp();
      ++acc_it;
    }
    if (leader) {
      if (lane == 0) {
        mma_commit_pair_local(&drain_bar);
        if (!mbar_wait(&drain_bar, 0, budget_ns, nullptr)) raise_flag(status, LRM_ERR_TIMEOUT);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                             // TMEM lane quarter this warp may access
    const int c_begin = ((warp - 2) >> 2) * (BNR / 2);  // this warp's half of the tile's rows
    uint16_t* tbuf = reinterpret_cast<uint16_t*>(smem + C::STAGES * C::STAGE_BYTES) + (warp - 2) * 32 * C::T_PITCH;
    const uint32_t tempty0 = mapa_shared(&tempty_bar[0], 0);
    uint32_t acc_it = 0;
    for (int tile = pair; tile < total_tiles; tile += npairs) {
      int e, nt, mt;
      decode(tile, e, nt, mt);
      const int start = s_start[e], len = s_len[e];
      const int n_cols = tile_rows(len, nt);
      const int rows_valid = len - nt * BNR;  // rows of this tile inside the segment
      const uint32_t acc = acc_it & 1u;
      const uint32_t aph = (acc_it >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull_bar[acc], aph, budget_ns, abort_flag))) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const int col0 = mt * 256 + static_cast<int>(rank) * 128 + q * 32;  // first I column of this warp
      const int row0 = start + nt * BNR;  // first compacted row of this tile
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BNR;
      const int c_end = min(n_cols, c_begin + BNR / 2);
      for (int c = c_begin; c < c_end; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c, r);  // lane = I column, r[j] = output row c + j
        tmem_ld_wait();
        __syncwarp();  // the previous chunk's reads of the buffer are done
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          // row j, I column `lane`: 16-byte chunk lane / 8 of the row, XOR-swizzled by row
          const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(r[j]));
          tbuf[j * C::T_PITCH + ((((lane >> 3) ^ (j >> 1)) & 3) << 3) + (lane & 7)] =
              *reinterpret_cast<const uint16_t*>(&b);
        }
        __syncwarp();
        if (c + lane < rows_valid) {  // lane = output row c + lane
          // compacted layout: row r of out; with a row map (the inverse mapping
          // of the selection), row row_map[r] of the [out_rows, I] array
          int r = row0 + c + lane;
          if (row_map != nullptr) {
            r = __ldg(row_map + r);
            if (r < 0 || r >= out_rows) {
              raise_flag(status, LRM_ERR_INDEX);
              r = -1;
            }
          }
          if (r >= 0) {
            const uint4* src = reinterpret_cast<const uint4*>(tbuf + lane * C::T_PITCH);
            uint16_t* orow = out + static_cast<size_t>(r) * I + col0;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              if (col0 + v * 8 < I) *reinterpret_cast<uint4*>(orow + v * 8) = src[(v ^ (lane >> 1)) & 3];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty_bar[acc]);
        else
          mbar_arrive_cluster(tempty0 + acc * 8);
      }
      ++acc_it;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its partner may still read its shared memory or TMEM
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
}

// Row-major 2-D bf16 tensor [rows][cols] with [box_rows][64] boxes.
lrm_status encode_2d(lrm_ctx* ctx, CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                     uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = ctx->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LRM_OK : LRM_ERR_CUDA;
}

// W [E][h][I] bf16 as a 3-D tensor (I, h, E) with [1][box_h][64] boxes.
lrm_status encode_w(lrm_ctx* ctx, CUtensorMap* map, const void* base, uint64_t I, uint64_t h, uint64_t E,
                    uint32_t box_h) {
  const cuuint64_t dims[3] = {I, h, E};
  const cuuint64_t strides[2] = {I * 2, h * I * 2};
  const cuuint32_t box[3] = {64, box_h, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = ctx->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LRM_OK : LRM_ERR_CUDA;
}

template <int BN, typename OutT>
lrm_status launch_wgrad_pair(lrm_ctx* ctx, const CUtensorMap& a, const CUtensorMap& b,
                             const int32_t* sel_offsets, const lrm_dims& d, int max_rows, int accumulate, OutT* out,
                             cudaStream_t s) {
  using C = CfgPair<BN>;
  auto kern = wgrad_pair_kernel<BN, OutT>;
  static thread_local int configured_device = -1;
  static thread_local int clusters = 0;
  if (configured_device != ctx->device) {
    if (ctx->smem_optin < C::SMEM_BYTES + 1024) return LRM_ERR_ARCH;
    LRM_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctx->sm_count & ~1, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    int n = 0;
    LRM_CHECK_CUDA(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
    if (n < 1) return LRM_ERR_ARCH;
    clusters = n;
    configured_device = ctx->device;
  }
  kern<<<2 * clusters, C::THREADS, C::SMEM_BYTES, s>>>(a, b, sel_offsets, d.E, d.h, d.I, max_rows, accumulate,
                                                         out, ctx->d_status, ctx->wait_budget_ns);
  return launch_status();
}

// a = W_e^T operand (W map), b = segment rows operand (delta_c map)
template <int BNR>
lrm_status launch_dgrad_pair(lrm_ctx* ctx, const CUtensorMap& a, const CUtensorMap& b, const int32_t* sel_offsets,
                             const lrm_dims& d, int max_rows, uint16_t* out, const int32_t* row_map, int out_rows,
                             cudaStream_t s) {
  using C = CfgDgradPair<BNR>;
  auto kern = dgrad_pair_kernel<BNR>;
  static thread_local int configured_device = -1;
  static thread_local int clusters = 0;
  if (configured_device != ctx->device) {
    if (ctx->smem_optin < C::SMEM_BYTES + 8 * 1024) return LRM_ERR_ARCH;
    LRM_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctx->sm_count & ~1, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    int n = 0;
    LRM_CHECK_CUDA(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
    if (n < 1) return LRM_ERR_ARCH;
    clusters = n;
    configured_device = ctx->device;
  }
  kern<<<2 * clusters, C::THREADS, C::SMEM_BYTES, s>>>(a, b, sel_offsets, d.E, d.h, d.I, max_rows, out, row_map,
                                                       out_rows, ctx->d_status, ctx->wait_budget_ns);
  return launch_status();
}

}  // namespace
}  // namespace lrm

using namespace lrm;

namespace {

// Both dgrad entry points: rows go to `out` in the compacted order, or through
// `row_map` to rows of an [out_rows, I] array.
lrm_status grouped_dgrad(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* W, const int32_t* sel_offsets,
                         lrm_dims dims, int32_t max_rows, uint16_t* out, const int32_t* row_map, int out_rows,
                         void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0 || sel_offsets == nullptr) return LRM_ERR_INVALID_ARG;
  if (max_rows == 0) return LRM_OK;
  if (delta_c == nullptr || W == nullptr || out == nullptr) return LRM_ERR_INVALID_ARG;
  if (!aligned(delta_c, 16) || !aligned(W, 16) || !aligned(out, 16) || !aligned(sel_offsets, 4) ||
      (row_map != nullptr && !aligned(row_map, 4)))
    return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  alignas(64) CUtensorMap ma, mb;
  using CD = CfgDgradPair<256>;
  if ((st = encode_2d(ctx, &ma, delta_c, dims.h, max_rows, 256 / 2)) != LRM_OK) return st;
  if ((st = encode_w(ctx, &mb, W, dims.I, dims.h, dims.E, CD::BKS / 2)) != LRM_OK) return st;  // half-stage boxes
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launch_dgrad_pair<256>(ctx, mb, ma, sel_offsets, dims, max_rows, out, row_map, out_rows, s);
}

}  // namespace

extern "C" lrm_status lrm_grouped_dgrad(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* W,
                                        const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows,
                                        uint16_t* dphi_c, void* stream) {
  return grouped_dgrad(ctx, delta_c, W, sel_offsets, dims, max_rows, dphi_c, nullptr, 0, stream);
}

extern "C" lrm_status lrm_grouped_dgrad_scatter(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* W,
                                                const int32_t* sel_offsets, const int32_t* sel_ids, lrm_dims dims,
                                                int32_t max_rows, uint16_t* dphi_rows, void* stream) {
  if (sel_ids == nullptr && max_rows > 0) return LRM_ERR_INVALID_ARG;
  return grouped_dgrad(ctx, delta_c, W, sel_offsets, dims, max_rows, dphi_rows, sel_ids, dims.T * dims.k, stream);
}

namespace {

template <typename OutT>
lrm_status grouped_wgrad(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* phi_c, const int32_t* sel_offsets,
                         lrm_dims dims, int32_t max_rows, int32_t accumulate, OutT* dW, void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0 || sel_offsets == nullptr || dW == nullptr) return LRM_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return LRM_ERR_INVALID_ARG;
  if (max_rows > 0 && (delta_c == nullptr || phi_c == nullptr)) return LRM_ERR_INVALID_ARG;
  if (!aligned(delta_c, 16) || !aligned(phi_c, 16) || !aligned(dW, 16) || !aligned(sel_offsets, 4))
    return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  // A map needs a non-null, 16-byte aligned base even when no row exists.
  const void* a_base = max_rows > 0 ? static_cast<const void*>(delta_c) : static_cast<const void*>(dW);
  const void* b_base = max_rows > 0 ? static_cast<const void*>(phi_c) : static_cast<const void*>(dW);
  const uint64_t rows = max_rows > 0 ? static_cast<uint64_t>(max_rows) : 1;
  alignas(64) CUtensorMap ma, mb;
  if ((st = encode_2d(ctx, &ma, a_base, dims.h, rows, CfgPair<256>::BKS)) != LRM_OK) return st;
  if ((st = encode_2d(ctx, &mb, b_base, dims.I, rows, CfgPair<256>::BKS)) != LRM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launch_wgrad_pair<256, OutT>(ctx, ma, mb, sel_offsets, dims, max_rows, accumulate, dW, s);
}

}  // namespace

extern "C" lrm_status lrm_grouped_wgrad(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* phi_c,
                                        const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows,
                                        int32_t accumulate, float* dW, void* stream) {
  return grouped_wgrad<float>(ctx, delta_c, phi_c, sel_offsets, dims, max_rows, accumulate, dW, stream);
}

extern "C" lrm_status lrm_grouped_wgrad_bf16(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* phi_c,
                                             const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows,
                                             int32_t accumulate, uint16_t* dW, void* stream) {
  return grouped_wgrad<uint16_t>(ctx, delta_c, phi_c, sel_offsets, dims, max_rows, accumulate, dW, stream);
}
