// Step 5 of the path: the packed expert backward of FC2 as variable-size
// grouped GEMMs without padding (LRMoE sec. 3.3: "m determines the row
// dimension of input-gradient products and the reduction dimension of
// weight-gradient products, while parameter dimensions remain unchanged";
// sec. 3.4 and Fig. 4: variable M, no padding rows; appendix 7.1 eq. (6),
// (8), (9)).  With the compacted, expert-major rows of step 4:
//   dgrad  dphi_c[seg e] = delta_c[seg e] . W_e      M = Q_e (ragged), N = I, K = h
//   wgrad  dW_e          = delta_c[seg e]^T . phi_c  M = h, N = I, K = Q_e (ragged)
//
// Blackwell design: one persistent CTA per SM, 6 warps.
//   warp 0      TMA producer: 128-byte-swizzled tiles into a STAGES-deep
//               shared-memory ring (full/empty mbarriers);
//   warp 1      owns TMEM (2 accumulators of BM x BN fp32) and issues
//               tcgen05.mma kind::f16 (bf16 in, fp32 accumulate), one elected
//               lane, committing to the ring's empty barriers and to the
//               accumulator's full barrier;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane TMEM quarter, convert
//               and store, then release the accumulator.
// The tile schedule is static and computed on the device from sel_offsets:
// every role walks the same list (expert, m-tile, n-tile), so the ragged
// sizes never travel to the host.  Tiles of the wgrad beyond an expert's last
// retained row are zero-filled in shared memory before the MMA reads them;
// experts with no retained row get exact zeros without touching TMEM.
//
// Operand layouts (bf16, 128-byte swizzle, 64-element atoms):
//   dgrad A = delta_c rows      K-major   [BM rows][64 K]        one TMA box
//   dgrad B = W_e [h, I]        MN-major  BN/64 boxes [64 K][64 N]
//   wgrad A = delta_c^T         MN-major  2 boxes [64 K][64 M]
//   wgrad B = phi_c             MN-major  BN/64 boxes [64 K][64 N]
// Every wait is bounded (lrm_set_wait_budget); a wait that runs out raises
// LRM_ERR_TIMEOUT, the block winds down, drains its tensor-core work and
// frees its TMEM before returning.
#include <cuda_bf16.h>

#include "lrm_internal.cuh"

namespace lrm {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int GEMM_THREADS = 192;
constexpr int MAX_E = 1024;
constexpr uint32_t ATOM_BYTES = 64 * 64 * 2;  // one [64][64] bf16 swizzle box

enum Mode { DGRAD = 0, WGRAD = 1 };

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int STAGING_BYTES = 4 * 32 * 128;  // one [32][32] fp32 store box per epilogue warp
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024;
};

struct Tile {
  int e, mt, nt, start, len;
};

template <int MODE, int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut, const int32_t* __restrict__ sel_offsets, int E, int h, int I, int max_rows,
                        int accumulate, void* __restrict__ out, unsigned int* status,
                        unsigned long long budget_ns) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t dsmem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_start[MAX_E];
  __shared__ int s_len[MAX_E];
  __shared__ int s_prefix[MAX_E + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tiles_n = (I + BN - 1) / BN;
  const int tiles_m_w = (h + BM - 1) / BM;  // wgrad: output rows are h

  // ragged segments, clamped to the buffers
  for (int e = tid; e < E; e += GEMM_THREADS) {
    int s = __ldg(sel_offsets + e), t = __ldg(sel_offsets + e + 1);
    s = min(max(s, 0), max_rows);
    t = min(max(t, s), max_rows);
    s_start[e] = s;
    s_len[e] = t - s;
  }
  if (tid == 0) {
    s_abort = 0;
    if (blockIdx.x == 0 && __ldg(sel_offsets + E) > max_rows) raise_flag(status, LRM_ERR_SHAPE);
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 4);
    }
    mbar_init(&drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  // tile prefix over experts (warp 0: 32 experts per lane, then a warp scan)
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int local = 0;
    for (int e = e0; e < min(E, e0 + per); ++e)
      local += (MODE == DGRAD) ? ((s_len[e] + BM - 1) / BM) * tiles_n : tiles_m_w * tiles_n;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - local;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      s_prefix[e] = run;
      run += (MODE == DGRAD) ? ((s_len[e] + BM - 1) / BM) * tiles_n : tiles_m_w * tiles_n;
    }
    if (lane == 31) s_prefix[E] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total_tiles = s_prefix[E];
  volatile int* abort_flag = &s_abort;

  auto decode = [&](int tile) -> Tile {
    int lo = 0, hi = E - 1;  // last e with s_prefix[e] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_prefix[mid] <= tile)
        lo = mid;
      else
        hi = mid - 1;
    }
    Tile t;
    t.e = lo;
    const int rem = tile - s_prefix[lo];
    t.mt = rem / tiles_n;
    t.nt = rem - t.mt * tiles_n;
    t.start = s_start[lo];
    t.len = s_len[lo];
    return t;
  };
  auto kblocks_of = [&](const Tile& t) -> int {
    return (MODE == DGRAD) ? (h + BK - 1) / BK : (t.len + BK - 1) / BK;
  };
  auto fail = [&]() {
    *abort_flag = 1;
    raise_flag(status, LRM_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const Tile t = decode(tile);
        const int nkb = kblocks_of(t);
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
          mbar_arrive_expect_tx(&full_bar[s], C::STAGE_BYTES);
          if (MODE == DGRAD) {
            tma_load_2d(a_dst, &tmA, &full_bar[s], kb * BK, t.start + t.mt * BM);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_3d(b_dst + c * ATOM_BYTES, &tmB, &full_bar[s], t.nt * BN + c * 64, kb * BK, t.e);
          } else {
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              tma_load_2d(a_dst + c * ATOM_BYTES, &tmA, &full_bar[s], t.mt * BM + c * 64, t.start + kb * BK);
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(b_dst + c * ATOM_BYTES, &tmB, &full_bar[s], t.nt * BN + c * 64, t.start + kb * BK);
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the block exits
        for (uint32_t j = (it >= C::STAGES ? it - C::STAGES : 0); j < it; ++j)
          mbar_wait(&full_bar[j % C::STAGES], (j / C::STAGES) & 1u, budget_ns, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, MODE == WGRAD ? 1u : 0u, 1u);
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
      const Tile t = decode(tile);
      const int nkb = kblocks_of(t);
      if (nkb == 0) continue;
      const uint32_t acc = acc_it & 1u;
      const uint32_t aph = (acc_it >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty_bar[acc], aph ^ 1u, budget_ns, abort_flag))) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const uint32_t s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], ph, budget_ns, abort_flag))) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* a_stage = smem + s * C::STAGE_BYTES;
        uint8_t* b_stage = a_stage + C::A_BYTES;
        int nk = BK / 16;
        if (MODE == WGRAD) {
          const int valid = t.len - kb * BK;  // rows of this K block inside the segment
          if (valid < BK) {
            nk = (valid + 15) / 16;
            const int z0 = valid, z1 = nk * 16;  // rows [z0, z1) are zeroed
            const int atoms = BM / 64 + BN / 64;
            const int units = (z1 - z0) * 8 * atoms;  // 16-byte units
            for (int i = lane; i < units; i += 32) {
              const int atom = i / ((z1 - z0) * 8);
              const int rem = i - atom * (z1 - z0) * 8;
              const int row = z0 + rem / 8;
              const int chunk = rem % 8;
              uint8_t* base = (atom < BM / 64) ? a_stage + atom * ATOM_BYTES : b_stage + (atom - BM / 64) * ATOM_BYTES;
              *reinterpret_cast<uint4*>(base + row * 128 + chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (lane == 0) {
          const uint32_t a_addr = smem_u32(a_stage);
          const uint32_t b_addr = smem_u32(b_stage);
          for (int kk = 0; kk < nk; ++kk) {
            uint64_t adesc;
            if (MODE == DGRAD)
              adesc = smem_desc_sw128(a_addr + kk * 32, 16, 1024);  // K-major: 32 B per 16-element K step
            else
              adesc = smem_desc_sw128(a_addr + kk * 2048, ATOM_BYTES, 1024);  // MN-major: 16 K rows
            const uint64_t bdesc = smem_desc_sw128(b_addr + kk * 2048, ATOM_BYTES, 1024);
            mma_bf16_ss(d_tmem, adesc, bdesc, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty_bar[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&tfull_bar[acc]);
      __syncwarp();
      ++acc_it;
    }
    // drain: wait until every MMA issued by this warp has completed
    if (lane == 0) {
      mma_commit(&drain_bar);
      if (!mbar_wait(&drain_bar, 0, budget_ns, nullptr)) raise_flag(status, LRM_ERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    uint8_t* stg = smem + C::STAGES * C::STAGE_BYTES + (warp - 2) * (32 * 128);
    uint32_t acc_it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const Tile t = decode(tile);
      if (MODE == WGRAD && t.len == 0) {
        if (!accumulate) {
          const int i = t.mt * BM + row_in_tile;
          if (i < h) {
            float* orow = static_cast<float*>(out) + (static_cast<size_t>(t.e) * h + i) * I;
            for (int c = 0; c < BN; c += 4) {
              const int col = t.nt * BN + c;
              if (col < I) *reinterpret_cast<float4*>(orow + col) = make_float4(0.f, 0.f, 0.f, 0.f);
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
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c, r);
        tmem_ld_wait();
        const int col0 = t.nt * BN + c;
        if (MODE == DGRAD) {
          const int m = t.mt * BM + row_in_tile;
          if (m < t.len) {
            uint16_t* orow = static_cast<uint16_t*>(out) + static_cast<size_t>(t.start + m) * I;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (col0 + v * 8 < I) {
                uint4 pk;
                uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(r[v * 8 + 2 * j]),
                                                                  __uint_as_float(r[v * 8 + 2 * j + 1]));
                  w[j] = *reinterpret_cast<const uint32_t*>(&b2);
                }
                *reinterpret_cast<uint4*>(orow + col0 + v * 8) = pk;
              }
            }
          }
        } else if (!accumulate) {
          // stage the warp's [32 rows][32 cols] fp32 block with the 128-byte
          // swizzle (16-byte chunk j of row r at chunk j ^ (r % 8)), then one
          // tensor store; rows past h and columns past I are clipped by TMA
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmOut, stg, col0, t.mt * BM + q * 32, t.e);
            bulk_commit_group();
          }
        } else {
          const int i = t.mt * BM + row_in_tile;
          if (i < h) {
            float* orow = static_cast<float*>(out) + (static_cast<size_t>(t.e) * h + i) * I;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const int col = col0 + v * 4;
              if (col < I) {
                const float4 o = *reinterpret_cast<const float4*>(orow + col);
                *reinterpret_cast<float4*>(orow + col) =
                    make_float4(o.x + __uint_as_float(r[4 * v]), o.y + __uint_as_float(r[4 * v + 1]),
                                o.z + __uint_as_float(r[4 * v + 2]), o.w + __uint_as_float(r[4 * v + 3]));
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
      ++acc_it;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// wgrad on CTA pairs: dW_e [h, I] in 256 x BN output tiles, one per cluster of
// two CTAs.  CTA r of a pair loads rows [128r, 128r + 128) of the tile's M
// (= h) range of delta_c^T and columns [r BN/2, (r+1) BN/2) of phi_c into its
// own 6-stage ring (32 KiB per stage); the even CTA issues the M = 256
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
//            prefetched one ahead), TMA tensor stores, then release the
//            accumulator on the even CTA's barrier (16 arrivals)
//   warp 10  tail fixer: waits for the CTA's own tail load, zeroes the rows
//            of its halves that lie past the expert's segment (the MMA reads
//            whole 16-row K steps) and arrives on the even CTA's full barrier
//            (release at cluster scope), off the MMA warp's path

template <int BN>
struct CfgPair {
  static constexpr int A_BYTES = 128 * BK * 2;       // this CTA's 128 rows of M
  static constexpr int B_BYTES = (BN / 2) * BK * 2;  // this CTA's BN/2 columns of N
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 5;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int EPI_WARPS = 8;                       // two per TMEM lane quarter
  static constexpr int THREADS = 64 + 32 * EPI_WARPS + 32;  // + the tail fixer warp
  static constexpr int FIXER_WARP = 2 + EPI_WARPS;
  static constexpr int STAGING_BYTES = EPI_WARPS * 32 * 128;  // one [32][32] fp32 store box per epilogue warp
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024;
};

// Start row and length of expert e's segment, clamped to the buffers.
__device__ __forceinline__ void segment(const int32_t* __restrict__ sel_offsets, int e, int max_rows, int& start,
                                        int& len) {
  int st = __ldg(sel_offsets + e), en = __ldg(sel_offsets + e + 1);
  st = min(max(st, 0), max_rows);
  en = min(max(en, st), max_rows);
  start = st;
  len = en - st;
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(CfgPair<BN>::THREADS, 1)
    wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmOut, const int32_t* __restrict__ sel_offsets, int E,
                      int h, int I, int max_rows, int accumulate, float* __restrict__ out, unsigned int* status,
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

  // Schedule: the pair tiles of all experts, heaviest expert first, dealt to
  // the pairs in a snake order (round r goes forward for even r, backward for
  // odd r), which balances the ragged K loops across pairs.
  for (int e = tid; e < E; e += C::THREADS) {
    int st, ln;
    segment(sel_offsets, e, max_rows, st, ln);
    s_len[e] = ln;
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
      for (int round = 0, tile = tile_of(0); tile < total_tiles && ok; tile = tile_of(++round)) {
        int e, mt, nt;
        decode(tile, e, mt, nt);
        int start, len;
        segment(sel_offsets, e, max_rows, start, len);
        const int nkb = (len + BK - 1) / BK;
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
          const int y = start + kb * BK;
          if (len - kb * BK >= BK) {
            if (leader) {
              // both arrivals of a full block come from here; the odd CTA's
              // loads only add their bytes
              mbar_arrive_expect_tx(&full_bar[s], 2 * C::STAGE_BYTES);
              mbar_arrive(&full_bar[s]);
            }
            const uint32_t bar = full0 + s * 8;
#pragma unroll
            for (int c = 0; c < 2; ++c) tma_load_2d_pair(a_dst + c * ATOM_BYTES, &tmA, bar, xa + c * 64, y);
#pragma unroll
            for (int c = 0; c < BN / 128; ++c) tma_load_2d_pair(b_dst + c * ATOM_BYTES, &tmB, bar, xb + c * 64, y);
          } else {
            mbar_arrive_expect_tx(&tail_bar[s], C::STAGE_BYTES);
#pragma unroll
            for (int c = 0; c < 2; ++c) tma_load_2d(a_dst + c * ATOM_BYTES, &tmA, &tail_bar[s], xa + c * 64, y);
#pragma unroll
            for (int c = 0; c < BN / 128; ++c)
              tma_load_2d(b_dst + c * ATOM_BYTES, &tmB, &tail_bar[s], xb + c * 64, y);
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
    for (int round = 0, tile = tile_of(0); tile < total_tiles && ok; tile = tile_of(++round)) {
      int e, mt, nt;
      decode(tile, e, mt, nt);
      int start, len;
      segment(sel_offsets, e, max_rows, start, len);
      const int nkb = (len + BK - 1) / BK;
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
        const int valid = len - kb * BK;
        const bool tail = valid < BK;
        const int nk = tail ? (valid + 15) / 16 : BK / 16;
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
          const uint32_t b_addr = a_addr + C::A_BYTES;
          for (int kk = 0; kk < nk; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_addr + kk * 2048, ATOM_BYTES, 1024);
            const uint64_t bdesc = smem_desc_sw128(b_addr + kk * 2048, ATOM_BYTES, 1024);
            mma_bf16_ss_pair(d_tmem, adesc, bdesc, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
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
    for (int round = 0, tile = tile_of(0); tile < total_tiles && ok; tile = tile_of(++round)) {
      int e, mt, nt;
      decode(tile, e, mt, nt);
      int start, len;
      segment(sel_offsets, e, max_rows, start, len);
      const int nkb = (len + BK - 1) / BK;
      if (nkb == 0) continue;
      it += nkb - 1;  // full blocks need no fixing
      const int valid = len - (nkb - 1) * BK;
      if (valid < BK) {
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
          uint8_t* base = atom < 2 ? a_stage + atom * ATOM_BYTES : b_stage + (atom - 2) * ATOM_BYTES;
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
    const int row_in_half = q * 32 + lane;
    uint8_t* stg = smem + C::STAGES * C::STAGE_BYTES + (warp - 2) * (32 * 128);
    const uint32_t tempty0 = mapa_shared(&tempty_bar[0], 0);
    uint32_t acc_it = 0;
    for (int round = 0, tile = tile_of(0); tile < total_tiles; tile = tile_of(++round)) {
      int e, mt, nt;
      decode(tile, e, mt, nt);
      const int row0 = mt * 256 + static_cast<int>(rank) * 128;  // first dW row of this CTA's half
      int start, len;
      segment(sel_offsets, e, max_rows, start, len);
      if (len == 0) {
        if (!accumulate) {
          const int i = row0 + row_in_half;
          if (i < h) {
            float* orow = out + (static_cast<size_t>(e) * h + i) * I;
            for (int c = c_begin; c < c_begin + BN / 2; c += 4) {
              const int col = nt * BN + c;
              if (col < I) *reinterpret_cast<float4*>(orow + col) = make_float4(0.f, 0.f, 0.f, 0.f);
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
        const int col0 = nt * BN + c_begin + c;
        if (!accumulate) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmOut, stg, col0, row0 + q * 32, e);
            bulk_commit_group();
          }
        } else {
          const int i = row0 + row_in_half;
          if (i < h) {
            float* orow = out + (static_cast<size_t>(e) * h + i) * I;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const int col = col0 + v * 4;
              if (col < I) {
                const float4 o = *reinterpret_cast<const float4*>(orow + col);
                *reinterpret_cast<float4*>(orow + col) =
                    make_float4(o.x + __uint_as_float(r[4 * v]), o.y + __uint_as_float(r[4 * v + 1]),
                                o.z + __uint_as_float(r[4 * v + 2]), o.w + __uint_as_float(r[4 * v + 3]));
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
    if (lane == 0) bulk_wait_all();
    __syncwarp();
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

// W [E][h][I] bf16 as a 3-D tensor (I, h, E) with [1][64][64] boxes.
lrm_status encode_w(lrm_ctx* ctx, CUtensorMap* map, const void* base, uint64_t I, uint64_t h, uint64_t E) {
  const cuuint64_t dims[3] = {I, h, E};
  const cuuint64_t strides[2] = {I * 2, h * I * 2};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = ctx->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LRM_OK : LRM_ERR_CUDA;
}

// dW [E][h][I] fp32 as a 3-D tensor (I, h, E) with [1][32][32] boxes, 128-byte swizzle.
lrm_status encode_dw(lrm_ctx* ctx, CUtensorMap* map, const void* base, uint64_t I, uint64_t h, uint64_t E) {
  const cuuint64_t dims[3] = {I, h, E};
  const cuuint64_t strides[2] = {I * 4, h * I * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = ctx->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LRM_OK : LRM_ERR_CUDA;
}

template <int MODE, int BN>
lrm_status launch(lrm_ctx* ctx, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                  const int32_t* sel_offsets,
                  const lrm_dims& d, int max_rows, int accumulate, void* out, cudaStream_t s) {
  using C = Cfg<BN>;
  auto kern = grouped_gemm_kernel<MODE, BN>;
  static thread_local int configured_device = -1;
  if (configured_device != ctx->device) {
    if (ctx->smem_optin < C::SMEM_BYTES + 16 * 1024) return LRM_ERR_ARCH;
    LRM_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES));
    configured_device = ctx->device;
  }
  kern<<<ctx->sm_count, GEMM_THREADS, C::SMEM_BYTES, s>>>(a, b, o, sel_offsets, d.E, d.h, d.I, max_rows,
                                                          accumulate, out, ctx->d_status, ctx->wait_budget_ns);
  return launch_status();
}

template <int BN>
lrm_status launch_wgrad_pair(lrm_ctx* ctx, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                             const int32_t* sel_offsets, const lrm_dims& d, int max_rows, int accumulate, float* out,
                             cudaStream_t s) {
  using C = CfgPair<BN>;
  auto kern = wgrad_pair_kernel<BN>;
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
  kern<<<2 * clusters, C::THREADS, C::SMEM_BYTES, s>>>(a, b, o, sel_offsets, d.E, d.h, d.I, max_rows, accumulate,
                                                         out, ctx->d_status, ctx->wait_budget_ns);
  return launch_status();
}

}  // namespace
}  // namespace lrm

using namespace lrm;

namespace {

// The N tile: 256 when the expert width fills it, 128 otherwise.
inline bool use_bn256(int I) { return I >= 256 && (I % 256 == 0 || I % 128 != 0); }

}  // namespace

extern "C" lrm_status lrm_grouped_dgrad(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* W,
                                        const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows,
                                        uint16_t* dphi_c, void* stream) {
  if (ctx == nullptr) return LRM_ERR_INVALID_ARG;
  lrm_status st = check_dims(dims);
  if (st != LRM_OK) return st;
  if (max_rows < 0 || sel_offsets == nullptr) return LRM_ERR_INVALID_ARG;
  if (max_rows == 0) return LRM_OK;
  if (delta_c == nullptr || W == nullptr || dphi_c == nullptr) return LRM_ERR_INVALID_ARG;
  if (!aligned(delta_c, 16) || !aligned(W, 16) || !aligned(dphi_c, 16) || !aligned(sel_offsets, 4))
    return LRM_ERR_ALIGN;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return LRM_ERR_CUDA;
  alignas(64) CUtensorMap ma, mb;
  if ((st = encode_2d(ctx, &ma, delta_c, dims.h, max_rows, BM)) != LRM_OK) return st;
  if ((st = encode_w(ctx, &mb, W, dims.I, dims.h, dims.E)) != LRM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return use_bn256(dims.I) ? launch<DGRAD, 256>(ctx, ma, mb, ma, sel_offsets, dims, max_rows, 0, dphi_c, s)
                           : launch<DGRAD, 128>(ctx, ma, mb, ma, sel_offsets, dims, max_rows, 0, dphi_c, s);
}

extern "C" lrm_status lrm_grouped_wgrad(lrm_ctx* ctx, const uint16_t* delta_c, const uint16_t* phi_c,
                                        const int32_t* sel_offsets, lrm_dims dims, int32_t max_rows,
                                        int32_t accumulate, float* dW, void* stream) {
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
  alignas(64) CUtensorMap ma, mb, mo;
  if ((st = encode_2d(ctx, &ma, a_base, dims.h, rows, 64)) != LRM_OK) return st;
  if ((st = encode_2d(ctx, &mb, b_base, dims.I, rows, 64)) != LRM_OK) return st;
  if ((st = encode_dw(ctx, &mo, dW, dims.I, dims.h, dims.E)) != LRM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launch_wgrad_pair<256>(ctx, ma, mb, mo, sel_offsets, dims, max_rows, accumulate, dW, s);
}
