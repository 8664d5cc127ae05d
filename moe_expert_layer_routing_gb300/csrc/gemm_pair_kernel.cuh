// Grouped GEMM over CTA pairs (clusters of two): the 5th-generation tensor cores' cta_group::2 MMA
// computes a 256 x 256 tile per pair, each CTA holding 128 rows of A, 128 of the 256 rows of B and
// its own 128 x 256 fp32 accumulator in TMEM.  Per k-block a CTA loads 32 KB of operands instead of
// the 48 KB a 128 x 256 single-CTA tile needs, which cuts the L2 -> SM traffic per FLOP by a third.
//
//   C[m, n] = sum_k A[m, k] * B[n, k]        A, B K-major in global memory (bf16 or fp8 + E8M0)
//
// Work decomposition (a "pair tile" is 256 rows x 256 columns of the output):
//   M-grouped: expert e's 128-row tiles are paired in order (2j, 2j+1); an odd last tile is paired
//              with an idle partner whose A rows are read out of range (zero fill) and not stored.
//              pair_offsets[e] is the prefix of ceil(tiles_e / 2) (null: one expert).
//   K-grouped: 256-row blocks of M (M % 256 == 0) for every expert, contraction over the expert's
//              tile rows, as in the single-CTA kernel.
//
// Roles (same warp layout in both CTAs):
//   warp 0 lane 0   TMA producer.  The leader (cluster rank 0) claims pair tiles from a global counter
//                   and publishes each index to both CTAs' rings; each CTA loads its own halves with
//                   TMA whose completion is counted on the leader's stage barrier.
//   warp 1          TMEM allocation of the pair (both CTAs); on the leader, lane 0 issues the pair
//                   MMAs (and the scale copies of both CTAs) and commits to both CTAs' barriers.
//   warps 2-9       epilogue: drain this CTA's accumulator, release it to the leader, store.
// Every wait is bounded; a timeout raises MOE_STATUS_TIMEOUT and the abort flags of both CTAs.
#pragma once
#include "gemm_kernel.cuh"

namespace moebwd {

template <bool MX, int BN_, int EPI>
struct PairCfg {
  static constexpr int BM = 128;                   // rows per CTA
  static constexpr int BN = BN_;                   // columns of the pair tile (128 or 256)
  static constexpr int BK_BYTES = 128;
  static constexpr int BKE = MX ? 128 : 64;
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = (BN / 2) * BK_BYTES;
  static constexpr int SFA_BYTES = MX ? 512 : 0;
  static constexpr int SFB_BYTES = MX ? (BN / 128) * 512 : 0;  // scales of all BN rows of B in every CTA
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGING_BYTES = BM * 64 * 2;
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int BAR_BYTES = 512;
  static constexpr int RING = 4;
  static constexpr int STAGES_FIT = (kSmemLimit - 1024 - BAR_BYTES - STAGING_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int ACC_STAGES = (MX && BN == 256) ? 1 : 2;
  static constexpr int SF_COLS = MX ? 4 + 4 * (BN / 128) : 0;
  static constexpr int SF_BASE = ACC_STAGES * BN;
  static constexpr int COLS_NEEDED = SF_BASE + STAGES * SF_COLS;
  static constexpr int TMEM_COLS = 512;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + BAR_BYTES;
  static_assert(STAGES >= 3, "shared memory too small");
  static_assert(COLS_NEEDED <= TMEM_COLS, "TMEM overflow");
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory overflow");
  static_assert(EPI == kEpiStore || EPI == kEpiCkpt, "pair kernel epilogues: store, checkpoint");
  static_assert(BN == 128 || BN == 256, "pair tile width");
};

struct PairTile {
  int e, nt, mt, valid, a_row, b_base, k0, nk;
  int64_t out_row;
};

__device__ __forceinline__ int pair_total_tiles(const GemmParams& p) {
  if (p.mode == kMGrouped) {
    const int np = p.pair_offsets ? *p.num_pairs : (p.m_tiles + 1) / 2;
    return np * p.n_tiles;
  }
  return p.num_experts * (p.m_tiles / 2) * p.n_tiles;
}

// Tile t of the pair schedule as seen by CTA `rank` of the pair.
template <int BN, int BKE>
__device__ __forceinline__ PairTile pair_decode(const GemmParams& p, int t, int rank) {
  PairTile ti;
  if (p.mode == kMGrouped) {
    const int pi = t / p.n_tiles;
    ti.nt = t - pi * p.n_tiles;
    int first, end;
    ti.e = 0;
    if (p.pair_offsets) {  // largest e with pair_offsets[e] <= pi
      int lo = 0, hi = p.num_experts;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.pair_offsets[mid] <= pi) lo = mid; else hi = mid;
      }
      ti.e = lo;
      first = p.e_tile_offsets[lo] / kTileM + 2 * (pi - p.pair_offsets[lo]);
      end = p.e_tile_offsets[lo + 1] / kTileM;
    } else {
      first = 2 * pi;
      end = p.m_tiles;
    }
    ti.mt = first + rank;
    ti.valid = ti.mt < end;
    ti.a_row = ti.valid ? ti.mt * kTileM : p.m_tiles * kTileM;  // idle partner: rows past the end
    ti.b_base = ti.e * p.b_rows_per_expert + ti.nt * BN;
    ti.k0 = 0;
    ti.nk = p.K / BKE;
    ti.out_row = (int64_t)ti.mt * kTileM;
  } else {
    const int mp = p.m_tiles / 2;
    const int per = mp * p.n_tiles;
    const int ei = t / per;
    const int r = t - ei * per;
    const int mb = r / p.n_tiles;
    ti.nt = r - mb * p.n_tiles;
    ti.e = p.expert_order ? p.expert_order[ei] : ei;
    ti.mt = mb * 2 + rank;
    ti.valid = 1;
    ti.a_row = ti.mt * kTileM;
    ti.b_base = ti.nt * BN;
    ti.k0 = p.tile_offsets[ti.e];
    ti.nk = (p.tile_offsets[ti.e + 1] - ti.k0) / BKE;
    ti.out_row = (int64_t)ti.e * p.M + ti.a_row;
  }
  return ti;
}

// Bounded wait on a local mbarrier (arrivals may come from the peer).  CLUSTER_ACQUIRE: for data the
// peer wrote with generic stores (the tile ring); the stage and accumulator barriers guard data moved
// by TMA / tcgen05 and take the CTA-scope form.  On timeout the status word gets MOE_STATUS_TIMEOUT
// and both CTAs' abort flags are raised.
template <bool CLUSTER_ACQUIRE = false>
__device__ __forceinline__ bool pair_wait(uint64_t* bar, uint32_t parity, int* status, volatile int* abort_flag,
                                          uint32_t peer_abort, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  auto poll = [&]() { return CLUSTER_ACQUIRE ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity); };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (poll()) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        if (status) atomicOr(status, MOE_STATUS_TIMEOUT);
        *abort_flag = 1;
        st_shared_cluster_u32(peer_abort, 1u);
        return false;
      }
    }
  }
}

template <bool MX, int BN, int EPI>
__global__ void __launch_bounds__(PairCfg<MX, BN, EPI>::THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmSFA,
                     const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ GemmParams p) {
  using C = PairCfg<MX, BN, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smA + C::STAGES * C::A_BYTES;
  uint8_t* smStage = smB + C::STAGES * C::B_BYTES;
  uint8_t* smSFA = smStage + C::STAGING_BYTES;
  uint8_t* smSFB = smSFA + C::STAGES * C::SFA_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smSFB + C::STAGES * C::SFB_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint64_t* tile_full = done + 1;
  uint64_t* tile_empty = tile_full + C::RING;
  volatile int* tile_ring = reinterpret_cast<volatile int*>(tile_empty + C::RING);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tile_ring) + C::RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t peer = rank ^ 1u;
  const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int*>(abort_flag)), peer);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * C::EPI_WARPS);
    }
    mbar_init(done, 1);
    for (int r = 0; r < C::RING; ++r) {
      mbar_init(&tile_full[r], 1);
      mbar_init(&tile_empty[r], 2 + 2 * C::EPI_WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    if (MX) {
      prefetch_tmap(&tmSFA);
      prefetch_tmap(&tmSFB);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the prologue above (barriers, TMEM, tensor-map prefetch) overlaps the previous kernel's tail;
  // nothing written by earlier work is read before this point
  pdl_wait();
  pdl_trigger();
  const int total = pair_total_tiles(p);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      const uint32_t lead_full = mapa_shared(smem_u32(full), 0);
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      int rs = 0;
      uint32_t rph = 0;
      for (;;) {
        int t;
        if (leader) {
          t = atomicAdd(p.tile_counter, 1);
          if (t >= total) t = -1;
          if (!pair_wait(&tile_empty[rs], rph ^ 1u, p.status, abort_flag, peer_abort, p.wait_ns)) break;
          tile_ring[rs] = t;
          st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(&tile_ring[rs])), peer), (uint32_t)t);
          mbar_arrive(&tile_full[rs]);
          mbar_arrive_cluster(mapa_shared(smem_u32(&tile_full[rs]), peer));
        } else {
          if (!pair_wait<true>(&tile_full[rs], rph, p.status, abort_flag, peer_abort, p.wait_ns)) break;
          t = tile_ring[rs];
          mbar_arrive_cluster(mapa_shared(smem_u32(&tile_empty[rs]), 0));
        }
        if (++rs == C::RING) {
          rs = 0;
          rph ^= 1u;
        }
        if (t < 0) break;
        const PairTile ti = pair_decode<BN, C::BKE>(p, t, (int)rank);
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!pair_wait(&empty[s], ph ^ 1u, p.status, abort_flag, peer_abort, p.wait_ns)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
          const uint32_t fb = lead_full + (uint32_t)(s * 8);
          const int kc = ti.k0 + kb * C::BKE;
          if (!MX && p.a_mn) {  // [K, M] operand: 64 x 64 boxes, 8 KB apart along M
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_2d_pair(smA + s * C::A_BYTES + j * 8192, &tmA, fb, ti.a_row + 64 * j, kc);
          } else {
            tma_load_2d_pair(smA + s * C::A_BYTES, &tmA, fb, kc, ti.a_row);
          }
          if (!MX && p.b_mn) {  // this CTA's BN / 2 columns of the [K, N] operand
#pragma unroll
            for (int j = 0; j < BN / 128; ++j)
              tma_load_2d_pair(smB + s * C::B_BYTES + j * 8192, &tmB, fb, ti.b_base + (BN / 2) * (int)rank + 64 * j,
                               kc);
          } else {
            tma_load_2d_pair(smB + s * C::B_BYTES, &tmB, fb, kc, ti.b_base + (BN / 2) * (int)rank);
          }
          if constexpr (MX) {
            const int kt = kc / 128;
            tma_load_2d_pair(smSFA + s * C::SFA_BYTES, &tmSFA, fb, 0, (ti.a_row / 128) * p.sfa_ktiles + kt);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tma_load_2d_pair(smSFB + s * C::SFB_BYTES + h * 512, &tmSFB, fb, 0,
                               (ti.b_base / 128 + h) * p.sfb_ktiles + kt);
          }
          ++issued;
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Drain: the leader's stage barriers count both CTAs' copies; every copy issued must land
      // before either CTA exits (the final cluster barrier holds the partner until then).
      if (leader) {
        const int64_t n = issued < C::STAGES ? issued : C::STAGES;
        for (int64_t i = 1; i <= n; ++i) {
          const int64_t q = issued - i;
          mbar_wait_drain(&full[q % C::STAGES], (uint32_t)((q / C::STAGES) & 1), p.status);
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ---------------- pair MMA issuer (leader) ----------------
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      int rs = 0;
      uint32_t rph = 0;
      while (ok) {
        if (!pair_wait<true>(&tile_full[rs], rph, p.status, abort_flag, peer_abort, p.wait_ns)) break;
        const int t = tile_ring[rs];
        mbar_arrive(&tile_empty[rs]);
        if (++rs == C::RING) {
          rs = 0;
          rph ^= 1u;
        }
        if (t < 0) break;
        const PairTile ti = pair_decode<BN, C::BKE>(p, t, 0);
        if (!pair_wait(&tempty[acc], aph ^ 1u, p.status, abort_flag, peer_abort, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * C::BN);
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!pair_wait(&full[s], ph, p.status, abort_flag, peer_abort, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smA + s * C::A_BYTES);
          const uint32_t b0 = smem_u32(smB + s * C::B_BYTES);
          if constexpr (MX) {
            const uint32_t sfa_t = tmem_base + (uint32_t)(C::SF_BASE + s * C::SF_COLS);
            const uint32_t sfb_t = sfa_t + 4;
            tmem_cp_pair_32x128b_warpx4(sfa_t, make_smem_desc(smem_u32(smSFA + s * C::SFA_BYTES), 0, 128, kSwizzleNone));
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tmem_cp_pair_32x128b_warpx4(sfb_t + 4 * h, make_smem_desc(smem_u32(smSFB + s * C::SFB_BYTES + h * 512), 0,
                                                                        128, kSwizzleNone));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_mxf8_pair(d, kmajor_sw128_desc(a0 + kk * 32), kmajor_sw128_desc(b0 + kk * 32),
                            idesc_mxf8(256, C::BN, (uint32_t)p.fmt_a, (uint32_t)p.fmt_b, (uint32_t)kk, (uint32_t)kk),
                            sfa_t, sfb_t, (kb | kk) != 0);
          } else {
            // K step kk: 32 bytes into each 128-byte K-major row, or two 8-row atoms of an MN-major tile
            const uint32_t idesc = idesc_bf16(256, C::BN, (uint32_t)p.a_mn, (uint32_t)p.b_mn);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_pair(d, p.a_mn ? mnmajor_sw128_desc(a0 + kk * 2048, 8192) : kmajor_sw128_desc(a0 + kk * 32),
                            p.b_mn ? mnmajor_sw128_desc(b0 + kk * 2048, 8192) : kmajor_sw128_desc(b0 + kk * 32), idesc,
                            (kb | kk) != 0);
          }
          mma_commit_pair(mapa_shared(smem_u32(&empty[s]), 0));
          mma_commit_pair(mapa_shared(smem_u32(&empty[s]), 1));
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (ti.nk > 0) {
          mma_commit_pair(mapa_shared(smem_u32(&tfull[acc]), 0));
          mma_commit_pair(mapa_shared(smem_u32(&tfull[acc]), 1));
        } else {
          mbar_arrive(&tfull[acc]);
          mbar_arrive_cluster(mapa_shared(smem_u32(&tfull[acc]), 1));
        }
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          aph ^= 1u;
        }
      }
      mma_commit_pair(mapa_shared(smem_u32(done), 0));
      mbar_wait_drain(done, 0, p.status);
    }
  } else {
    // ---------------- epilogue warps 2..9 (both CTAs) ----------------
    const int q = warp & 3;
    const int m = 32 * q + lane;
    const int half = (warp - 2) >> 2;
    const uint32_t lead_tempty = mapa_shared(smem_u32(tempty), 0);
    const uint32_t lead_tile_empty = mapa_shared(smem_u32(tile_empty), 0);
    int acc = 0;
    uint32_t aph = 0;
    int rs = 0;
    uint32_t rph = 0;
    for (;;) {
      const bool gt = pair_wait<true>(&tile_full[rs], rph, p.status, abort_flag, peer_abort, p.wait_ns);
      const int t = gt ? tile_ring[rs] : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead_tile_empty + (uint32_t)(rs * 8));
      if (++rs == C::RING) {
        rs = 0;
        rph ^= 1u;
      }
      // exit decisions are taken together: the OR of the abort flag over the epilogue warps at a barrier
      if (epilogue_bar_any<32 * C::EPI_WARPS>(*abort_flag != 0)) break;
      if (t < 0) break;
      const PairTile ti = pair_decode<BN, C::BKE>(p, t, (int)rank);
      pair_wait(&tfull[acc], aph, p.status, abort_flag, peer_abort, p.wait_ns);
      if (epilogue_bar_any<32 * C::EPI_WARPS>(*abort_flag != 0)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * C::BN);
      // this CTA's 128 x 256 accumulator -> registers (bf16), then release it to the leader
      uint32_t pk[C::BN / 64][16];
#pragma unroll
      for (int sl = 0; sl < C::BN / 64; ++sl) {
        uint32_t r[32];
        if (ti.nk > 0) {
          tmem_ld_32x32b_x32(taddr + (sl * 2 + half) * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        if constexpr (EPI == kEpiCkpt) {
          if (p.b1) {  // h = acc + b1_e for the 32 gate|up features of this chunk
            const int n0 = ti.nt * C::BN + (sl * 2 + half) * 32;
            const uint4* bp = reinterpret_cast<const uint4*>(p.b1 + (int64_t)ti.e * 2 * p.I + n0);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint4 bv = __ldg(bp + q4);
              const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                r[8 * q4 + 2 * j] = __float_as_uint(__uint_as_float(r[8 * q4 + 2 * j]) + __uint_as_float(bw[j] << 16));
                r[8 * q4 + 2 * j + 1] =
                    __float_as_uint(__uint_as_float(r[8 * q4 + 2 * j + 1]) + __uint_as_float(bw[j] & 0xFFFF0000u));
              }
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[sl][j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_remote(lead_tempty + (uint32_t)(acc * 8));
      }
      if (++acc == C::ACC_STAGES) {
        acc = 0;
        aph ^= 1u;
      }
      if constexpr (EPI == kEpiStore) {
        // 64-column slabs through the 128B-swizzled staging tile, TMA-stored (or reduce-added)
#pragma unroll
        for (int sl = 0; sl < C::BN / 64; ++sl) {
          if (warp == 2 && lane == 0) bulk_wait_read_all();
          epilogue_bar<32 * C::EPI_WARPS>();
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = half * 4 + q4;
            *reinterpret_cast<uint4*>(smStage + m * 128 + ((chunk ^ (m & 7)) << 4)) =
                make_uint4(pk[sl][4 * q4 + 0], pk[sl][4 * q4 + 1], pk[sl][4 * q4 + 2], pk[sl][4 * q4 + 3]);
          }
          fence_proxy_async_smem();
          epilogue_bar<32 * C::EPI_WARPS>();
          if (warp == 2 && lane == 0 && ti.valid) {
            if (p.accumulate)
              tma_reduce_add_2d(&tmC, smStage, ti.nt * C::BN + sl * 64, (int)ti.out_row);
            else
              tma_store_2d(&tmC, smStage, ti.nt * C::BN + sl * 64, (int)ti.out_row);
            bulk_commit();
          }
        }
      } else {
        // gate|up chunks of 32 features x 128 rows into the block checkpoint [N*2*I, B]
        int64_t blk = 0;
        int b0 = 0;
        if (ti.valid) {
          TileInfo t1;
          t1.e = ti.e;
          t1.mt = ti.mt;
          tile_ckpt_origin(p, t1, blk, b0);
        }
        uint16_t* stg = reinterpret_cast<uint16_t*>(smStage) + half * (32 * 128);
#pragma unroll
        for (int cp = 0; cp < C::BN / 64; ++cp) {
          if (warp == 2 && lane == 0) bulk_wait_read_all();
          epilogue_bar<32 * C::EPI_WARPS>();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            stg[(2 * j) * 128 + m] = (uint16_t)(pk[cp][j] & 0xFFFFu);
            stg[(2 * j + 1) * 128 + m] = (uint16_t)(pk[cp][j] >> 16);
          }
          fence_proxy_async_smem();
          epilogue_bar<32 * C::EPI_WARPS>();
          if (warp == 2 && lane == 0 && ti.valid) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int n = ti.nt * C::BN + (cp * 2 + hh) * 32;
              const int g = n >= p.I ? 1 : 0;
              tma_store_2d(&tmC, smStage + hh * (32 * 128 * 2), b0, (int)((blk * 2 + g) * p.I + (n - g * p.I)));
            }
            bulk_commit();
          }
        }
      }
    }
    if (warp == 2 && lane == 0) bulk_wait_all();  // stores complete before exit
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves (or frees TMEM) while its partner may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <bool MX, int BN, int EPI>
int gemm_pair_launch_instance(const GemmParams& p, const void* tmA, const void* tmB, const void* tmC,
                              const void* tmSFA, const void* tmSFB, int max_pairs, cudaStream_t st) {
  using C = PairCfg<MX, BN, EPI>;
  auto kern = gemm_pair_kernel<MX, BN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(gemm pair)");
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2, 1, 1);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (e != cudaSuccess) return cuda_check(e, "cudaOccupancyMaxActiveClusters");
  if (clusters <= 0) return fail(MOE_ERR_CUDA, "gemm pair kernel: no cluster of two fits on this device");
  const int pairs = max_pairs < clusters ? max_pairs : clusters;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.numAttrs = option(MOE_OPT_PDL) ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, *static_cast<const CUtensorMap*>(tmA), *static_cast<const CUtensorMap*>(tmB),
                         *static_cast<const CUtensorMap*>(tmC), *static_cast<const CUtensorMap*>(tmSFA),
                         *static_cast<const CUtensorMap*>(tmSFB), p);
  count_launch();
  if (e != cudaSuccess) return cuda_check(e, "gemm pair launch");
  return cuda_check(cudaGetLastError(), "gemm pair launch");
}

}  // namespace moebwd
