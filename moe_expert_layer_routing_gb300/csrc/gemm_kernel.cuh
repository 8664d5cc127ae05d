// Persistent, warp-specialised grouped GEMM on the 5th-generation tensor cores (tcgen05).
//
//   C[m, n] = sum_k A[m, k] * B[n, k]        A, B K-major in global memory (bf16 or fp8 + E8M0)
//
// Two grouping modes cover the four GEMMs of the MoE backward and the dense linear backward:
//   M-grouped: A rows are tile rows (128-row tiles, each owned by one expert); B is the weight
//              block of that tile's expert; the contraction length is fixed (G1: dA = dout_g W2_e^T,
//              G2: dx_expanded = dh W1_e, dense dX / dW).
//   K-grouped: every expert e contracts over its own tile-row range [tile_offsets[e],
//              tile_offsets[e+1]) of the transposed operands (G3: dW2_e = a'^T dout_g,
//              G4: dW1_e = x_g^T dh); an expert without rows writes zeros.
//
// CTA = 6 warps: warp 0 issues TMA loads into a STAGES-deep shared-memory ring, warp 1 owns TMEM
// and issues tcgen05.mma (one elected lane), warps 2-5 drain the TMEM accumulator (double
// buffered where TMEM allows) through the epilogue.  One CTA per SM walks a static tile schedule.
// Every wait is bounded (MOE_STATUS_TIMEOUT on expiry, then an orderly drain and exit).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "moebwd_internal.h"
#include "mx_device.cuh"
#include "ptx.cuh"

namespace moebwd {

constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per block on sm_103a

template <bool MX, int BN, int EPI>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int BK_BYTES = 128;              // one 128-byte swizzle row of K per stage
  static constexpr int BKE = MX ? 128 : 64;         // K elements per stage
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = BN * BK_BYTES;
  static constexpr int SFA_BYTES = MX ? 512 : 0;
  static constexpr int SFB_BYTES = MX ? (BN / 128) * 512 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int EPI_WARP_BYTES = (EPI == kEpiDSwiGLU) ? (MX ? 3 * 32 * 32 : 3 * 32 * 40 * 2) : 0;
  static constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int STAGES_FIT = (kSmemLimit - 1024 - BAR_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int ACC_STAGES = (MX && BN == 256) ? 1 : 2;
  static constexpr int SF_COLS = MX ? 4 + 4 * (BN / 128) : 0;   // TMEM columns of scales per stage
  static constexpr int SF_BASE = ACC_STAGES * BN;
  static constexpr int COLS_NEEDED = SF_BASE + STAGES * SF_COLS;
  static constexpr int TMEM_COLS = COLS_NEEDED <= 32 ? 32 : COLS_NEEDED <= 64 ? 64 : COLS_NEEDED <= 128 ? 128
                                 : COLS_NEEDED <= 256 ? 256 : 512;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(STAGES >= 2, "shared memory too small for a 2-stage pipeline");
  static_assert(COLS_NEEDED <= 512, "TMEM overflow");
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory overflow");
};

struct TileInfo {
  int e, mt, nt, a_row, b_row, k0, nk;
};

__device__ __forceinline__ int gemm_total_tiles(const GemmParams& p) {
  if (p.mode == kMGrouped) {
    const int mt = p.num_tiles ? *p.num_tiles : p.m_tiles;
    return mt * p.n_tiles;
  }
  return p.num_experts * p.m_tiles * p.n_tiles;
}

template <int BN, int BKE>
__device__ __forceinline__ TileInfo gemm_decode_tile(const GemmParams& p, int t) {
  TileInfo ti;
  if (p.mode == kMGrouped) {
    ti.mt = t / p.n_tiles;
    ti.nt = t - ti.mt * p.n_tiles;
    ti.e = p.tile_expert ? p.tile_expert[ti.mt] : 0;
    ti.a_row = ti.mt * 128;
    ti.b_row = ti.e * p.b_rows_per_expert + ti.nt * BN;
    ti.k0 = 0;
    ti.nk = p.K / BKE;
  } else {
    const int per = p.m_tiles * p.n_tiles;
    const int ei = t / per;
    const int r = t - ei * per;
    ti.mt = r / p.n_tiles;
    ti.nt = r - ti.mt * p.n_tiles;
    ti.e = p.expert_order ? p.expert_order[ei] : ei;
    ti.a_row = ti.mt * 128;
    ti.b_row = ti.nt * BN;
    ti.k0 = p.tile_offsets[ti.e];
    ti.nk = (p.tile_offsets[ti.e + 1] - ti.k0) / BKE;
  }
  return ti;
}

// Wait without giving up when another role aborted (used to drain copies / MMAs in flight).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int* status) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 255u) == 255u && globaltimer_ns() - t0 > kWaitLimitNs) {
      if (status) atomicOr(status, MOE_STATUS_TIMEOUT);
      return false;
    }
  }
}

// ------------------------------------------------------------------------------------------
// epilogues
// ------------------------------------------------------------------------------------------

// Plain BF16 store of the fp32 accumulator tile (zeros when the contraction was empty).
template <int BN>
__device__ __forceinline__ void epi_store(const GemmParams& p, const TileInfo& ti, uint32_t taddr, int m) {
  uint16_t* out = static_cast<uint16_t*>(p.out);
  const int64_t row = (int64_t)ti.mt * 128 + m;
  uint16_t* dst = out + (p.mode == kMGrouped ? row * p.ldo : (int64_t)ti.e * p.out_expert_stride + row * p.ldo) +
                  (int64_t)ti.nt * BN;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    if (ti.nk > 0) {
      tmem_ld_32x32b_x32(taddr + c * 32, r);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 w;
      w.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]));
      w.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
      w.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
      w.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
      d4[q] = w;
    }
  }
}

// 32 rows (the warp's lanes) x 32 columns (v[]) written transposed: out[(row0 + c) * P + p0 + lane].
__device__ __forceinline__ void store_transposed_bf16(uint16_t* buf, const float (&v)[32], uint16_t* out,
                                                      int64_t P, int64_t row0, int64_t p0, int lane) {
#pragma unroll
  for (int j = 0; j < 32; ++j) buf[j * 40 + lane] = float_to_bf16_bits(v[j]);
  __syncwarp();
  const uint4* src = reinterpret_cast<const uint4*>(buf + lane * 40);
  uint4* dst = reinterpret_cast<uint4*>(out + (row0 + lane) * P + p0);
  const uint4 a = src[0], b = src[1], c = src[2], d = src[3];
  dst[0] = a;
  dst[1] = b;
  dst[2] = c;
  dst[3] = d;
  __syncwarp();
}

// Same, quantised along the 32 rows (groups of 32 tile rows) with one scale per output row.
__device__ __forceinline__ void store_transposed_mx(uint8_t* buf, const float (&v)[32], uint8_t* out, uint8_t* sf,
                                                    int64_t P, int64_t row0, int64_t p0, int lane, int fmt) {
  uint32_t mybyte = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t am = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[j])));
    const uint32_t byte = e8m0_byte(am, fmt);
    buf[j * 32 + lane] = (uint8_t)fp8_code(v[j] * e8m0_inv_scale(byte), fmt);
    if (lane == j) mybyte = byte;
  }
  __syncwarp();
  const uint4* src = reinterpret_cast<const uint4*>(buf + lane * 32);
  uint4* dst = reinterpret_cast<uint4*>(out + (row0 + lane) * P + p0);
  const uint4 a = src[0], b = src[1];
  dst[0] = a;
  dst[1] = b;
  sf[sf_tiled_offset(row0 + lane, p0, P)] = (uint8_t)mybyte;
  __syncwarp();
}

// G1 epilogue: from dA_raw (accumulator) and the checkpointed gate/up pre-activations compute
//   ds += <dA_raw, a>,  dA = s dA_raw,  dgate = dA up SiLU'(gate),  dup = dA SiLU(gate),  a' = s a
// and write dh [P,2I] (row-major), dh^T [2I,P], a'^T [I,P] (bf16, or fp8 + scales), plus this
// tile's partial ds.  Padding rows produce zeros.
template <bool MX, int BN>
__device__ __forceinline__ void epi_dswiglu(const GemmParams& p, const TileInfo& ti, uint32_t taddr, int m,
                                            int lane, uint8_t* wsm) {
  const int64_t prow = (int64_t)ti.mt * 128 + m;
  const int f = p.tile_row_flat[prow];
  const bool valid = f >= 0;
  const float sv = valid ? p.s[f] : 0.f;
  const int64_t j = prow - p.e_tile_offsets[ti.e];
  const int64_t slot = (int64_t)p.block_offsets[ti.e] * p.B + j;
  const int64_t blk = slot / p.B, b = slot - (slot / p.B) * p.B;
  const uint16_t* gb = p.ckpt + (blk * 2 + 0) * (int64_t)p.I * p.B + b;
  const uint16_t* ub = p.ckpt + (blk * 2 + 1) * (int64_t)p.I * p.B + b;
  const int I = p.I;
  const int64_t P = p.P;
  const int64_t p0 = (int64_t)ti.mt * 128 + (m & ~31);
  float ds_acc = 0.f;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int i0 = ti.nt * BN + c * 32;
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + c * 32, r);
    tmem_ld_wait();
    float dg[32], du[32], ap[32];
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      float v = __uint_as_float(r[jj]);
      float g = 0.f, u = 0.f;
      if (valid) {
        g = bf16_bits_to_float(gb[(int64_t)(i0 + jj) * p.B]);
        u = bf16_bits_to_float(ub[(int64_t)(i0 + jj) * p.B]);
      } else {
        v = 0.f;
      }
      const float sg = 1.f / (1.f + __expf(-g));
      const float sl = g * sg;
      const float a = sl * u;
      ds_acc = fmaf(v, a, ds_acc);
      const float dA = sv * v;
      dg[jj] = dA * u * (sg * (1.f + g * (1.f - sg)));
      du[jj] = dA * sl;
      ap[jj] = p.affinity_on_i ? sv * a : a;
    }
    if constexpr (MX) {
      uint8_t* dh = static_cast<uint8_t*>(p.dh) + prow * (2 * (int64_t)I);
      uint32_t w[8];
      uint32_t byte = quantize_group32(dg, p.fmt_act, w);
      reinterpret_cast<uint4*>(dh + i0)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(dh + i0)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      p.dh_sf[sf_tiled_offset(prow, i0, 2 * (int64_t)I)] = (uint8_t)byte;
      byte = quantize_group32(du, p.fmt_act, w);
      reinterpret_cast<uint4*>(dh + I + i0)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(dh + I + i0)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      p.dh_sf[sf_tiled_offset(prow, I + i0, 2 * (int64_t)I)] = (uint8_t)byte;
      store_transposed_mx(wsm, dg, static_cast<uint8_t*>(p.dht), p.dht_sf, P, i0, p0, lane, p.fmt_act);
      store_transposed_mx(wsm + 1024, du, static_cast<uint8_t*>(p.dht), p.dht_sf, P, I + i0, p0, lane, p.fmt_act);
      store_transposed_mx(wsm + 2048, ap, static_cast<uint8_t*>(p.apt), p.apt_sf, P, i0, p0, lane, p.fmt_act);
    } else {
      uint16_t* dh = static_cast<uint16_t*>(p.dh) + prow * (2 * (int64_t)I);
      uint4* dgp = reinterpret_cast<uint4*>(dh + i0);
      uint4* dup = reinterpret_cast<uint4*>(dh + I + i0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dgp[q] = make_uint4(pack_bf16x2(dg[8 * q + 0], dg[8 * q + 1]), pack_bf16x2(dg[8 * q + 2], dg[8 * q + 3]),
                            pack_bf16x2(dg[8 * q + 4], dg[8 * q + 5]), pack_bf16x2(dg[8 * q + 6], dg[8 * q + 7]));
        dup[q] = make_uint4(pack_bf16x2(du[8 * q + 0], du[8 * q + 1]), pack_bf16x2(du[8 * q + 2], du[8 * q + 3]),
                            pack_bf16x2(du[8 * q + 4], du[8 * q + 5]), pack_bf16x2(du[8 * q + 6], du[8 * q + 7]));
      }
      uint16_t* buf = reinterpret_cast<uint16_t*>(wsm);
      store_transposed_bf16(buf, dg, static_cast<uint16_t*>(p.dht), P, i0, p0, lane);
      store_transposed_bf16(buf + 32 * 40, du, static_cast<uint16_t*>(p.dht), P, I + i0, p0, lane);
      store_transposed_bf16(buf + 2 * 32 * 40, ap, static_cast<uint16_t*>(p.apt), P, i0, p0, lane);
    }
  }
  p.ds_part[prow * (int64_t)(I / BN) + ti.nt] = valid ? ds_acc : 0.f;
}

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------
template <bool MX, int BN, int EPI>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ GemmParams p) {
  using C = GemmCfg<MX, BN, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smA + C::STAGES * C::A_BYTES;
  uint8_t* smSFA = smB + C::STAGES * C::B_BYTES;
  uint8_t* smSFB = smSFA + C::STAGES * C::SFA_BYTES;
  uint8_t* smEPI = smSFB + C::STAGES * C::SFB_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smEPI + C::EPI_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = gemm_total_tiles(p);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TileInfo ti = gemm_decode_tile<BN, C::BKE>(p, t);
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          const int kc = ti.k0 + kb * C::BKE;
          tma_load_2d(smA + s * C::A_BYTES, &tmA, &full[s], kc, ti.a_row);
          tma_load_2d(smB + s * C::B_BYTES, &tmB, &full[s], kc, ti.b_row);
          if constexpr (MX) {
            const int kt = kc / 128;
            bulk_load(smSFA + s * C::SFA_BYTES, p.sfa + ((int64_t)(ti.a_row / 128) * p.sfa_ktiles + kt) * 512, 512,
                      &full[s]);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              bulk_load(smSFB + s * C::SFB_BYTES + h * 512,
                        p.sfb + ((int64_t)(ti.b_row / 128 + h) * p.sfb_ktiles + kt) * 512, 512, &full[s]);
          }
          ++issued;
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Drain: every copy issued must have landed before the CTA may exit.
      const int64_t n = issued < C::STAGES ? issued : C::STAGES;
      for (int64_t i = 1; i <= n; ++i) {
        const int64_t q = issued - i;
        mbar_wait_drain(&full[q % C::STAGES], (uint32_t)((q / C::STAGES) & 1), p.status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileInfo ti = gemm_decode_tile<BN, C::BKE>(p, t);
        if (!mbar_wait_bounded(&tempty[acc], aph ^ 1u, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait_bounded(&full[s], ph, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smA + s * C::A_BYTES);
          const uint32_t b0 = smem_u32(smB + s * C::B_BYTES);
          if constexpr (MX) {
            const uint32_t sfa_t = tmem_base + (uint32_t)(C::SF_BASE + s * C::SF_COLS);
            const uint32_t sfb_t = sfa_t + 4;
            tmem_cp_32x128b_warpx4(sfa_t, make_smem_desc(smem_u32(smSFA + s * C::SFA_BYTES), 0, 128, kSwizzleNone));
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tmem_cp_32x128b_warpx4(sfb_t + 4 * h, make_smem_desc(smem_u32(smSFB + s * C::SFB_BYTES + h * 512), 0,
                                                                   128, kSwizzleNone));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = kmajor_sw128_desc(a0 + kk * 32);
#pragma unroll
              for (int h = 0; h < BN / 128; ++h) {
                const uint64_t bdesc = kmajor_sw128_desc(b0 + h * 128 * 128 + kk * 32);
                mma_mxf8(d + h * 128, adesc, bdesc,
                         idesc_mxf8(128, 128, (uint32_t)p.fmt_a, (uint32_t)p.fmt_b, (uint32_t)kk, (uint32_t)kk),
                         sfa_t, sfb_t + 4 * h, (kb | kk) != 0);
              }
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(d, kmajor_sw128_desc(a0 + kk * 32), kmajor_sw128_desc(b0 + kk * 32), idesc_bf16(128, BN),
                       (kb | kk) != 0);
          }
          mma_commit(&empty[s]);
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (ti.nk > 0)
          mma_commit(&tfull[acc]);
        else
          mbar_arrive(&tfull[acc]);
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          aph ^= 1u;
        }
      }
      // Drain: all tensor-core work of this CTA completes before TMEM is released.
      mma_commit(done);
      mbar_wait_drain(done, 0, p.status);
    }
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int m = 32 * q + lane;
    uint8_t* wsm = smEPI + (warp - 2) * C::EPI_WARP_BYTES;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = gemm_decode_tile<BN, C::BKE>(p, t);
      if (!mbar_wait_bounded(&tfull[acc], aph, p.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      if constexpr (EPI == kEpiStore) {
        epi_store<BN>(p, ti, taddr, m);
      } else {
        epi_dswiglu<MX, BN>(p, ti, taddr, m, lane, wsm);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == C::ACC_STAGES) {
        acc = 0;
        aph ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <bool MX, int BN, int EPI>
int gemm_launch_instance(const GemmParams& p, const void* tmA, const void* tmB, int grid, cudaStream_t st) {
  using C = GemmCfg<MX, BN, EPI>;
  auto kern = gemm_kernel<MX, BN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(gemm)");
  kern<<<grid, 192, C::SMEM_BYTES, st>>>(*static_cast<const CUtensorMap*>(tmA),
                                        *static_cast<const CUtensorMap*>(tmB), p);
  count_launch();
  return cuda_check(cudaGetLastError(), "gemm launch");
}

}  // namespace moebwd
