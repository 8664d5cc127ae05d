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
// One persistent CTA per SM.  Warp 0 (one lane) claims tiles from a global counter, publishes them
// through a small ring and issues the TMA loads into a STAGES-deep shared-memory ring; warp 1 owns
// TMEM and issues tcgen05.mma (one lane); the epilogue warps drain the TMEM accumulator (double
// buffered where TMEM allows): 4 for the plain store, 8 for the staged store / checkpoint epilogues
// and for the dSwiGLU epilogue, which also has a checkpoint-loader warp.  Every wait is bounded
// (MOE_STATUS_TIMEOUT on expiry, then an orderly drain and exit).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "moebwd_internal.h"
#include "mx_device.cuh"
#include "ptx.cuh"

namespace moebwd {

constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per block on sm_103a
constexpr int kTransPitch = 36;   // fp32 row pitch of the epilogue transpose buffers (16-byte rows, no bank conflicts)

template <bool MX, int BN, int EPI>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int BK_BYTES = 128;              // one 128-byte swizzle row of K per stage
  static constexpr int BKE = MX ? 128 : 64;         // K elements per stage
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = BN * BK_BYTES;
  static constexpr int SFA_BYTES = MX ? 512 : 0;
  // scales of B: one 512-byte atom per 128 rows; a 192-column tile takes two atoms (the second half
  // padding), so its scales come re-tiled per tile (see sf_retile_tiles)
  static constexpr int SFB_ATOMS = (BN + 127) / 128;
  static constexpr int SFB_BYTES = MX ? SFB_ATOMS * 512 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // dSwiGLU epilogue: 4 * kG1Subs warps (kG1Subs per TMEM lane quarter, each taking NC = 32 / kG1Subs
  // of every 32 columns), three NC x 32 fp32 transposition buffers per warp, the row-wise amax
  // exchange of each quarter (double-buffered by chunk parity) and a double-buffered checkpoint chunk
  // (gate and up, 32 features x 128 tile rows each) refilled by the loader warp's TMA copies.
  static constexpr int G1_NC = 32 / kG1Subs;
  // dSwiGLU epilogues; kEpiDSwiGLU2 runs two groups of 4 * kG1Subs warps, group g taking the chunks
  // c = g, g + 2, ... of every tile, with three checkpoint buffers (each group one chunk ahead)
  static constexpr bool DSW = EPI == kEpiDSwiGLU || EPI == kEpiDSwiGLU2;
  static constexpr int G1_GROUPS = EPI == kEpiDSwiGLU2 ? 2 : 1;
  static constexpr int CK_BUFS = G1_GROUPS == 2 ? 3 : 2;
  // fp32 transpose buffers per warp: MXFP8, and BF16 at 256 columns, share one between the three
  // transposes (the shared memory saved buys a pipeline stage); BF16 at 128 columns has stages enough
  // and keeps three, which overlap
  static constexpr int G1_TBUFS = (MX || BN == 256) ? 1 : 3;
  static constexpr int EPI_WARP_BYTES = DSW ? G1_TBUFS * G1_NC * kTransPitch * 4 : 0;
  static constexpr int XCHG_QUARTER = kG1Subs * 2 * 32;  // floats: [slice][gate|up][lane]
  static constexpr int XCHG_BYTES = DSW ? G1_GROUPS * 2 * 4 * XCHG_QUARTER * 4 : 0;
  // MXFP8 row-wise dh: the two column slices of a quarter swap 16-byte halves of their quantised gate
  // and up columns ([quarter][slice][lane] uint4), so that each writes one whole 32-byte sector
  static constexpr int QX_BYTES = (DSW && MX && G1_NC == 16) ? G1_GROUPS * 4 * 2 * 32 * 16 : 0;
  static constexpr int CK_CHUNK_BYTES = 2 * 32 * 128 * 2;
  static constexpr int CK_BYTES = DSW ? CK_BUFS * CK_CHUNK_BYTES : 0;
  // Store epilogue with a single TMEM accumulator: the tile is drained into a 128B-swizzled bf16
  // staging tile in shared memory (TMEM released at once) and written by TMA stores.
#ifdef MOEBWD_NO_TMA_STORE
  static constexpr bool TMA_STORE = false;
#else
  static constexpr bool TMA_STORE = (EPI == kEpiStore) && ((MX && BN == 256) ? 1 : 2) == 1;
#endif
  // Checkpoint epilogue (G0): the tile is written as bf16 into the block checkpoint [N,2,I,B]
  // through two [32 features][128 rows] staging slabs and TMA stores.
  static constexpr bool CKPT_STORE = EPI == kEpiCkpt;
  static constexpr bool STAGED = TMA_STORE || CKPT_STORE;
  // one 64-column staging slab (16 KB) keeps a fourth pipeline stage in shared memory
  static constexpr int STAGING_BYTES = STAGED ? BM * 64 * 2 : 0;
  // staged epilogues: 8 warps, two per TMEM lane quarter, splitting the columns
  static constexpr int EPI_WARPS = DSW ? 4 * kG1Subs * G1_GROUPS : STAGED ? 8 : 4;
  // dSwiGLU: one more warp whose lane 0 streams the checkpoint chunks into their two buffers, each as
  // soon as every epilogue warp has released it (ten or eleven warps share the 168-register cap)
  static constexpr bool CK_LOADER = DSW;
  static constexpr int CK_LOADER_WARP = 2 + EPI_WARPS;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS + (CK_LOADER ? 32 : 0);
  // registers per thread: the launch bound's share of the register file (multiples of 8), which the
  // sixteen-warp dSwiGLU epilogue needs stated (ptxas would otherwise settle below it)
  static constexpr int MAX_REGS = (65536 / THREADS) / 8 * 8 > 255 ? 255 : (65536 / THREADS) / 8 * 8;
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES + XCHG_BYTES + QX_BYTES + CK_BYTES + STAGING_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int RING = 4;  // tile indices published by the producer ahead of the consumers
  static constexpr int STAGES_FIT = (kSmemLimit - 1024 - BAR_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int ACC_STAGES = (MX && BN == 256) ? 1 : 2;
  static constexpr int SF_COLS = MX ? 4 + 4 * SFB_ATOMS : 0;   // TMEM columns of scales per stage
  // TMEM column distance of the two accumulators: 192-column tiles keep them 256 apart
  static constexpr int ACC_STRIDE = BN == 192 ? 256 : BN;
  static constexpr int SF_BASE = (ACC_STAGES - 1) * ACC_STRIDE + BN;
  static constexpr int COLS_NEEDED = SF_BASE + STAGES * SF_COLS;
  static constexpr int TMEM_COLS = COLS_NEEDED <= 32 ? 32 : COLS_NEEDED <= 64 ? 64 : COLS_NEEDED <= 128 ? 128
                                 : COLS_NEEDED <= 256 ? 256 : 512;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static constexpr int NCHUNK = BN / 32;
  static_assert(STAGES >= 2, "shared memory too small for a 2-stage pipeline");
  static_assert(COLS_NEEDED <= 512, "TMEM overflow");
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory overflow");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && STAGING_BYTES % 1024 == 0, "tile alignment");
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

// Wait without giving up when another role aborted (used to drain copies / MMAs in flight).  It keeps
// the fixed 2 s limit whatever the launch's pipeline-wait limit, so that copies and tensor-core work
// in flight land before a CTA frees its shared memory and TMEM.
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
    if (p.accumulate) {  // read-add-write of the bf16 output
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 o = d4[q];
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          r[8 * q + 2 * j] = __float_as_uint(__uint_as_float(r[8 * q + 2 * j]) + __uint_as_float(ow[j] << 16));
          r[8 * q + 2 * j + 1] =
              __float_as_uint(__uint_as_float(r[8 * q + 2 * j + 1]) + __uint_as_float(ow[j] & 0xFFFF0000u));
        }
      }
    }
    auto pk = [&](int j) { return pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])); };
#pragma unroll
    for (int q = 0; q < 2; ++q)  // whole 32-byte sectors (the output is caller-owned: 16-byte alignment)
      st_global_32b_or_halves(d4 + 2 * q, pk(16 * q), pk(16 * q + 2), pk(16 * q + 4), pk(16 * q + 6), pk(16 * q + 8),
                    pk(16 * q + 10), pk(16 * q + 12), pk(16 * q + 14));
  }
}

// Location of a tile's rows in the block checkpoint [N, 2, I, B]: block index and the slot of its first
// row inside that block (the 128 rows of a tile never straddle a block since B % 128 == 0).
__device__ __forceinline__ void tile_ckpt_origin(const GemmParams& p, const TileInfo& ti, int64_t& blk, int& b0) {
  const int64_t j0 = (int64_t)ti.mt * 128 - p.e_tile_offsets[ti.e];
  const int64_t slot0 = (int64_t)p.block_offsets[ti.e] * p.B + j0;
  blk = slot0 / p.B;
  b0 = (int)(slot0 - blk * p.B);
}

// Transposed store of NC columns x 32 rows (NC = 8 or 16): v[j] of lane r is element (r, j).  The
// block is transposed through shared memory as fp32 (pitch kTransPitch = 36: the column-wise writes
// and the 16-byte row reads are both free of bank conflicts); lane l then handles
// column l % NC, rows NC*(l / NC) .. +NC-1, so output row row0 + (l % NC) * rstride gets columns
// p0..p0+31 from 32/NC lanes (bf16, or fp8 codes with one scale quantised along all 32: those lanes
// combine their amax).  With `colsum`: the sum of the 32 (unquantised) rows of every output row
// (column) goes to colsum[output row] as well (the bias gradient's share of these rows).
template <bool MX, int NC, int AF>
__device__ __forceinline__ void store_transposed(float* buf, const float (&v)[NC], void* out, uint8_t* sf,
                                                 int64_t P, int64_t row0, int rstride, int64_t p0, int lane,
                                                 float* colsum = nullptr) {
#pragma unroll
  for (int j = 0; j < NC; ++j) buf[j * kTransPitch + lane] = v[j];
  __syncwarp();
  const int c = lane % NC, rg = lane / NC;
  float col[NC];
#pragma unroll
  for (int i = 0; i < NC; i += 4) {
    const float4 f = *reinterpret_cast<const float4*>(buf + c * kTransPitch + rg * NC + i);
    col[i] = f.x;
    col[i + 1] = f.y;
    col[i + 2] = f.z;
    col[i + 3] = f.w;
  }
  if (colsum) {  // with biases: the sum of the 32 rows of this output row (column)
    float cs = 0.f;
#pragma unroll
    for (int i = 0; i < NC; ++i) cs += col[i];  // in order: the same sums as before
#pragma unroll
    for (int o = NC; o < 32; o <<= 1) cs += __shfl_xor_sync(0xffffffffu, cs, o);
    if (rg == 0) colsum[row0 + (int64_t)c * rstride] = cs;
  }
  if constexpr (MX) {
    float am = amax_tree<NC>(col);
#pragma unroll
    for (int o = NC; o < 32; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const uint32_t byte = e8m0_byte(__float_as_uint(am), AF);
    const uint64_t inv2 = f2_splat(e8m0_inv_scale(byte));
    uint32_t q[NC / 4];
#pragma unroll
    for (int w = 0; w < NC / 4; ++w)
      q[w] = fp8x4_scaled<AF>(col[4 * w], col[4 * w + 1], col[4 * w + 2], col[4 * w + 3], inv2);
    uint8_t* dst = static_cast<uint8_t*>(out) + (row0 + (int64_t)c * rstride) * P + p0 + rg * NC;
    if constexpr (NC == 16)
      *reinterpret_cast<uint4*>(dst) = make_uint4(q[0], q[1], q[2], q[3]);
    else
      *reinterpret_cast<uint2*>(dst) = make_uint2(q[0], q[1]);
    if (rg == 0) {  // tiled scale layout of the [rows, P] operand (see sf_tiled_offset)
      const int64_t r = row0 + (int64_t)c * rstride;
      sf[((r >> 7) * (P >> 7) + (p0 >> 7)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + ((p0 >> 5) & 3)] =
          (uint8_t)byte;
    }
  } else {
    uint16_t* dst = static_cast<uint16_t*>(out) + (row0 + (int64_t)c * rstride) * P + p0 + rg * NC;
    auto pk = [&](int j) { return pack_bf16x2(col[j], col[j + 1]); };
    if constexpr (NC == 16)  // one whole 32-byte sector
      st_global_32b(dst, pk(0), pk(2), pk(4), pk(6), pk(8), pk(10), pk(12), pk(14));
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(pk(0), pk(2), pk(4), pk(6));
  }
  __syncwarp();
}

// Column sums over the warp's 32 lanes (rows) of 2 * NC values per lane (a, then b), by a butterfly
// reduce-scatter: lane l returns the sum of value l % (2 NC) (2 NC = 16: the lane halves folded first).
template <int NC>
__device__ __forceinline__ float colsum_butterfly(const float (&a)[NC], const float (&b)[NC], int lane) {
  constexpr int NV = 2 * NC;
  static_assert(NV == 16 || NV == 32, "16 or 32 values");
  float v[NV];
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    v[i] = a[i];
    v[NC + i] = b[i];
  }
  if constexpr (NV == 16) {
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], 16);
  }
#pragma unroll
  for (int w = NV / 2; w >= 1; w >>= 1) {  // lane bit w picks the half of the values this lane keeps
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

template <int NTHREADS>
__device__ __forceinline__ void group_bar(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(NTHREADS) : "memory");
}

// G1 epilogue, NC columns (slice `sub` of a 32-column chunk starting at feature i0) of one warp:
// from dA_raw (accumulator) and the checkpointed gate/up pre-activations (staged in shared memory,
// [gate|up][32 features][128 rows]) compute
//   ds += <dA_raw, a>,  dA = s dA_raw,  dgate = dA up SiLU'(gate),  dup = dA SiLU(gate),  a' = s a
// and write dh [P,2I] (row-major), dh^T [2I,P], a'^T [I,P] (bf16, or fp8 + scales).  The row-wise
// MXFP8 groups of dh (32 features) span the 32/NC warps of a TMEM lane quarter: partial amax values
// are exchanged through `xchg` ([slice][gate|up][32 lanes]) with a barrier over those warps.
// GENERIC with `ga` (this row's slot in a saved act(gate) checkpoint [N,I,B], feature stride B):
// act(gate) is read from it, act'(gate) still computed from the pre-activation.
// Padding rows produce zeros.
template <bool MX, int NC, int AF, bool GENERIC, bool SHARED_TBUF>
__device__ __forceinline__ void epi_dswiglu_part(const GemmParams& p, uint32_t taddr, int64_t prow, int m, int lane,
                                                 bool valid, float sv, int i0, int sub, const uint16_t* ck,
                                                 const uint16_t* ga, float* tbuf, float* xchg, uint4* qx,
                                                 int bar_id, float& ds_acc) {
  constexpr int SUBS = 32 / NC;
  const int I = p.I;
  const int64_t P = p.P;
  const int64_t p0 = prow - lane;
  // the accumulator load is in flight while the checkpoint-only terms are computed
  uint32_t r[NC];
  if constexpr (NC == 16)
    tmem_ld_32x32b_x16(taddr, r);
  else
    tmem_ld_32x32b_x8(taddr, r);
  float dg[NC], du[NC], ap[NC];  // act(g), a and up * act'(g) first, the gradients after the load
  // GENERIC: the activation, the gate/up layout and a saved act(gate) are read at run time;
  // otherwise SwiGLU, concat
  float sa[GENERIC ? NC : 1];
  const bool saved = GENERIC && ga != nullptr;
  if constexpr (GENERIC) {
    if (saved) {
#pragma unroll
      for (int jj = 0; jj < NC; ++jj)
        sa[jj] = valid ? bf16_bits_to_float(__ldg(ga + (int64_t)(i0 + sub * NC + jj) * p.B)) : 0.f;
    }
  }
  if (GENERIC && p.glu == MOE_GLU_GEGLU) {  // GELU(g) = g Phi(g), GELU'(g) = Phi(g) + g phi(g)
#pragma unroll
    for (int jj = 0; jj < NC; ++jj) {
      float g = bf16_bits_to_float(ck[(sub * NC + jj) * 128 + m]);
      float u = bf16_bits_to_float(ck[32 * 128 + (sub * NC + jj) * 128 + m]);
      if (!valid) g = u = 0.f;
      const float cdf = 0.5f * (1.f + erff(g * 0.70710678118654752f));
      const float pdf = 0.39894228040143268f * __expf(-0.5f * g * g);
      float act = g * cdf;
      if constexpr (GENERIC) act = saved ? sa[jj] : act;
      du[jj] = act;
      ap[jj] = act * u;
      dg[jj] = u * (cdf + g * pdf);
    }
  } else if constexpr (GENERIC) {  // SiLU(g) = g sigma(g), SiLU'(g) = sigma(g) (1 + g (1 - sigma(g)))
#pragma unroll
    for (int jj = 0; jj < NC; ++jj) {
      float g = bf16_bits_to_float(ck[(sub * NC + jj) * 128 + m]);
      float u = bf16_bits_to_float(ck[32 * 128 + (sub * NC + jj) * 128 + m]);
      if (!valid) g = u = 0.f;
      const float sg = __fdividef(1.f, 1.f + __expf(-g));
      float sl = g * sg;
      sl = saved ? sa[jj] : sl;
      du[jj] = sl;
      ap[jj] = sl * u;
      dg[jj] = u * (sg * (1.f + g * (1.f - sg)));
    }
  } else {
    // the same SwiGLU terms two features at a time in paired fp32 arithmetic; sigma(g) = 1 / (1 +
    // 2^(-g log2(e))) from the exp2 and reciprocal approximations, one value per instruction
    const uint64_t one2 = f2_splat(1.f), neg1 = f2_splat(-1.f), nl2e = f2_splat(-1.4426950408889634f);
#pragma unroll
    for (int jj = 0; jj < NC; jj += 2) {
      float g0 = bf16_bits_to_float(ck[(sub * NC + jj) * 128 + m]);
      float g1 = bf16_bits_to_float(ck[(sub * NC + jj + 1) * 128 + m]);
      float u0 = bf16_bits_to_float(ck[32 * 128 + (sub * NC + jj) * 128 + m]);
      float u1 = bf16_bits_to_float(ck[32 * 128 + (sub * NC + jj + 1) * 128 + m]);
      if (!valid) g0 = g1 = u0 = u1 = 0.f;
      const uint64_t G = f2_pack(g0, g1), U = f2_pack(u0, u1);
      float x0, x1;
      f2_unpack(f2_mul(G, nl2e), x0, x1);
      float e0, e1, s0, s1;
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(x0));
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(x1));
      f2_unpack(f2_add(f2_pack(e0, e1), one2), x0, x1);
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(s0) : "f"(x0));
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(s1) : "f"(x1));
      const uint64_t SG = f2_pack(s0, s1);
      const uint64_t SL = f2_mul(G, SG);
      const uint64_t T = f2_fma(G, f2_fma(SG, neg1, one2), one2);  // 1 + g (1 - sigma)
      f2_unpack(SL, du[jj], du[jj + 1]);
      f2_unpack(f2_mul(SL, U), ap[jj], ap[jj + 1]);
      f2_unpack(f2_mul(U, f2_mul(SG, T)), dg[jj], dg[jj + 1]);
    }
  }
  tmem_ld_wait_regs<NC>(r);
  if constexpr (GENERIC) {
#pragma unroll
    for (int jj = 0; jj < NC; ++jj) {
      const float v = valid ? __uint_as_float(r[jj]) : 0.f;
      const float a = ap[jj];
      ds_acc = fmaf(v, a, ds_acc);
      const float dA = sv * v;
      dg[jj] = dA * dg[jj];
      du[jj] = dA * du[jj];
      ap[jj] = (p.affinity_on_i || p.ap_s) ? sv * a : a;
    }
  } else {
    const uint64_t sv2 = f2_splat(sv);
    // a' = s a (affinity on I, or on H with s moved from dout to a') or a (x 1, exact)
    const uint64_t sa2 = f2_splat((p.affinity_on_i || p.ap_s) ? sv : 1.f);
    uint64_t DS = f2_splat(0.f);
#pragma unroll
    for (int jj = 0; jj < NC; jj += 2) {
      const uint64_t V = valid ? f2_pack(__uint_as_float(r[jj]), __uint_as_float(r[jj + 1])) : f2_splat(0.f);
      const uint64_t A = f2_pack(ap[jj], ap[jj + 1]);
      DS = f2_fma(V, A, DS);
      const uint64_t DA = f2_mul(sv2, V);
      f2_unpack(f2_mul(DA, f2_pack(dg[jj], dg[jj + 1])), dg[jj], dg[jj + 1]);
      f2_unpack(f2_mul(DA, f2_pack(du[jj], du[jj + 1])), du[jj], du[jj + 1]);
      f2_unpack(f2_mul(sa2, A), ap[jj], ap[jj + 1]);
    }
    float d0, d1;
    f2_unpack(DS, d0, d1);
    ds_acc += d0 + d1;
  }
  const int c0 = i0 + sub * NC;  // first feature of this warp's columns
  const bool il = GENERIC && NC == 16 && p.interleaved;  // gate_i, up_i at columns 2i, 2i+1 (host: NC == 16)
  if (il) {
    // this warp's 16 (gate, up) pairs are the 32 consecutive columns 2*c0.. of dh: one MX group
    // (the layout is fixed per launch: a quarter's warps take the same branch and meet at the same
    // named barriers)
    group_bar<32 * SUBS>(bar_id);
    if constexpr (MX) {
      const float am = fmaxf(amax_tree<NC>(dg), amax_tree<NC>(du));
      const uint32_t byte = e8m0_byte(__float_as_uint(am), AF);
      const float inv = e8m0_inv_scale(byte);
      uint32_t q[NC / 2];
#pragma unroll
      for (int w = 0; w < NC / 2; ++w)
        q[w] = fp8x4_t<AF>(dg[2 * w] * inv, du[2 * w] * inv, dg[2 * w + 1] * inv, du[2 * w + 1] * inv);
      uint8_t* dst = static_cast<uint8_t*>(p.dh) + prow * (2 * (int64_t)I) + 2 * c0;
      if constexpr (NC == 16)  // one whole 32-byte sector
        st_global_32b(dst, q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(q[0], q[1], q[2], q[3]);
      p.dh_sf[sf_tiled_offset(prow, 2 * c0, 2 * (int64_t)I)] = (uint8_t)byte;
    } else {
      uint16_t* dst = static_cast<uint16_t*>(p.dh) + prow * (2 * (int64_t)I) + 2 * c0;
      auto pk = [&](int j) { return pack_bf16x2(dg[j], du[j]); };
#pragma unroll
      for (int w = 0; w < NC / 8; ++w)  // whole 32-byte sectors
        st_global_32b(dst + 16 * w, pk(8 * w), pk(8 * w + 1), pk(8 * w + 2), pk(8 * w + 3), pk(8 * w + 4),
                      pk(8 * w + 5), pk(8 * w + 6), pk(8 * w + 7));
    }
  } else if constexpr (MX) {
    float amg = amax_tree<NC>(dg), amu = amax_tree<NC>(du);
    xchg[(sub * 2 + 0) * 32 + lane] = amg;
    xchg[(sub * 2 + 1) * 32 + lane] = amu;
    group_bar<32 * SUBS>(bar_id);
#pragma unroll
    for (int o = 0; o < SUBS; ++o) {
      if (o == sub) continue;
      amg = fmaxf(amg, xchg[(o * 2 + 0) * 32 + lane]);
      amu = fmaxf(amu, xchg[(o * 2 + 1) * 32 + lane]);
    }
    uint8_t* dh = static_cast<uint8_t*>(p.dh) + prow * (2 * (int64_t)I);
    const uint32_t bg = e8m0_byte(__float_as_uint(amg), AF), bu = e8m0_byte(__float_as_uint(amu), AF);
    const uint64_t ig = f2_splat(e8m0_inv_scale(bg)), iu = f2_splat(e8m0_inv_scale(bu));
    uint32_t qg[NC / 4], qu[NC / 4];
#pragma unroll
    for (int w = 0; w < NC / 4; ++w) {
      qg[w] = fp8x4_scaled<AF>(dg[4 * w], dg[4 * w + 1], dg[4 * w + 2], dg[4 * w + 3], ig);
      qu[w] = fp8x4_scaled<AF>(du[4 * w], du[4 * w + 1], du[4 * w + 2], du[4 * w + 3], iu);
    }
    if constexpr (NC == 16) {
      // slice 0 writes the row's 32 gate columns i0.., slice 1 its 32 up columns I + i0..: each takes
      // the other's half from shared memory (one more barrier of the quarter's two warps)
      qx[sub * 32 + lane] = sub == 0 ? make_uint4(qu[0], qu[1], qu[2], qu[3]) : make_uint4(qg[0], qg[1], qg[2], qg[3]);
      group_bar<32 * SUBS>(bar_id);
      const uint4 o = qx[(1 - sub) * 32 + lane];
      if (sub == 0)
        st_global_32b(dh + i0, qg[0], qg[1], qg[2], qg[3], o.x, o.y, o.z, o.w);
      else
        st_global_32b(dh + I + i0, o.x, o.y, o.z, o.w, qu[0], qu[1], qu[2], qu[3]);
    } else {
      *reinterpret_cast<uint2*>(dh + c0) = make_uint2(qg[0], qg[1]);
      *reinterpret_cast<uint2*>(dh + I + c0) = make_uint2(qu[0], qu[1]);
    }
    if (sub == 0) {
      p.dh_sf[sf_tiled_offset(prow, i0, 2 * (int64_t)I)] = (uint8_t)bg;
      p.dh_sf[sf_tiled_offset(prow, I + i0, 2 * (int64_t)I)] = (uint8_t)bu;
    }
  } else {
    group_bar<32 * SUBS>(bar_id);  // the amax exchange's barrier on the MXFP8 branch (its partner's reads)
    uint16_t* dh = static_cast<uint16_t*>(p.dh) + prow * (2 * (int64_t)I);
    auto pg = [&](int j) { return pack_bf16x2(dg[j], dg[j + 1]); };
    auto pu = [&](int j) { return pack_bf16x2(du[j], du[j + 1]); };
    if constexpr (NC == 16) {  // whole 32-byte sectors
      st_global_32b(dh + c0, pg(0), pg(2), pg(4), pg(6), pg(8), pg(10), pg(12), pg(14));
      st_global_32b(dh + I + c0, pu(0), pu(2), pu(4), pu(6), pu(8), pu(10), pu(12), pu(14));
    } else {
      *reinterpret_cast<uint4*>(dh + c0) = make_uint4(pg(0), pg(2), pg(4), pg(6));
      *reinterpret_cast<uint4*>(dh + I + c0) = make_uint4(pu(0), pu(2), pu(4), pu(6));
    }
  }
  // dh^T rows in W1's gate/up layout, a'^T rows by feature
  // SHARED_TBUF: the three transposes share the warp's buffer (each ends with the warp's reads done)
  constexpr int TB = SHARED_TBUF ? 0 : NC * kTransPitch;
  // db1 (BF16 with biases): this tile's and lane quarter's column sums of dh, in W1's layout
  float* db1p = p.db1_part ? p.db1_part + ((prow >> 7) * 4 + (m >> 5)) * (2 * (int64_t)I) : nullptr;
  if (p.dht) {
    store_transposed<MX, NC, AF>(tbuf, dg, p.dht, p.dht_sf, P, il ? 2 * c0 : c0, il ? 2 : 1, p0, lane, db1p);
    store_transposed<MX, NC, AF>(tbuf + TB, du, p.dht, p.dht_sf, P, il ? 2 * c0 + 1 : I + c0, il ? 2 : 1, p0, lane,
                                 db1p);
  } else if (db1p) {  // no dh^T (BF16: the weight-gradient GEMM reads dh): the quarter's column sums
    const float v = colsum_butterfly<NC>(dg, du, lane);
    const int idx = lane, f = idx % NC, gu = idx / NC;  // value idx: dg[f] (gu = 0) or du[f] (gu = 1)
    if (idx < 2 * NC) db1p[il ? 2 * (c0 + f) + gu : gu * I + c0 + f] = v;
  }
  if (p.apt) {  // a'^T (null: built from a saved checkpoint of a or s*a)
    if (!MX && p.ap_rows) {  // BF16 whose dW2 GEMM reads a' MN-major: the row's NC features of a'
      uint16_t* dst = static_cast<uint16_t*>(p.apt) + prow * (int64_t)I + c0;
      auto pa2 = [&](int j) { return pack_bf16x2(ap[j], ap[j + 1]); };
      if constexpr (NC == 16)
        st_global_32b(dst, pa2(0), pa2(2), pa2(4), pa2(6), pa2(8), pa2(10), pa2(12), pa2(14));
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(pa2(0), pa2(2), pa2(4), pa2(6));
    } else {
      store_transposed<MX, NC, AF>(tbuf + 2 * TB, ap, p.apt, p.apt_sf, P, c0, 1, p0, lane);
    }
  }
}


// Producer with a gathered A operand (the whole warp 0; dSwiGLU GEMM with p.a_gather).  Lane 0 claims
// and publishes tiles and loads B (and, for MXFP8, both operands' scale atoms) by TMA as the plain
// producer does; all 32 lanes copy A's 128 rows of each k-block from their source rows with 16-byte
// cp.async: piece c (16 bytes) of row r lands at r*128 + ((c ^ (r % 8)) * 16), where the 128-byte
// swizzle of a TMA tile load would put it (the stage is 1024-byte aligned).  A stage's copies are
// completed kLag stages later -- cp.async.wait_group, the proxy fence that makes them visible to the
// tensor core, then lane 0's second arrival on the stage's full barrier (initialised with two) -- so
// that each lane keeps kLag stages of gathers in flight.  kLag < STAGES: the stage the producer waits
// to refill was completed kLag stages after it was issued, so the MMA can always drain it.
template <typename C, int BN, bool MX>
__device__ __forceinline__ void producer_gather(const GemmParams& p, const CUtensorMap* tmB, uint8_t* smA,
                                                uint8_t* smB, uint8_t* smSFA, uint8_t* smSFB, uint64_t* full,
                                                uint64_t* empty, uint64_t* tile_full, uint64_t* tile_empty,
                                                volatile int* tile_ring, volatile int* abort_flag, int total,
                                                int lane) {
  constexpr int kLag = 2;
  static_assert(kLag <= C::STAGES - 1, "gathered A needs more stages than its completion lag");
  const char* src = static_cast<const char*>(p.a_gather);
  const int piece = lane & 7;
  int s = 0;
  uint32_t ph = 0;
  int64_t issued = 0, completed = 0;
  int rs = 0;
  uint32_t rph = 0;
  for (;;) {
    int t = 0;
    if (lane == 0) {
      t = atomicAdd(p.tile_counter, 1);
      if (t >= total) t = -1;
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(&tile_empty[rs], rph ^ 1u, p.status, abort_flag, p.wait_ns);
    if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    if (lane == 0) {
      tile_ring[rs] = t;
      mbar_arrive(&tile_full[rs]);
    }
    if (++rs == C::RING) {
      rs = 0;
      rph ^= 1u;
    }
    if (t < 0) break;
    const TileInfo ti = gemm_decode_tile<BN, C::BKE>(p, t);
    // source rows of this lane's tile rows r = (lane >> 3) + 4 i (padding rows read row 0)
    uint32_t rowi[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int f = p.tile_row_flat[(int64_t)ti.a_row + (lane >> 3) + 4 * i];
      rowi[i] = f >= 0 ? (uint32_t)(f / p.a_gather_div) : 0u;
    }
    for (int kb = 0; kb < ti.nk; ++kb) {
      int w = 1;
      if (lane == 0) w = mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, abort_flag, p.wait_ns);
      if (!__shfl_sync(0xffffffffu, w, 0)) {
        ok = 0;
        break;
      }
      const int kc = ti.k0 + kb * C::BKE;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES - C::A_BYTES);
        tma_load_2d(smB + s * C::B_BYTES, tmB, &full[s], kc, ti.b_row);
        if constexpr (MX) {
          const int kt = kc / 128;
          bulk_load(smSFA + s * C::SFA_BYTES, p.sfa + ((int64_t)(ti.a_row / 128) * p.sfa_ktiles + kt) * 512, 512,
                    &full[s]);
#pragma unroll
          for (int h = 0; h < C::SFB_ATOMS; ++h)
            bulk_load(smSFB + s * C::SFB_BYTES + h * 512,
                      p.sfb + ((int64_t)((ti.b_row / BN) * C::SFB_ATOMS + h) * p.sfb_ktiles + kt) * 512, 512,
                      &full[s]);
        }
      }
      const uint32_t dst0 = smem_u32(smA + s * C::A_BYTES);
      const int64_t koff = (int64_t)kc * (MX ? 1 : 2) + piece * 16;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = (lane >> 3) + 4 * i;
        cp_async_16(dst0 + r * 128 + ((piece ^ (r & 7)) << 4), src + (int64_t)rowi[i] * p.a_gather_ld + koff);
      }
      cp_async_commit();
      ++issued;
      if (issued - completed > kLag) {  // the stage issued kLag stages ago is complete for every lane
        cp_async_wait<kLag>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[completed % C::STAGES]);
        ++completed;
      }
      if (++s == C::STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (!ok) break;
  }
  // Drain: every gather completes and is released, then every TMA copy issued lands, before the CTA
  // may exit.
  cp_async_wait<0>();
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    for (; completed < issued; ++completed) mbar_arrive(&full[completed % C::STAGES]);
    const int64_t n = issued < C::STAGES ? issued : C::STAGES;
    for (int64_t i = 1; i <= n; ++i) {
      const int64_t q = issued - i;
      mbar_wait_drain(&full[q % C::STAGES], (uint32_t)((q / C::STAGES) & 1), p.status);
    }
  }
}

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------
template <bool MX, int BN, int EPI>
__global__ void __launch_bounds__((GemmCfg<MX, BN, EPI>::THREADS), 1) __maxnreg__((GemmCfg<MX, BN, EPI>::MAX_REGS))
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ GemmParams p) {
  using C = GemmCfg<MX, BN, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smA + C::STAGES * C::A_BYTES;
  uint8_t* smStage = smB + C::STAGES * C::B_BYTES;      // output staging (TMA-store epilogue), 1024-aligned
  uint8_t* smSFA = smStage + C::STAGING_BYTES;
  uint8_t* smSFB = smSFA + C::STAGES * C::SFA_BYTES;
  uint8_t* smCK = smSFB + C::STAGES * C::SFB_BYTES;     // checkpoint chunks (dSwiGLU epilogue), 512-aligned
  uint8_t* smEPI = smCK + C::CK_BYTES;
  float* smXchg = reinterpret_cast<float*>(smEPI + C::EPI_WARPS * C::EPI_WARP_BYTES);
  uint4* smQx = reinterpret_cast<uint4*>(smEPI + C::EPI_WARPS * C::EPI_WARP_BYTES + C::XCHG_BYTES);
  uint64_t* full =
      reinterpret_cast<uint64_t*>(smEPI + C::EPI_WARPS * C::EPI_WARP_BYTES + C::XCHG_BYTES + C::QX_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* ck_full = tempty + 2;
  uint64_t* ck_empty = ck_full + C::CK_BUFS;  // every warp of the chunk's group has consumed the buffer
  uint64_t* done = ck_empty + C::CK_BUFS;
  uint64_t* tile_full = done + 1;          // ring slot r holds a tile index (producer arrives)
  uint64_t* tile_empty = tile_full + C::RING;  // every consumer warp has read slot r
  volatile int* tile_ring = reinterpret_cast<volatile int*>(tile_empty + C::RING);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tile_ring) + C::RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // a gathered A operand arrives on a stage's full barrier a second time (see producer_gather)
    const uint32_t full_count = (C::DSW && p.a_gather) ? 2u : 1u;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], full_count);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], C::EPI_WARPS);
    }
    for (int a = 0; a < C::CK_BUFS; ++a) {
      mbar_init(&ck_full[a], 1);
      mbar_init(&ck_empty[a], C::EPI_WARPS / C::G1_GROUPS);
    }
    mbar_init(done, 1);
    for (int r = 0; r < C::RING; ++r) {
      mbar_init(&tile_full[r], 1);
      mbar_init(&tile_empty[r], 1 + C::EPI_WARPS + (C::CK_LOADER ? 1 : 0));
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (C::DSW || C::STAGED) prefetch_tmap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the prologue above (barriers, TMEM, tensor-map prefetch) overlaps the previous kernel's tail;
  // nothing written by earlier work is read before this point
  pdl_wait();
  pdl_trigger();
  const int total = gemm_total_tiles(p);
  // Dynamic schedule: the producer claims tiles from a global counter (heaviest experts first in
  // the K-grouped order) and publishes each index, then -1, through the ring.

  if (warp == 0) {
    if (C::DSW && p.a_gather) {
      // ---------------- producer with gathered A rows (whole warp) ----------------
      producer_gather<C, BN, MX>(p, &tmB, smA, smB, smSFA, smSFB, full, empty, tile_full, tile_empty, tile_ring,
                                 abort_flag, total, lane);
    } else if (lane == 0) {
      // ---------------- TMA producer ----------------
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      int rs = 0;
      uint32_t rph = 0;
      for (;;) {
        int t = atomicAdd(p.tile_counter, 1);
        if (t >= total) t = -1;
        if (!mbar_wait_bounded(&tile_empty[rs], rph ^ 1u, p.status, abort_flag, p.wait_ns)) break;
        tile_ring[rs] = t;
        mbar_arrive(&tile_full[rs]);
        if (++rs == C::RING) {
          rs = 0;
          rph ^= 1u;
        }
        if (t < 0) break;
        const TileInfo ti = gemm_decode_tile<BN, C::BKE>(p, t);
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          const int kc = ti.k0 + kb * C::BKE;
          if (!MX && p.a_mn) {  // [K, M] operand: 64 x 64 boxes, 8 KB apart along M
#pragma unroll
            for (int j = 0; j < 2; ++j) tma_load_2d(smA + s * C::A_BYTES + j * 8192, &tmA, &full[s], ti.a_row + 64 * j, kc);
          } else {
            tma_load_2d(smA + s * C::A_BYTES, &tmA, &full[s], kc, ti.a_row);
          }
          if (!MX && p.b_mn) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(smB + s * C::B_BYTES + j * 8192, &tmB, &full[s], ti.b_row + 64 * j, kc);
          } else {
            tma_load_2d(smB + s * C::B_BYTES, &tmB, &full[s], kc, ti.b_row);
          }
          if constexpr (MX) {
            const int kt = kc / 128;
            bulk_load(smSFA + s * C::SFA_BYTES, p.sfa + ((int64_t)(ti.a_row / 128) * p.sfa_ktiles + kt) * 512, 512,
                      &full[s]);
#pragma unroll
            for (int h = 0; h < C::SFB_ATOMS; ++h)
              bulk_load(smSFB + s * C::SFB_BYTES + h * 512,
                        p.sfb + ((int64_t)((ti.b_row / BN) * C::SFB_ATOMS + h) * p.sfb_ktiles + kt) * 512, 512,
                        &full[s]);
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
      int rs = 0;
      uint32_t rph = 0;
      while (ok) {
        if (!mbar_wait_bounded(&tile_full[rs], rph, p.status, abort_flag, p.wait_ns)) break;
        const int t = tile_ring[rs];
        mbar_arrive(&tile_empty[rs]);
        if (++rs == C::RING) {
          rs = 0;
          rph ^= 1u;
        }
        if (t < 0) break;
        const TileInfo ti = gemm_decode_tile<BN, C::BKE>(p, t);
        if (!mbar_wait_bounded(&tempty[acc], aph ^ 1u, p.status, abort_flag, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * C::ACC_STRIDE);
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait_bounded(&full[s], ph, p.status, abort_flag, p.wait_ns)) {
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
            for (int h = 0; h < C::SFB_ATOMS; ++h)
              tmem_cp_32x128b_warpx4(sfb_t + 4 * h, make_smem_desc(smem_u32(smSFB + s * C::SFB_BYTES + h * 512), 0,
                                                                   128, kSwizzleNone));
// one MMA per 32-wide K step over all BN columns; the scales of B rows 128..255 sit in the four
// TMEM columns after those of rows 0..127
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_mxf8(d, kmajor_sw128_desc(a0 + kk * 32), kmajor_sw128_desc(b0 + kk * 32),
                       idesc_mxf8(128, BN, (uint32_t)p.fmt_a, (uint32_t)p.fmt_b, (uint32_t)kk, (uint32_t)kk), sfa_t,
                       sfb_t, (kb | kk) != 0);
          } else {
            // K step kk: 32 bytes into each 128-byte K-major row, or two 8-row atoms of an MN-major tile
            const uint32_t idesc = idesc_bf16(128, BN, (uint32_t)p.a_mn, (uint32_t)p.b_mn);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(d, p.a_mn ? mnmajor_sw128_desc(a0 + kk * 2048, 8192) : kmajor_sw128_desc(a0 + kk * 32),
                       p.b_mn ? mnmajor_sw128_desc(b0 + kk * 2048, 8192) : kmajor_sw128_desc(b0 + kk * 32), idesc,
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
  } else if (C::CK_LOADER && warp == C::CK_LOADER_WARP) {
    if (lane == 0) {
      // ---------------- checkpoint loader (dSwiGLU) ----------------
      // chunk n of the schedule (the tiles in ring order, NCHUNK chunks each) goes to buffer
      // n % CK_BUFS once every warp of its group has released chunk n - CK_BUFS
      int64_t issued = 0;
      int rs = 0;
      uint32_t rph = 0;
      bool ok = true;
      while (ok) {
        if (!mbar_wait_bounded(&tile_full[rs], rph, p.status, abort_flag, p.wait_ns)) break;
        const int t = tile_ring[rs];
        mbar_arrive(&tile_empty[rs]);
        if (++rs == C::RING) {
          rs = 0;
          rph ^= 1u;
        }
        if (t < 0) break;
        const TileInfo tn = gemm_decode_tile<BN, C::BKE>(p, t);
        int64_t blk;
        int b0;
        tile_ckpt_origin(p, tn, blk, b0);
        for (int c = 0; c < C::NCHUNK; ++c) {
          const int buf = (int)(issued % C::CK_BUFS);
          if (issued >= C::CK_BUFS &&
              !mbar_wait_bounded(&ck_empty[buf], (uint32_t)(((issued - C::CK_BUFS) / C::CK_BUFS) & 1), p.status,
                                 abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          uint8_t* dst = smCK + buf * C::CK_CHUNK_BYTES;
          const int i0 = tn.nt * BN + c * 32;
          mbar_arrive_expect_tx(&ck_full[buf], C::CK_CHUNK_BYTES);
          tma_load_2d(dst, &tmC, &ck_full[buf], b0, (int)((blk * 2 + 0) * p.I + i0));
          tma_load_2d(dst + C::CK_CHUNK_BYTES / 2, &tmC, &ck_full[buf], b0, (int)((blk * 2 + 1) * p.I + i0));
          ++issued;
        }
      }
      // Drain: the last CK_BUFS chunks' copies land before the CTA may exit.
      for (int64_t n = issued > C::CK_BUFS ? issued - C::CK_BUFS : 0; n < issued; ++n)
        mbar_wait_drain(&ck_full[n % C::CK_BUFS], (uint32_t)((n / C::CK_BUFS) & 1), p.status);
    }
  } else {
    // ---------------- epilogue warps (2..5, 2..9, or 2..17) ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int m = 32 * q + lane;
    // dSwiGLU: column slice of every 32 columns and (two groups) the warp's chunk group; staged: which half
    const int half = ((warp - 2) >> 2) & 1;
    const int grp = (warp - 2) >> 3;
    uint8_t* wsm = smEPI + (warp - 2) * C::EPI_WARP_BYTES;
    // the amax exchange of the group's quarter: [group][chunk parity][quarter][XCHG_QUARTER]
    float* xchg = smXchg + grp * (8 * C::XCHG_QUARTER) + q * C::XCHG_QUARTER;
    // checkpoint chunk n of the schedule (n = tiles before this one * NCHUNK + c) is read from buffer
    // n % CK_BUFS (filled by the loader warp); `done_chunks` counts this warp's chunks (pair parity)
    int64_t tile_seq = 0, done_chunks = 0;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    int rs = 0;
    uint32_t rph = 0;
    while (ok) {
      const bool gt = mbar_wait_bounded(&tile_full[rs], rph, p.status, abort_flag, p.wait_ns);
      const int t = gt ? tile_ring[rs] : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&tile_empty[rs]);
      if (++rs == C::RING) {
        rs = 0;
        rph ^= 1u;
      }
      if constexpr (C::DSW || C::STAGED) {
        // uniform exit decision (see below)
        if (epilogue_bar_any<32 * C::EPI_WARPS>(*abort_flag != 0)) break;
      }
      if (t < 0) break;
      const TileInfo ti = gemm_decode_tile<BN, C::BKE>(p, t);
      // dSwiGLU: the row's flat index and score, loaded while the accumulator is still being computed
      int row_f = -1;
      float row_s = 0.f;
      if constexpr (C::DSW) {
        row_f = p.tile_row_flat[(int64_t)ti.mt * 128 + m];
        if (row_f >= 0) row_s = p.s[row_f];
      }
      const bool got = mbar_wait_bounded(&tfull[acc], aph, p.status, abort_flag, p.wait_ns);
      if constexpr (C::DSW || C::STAGED) {
        // these epilogues synchronise their warps with named barriers: every exit decision is the
        // OR of the shared abort flag over all of them, taken at a barrier, so no warp is left waiting
        if (epilogue_bar_any<32 * C::EPI_WARPS>(*abort_flag != 0)) break;
      } else if (!got) {
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * C::ACC_STRIDE);
      if constexpr (C::CKPT_STORE) {
        // two 32-feature chunks per step, one per warp half: h = acc + b1_e (bf16) staged as
        // [32 features][128 rows] and stored to the checkpoint rows of the tile's block
        int64_t blk;
        int b0;
        tile_ckpt_origin(p, ti, blk, b0);
        uint16_t* stg = reinterpret_cast<uint16_t*>(smStage) + half * (32 * 128);
        // the warp's four 32-column chunks come out of TMEM under one wait and the accumulator is
        // released at once; bias, staging and stores then run from registers
        uint32_t rr[BN / 64][32];
        if (ti.nk > 0) {
#pragma unroll
          for (int cp = 0; cp < BN / 64; ++cp) tmem_ld_32x32b_x32(taddr + (cp * 2 + half) * 32, rr[cp]);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int cp = 0; cp < BN / 64; ++cp)
#pragma unroll
            for (int j = 0; j < 32; ++j) rr[cp][j] = 0u;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
#pragma unroll
        for (int cp = 0; cp < BN / 64; ++cp) {
          if (warp == 2 && lane == 0) bulk_wait_read_all();
          epilogue_bar<32 * C::EPI_WARPS>();
          const int n0 = ti.nt * BN + (cp * 2 + half) * 32;  // first gate|up feature of the chunk
          uint32_t (&r)[32] = rr[cp];
          if (p.b1) {
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
#pragma unroll
          for (int j = 0; j < 32; ++j) stg[j * 128 + m] = float_to_bf16_bits(__uint_as_float(r[j]));
          fence_proxy_async_smem();
          epilogue_bar<32 * C::EPI_WARPS>();
          if (warp == 2 && lane == 0) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int n = ti.nt * BN + (cp * 2 + hh) * 32;
              const int g = n >= p.I ? 1 : 0;
              tma_store_2d(&tmC, smStage + hh * (32 * 128 * 2), b0, (int)((blk * 2 + g) * p.I + (n - g * p.I)));
            }
            bulk_commit();
          }
        }
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          aph ^= 1u;
        }
        continue;
      } else if constexpr (C::TMA_STORE) {
        // The warp's 128 columns (4 slabs x 32) are read from TMEM under one wait and the accumulator
        // is released at once; packed to bf16 in registers, the slabs then go out one at a time
        // through the staging slab while the next tile's MMAs run.
        uint32_t pk[BN / 64][16];
        {  // all of the warp's slabs in flight under one wait; TMEM is released before the packing
          uint32_t r[BN / 64][32];
          if (ti.nk > 0) {
#pragma unroll
            for (int sl = 0; sl < BN / 64; ++sl) tmem_ld_32x32b_x32(taddr + (sl * 2 + half) * 32, r[sl]);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int sl = 0; sl < BN / 64; ++sl)
#pragma unroll
              for (int j = 0; j < 32; ++j) r[sl][j] = 0u;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
#pragma unroll
          for (int sl = 0; sl < BN / 64; ++sl)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[sl][j] = pack_bf16x2(__uint_as_float(r[sl][2 * j]), __uint_as_float(r[sl][2 * j + 1]));
        }
#pragma unroll
        for (int sl = 0; sl < BN / 64; ++sl) {
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
          if (warp == 2 && lane == 0) {
            const int orow = (p.mode == kMGrouped ? 0 : ti.e * p.M) + ti.mt * 128;
            if (p.accumulate)
              tma_reduce_add_2d(&tmC, smStage, ti.nt * BN + sl * 64, orow);
            else
              tma_store_2d(&tmC, smStage, ti.nt * BN + sl * 64, orow);
            bulk_commit();
          }
        }
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          aph ^= 1u;
        }
        continue;
      } else if constexpr (EPI == kEpiStore) {
        epi_store<BN>(p, ti, taddr, m);
      } else {
        const int64_t prow = (int64_t)ti.mt * 128 + m;
        const bool valid = row_f >= 0;
        const float sv = row_s;
        float ds_acc = 0.f;
        const uint16_t* ga = nullptr;  // this row's slot in the saved act(gate) checkpoint
        if (p.gate_act) {
          int64_t blk;
          int b0;
          tile_ckpt_origin(p, ti, blk, b0);
          ga = p.gate_act + blk * (int64_t)p.I * p.B + b0 + m;
        }
        const int bar_id = 2 + q + 4 * grp;  // the pair of this quarter and group
#pragma unroll 1
        for (int c = grp; c < C::NCHUNK; c += C::G1_GROUPS) {
          const int64_t n = tile_seq * C::NCHUNK + c;  // the chunk's place in the loader's schedule
          const int buf = (int)(n % C::CK_BUFS);
          // on a failed wait the chunk is still walked (garbage in, flagged by the status word) so
          // that both warps of a pair reach the same barriers
          const bool ck_ok = mbar_wait_bounded(&ck_full[buf], (uint32_t)((n / C::CK_BUFS) & 1), p.status, abort_flag,
                                               p.wait_ns);
          {
            const uint32_t ta = taddr + c * 32 + half * C::G1_NC;
            const int i0 = ti.nt * BN + c * 32;
            const uint16_t* ckb = reinterpret_cast<const uint16_t*>(smCK + buf * C::CK_CHUNK_BYTES);
            float* xc = xchg + (int)(done_chunks & 1) * (4 * C::XCHG_QUARTER);
            uint4* qx = smQx + (grp * 4 + q) * 64;
            // the activation format fixed per instantiation; SwiGLU with concat gate/up specialised
            const bool generic = p.glu != MOE_GLU_SWIGLU || p.interleaved || p.gate_act != nullptr;
            float* tb = reinterpret_cast<float*>(wsm);
            if (!MX || p.fmt_act == MOE_FP8_E5M2) {
              if (generic)
                epi_dswiglu_part<MX, C::G1_NC, MOE_FP8_E5M2, true, C::G1_TBUFS == 1>(p, ta, prow, m, lane, valid, sv, i0, half, ckb, ga, tb,
                                                                  xc, qx, bar_id, ds_acc);
              else
                epi_dswiglu_part<MX, C::G1_NC, MOE_FP8_E5M2, false, C::G1_TBUFS == 1>(p, ta, prow, m, lane, valid, sv, i0, half, ckb, ga, tb,
                                                                   xc, qx, bar_id, ds_acc);
            } else {
              if (generic)
                epi_dswiglu_part<MX, C::G1_NC, MOE_FP8_E4M3, true, C::G1_TBUFS == 1>(p, ta, prow, m, lane, valid, sv, i0, half, ckb, ga, tb,
                                                                  xc, qx, bar_id, ds_acc);
              else
                epi_dswiglu_part<MX, C::G1_NC, MOE_FP8_E4M3, false, C::G1_TBUFS == 1>(p, ta, prow, m, lane, valid, sv, i0, half, ckb, ga, tb,
                                                                   xc, qx, bar_id, ds_acc);
            }
          }
          __syncwarp();
          // this warp no longer reads the buffer; a chunk whose copy was not seen to land is never
          // released, so the loader cannot refill a buffer while a copy into it is still in flight
          if (lane == 0 && ck_ok) mbar_arrive(&ck_empty[buf]);
          ++done_chunks;
        }
        ++tile_seq;
        // one ds partial per (row, N tile, group, column slice)
        constexpr int kParts = kG1Subs * C::G1_GROUPS;
        p.ds_part[prow * (int64_t)(kParts * (p.I / BN)) + kParts * ti.nt + grp * kG1Subs + half] = valid ? ds_acc : 0.f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == C::ACC_STAGES) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if (C::STAGED && warp == 2 && lane == 0) bulk_wait_all();  // stores complete before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <bool MX, int BN, int EPI>
int gemm_launch_instance(const GemmParams& p, const void* tmA, const void* tmB, const void* tmC, int grid,
                         cudaStream_t st) {
  using C = GemmCfg<MX, BN, EPI>;
  auto kern = gemm_kernel<MX, BN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(gemm)");
  return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, st, "gemm launch",
                    *static_cast<const CUtensorMap*>(tmA), *static_cast<const CUtensorMap*>(tmB),
                    *static_cast<const CUtensorMap*>(tmC), p);
}

}  // namespace moebwd
