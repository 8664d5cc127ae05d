// Operand preparation for the grouped GEMMs, and the public mxfp8_quantize.
//
// prep_kernel (one CTA per 128-row tile of the tile-row space, H walked in 256-column chunks)
// gathers the token rows of every routed (t, k) once and writes, in one pass over dout and x:
//   dout_g  [P, H]  gathered dout rows                      (G1 A operand, groups along H; when G1
//                   gathers its rows itself, nothing for BF16 and only the tiled scales for MXFP8)
//   dout_gt [H, P]  gathered dout transposed, s-scaled for affinity on H (G3 B operand)
//   x_gt    [H, P]  gathered x transposed                   (G4 A operand)
//   ds_bias [P]     <dout_t, b2_e>, the bias term of ds      (sonic-moe db2_and_ds_kernel)
// as BF16, or as MXFP8 with E8M0 scales in the tiled layout (transposed operands are quantised
// in groups of 32 tile rows, i.e. along the GEMM contraction).  Padding rows are zero.  When the
// gate/up pre-activations are recomputed, a row-major gathered x [P,H] (G0's A operand) is written too.
#include <cuda_runtime.h>

#include "moebwd_internal.h"
#include "mx_device.cuh"

namespace moebwd {

constexpr int kPrepPitch = 66;       // bf16 row pitch of the 64-column tiles of the generic quantiser
constexpr int kPrepCols = 256;       // H columns per step of the MoE prep kernel
constexpr int kPrepTilePitch = 264;  // bf16 row pitch of its [128][256] tile (528 B: 16 B aligned)
constexpr int kPrepSmem = 128 * kPrepTilePitch * 2;

// Per 256-column chunk and per tensor (dout, then x): phase 1, each warp reads whole 512-byte row
// segments of 16 gathered rows (16-byte vectors, 16 in flight per thread), writes the row-major
// dout_g chunk and stages the tile in shared memory; phase 2 writes the transposed output in 32-row
// groups (128 contiguous bytes for fp8, 256 for bf16, per output row): for MXFP8 each thread owns
// one column and its four groups, for BF16 a column pair (32-bit shared-memory reads) and two groups.
// Gathered rows in flight per thread in phase 1: 8 (two batches per 16 rows) measured as fast as 16
// at 2 CTAs per SM with half the registers; 3 CTAs per SM measured slower.
constexpr int kPrepBatch = 8;

template <bool MX, bool SCALE_T, bool BIAS, int AF>
__global__ void __launch_bounds__(256, 2) prep_kernel(const PrepArgs a) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  if ((int)blockIdx.x >= *a.num_tiles) return;
  const int tile = a.tile_order ? a.tile_order[blockIdx.x] : (int)blockIdx.x;
  extern __shared__ uint4 prep_smem[];
  uint16_t* st = reinterpret_cast<uint16_t*>(prep_smem);
  __shared__ int32_t s_tok[128];
  __shared__ float s_s[128];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H;
  const int64_t P = a.P;
  const int64_t prow0 = (int64_t)tile * 128;
  if (tid < 128) {
    const int f = a.tile_row_flat[prow0 + tid];
    s_tok[tid] = f >= 0 ? f / a.K : -1;
    s_s[tid] = f >= 0 ? a.s[f] : 0.f;
  }
  const int e = BIAS ? a.tile_expert[tile] : 0;
  __syncthreads();
  float bias_acc[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) bias_acc[r] = 0.f;
  for (int h0 = 0; h0 < H; h0 += kPrepCols) {
    const int ncol = min(kPrepCols, H - h0);
    const int col = h0 + lane * 8;
    const bool colok = lane * 8 < ncol;
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      const uint16_t* src = which == 0 ? a.dout : a.x;
      // ---- phase 1 ----
      uint4 bv = make_uint4(0, 0, 0, 0);
      if (BIAS && which == 0 && colok) bv = *reinterpret_cast<const uint4*>(a.b2 + (int64_t)e * H + col);
#pragma unroll
      for (int rb = 0; rb < 16; rb += kPrepBatch) {
      uint4 v[kPrepBatch];
#pragma unroll
      for (int i = 0; i < kPrepBatch; ++i) {
        const int row = warp + 8 * (rb + i);
        const int t = s_tok[row];
        v[i] = make_uint4(0, 0, 0, 0);
        if (t >= 0 && colok) v[i] = *reinterpret_cast<const uint4*>(src + (int64_t)t * H + col);
      }
#pragma unroll
      for (int i = 0; i < kPrepBatch; ++i) {
        const int r = rb + i;
        const int row = warp + 8 * r;
        const int64_t prow = prow0 + row;
        if (colok) *reinterpret_cast<uint4*>(st + row * kPrepTilePitch + lane * 8) = v[i];
        if (which != 0 && !a.x_g) continue;  // row-major copy: dout always, x when recomputing h
        void* rowdst = which == 0 ? a.dout_g : a.x_g;
        uint8_t* rowsf = which == 0 ? a.dout_g_sf : a.x_g_sf;
        const uint32_t dw[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        float d8[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          d8[2 * j] = __uint_as_float(dw[j] << 16);
          d8[2 * j + 1] = __uint_as_float(dw[j] & 0xFFFF0000u);
        }
        if (BIAS && which == 0) {
          const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            bias_acc[r] = fmaf(d8[2 * j], __uint_as_float(bw[j] << 16), bias_acc[r]);
            bias_acc[r] = fmaf(d8[2 * j + 1], __uint_as_float(bw[j] & 0xFFFF0000u), bias_acc[r]);
          }
        }
        if constexpr (MX) {
          float am = amax_tree<8>(d8);
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
          if (!colok) continue;
          const uint32_t byte = e8m0_byte(__float_as_uint(am), AF);
          if (rowdst) {  // no codes when G1 gathers its rows from dout quantised per token
            const float inv = e8m0_inv_scale(byte);
            uint2 q;
            q.x = fp8x4_t<AF>(d8[0] * inv, d8[1] * inv, d8[2] * inv, d8[3] * inv);
            q.y = fp8x4_t<AF>(d8[4] * inv, d8[5] * inv, d8[6] * inv, d8[7] * inv);
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(rowdst) + prow * H + col) = q;
          }
          if ((lane & 3) == 0) rowsf[sf_tiled_offset(prow, col, H)] = (uint8_t)byte;
        } else {
          if (colok && rowdst) *reinterpret_cast<uint4*>(static_cast<uint16_t*>(rowdst) + prow * H + col) = v[i];
        }
      }
      }
      __syncthreads();
      // ---- phase 2 ---- (dout^T comes from a saved s*dout checkpoint when skip_dout_t)
      // MXFP8: thread = one column, its four 32-row groups.  BF16: thread = a column pair (one 32-bit
      // shared-memory word per row) and two of the groups; ncol is a multiple of 128, so a pair is whole.
      if constexpr (MX) {
        if (tid < ncol && !(which == 0 && a.skip_dout_t)) {
          const int h = tid;
          const int64_t orow = h0 + h;
          uint8_t* outp = static_cast<uint8_t*>(which == 0 ? a.dout_gt : a.x_gt);
          uint8_t* outsf = which == 0 ? a.dout_gt_sf : a.x_gt_sf;
          // the tile's four 32-row groups have adjacent scale bytes (k = g in the tiled layout, the
          // tile's first row a multiple of 128): one 32-bit store per column
          uint32_t sfw = 0u;
          // with biases: this column's sums of s*dout over the tile's row halves (db2's partials)
          const bool db2 = BIAS && which == 0 && a.db2_part != nullptr;
          float cs[2] = {0.f, 0.f};
#pragma unroll 2
          for (int g = 0; g < 4; ++g) {
            float c32[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int row = g * 32 + j;
              float x = bf16_bits_to_float(st[row * kPrepTilePitch + h]);
              if (SCALE_T && which == 0) x *= s_s[row];
              c32[j] = x;
              if (db2) cs[g >> 1] = fmaf(x, SCALE_T ? 1.f : s_s[row], cs[g >> 1]);
            }
            const int64_t ocol = prow0 + g * 32;
            uint32_t w[8];
            const uint32_t byte = quantize_group32_t<AF>(c32, w);
            st_global_32b(outp + orow * P + ocol, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            sfw |= byte << (8 * g);
          }
          *reinterpret_cast<uint32_t*>(outsf + sf_tiled_offset(orow, prow0, P)) = sfw;
          if (db2) {
            a.db2_part[((int64_t)tile * 2 + 0) * H + orow] = cs[0];
            a.db2_part[((int64_t)tile * 2 + 1) * H + orow] = cs[1];
          }
        }
      } else {
        const int cp = tid & 127;
        if (2 * cp < ncol && !(which == 0 && a.skip_dout_t)) {
          uint16_t* outp = static_cast<uint16_t*>(which == 0 ? a.dout_gt : a.x_gt);
          // db2: this thread's share of the tile's column sums of s*dout (its two 32-row groups)
          const bool db2 = BIAS && which == 0 && a.db2_part != nullptr;
          float cs0 = 0.f, cs1 = 0.f;
#pragma unroll 1
          for (int g = 2 * (tid >> 7); g < 2 * (tid >> 7) + 2; ++g) {
            uint32_t wv[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
              wv[j] = *reinterpret_cast<const uint32_t*>(st + (g * 32 + j) * kPrepTilePitch + 2 * cp);
            auto elem = [&](int j, int half) {  // column 2*cp + half, row g*32 + j
              float x = __uint_as_float(half ? (wv[j] & 0xFFFF0000u) : (wv[j] << 16));
              if (SCALE_T && which == 0) x *= s_s[g * 32 + j];
              return x;
            };
            if (db2) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float w = SCALE_T ? 1.f : s_s[g * 32 + j];  // s*dout (already scaled when SCALE_T)
                cs0 = fmaf(elem(j, 0), w, cs0);
                cs1 = fmaf(elem(j, 1), w, cs1);
              }
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint16_t* dst = outp + (h0 + 2 * cp + half) * P + prow0 + g * 32;
#pragma unroll
              for (int q = 0; q < 2; ++q)
                st_global_32b(dst + 16 * q, pack_bf16x2(elem(16 * q + 0, half), elem(16 * q + 1, half)),
                              pack_bf16x2(elem(16 * q + 2, half), elem(16 * q + 3, half)),
                              pack_bf16x2(elem(16 * q + 4, half), elem(16 * q + 5, half)),
                              pack_bf16x2(elem(16 * q + 6, half), elem(16 * q + 7, half)),
                              pack_bf16x2(elem(16 * q + 8, half), elem(16 * q + 9, half)),
                              pack_bf16x2(elem(16 * q + 10, half), elem(16 * q + 11, half)),
                              pack_bf16x2(elem(16 * q + 12, half), elem(16 * q + 13, half)),
                              pack_bf16x2(elem(16 * q + 14, half), elem(16 * q + 15, half)));
            }
          }
          if (db2)
            *reinterpret_cast<float2*>(a.db2_part + ((int64_t)tile * 2 + (tid >> 7)) * H + h0 + 2 * cp) =
                make_float2(cs0, cs1);
        }
      }
      __syncthreads();
    }
  }
  if constexpr (BIAS) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float v = bias_acc[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      const int row = warp + 8 * r;
      if (lane == 0) a.ds_bias[prow0 + row] = s_tok[row] >= 0 ? v : 0.f;
    }
  }
}

template <bool MX, bool SCALE_T, bool BIAS>
static int prep_launch(const PrepArgs& a, int grid, cudaStream_t st) {
  auto k = (!MX || a.fmt == MOE_FP8_E5M2) ? prep_kernel<MX, SCALE_T, BIAS, MOE_FP8_E5M2>
                                          : prep_kernel<MX, SCALE_T, BIAS, MOE_FP8_E4M3>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
  if (e != cudaSuccess) return cuda_check(e, "prep attribute");
  return launch_pdl(k, dim3(grid), dim3(256), kPrepSmem, st, "prep", a);
}

int launch_prep(const PrepArgs& a, cudaStream_t st) {
  const int grid = (int)(a.P / 128);
  if (grid == 0) return MOE_OK;
  const bool bias = a.ds_bias != nullptr;
  if (a.mx) {
    if (a.scale_t) return bias ? prep_launch<true, true, true>(a, grid, st) : prep_launch<true, true, false>(a, grid, st);
    return bias ? prep_launch<true, false, true>(a, grid, st) : prep_launch<true, false, false>(a, grid, st);
  }
  if (a.scale_t) return bias ? prep_launch<false, true, true>(a, grid, st) : prep_launch<false, true, false>(a, grid, st);
  return bias ? prep_launch<false, false, true>(a, grid, st) : prep_launch<false, false, false>(a, grid, st);
}

// ------------------------------------------------------------------------------------------
// operands from saved forward values ([N, I, B] and [N, B, H] block checkpoints)
// ------------------------------------------------------------------------------------------

// a'^T [I, P] (dW_down's token-side operand) from a feature-major block checkpoint [N, I, B] of a (or
// s*a): tile row p of expert e is slot block_offsets[e]*B + (p - tile_offsets[e]), and a tile's 128
// rows are 128 consecutive slots of one block.  Thread (feature i, 32-row group g) reads 64
// contiguous bytes, multiplies by s when SCALE, zeroes padding rows, and writes one group (bf16, or
// fp8 codes with their scale).
template <bool MX, bool SCALE, int AF>
__global__ void __launch_bounds__(256) apt_from_ckpt_kernel(const uint16_t* __restrict__ ckpt, int I, int B,
                                                            int64_t P, const int32_t* __restrict__ num_tiles,
                                                            const int32_t* __restrict__ tile_expert,
                                                            const int32_t* __restrict__ tile_offsets,
                                                            const int32_t* __restrict__ block_offsets,
                                                            const int32_t* __restrict__ tile_row_flat,
                                                            const float* __restrict__ s, void* out, uint8_t* out_sf) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int tile = blockIdx.x;
  if (tile >= *num_tiles) return;
  const int i = blockIdx.y * 64 + (threadIdx.x >> 2);
  const int g = threadIdx.x & 3;
  if (i >= I) return;
  const int e = tile_expert[tile];
  const int64_t p0 = (int64_t)tile * 128 + g * 32;
  const int64_t slot = (int64_t)block_offsets[e] * B + ((int64_t)tile * 128 - tile_offsets[e]) + g * 32;
  const int64_t blk = slot / B, b = slot - blk * B;
  const uint4* src = reinterpret_cast<const uint4*>(ckpt + (blk * I + i) * B + b);
  float v[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = src[q];
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * q + 2 * j] = __uint_as_float(ww[j] << 16);
      v[8 * q + 2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int f = tile_row_flat[p0 + r];
    if (f < 0)
      v[r] = 0.f;
    else if (SCALE)
      v[r] *= s[f];
  }
  if constexpr (MX) {
    uint32_t w[8];
    const uint32_t byte = quantize_group32_t<AF>(v, w);
    st_global_32b(static_cast<uint8_t*>(out) + (int64_t)i * P + p0, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
    out_sf[sf_tiled_offset(i, p0, P)] = (uint8_t)byte;
  } else {
    uint16_t* dst = static_cast<uint16_t*>(out) + (int64_t)i * P + p0;
    auto pk = [&](int j) { return pack_bf16x2(v[j], v[j + 1]); };
#pragma unroll
    for (int q = 0; q < 2; ++q)  // whole 32-byte sectors
      st_global_32b(dst + 16 * q, pk(16 * q), pk(16 * q + 2), pk(16 * q + 4), pk(16 * q + 6), pk(16 * q + 8),
                    pk(16 * q + 10), pk(16 * q + 12), pk(16 * q + 14));
  }
}

int launch_apt_from_ckpt(const uint16_t* ckpt, int I, int B, int64_t P, const int32_t* num_tiles,
                         const int32_t* tile_expert, const int32_t* tile_offsets, const int32_t* block_offsets,
                         const int32_t* tile_row_flat, const float* s_or_null, int mx, int fmt, void* out,
                         uint8_t* out_sf, cudaStream_t st) {
  const dim3 grid((unsigned)(P / 128), (unsigned)((I + 63) / 64));
  if (grid.x == 0) return MOE_OK;
  const bool sc = s_or_null != nullptr;
#define APT_LAUNCH(MXV, SCV, AFV)                                                                          \
  apt_from_ckpt_kernel<MXV, SCV, AFV><<<grid, 256, 0, st>>>(ckpt, I, B, P, num_tiles, tile_expert, tile_offsets, \
                                                             block_offsets, tile_row_flat, s_or_null, out, out_sf)
  if (mx) {
    if (fmt == MOE_FP8_E4M3) {
      if (sc) APT_LAUNCH(true, true, MOE_FP8_E4M3); else APT_LAUNCH(true, false, MOE_FP8_E4M3);
    } else {
      if (sc) APT_LAUNCH(true, true, MOE_FP8_E5M2); else APT_LAUNCH(true, false, MOE_FP8_E5M2);
    }
  } else {
    if (sc) APT_LAUNCH(false, true, MOE_FP8_E5M2); else APT_LAUNCH(false, false, MOE_FP8_E5M2);
  }
#undef APT_LAUNCH
  count_launch();
  return cuda_check(cudaGetLastError(), "apt_from_ckpt");
}

// Slot of every tile row in the block layout (-1 for padding rows and unused tiles).
__global__ void tile_row_slot_kernel(int64_t P, int B, const int32_t* __restrict__ num_tiles,
                                     const int32_t* __restrict__ tile_expert, const int32_t* __restrict__ tile_offsets,
                                     const int32_t* __restrict__ block_offsets,
                                     const int32_t* __restrict__ tile_row_flat, int32_t* __restrict__ slot) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= P) return;
  const int tile = (int)(p / 128);
  if (tile >= *num_tiles || tile_row_flat[p] < 0) {
    slot[p] = -1;
    return;
  }
  const int e = tile_expert[tile];
  slot[p] = (int32_t)((int64_t)block_offsets[e] * B + (p - tile_offsets[e]));
}

int launch_tile_row_slot(int64_t P, int B, const int32_t* num_tiles, const int32_t* tile_expert,
                         const int32_t* tile_offsets, const int32_t* block_offsets, const int32_t* tile_row_flat,
                         int32_t* slot, cudaStream_t st) {
  if (P == 0) return MOE_OK;
  tile_row_slot_kernel<<<(unsigned)((P + 255) / 256), 256, 0, st>>>(P, B, num_tiles, tile_expert, tile_offsets,
                                                                     block_offsets, tile_row_flat, slot);
  count_launch();
  return cuda_check(cudaGetLastError(), "tile_row_slot");
}

// Scales of a [R, C] MXFP8 operand (tiled layout, 128-row atoms) re-tiled for B tiles of `bn` rows
// (bn % 128 != 0): tile j's scales fill ceil(bn / 128) whole atoms, rows j*bn .. j*bn + bn - 1 in
// order and the rest of the last atom zero.  The four scale bytes of one row inside an atom are
// contiguous in both layouts, so each thread moves one 32-bit word.
__global__ void __launch_bounds__(256) sf_retile_kernel(const uint32_t* __restrict__ src, int64_t R, int64_t C,
                                                        int bn, int atoms, uint32_t* __restrict__ dst) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int64_t ktiles = C / 128;
  const int64_t words = (R / bn) * atoms * ktiles * 128;
  const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= words) return;
  const int r = (int)(w & 127);           // row inside the destination atom
  const int64_t a = w >> 7;               // destination atom: ((tile * atoms + h) * ktiles + kt)
  const int64_t kt = a % ktiles;
  const int64_t th = a / ktiles;
  const int h = (int)(th % atoms);
  const int64_t tile = th / atoms;
  const int tr = h * 128 + r;              // row inside the tile
  uint32_t v = 0u;
  if (tr < bn) {
    const int64_t sr = tile * bn + tr;     // source row
    v = src[(((sr >> 7) * ktiles + kt) * 512 + (sr & 31) * 16 + ((sr & 127) >> 5) * 4) >> 2];
  }
  dst[(a * 512 + (r & 31) * 16 + (r >> 5) * 4) >> 2] = v;
}

int launch_sf_retile(const uint8_t* src, int64_t R, int64_t C, int bn, uint8_t* dst, cudaStream_t st) {
  if (bn <= 0 || R % bn || R % 128 || C % 128) return fail(MOE_ERR_INVALID, "sf_retile: bad sizes");
  const int atoms = (bn + 127) / 128;
  const int64_t words = (R / bn) * atoms * (C / 128) * 128;
  if (words == 0) return MOE_OK;
  return launch_pdl(sf_retile_kernel, dim3((unsigned)((words + 255) / 256)), dim3(256), 0, st, "sf_retile",
                    reinterpret_cast<const uint32_t*>(src), R, C, bn, atoms, reinterpret_cast<uint32_t*>(dst));
}

// ------------------------------------------------------------------------------------------
// generic quantisers
// ------------------------------------------------------------------------------------------

// Row-wise: 8 elements per thread, 4 threads per 32-group.
__global__ void __launch_bounds__(256) quant_rowwise_kernel(const uint16_t* __restrict__ in, int64_t src_rows,
                                                            int64_t rows, int64_t cols, int64_t ld,
                                                            const int32_t* __restrict__ row_index, int fmt,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                            int tiled) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int64_t vpr = cols / 8;
  const int64_t total = rows * vpr;
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x - lane; base < total; base += stride) {
    const int64_t idx = base + lane;
    const bool in_range = idx < total;
    const int64_t r = in_range ? idx / vpr : 0;
    const int64_t c = in_range ? (idx - r * vpr) * 8 : 0;
    int64_t sr = r;
    if (row_index) sr = in_range ? row_index[r] : -1;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (in_range && sr >= 0 && sr < src_rows) v = *reinterpret_cast<const uint4*>(in + sr * ld + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float d[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      d[2 * j] = __uint_as_float(w[j] << 16);
      d[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    float am = amax_tree<8>(d);
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    if (!in_range) continue;
    const uint32_t byte = e8m0_byte(__float_as_uint(am), fmt);
    const float inv = e8m0_inv_scale(byte);
    uint2 o;
    o.x = fp8x4(d[0] * inv, d[1] * inv, d[2] * inv, d[3] * inv, fmt);
    o.y = fp8x4(d[4] * inv, d[5] * inv, d[6] * inv, d[7] * inv, fmt);
    *reinterpret_cast<uint2*>(q + r * cols + c) = o;
    if (sf && ((c >> 3) & 3) == 0) sf[tiled ? sf_tiled_offset(r, c, cols) : r * (cols / 32) + c / 32] = (uint8_t)byte;
  }
}

// Column-wise: a CTA stages a 128-row x 64-column tile, then each thread writes one 32-row group of
// one column into the transposed output [cols, rows] (fp8 + scale, or bf16).
template <bool MX>
__global__ void __launch_bounds__(256) quant_colwise_kernel(const uint16_t* __restrict__ in, int64_t src_rows,
                                                            int64_t rows, int64_t cols, int64_t ld,
                                                            const int32_t* __restrict__ row_index, int fmt,
                                                            void* __restrict__ q, uint8_t* __restrict__ sf,
                                                            int tiled) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  __shared__ uint16_t tile[128 * kPrepPitch];
  const int tid = threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.x * 128;
  const int64_t c0 = (int64_t)blockIdx.y * 64;
  const int vec = tid & 7;
#pragma unroll
  for (int r4 = 0; r4 < 4; ++r4) {
    const int row = (tid >> 3) + 32 * r4;
    const int64_t r = r0 + row;
    const int64_t c = c0 + vec * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows && c < cols) {
      const int64_t sr = row_index ? row_index[r] : r;
      if (sr >= 0 && sr < src_rows) v = *reinterpret_cast<const uint4*>(in + sr * ld + c);
    }
    uint32_t* tw = reinterpret_cast<uint32_t*>(tile + row * kPrepPitch + vec * 8);
    tw[0] = v.x; tw[1] = v.y; tw[2] = v.z; tw[3] = v.w;
  }
  __syncthreads();
  const int h = tid & 63;
  const int g = tid >> 6;
  const int64_t oc = c0 + h;          // output row = input column
  const int64_t orr = r0 + g * 32;    // first output column = input row
  if (oc >= cols || orr >= rows) return;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = bf16_bits_to_float(tile[(g * 32 + j) * kPrepPitch + h]);
  if constexpr (MX) {
    uint32_t w[8];
    const uint32_t byte = quantize_group32(v, fmt, w);
    st_global_32b_or_halves(static_cast<uint8_t*>(q) + oc * rows + orr, w[0], w[1], w[2], w[3], w[4], w[5], w[6],
                            w[7]);
    sf[tiled ? sf_tiled_offset(oc, orr, rows) : oc * (rows / 32) + orr / 32] = (uint8_t)byte;
  } else {
    uint16_t* dst = static_cast<uint16_t*>(q) + oc * rows + orr;
    auto pk = [&](int j) { return pack_bf16x2(v[j], v[j + 1]); };
#pragma unroll
    for (int k = 0; k < 2; ++k)  // whole 32-byte sectors (q is caller-owned: 16-byte alignment)
      st_global_32b_or_halves(dst + 16 * k, pk(16 * k), pk(16 * k + 2), pk(16 * k + 4), pk(16 * k + 6), pk(16 * k + 8),
                    pk(16 * k + 10), pk(16 * k + 12), pk(16 * k + 14));
  }
}

int launch_quant_rowwise(const uint16_t* in, int64_t src_rows, int64_t rows, int64_t cols, int64_t ld,
                         const int32_t* row_index, int fmt, uint8_t* q, uint8_t* sf, int tiled, cudaStream_t st) {
  const int64_t total = rows * (cols / 8);
  if (total == 0) return MOE_OK;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(quant_rowwise_kernel, dim3((unsigned)blocks), dim3(256), 0, st, "quant_rowwise", in, src_rows, rows,
                    cols, ld, row_index, fmt, q, sf, tiled);
}

int launch_quant_colwise(const uint16_t* in, int64_t src_rows, int64_t rows, int64_t cols, int64_t ld,
                         const int32_t* row_index, int mx, int fmt, void* q, uint8_t* sf, int tiled, cudaStream_t st) {
  if (rows == 0 || cols == 0) return MOE_OK;
  dim3 grid((unsigned)((rows + 127) / 128), (unsigned)((cols + 63) / 64));
  if (mx)
    quant_colwise_kernel<true><<<grid, 256, 0, st>>>(in, src_rows, rows, cols, ld, row_index, fmt, q, sf, tiled);
  else
    quant_colwise_kernel<false><<<grid, 256, 0, st>>>(in, src_rows, rows, cols, ld, row_index, fmt, q, sf, tiled);
  count_launch();
  return cuda_check(cudaGetLastError(), "quant_colwise");
}

}  // namespace moebwd

using namespace moebwd;

extern "C" int mxfp8_quantize(const void* in, int64_t src_rows, int64_t rows, int64_t cols, int64_t ld,
                              const int32_t* row_index, int axis, int fp8_fmt, uint8_t* q, uint8_t* scales,
                              int scale_layout, moe_stream_t stream) {
  clear_error();
  if (!in || !q || !scales) return fail(MOE_ERR_INVALID, "mxfp8_quantize: null pointer");
  if (rows < 0 || cols < 0 || src_rows < 0) return fail(MOE_ERR_INVALID, "mxfp8_quantize: negative size");
  if (ld < cols || ld % 8 != 0) return fail(MOE_ERR_INVALID, "mxfp8_quantize: ld must be >= cols and a multiple of 8");
  if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(q) & 15))
    return fail(MOE_ERR_INVALID, "mxfp8_quantize: in and q must be 16-byte aligned");
  if (fp8_fmt != MOE_FP8_E4M3 && fp8_fmt != MOE_FP8_E5M2) return fail(MOE_ERR_INVALID, "mxfp8_quantize: bad fp8_fmt");
  if (scale_layout != MOE_SF_PLAIN && scale_layout != MOE_SF_TILED)
    return fail(MOE_ERR_INVALID, "mxfp8_quantize: bad scale_layout");
  if (!row_index && rows > src_rows) return fail(MOE_ERR_INVALID, "mxfp8_quantize: rows > src_rows without row_index");
  const int tiled = scale_layout == MOE_SF_TILED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (axis == MOE_QUANT_ROWWISE) {
    if (cols % 32) return fail(MOE_ERR_UNSUPPORTED, "mxfp8_quantize: cols must be a multiple of 32 (rowwise)");
    if (tiled && (rows % 128 || cols % 128))
      return fail(MOE_ERR_UNSUPPORTED, "mxfp8_quantize: tiled scales need rows, cols multiples of 128");
    return launch_quant_rowwise(static_cast<const uint16_t*>(in), src_rows, rows, cols, ld, row_index, fp8_fmt, q,
                                scales, tiled, st);
  }
  if (axis == MOE_QUANT_COLWISE) {
    if (rows % 32) return fail(MOE_ERR_UNSUPPORTED, "mxfp8_quantize: rows must be a multiple of 32 (colwise)");
    if (cols % 8) return fail(MOE_ERR_UNSUPPORTED, "mxfp8_quantize: cols must be a multiple of 8 (colwise)");
    if (reinterpret_cast<uintptr_t>(q) & 15 || rows % 16)
      return fail(MOE_ERR_UNSUPPORTED, "mxfp8_quantize: colwise output rows must be 16-byte aligned");
    if (tiled && (rows % 128 || cols % 128))
      return fail(MOE_ERR_UNSUPPORTED, "mxfp8_quantize: tiled scales need rows, cols multiples of 128");
    return launch_quant_colwise(static_cast<const uint16_t*>(in), src_rows, rows, cols, ld, row_index, 1, fp8_fmt, q,
                                scales, tiled, st);
  }
  return fail(MOE_ERR_INVALID, "mxfp8_quantize: bad axis");
}
