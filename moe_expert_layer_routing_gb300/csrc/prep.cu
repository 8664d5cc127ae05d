// Operand preparation for the grouped GEMMs, and the public mxfp8_quantize.
//
// prep_kernel (persistent; 128-row tiles of the tile-row space, H walked in 128-column chunks)
// gathers the token rows of every routed (t, k) once and writes, in one pass over dout and x:
//   dout_g  [P, H]  gathered dout rows                      (G1 A operand, groups along H; when G1
//                   gathers its rows itself, nothing for BF16 and only the tiled scales for MXFP8)
//   dout_gt [H, P]  gathered dout transposed, s-scaled for affinity on H (G3 B operand)
//   x_gt    [H, P]  gathered x transposed                   (G4 A operand)
//   ds_bias [P]     <dout_t, b2_e>, the bias term of ds      (sonic-moe db2_and_ds_kernel)
// as BF16, or as MXFP8 with E8M0 scales in the tiled layout (transposed operands are quantised
// in groups of 32 tile rows, i.e. along the GEMM contraction).  Padding rows are zero.  When the
// gate/up pre-activations are recomputed, a row-major gathered x [P,H] (G0's A operand) is written too.
// BF16 whose weight-gradient GEMMs read MN-major operands (no_t): no transposed outputs; x's gathered
// rows go to x_g and, where the dW2 GEMM cannot read dout_g itself, dout (or s*dout) rows to dout_b.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "moebwd_internal.h"
#include "mx_device.cuh"
#include "ptx.cuh"

namespace moebwd {

constexpr int kPrepPitch = 66;       // bf16 row pitch of the 64-column tiles of the generic quantiser
// ---- MoE prep kernel ----
// Persistent CTAs (two per SM) walk work items: a whole tile (128 tile rows x all of H) when the bias
// term of ds is wanted (its row dot products span H), else one 128-column chunk of a tile.  An item
// is a sequence of units, one per chunk and tensor (dout when anything is built from it, then x);
// a unit's [128 rows x 128 columns] bf16 tile is gathered by cp.async (16-byte pieces, padding rows
// zero-filled) into one of two shared buffers one unit ahead, so the gather of unit u+1 overlaps
// the quantisation of unit u.  Per unit:
//   phase A (dout; x too when h is recomputed): each thread quantises the 16-byte pieces of eight
//     rows row-wise (MXFP8 groups of 32 columns = 4 lanes) into the row-major copy and its scales,
//     and accumulates the rows' dot products with b2;
//     (no_t: also the dout_b rows and db2's per-tile column sums: lane pairs, then eight warps through
//     shared memory);
//   phase B (not with no_t): thread (column pair, 32-row quarter) reads 32 words, quantises (MXFP8) or
//     rounds (BF16) the two transposed 32-element groups — MXFP8 into a staging tile in the 128-byte
//     swizzled layout of the output's tensor map (16-byte piece c of staging row r at
//     r * 128 + ((c ^ (r % 8)) * 16)), written by one elected thread's tiled bulk stores, its scale
//     bytes into one staged 512-byte atom of the tiled layout written by a plain bulk copy; BF16 as
//     whole 32-byte sectors straight to global memory — and adds db2's quarter sums.
// Rows and tokens: tile row p holds flat index f = tile_row_flat[p] (token f / K, or padding when
// f < 0); the divide is a multiply by a constant from the host.
constexpr int kPrepCols = 128;                       // H columns per unit
constexpr int kPrepTilePitch = 136;                  // bf16 row pitch of a unit tile (272 B: 16-B aligned,
                                                     // consecutive rows four banks apart)
constexpr int kPrepTile = 128 * kPrepTilePitch * 2;  // bytes of one unit buffer
// MXFP8 staging: two buffers (by unit parity) of a unit's transposed fp8 codes (16 KB) and its scale
// atom (512 B), 17 KB apart.  (BF16 writes its transposed rows directly: 64 contiguous bytes per
// output row and group.)
constexpr int kPrepStageMx = 128 * 128;
constexpr int kPrepStageMxStride = 17 * 1024;
template <bool MX>
constexpr int prep_smem_bytes() {  // 1024-byte alignment slack, staging (MXFP8) or the column-sum scratch
                                   // (BF16), two unit buffers, s and b2 per buffer
  return 1024 + (MX ? 2 * kPrepStageMxStride : 8 * 128 * 4) + 2 * kPrepTile + 2 * 128 * 4 + 2 * 128 * 2;
}

__device__ __forceinline__ int prep_token(const PrepArgs& a, int f) {
  if (f < 0) return -1;
  return a.k_shift == 0 ? f : (int)(__umulhi((uint32_t)f, a.k_mul) >> (a.k_shift - 1));
}

template <bool MX, bool SCALE_T, bool BIAS, int AF>
__global__ void __launch_bounds__(256, 2)
    prep_kernel(const PrepArgs a, const __grid_constant__ CUtensorMap tm_dout_gt,
                const __grid_constant__ CUtensorMap tm_x_gt) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int H = a.H, nch = H / kPrepCols;
  const int64_t P = a.P;
  const int ntiles = *a.num_tiles;
  const int nitems = BIAS ? ntiles : ntiles * nch;
  if ((int)blockIdx.x >= nitems) return;
  extern __shared__ uint4 prep_smem[];
  uint8_t* const stage0 =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(prep_smem) + 1023) & ~uintptr_t(1023));
  uint16_t* const tiles = reinterpret_cast<uint16_t*>(stage0 + (MX ? 2 * kPrepStageMxStride : 8 * 128 * 4));
  float* const colred = reinterpret_cast<float*>(stage0);  // BF16: [8 warps][128] column partial sums
  float* const s_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tiles) + 2 * kPrepTile);  // [2][128]
  uint16_t* const s_b2 = reinterpret_cast<uint16_t*>(s_s + 2 * 128);                                 // [2][128]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rl = tid >> 4;  // this thread gathers and row-quantises rows rl + 16k (k < 8) of a unit ...
  const int pc = tid & 15;  // ... their 16-byte piece pc (columns 8pc .. 8pc+7 of the chunk)
  const bool need_s = SCALE_T || (BIAS && a.db2_part != nullptr);  // s per tile row in dout's phase B
  const bool dout_t = !a.skip_dout_t && !a.no_t;
  const bool dout_rows = MX || a.dout_g != nullptr || BIAS || a.dout_b != nullptr;  // phase A has work on dout
  const bool db2_rows = !MX && BIAS && a.no_t && a.db2_part != nullptr;  // db2's partials in phase A
  const int nw = (dout_t || dout_rows) ? 2 : 1;             // units per chunk: dout (if any work), x
  const int nu = (BIAS ? nch : 1) * nw;                      // units per item
  const int G = (int)gridDim.x;
  // item it -> (tile list index ti, first chunk c), chunk-major without biases (it = c * ntiles + ti:
  // the items in flight are one chunk of consecutive tiles of the token-ordered schedule, so the K
  // gathers of a token's row segment come close together and hit L2); the CTA's items are it, it + G, ...
  const int dgi = BIAS ? G : G % ntiles, dgc = BIAS ? 0 : G / ntiles;
  auto next_item = [&](int& it, int& ti, int& c) {
    it += G;
    ti += dgi;
    c += dgc;
    if (!BIAS && ti >= ntiles) {
      ti -= ntiles;
      ++c;
    }
  };
  auto tile_of = [&](int ti) { return a.tile_order ? a.tile_order[ti] : ti; };

  // loader: item l_* (tokens lt[], the flat index l_fs of row rl + 16pc for s, expert l_e), unit l_j;
  // the next item p_* has its flat indices pf[] and expert in flight; the tile of the one after, q_tile
  int l_it = (int)blockIdx.x, l_ti = BIAS ? l_it : l_it % ntiles, l_c = BIAS ? 0 : l_it / ntiles;
  int l_tile = tile_of(l_ti), l_e = 0, l_fs = -1, l_j = 0;
  int lt[8], pf[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) pf[k] = a.tile_row_flat[(int64_t)l_tile * 128 + rl + 16 * k];
  if (BIAS) l_e = a.tile_expert[l_tile];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    lt[k] = prep_token(a, pf[k]);
    if (k == pc) l_fs = pf[k];
  }
  int p_it = l_it, p_ti = l_ti, p_c = l_c;
  next_item(p_it, p_ti, p_c);
  int p_tile = p_it < nitems ? tile_of(p_ti) : 0, p_e = 0;
  if (p_it < nitems) {
#pragma unroll
    for (int k = 0; k < 8; ++k) pf[k] = a.tile_row_flat[(int64_t)p_tile * 128 + rl + 16 * k];
    if (BIAS) p_e = a.tile_expert[p_tile];
  }
  int q_tile = 0;
  {
    int q_it = p_it, q_ti = p_ti, q_c = p_c;
    next_item(q_it, q_ti, q_c);
    if (q_it < nitems) q_tile = tile_of(q_ti);
  }

  // gathers unit (chunk c, tensor w) of the loader's item into buffer b
  auto issue = [&](int b, int c, int w) {
    const uint16_t* src = w == 0 ? a.dout : a.x;
    const uint32_t dst = smem_u32(tiles + b * (128 * kPrepTilePitch) + rl * kPrepTilePitch + pc * 8);
    const int col = c * kPrepCols + pc * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const bool ok = lt[k] >= 0;
      cp_async_16_zfill(dst + k * 16 * kPrepTilePitch * 2, ok ? src + (int64_t)lt[k] * H + col : src,
                        ok ? 16u : 0u);
    }
    if (w == 0) {
      if (need_s && pc < 8)
        cp_async_4_zfill(smem_u32(s_s + b * 128 + rl + 16 * pc), l_fs >= 0 ? a.s + l_fs : a.s, l_fs >= 0 ? 4u : 0u);
      if (BIAS && tid < 16)
        cp_async_16(smem_u32(s_b2 + b * 128 + tid * 8), a.b2 + (int64_t)l_e * H + c * kPrepCols + tid * 8);
    }
    cp_async_commit();
  };

  float bias_acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) bias_acc[k] = 0.f;
  // the unit being processed (tile, chunk, tensor) and the one gathered ahead of it
  int cur_tile = l_tile, cur_c = l_c, cur_w = nw == 2 ? 0 : 1;
  issue(0, cur_c, cur_w);
  int buf = 0;
  while (true) {
    // ---- advance the loader one unit and gather it into the other buffer ----
    int nx_tile = 0, nx_c = 0, nx_w = 0;
    bool has_next = true;
    if (++l_j == nu) {  // next item: its tokens were fetched one item ago
      l_j = 0;
      l_it = p_it;
      l_ti = p_ti;
      l_c = p_c;
      has_next = l_it < nitems;
      if (has_next) {
        l_tile = p_tile;
        l_e = p_e;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          lt[k] = prep_token(a, pf[k]);
          if (k == pc) l_fs = pf[k];
        }
        next_item(p_it, p_ti, p_c);
        p_tile = q_tile;
        if (p_it < nitems) {
#pragma unroll
          for (int k = 0; k < 8; ++k) pf[k] = a.tile_row_flat[(int64_t)p_tile * 128 + rl + 16 * k];
          if (BIAS) p_e = a.tile_expert[p_tile];
          int q_it = p_it, q_ti = p_ti, q_c = p_c;
          next_item(q_it, q_ti, q_c);
          if (q_it < nitems) q_tile = tile_of(q_ti);
        }
      }
    }
    if (has_next) {
      nx_tile = l_tile;
      nx_c = l_c + (nw == 2 ? l_j >> 1 : l_j);
      nx_w = nw == 2 ? (l_j & 1) : 1;
      issue(buf ^ 1, nx_c, nx_w);
      cp_async_wait<1>();  // this thread's pieces of the current unit have landed
    } else {
      cp_async_wait<0>();
    }
    // MXFP8: the staging buffer of this unit's parity was last read by the stores of unit u - 2
    if (MX && tid == 0) bulk_wait_read<1>();
    __syncthreads();  // everyone's pieces of the current unit are in
    uint8_t* const stage = stage0 + (MX ? buf * kPrepStageMxStride : 0);
    uint8_t* const stage_sf = stage + kPrepStageMx;  // MXFP8

    const uint16_t* tb = tiles + buf * (128 * kPrepTilePitch);
    const int64_t prow0 = (int64_t)cur_tile * 128;
    // ---- phase A: row-major copy (codes and scales) and the rows' dot products with b2 ----
    if (cur_w == 0 ? dout_rows : a.x_g != nullptr) {
      void* rowdst = cur_w == 0 ? a.dout_g : a.x_g;
      uint8_t* rowsf = cur_w == 0 ? a.dout_g_sf : a.x_g_sf;
      const int col = cur_c * kPrepCols + pc * 8;
      uint4 bv = make_uint4(0, 0, 0, 0);
      if (BIAS && cur_w == 0) bv = *reinterpret_cast<const uint4*>(s_b2 + buf * 128 + pc * 8);
      // scale of row prow0 + rl + 16k, columns col.. (a 128-aligned tile): atom (tile, chunk), byte
      // (rl + 16 (k % 2)) * 16 + (k / 2) * 4 + pc / 4
      uint8_t* const sfrow = MX ? rowsf + ((int64_t)cur_tile * (H >> 7) + cur_c) * 512 + rl * 16 + (pc >> 2) : nullptr;
      float cs8[8];  // db2_rows: this thread's column sums of s*dout over its eight rows
#pragma unroll
      for (int j = 0; j < 8; ++j) cs8[j] = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t prow = prow0 + rl + 16 * k;
        const uint4 v = *reinterpret_cast<const uint4*>(tb + (rl + 16 * k) * kPrepTilePitch + pc * 8);
        const uint32_t dw[4] = {v.x, v.y, v.z, v.w};
        float d8[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          d8[2 * j] = __uint_as_float(dw[j] << 16);
          d8[2 * j + 1] = __uint_as_float(dw[j] & 0xFFFF0000u);
        }
        if (BIAS && cur_w == 0) {
          const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            bias_acc[k] = fmaf(d8[2 * j], __uint_as_float(bw[j] << 16), bias_acc[k]);
            bias_acc[k] = fmaf(d8[2 * j + 1], __uint_as_float(bw[j] & 0xFFFF0000u), bias_acc[k]);
          }
        }
        if constexpr (MX) {
          float am = amax_tree<8>(d8);
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
          const uint32_t byte = e8m0_byte(__float_as_uint(am), AF);
          if (rowdst) {  // no codes when G1 gathers its rows from dout quantised per token
            const float inv = e8m0_inv_scale(byte);
            uint2 q;
            q.x = fp8x4_t<AF>(d8[0] * inv, d8[1] * inv, d8[2] * inv, d8[3] * inv);
            q.y = fp8x4_t<AF>(d8[4] * inv, d8[5] * inv, d8[6] * inv, d8[7] * inv);
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(rowdst) + prow * H + col) = q;
          }
          if ((lane & 3) == 0) sfrow[(k & 1) * 256 + (k >> 1) * 4] = (uint8_t)byte;
        } else {
          if (rowdst) *reinterpret_cast<uint4*>(static_cast<uint16_t*>(rowdst) + prow * H + col) = v;
          if (cur_w == 0 && (a.dout_b || db2_rows)) {
            const float sr = s_s[buf * 128 + rl + 16 * k];
            if (a.dout_b) {  // the dW2 GEMM's B rows: s*dout in fp32, rounded (dout_b_s), else dout
              uint4 o = v;
              if (SCALE_T && a.dout_b_s)
                o = make_uint4(pack_bf16x2(d8[0] * sr, d8[1] * sr), pack_bf16x2(d8[2] * sr, d8[3] * sr),
                               pack_bf16x2(d8[4] * sr, d8[5] * sr), pack_bf16x2(d8[6] * sr, d8[7] * sr));
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dout_b) + prow * H + col) = o;
            }
            if (db2_rows) {
#pragma unroll
              for (int j = 0; j < 8; ++j) cs8[j] = fmaf(d8[j], sr, cs8[j]);
            }
          }
        }
      }
      if (db2_rows && cur_w == 0) {  // the tile's column sums of s*dout: lane pairs, then the eight warps
#pragma unroll
        for (int j = 0; j < 8; ++j) cs8[j] += __shfl_xor_sync(0xffffffffu, cs8[j], 16);
        if (lane < 16) {
#pragma unroll
          for (int j = 0; j < 8; ++j) colred[warp * 128 + pc * 8 + j] = cs8[j];
        }
        __syncthreads();
        if (tid < 128) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < 8; ++w) v += colred[w * 128 + tid];
          a.db2_part[(int64_t)cur_tile * H + cur_c * kPrepCols + tid] = v;
        }
      }
      if (BIAS && cur_w == 0 && cur_c == nch - 1) {  // the tile's last chunk: ds_bias of its rows
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float v = bias_acc[k];
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          // (the loader is still in this item: lt[] are this tile's tokens; padding rows give 0)
          if (pc == 0) a.ds_bias[prow0 + rl + 16 * k] = lt[k] >= 0 ? v : 0.f;
          bias_acc[k] = 0.f;
        }
      }
    }
    // ---- phase B: the transposed output through the staging tile ----
    const bool do_t = cur_w == 1 ? !a.no_t : dout_t;
    if (do_t) {
      const int cp = tid & 63, g = tid >> 6;  // columns 2cp, 2cp+1; tile rows 32g .. 32g+31
      const bool db2 = BIAS && cur_w == 0 && a.db2_part != nullptr;
      const float* ss = s_s + buf * 128 + g * 32;
      uint32_t wv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        wv[j] = *reinterpret_cast<const uint32_t*>(tb + (g * 32 + j) * kPrepTilePitch + 2 * cp);
      // lanes with bit 2 of cp set write the two halves of a row's piece pair in the other order: with
      // the swizzle, a warp's 32 16-byte stores of one instruction then cover all eight pieces of a
      // 128-byte row position four times (no bank conflict)
      const int flip = (cp >> 2) & 1;
      // MXFP8 without the s factor: both columns' amax from the packed words
      uint32_t am2 = 0u;
      if (MX && !(SCALE_T && cur_w == 0)) am2 = bf16x2_absmax32(wv);
      float cs[2] = {0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 2; ++q) {  // column 2cp + q = staging row r
        float c32[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float x = __uint_as_float(q ? (wv[j] & 0xFFFF0000u) : (wv[j] << 16));
          if (SCALE_T && cur_w == 0) x *= ss[j];
          c32[j] = x;
          if (db2) cs[q] = fmaf(x, SCALE_T ? 1.f : ss[j], cs[q]);
        }
        const int r = 2 * cp + q;
        if constexpr (MX) {
          uint32_t w8[8];
          const uint32_t byte = (SCALE_T && cur_w == 0) ? quantize_group32_t<AF>(c32, w8)
                                                        : quantize_group32_am<AF>(c32, q ? am2 & 0xFFFF0000u : am2 << 16, w8);
          uint8_t* rowp = stage + r * 128;  // tile rows 32g.. are bytes 32g.. of the row: pieces 2g, 2g+1
          const uint4 lo = make_uint4(w8[0], w8[1], w8[2], w8[3]), hi = make_uint4(w8[4], w8[5], w8[6], w8[7]);
          *reinterpret_cast<uint4*>(rowp + (((2 * g + flip) ^ (r & 7)) << 4)) = flip ? hi : lo;
          *reinterpret_cast<uint4*>(rowp + (((2 * g + 1 - flip) ^ (r & 7)) << 4)) = flip ? lo : hi;
          // scale byte (row r of the chunk's atom, k-group g: the tile's first row is a multiple of 128)
          stage_sf[(r & 31) * 16 + (r >> 5) * 4 + g] = (uint8_t)byte;
        } else {
          // BF16: the group's 64 bytes of output row h straight to global memory, two whole sectors
          uint16_t* dst = static_cast<uint16_t*>(cur_w == 0 ? a.dout_gt : a.x_gt) +
                          ((int64_t)cur_c * kPrepCols + r) * P + prow0 + g * 32;
#pragma unroll
          for (int hq = 0; hq < 2; ++hq)
            st_global_32b(dst + 16 * hq, pack_bf16x2(c32[16 * hq + 0], c32[16 * hq + 1]),
                          pack_bf16x2(c32[16 * hq + 2], c32[16 * hq + 3]), pack_bf16x2(c32[16 * hq + 4], c32[16 * hq + 5]),
                          pack_bf16x2(c32[16 * hq + 6], c32[16 * hq + 7]), pack_bf16x2(c32[16 * hq + 8], c32[16 * hq + 9]),
                          pack_bf16x2(c32[16 * hq + 10], c32[16 * hq + 11]),
                          pack_bf16x2(c32[16 * hq + 12], c32[16 * hq + 13]),
                          pack_bf16x2(c32[16 * hq + 14], c32[16 * hq + 15]));
        }
      }
      if (db2)
        *reinterpret_cast<float2*>(a.db2_part + ((int64_t)cur_tile * 4 + g) * H + cur_c * kPrepCols + 2 * cp) =
            make_float2(cs[0], cs[1]);
    }
    if (MX) fence_proxy_async_smem();  // staged bytes are read by the bulk copies (async proxy)
    __syncthreads();                    // phase A and B reads of the buffer, and the staging writes, are done
    if (MX && do_t && tid == 0) {
      const void* tm = cur_w == 0 ? static_cast<const void*>(&tm_dout_gt) : static_cast<const void*>(&tm_x_gt);
      tma_store_2d(tm, stage, (int)prow0, cur_c * kPrepCols);
      uint8_t* outsf = cur_w == 0 ? a.dout_gt_sf : a.x_gt_sf;
      bulk_store(outsf + ((int64_t)cur_c * (P >> 7) + cur_tile) * 512, stage_sf, 512);
      bulk_commit();
    }
    if (!has_next) break;
    cur_tile = nx_tile;
    cur_c = nx_c;
    cur_w = nx_w;
    buf ^= 1;
  }
  if (MX && tid == 0) bulk_wait_all();  // the last bulk stores complete before the CTA exits
}

template <bool MX, bool SCALE_T, bool BIAS>
static int prep_launch(const PrepArgs& a, int grid, cudaStream_t st) {
  auto k = (!MX || a.fmt == MOE_FP8_E5M2) ? prep_kernel<MX, SCALE_T, BIAS, MOE_FP8_E5M2>
                                          : prep_kernel<MX, SCALE_T, BIAS, MOE_FP8_E4M3>;
  // MXFP8: tensor maps of the transposed [H, P] code matrices, boxes of 128 rows x 128 bytes, 128-byte swizzle
  alignas(64) CUtensorMap tm_dgt, tm_xgt;
  std::memset(&tm_dgt, 0, sizeof(tm_dgt));
  std::memset(&tm_xgt, 0, sizeof(tm_xgt));
  if (MX) {
    if (!a.skip_dout_t &&
        !make_tmap_2d(&tm_dgt, a.dout_gt, 1, (uint64_t)a.H, (uint64_t)a.P, (uint64_t)a.P, 128, 128, true))
      return MOE_ERR_INVALID;
    if (!make_tmap_2d(&tm_xgt, a.x_gt, 1, (uint64_t)a.H, (uint64_t)a.P, (uint64_t)a.P, 128, 128, true))
      return MOE_ERR_INVALID;
  }
  const int smem = prep_smem_bytes<MX>();
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_check(e, "prep attribute");
  return launch_pdl(k, dim3(grid), dim3(256), smem, st, "prep", a, tm_dgt, tm_xgt);
}

int launch_prep(const PrepArgs& args, cudaStream_t st) {
  const int64_t tiles = args.P / 128;
  if (tiles == 0) return MOE_OK;
  PrepArgs a = args;
  // f / K for 0 <= f < 2^31: with l = ceil(log2 K) and m = ceil(2^(31+l) / K) (< 2^32), the quotient
  // is floor(f m / 2^(31+l)): m K - 2^(31+l) < K <= 2^l keeps the error term below 1/K
  int l = 0;
  while ((1ll << l) < a.K) ++l;
  a.k_shift = l;
  a.k_mul = l == 0 ? 0u : (uint32_t)(((1ull << (31 + l)) + (uint64_t)a.K - 1) / (uint64_t)a.K);
  const bool bias = a.ds_bias != nullptr;
  const int64_t items = bias ? tiles : tiles * (a.H / kPrepCols);
  const int grid = (int)std::min<int64_t>(items, 2 * (int64_t)device_sm_count());
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

// Row-wise: one warp per row (rows strided over the grid's warps); a lane takes 16-byte pieces lane,
// lane + 32, ... of the row, two at a time, so an aligned quad of lanes holds each 32-column group.
// sf may be null (codes only: the per-token dout codes whose gathered scales prep writes).
__device__ __forceinline__ uint2 quant_piece(const uint4 v, int fmt, uint32_t& byte) {
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
  byte = e8m0_byte(__float_as_uint(am), fmt);
  const float inv = e8m0_inv_scale(byte);
  return make_uint2(fp8x4(d[0] * inv, d[1] * inv, d[2] * inv, d[3] * inv, fmt),
                    fp8x4(d[4] * inv, d[5] * inv, d[6] * inv, d[7] * inv, fmt));
}

__global__ void __launch_bounds__(256) quant_rowwise_kernel(const uint16_t* __restrict__ in, int64_t src_rows,
                                                            int64_t rows, int64_t cols, int64_t ld,
                                                            const int32_t* __restrict__ row_index, int fmt,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                            int tiled) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t pieces = cols >> 3;  // a multiple of 4: cols is a multiple of 32
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nw) {
    const int64_t sr = row_index ? row_index[r] : r;
    const bool have = sr >= 0 && sr < src_rows;
    const uint4* src = reinterpret_cast<const uint4*>(in + (have ? sr : 0) * ld);
    uint8_t* dst = q + r * cols;
    for (int64_t p0 = lane; p0 - lane < pieces; p0 += 64) {  // warp-uniform: every lane reaches the shuffles
      const int64_t p1 = p0 + 32;
      const uint4 z = make_uint4(0, 0, 0, 0);
      const uint4 v0 = (have && p0 < pieces) ? src[p0] : z;
      const uint4 v1 = (have && p1 < pieces) ? src[p1] : z;
      uint32_t b0, b1;
      const uint2 o0 = quant_piece(v0, fmt, b0);
      const uint2 o1 = quant_piece(v1, fmt, b1);
      if (p0 < pieces) {
        *reinterpret_cast<uint2*>(dst + 8 * p0) = o0;
        if (sf && (p0 & 3) == 0) sf[tiled ? sf_tiled_offset(r, 8 * p0, cols) : r * (cols / 32) + p0 / 4] = (uint8_t)b0;
      }
      if (p1 < pieces) {
        *reinterpret_cast<uint2*>(dst + 8 * p1) = o1;
        if (sf && (p1 & 3) == 0) sf[tiled ? sf_tiled_offset(r, 8 * p1, cols) : r * (cols / 32) + p1 / 4] = (uint8_t)b1;
      }
    }
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
  if (rows == 0 || cols == 0) return MOE_OK;
  int64_t blocks = (rows + 7) / 8;  // eight warps (rows) per block
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
  if (rows < 0 || cols < 0 || src_rows < 0) return fail(MOE_ERR_INVALID, "mxfp8_quantize: negative size");
  if (axis != MOE_QUANT_ROWWISE && axis != MOE_QUANT_COLWISE) return fail(MOE_ERR_INVALID, "mxfp8_quantize: bad axis");
  if (rows == 0 || cols == 0) return MOE_OK;  // nothing to write (the pointers may be null)
  if (!in || !q || !scales) return fail(MOE_ERR_INVALID, "mxfp8_quantize: null pointer");
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
