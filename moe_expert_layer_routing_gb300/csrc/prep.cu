// Operand preparation for the grouped GEMMs, and the public mxfp8_quantize.
//
// prep_kernel (one CTA per 128-row tile of the tile-row space, H walked in 64-column chunks)
// gathers the token rows of every routed (t, k) once and writes, in one pass over dout and x:
//   dout_g  [P, H]  gathered dout rows                      (G1 A operand, groups along H)
//   dout_gt [H, P]  gathered dout transposed, s-scaled for affinity on H (G3 B operand)
//   x_gt    [H, P]  gathered x transposed                   (G4 A operand)
//   ds_bias [P]     <dout_t, b2_e>, the bias term of ds      (sonic-moe db2_and_ds_kernel)
// as BF16, or as MXFP8 with E8M0 scales in the tiled layout (transposed operands are quantised
// in groups of 32 tile rows, i.e. along the GEMM contraction).  Padding rows are zero.
#include <cuda_runtime.h>

#include "moebwd_internal.h"
#include "mx_device.cuh"

namespace moebwd {

constexpr int kPrepChunk = 64;   // H columns per step
constexpr int kPrepPitch = 66;   // bf16 row pitch of the shared-memory tiles (bank-conflict free)

template <bool MX, bool SCALE_T, bool BIAS>
__global__ void __launch_bounds__(256) prep_kernel(const PrepArgs a) {
  const int tile = blockIdx.x;
  if (tile >= *a.num_tiles) return;
  __shared__ uint16_t sd[128 * kPrepPitch];
  __shared__ uint16_t sx[128 * kPrepPitch];
  __shared__ int32_t s_tok[128];
  __shared__ float s_s[128];
  const int tid = threadIdx.x;
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
  const int vec = tid & 7;
  float bias_acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int h0 = 0; h0 < H; h0 += kPrepChunk) {
    // ---- phase 1: gathered row loads, row-major dout_g, shared-memory staging ----
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
      const int row = (tid >> 3) + 32 * r4;
      const int t = s_tok[row];
      const int64_t col = h0 + vec * 8;
      uint4 dv = make_uint4(0, 0, 0, 0), xv = make_uint4(0, 0, 0, 0);
      if (t >= 0) {
        dv = *reinterpret_cast<const uint4*>(a.dout + (int64_t)t * H + col);
        xv = *reinterpret_cast<const uint4*>(a.x + (int64_t)t * H + col);
      }
      const int64_t prow = prow0 + row;
      uint32_t* sdw = reinterpret_cast<uint32_t*>(sd + row * kPrepPitch + vec * 8);
      uint32_t* sxw = reinterpret_cast<uint32_t*>(sx + row * kPrepPitch + vec * 8);
      sdw[0] = dv.x; sdw[1] = dv.y; sdw[2] = dv.z; sdw[3] = dv.w;
      sxw[0] = xv.x; sxw[1] = xv.y; sxw[2] = xv.z; sxw[3] = xv.w;
      float d8[8];
      const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        d8[2 * j] = __uint_as_float(dw[j] << 16);
        d8[2 * j + 1] = __uint_as_float(dw[j] & 0xFFFF0000u);
      }
      if constexpr (BIAS) {
        const uint4 bv = *reinterpret_cast<const uint4*>(a.b2 + (int64_t)e * H + col);
        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bias_acc[r4] = fmaf(d8[2 * j], __uint_as_float(bw[j] << 16), bias_acc[r4]);
          bias_acc[r4] = fmaf(d8[2 * j + 1], __uint_as_float(bw[j] & 0xFFFF0000u), bias_acc[r4]);
        }
      }
      if constexpr (MX) {
        float am = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(d8[j]));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        const uint32_t byte = e8m0_byte(__float_as_uint(am), a.fmt);
        const float inv = e8m0_inv_scale(byte);
        uint2 q;
        q.x = fp8_code(d8[0] * inv, a.fmt) | (fp8_code(d8[1] * inv, a.fmt) << 8) |
              (fp8_code(d8[2] * inv, a.fmt) << 16) | (fp8_code(d8[3] * inv, a.fmt) << 24);
        q.y = fp8_code(d8[4] * inv, a.fmt) | (fp8_code(d8[5] * inv, a.fmt) << 8) |
              (fp8_code(d8[6] * inv, a.fmt) << 16) | (fp8_code(d8[7] * inv, a.fmt) << 24);
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.dout_g) + prow * H + col) = q;
        if ((vec & 3) == 0) a.dout_g_sf[sf_tiled_offset(prow, col, H)] = (uint8_t)byte;
      } else {
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dout_g) + prow * H + col) = dv;
      }
    }
    __syncthreads();
    // ---- phase 2: transposed writes, one (column, 32-row group) per thread ----
    {
      const int h = tid & 63;
      const int g = tid >> 6;
      float dcol[32], xcol[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int row = g * 32 + j;
        float dvv = bf16_bits_to_float(sd[row * kPrepPitch + h]);
        if constexpr (SCALE_T) dvv *= s_s[row];
        dcol[j] = dvv;
        xcol[j] = bf16_bits_to_float(sx[row * kPrepPitch + h]);
      }
      const int64_t orow = h0 + h;
      const int64_t ocol = prow0 + g * 32;
      if constexpr (MX) {
        uint32_t w[8];
        uint32_t byte = quantize_group32(dcol, a.fmt, w);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.dout_gt) + orow * P + ocol);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        a.dout_gt_sf[sf_tiled_offset(orow, ocol, P)] = (uint8_t)byte;
        byte = quantize_group32(xcol, a.fmt, w);
        dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.x_gt) + orow * P + ocol);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        a.x_gt_sf[sf_tiled_offset(orow, ocol, P)] = (uint8_t)byte;
      } else {
        uint4* dd = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dout_gt) + orow * P + ocol);
        uint4* xd = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.x_gt) + orow * P + ocol);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dd[q] = make_uint4(pack_bf16x2(dcol[8 * q + 0], dcol[8 * q + 1]), pack_bf16x2(dcol[8 * q + 2], dcol[8 * q + 3]),
                             pack_bf16x2(dcol[8 * q + 4], dcol[8 * q + 5]), pack_bf16x2(dcol[8 * q + 6], dcol[8 * q + 7]));
          xd[q] = make_uint4(pack_bf16x2(xcol[8 * q + 0], xcol[8 * q + 1]), pack_bf16x2(xcol[8 * q + 2], xcol[8 * q + 3]),
                             pack_bf16x2(xcol[8 * q + 4], xcol[8 * q + 5]), pack_bf16x2(xcol[8 * q + 6], xcol[8 * q + 7]));
        }
      }
    }
    __syncthreads();
  }
  if constexpr (BIAS) {
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
      float v = bias_acc[r4];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      const int row = (tid >> 3) + 32 * r4;
      if (vec == 0) a.ds_bias[prow0 + row] = s_tok[row] >= 0 ? v : 0.f;
    }
  }
}

int launch_prep(const PrepArgs& a, cudaStream_t st) {
  const int grid = (int)(a.P / 128);
  if (grid == 0) return MOE_OK;
  const bool bias = a.ds_bias != nullptr;
#define MOE_PREP(MXV, ST, BI) prep_kernel<MXV, ST, BI><<<grid, 256, 0, st>>>(a)
  if (a.mx) {
    if (a.scale_t) { if (bias) MOE_PREP(true, true, true); else MOE_PREP(true, true, false); }
    else { if (bias) MOE_PREP(true, false, true); else MOE_PREP(true, false, false); }
  } else {
    if (a.scale_t) { if (bias) MOE_PREP(false, true, true); else MOE_PREP(false, true, false); }
    else { if (bias) MOE_PREP(false, false, true); else MOE_PREP(false, false, false); }
  }
#undef MOE_PREP
  count_launch();
  return cuda_check(cudaGetLastError(), "prep");
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
    float am = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(d[j]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    if (!in_range) continue;
    const uint32_t byte = e8m0_byte(__float_as_uint(am), fmt);
    const float inv = e8m0_inv_scale(byte);
    uint2 o;
    o.x = fp8_code(d[0] * inv, fmt) | (fp8_code(d[1] * inv, fmt) << 8) | (fp8_code(d[2] * inv, fmt) << 16) |
          (fp8_code(d[3] * inv, fmt) << 24);
    o.y = fp8_code(d[4] * inv, fmt) | (fp8_code(d[5] * inv, fmt) << 8) | (fp8_code(d[6] * inv, fmt) << 16) |
          (fp8_code(d[7] * inv, fmt) << 24);
    *reinterpret_cast<uint2*>(q + r * cols + c) = o;
    if (((c >> 3) & 3) == 0) sf[tiled ? sf_tiled_offset(r, c, cols) : r * (cols / 32) + c / 32] = (uint8_t)byte;
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
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(q) + oc * rows + orr);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    sf[tiled ? sf_tiled_offset(oc, orr, rows) : oc * (rows / 32) + orr / 32] = (uint8_t)byte;
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(q) + oc * rows + orr);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      dst[k] = make_uint4(pack_bf16x2(v[8 * k + 0], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                          pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
  }
}

int launch_quant_rowwise(const uint16_t* in, int64_t src_rows, int64_t rows, int64_t cols, int64_t ld,
                         const int32_t* row_index, int fmt, uint8_t* q, uint8_t* sf, int tiled, cudaStream_t st) {
  const int64_t total = rows * (cols / 8);
  if (total == 0) return MOE_OK;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  quant_rowwise_kernel<<<(unsigned)blocks, 256, 0, st>>>(in, src_rows, rows, cols, ld, row_index, fmt, q, sf, tiled);
  count_launch();
  return cuda_check(cudaGetLastError(), "quant_rowwise");
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
