// MXFP8 operands of the dense linear backward ("Matmul MXFP8 Backward Kernel API Reference": dX = dY W
// contracts over N, dW = dY^T X contracts over M; each GEMM operand is quantised in 32-element
// groups along that GEMM's contraction dimension) in one launch:
//   dY [M,N] -> dY codes [M,N] (groups along N, dX's A) and dY^T [N,M] (groups along M, dW's A)
//   W  [N,K] -> W^T [K,N] (groups along N, dX's B)
//   X  [M,K] -> X^T [K,M] (groups along M, dW's B)
// with every scale in the tiled layout of the block-scaled MMA.  The work is a list of 128 x 128 source
// tiles walked by persistent CTAs (three per SM); each CTA copies its next tile into the second of two
// shared buffers (16-byte cp.async, eight per thread) while it quantises the current one, so the loads
// of one tile overlap the arithmetic and stores of the previous.  dY's row-wise codes are taken from
// the staged rows (four threads per 32-column group), the transposed codes from the staged columns
// (one column and two 32-row groups per thread, each group one 32-byte store).  The 512 scale bytes of
// a 128 x 128 tile are one whole atom of the tiled layout: they are collected in shared memory and
// written as 16-byte stores.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "moebwd_internal.h"
#include "mx_device.cuh"
#include "ptx.cuh"

namespace moebwd {

namespace {

constexpr int kLinPitch = 136;  // bf16 pitch of the staged tile: 16-byte row pieces and 2-byte column reads conflict-free

struct LinQuantArgs {
  const uint16_t* src[3];  // dY [M,N], W [N,K], X [M,K]
  int64_t rows[3], cols[3];
  uint8_t* qt[3];          // transposed codes [cols, rows] of each source
  uint8_t* sft[3];         // their tiled scales
  uint8_t* qr;             // dY's row-wise codes [M,N]
  uint8_t* sfr;            // and their tiled scales
  int64_t end0, end1, total;  // tile index ranges: [0, end0) dY, [end0, end1) W, [end1, total) X
};

constexpr int kLinTileBytes = 128 * kLinPitch * 2;
constexpr int kLinSmemBytes = 2 * kLinTileBytes + 2 * 512;
constexpr int kLinCtasPerSm = 3;

// source tile `t` of the work list: its job and first row / column (tile counts below 2^31: 32-bit
// division)
__device__ __forceinline__ int lin_tile(const LinQuantArgs& a, int64_t t, int64_t& r0, int64_t& c0) {
  const int job = t < a.end0 ? 0 : t < a.end1 ? 1 : 2;
  const uint32_t u = (uint32_t)(t - (job == 0 ? 0 : job == 1 ? a.end0 : a.end1));
  const uint32_t ct = (uint32_t)(a.cols[job] >> 7);
  const uint32_t rt = u / ct;
  r0 = (int64_t)rt * 128;
  c0 = (int64_t)(u - rt * ct) * 128;
  return job;
}

// this thread's eight 16-byte pieces of tile `t` (rows tid/16 + 16 i, piece tid % 16) into `buf`
__device__ __forceinline__ void lin_issue(const LinQuantArgs& a, int64_t t, uint16_t* buf, int tid) {
  int64_t r0, c0;
  const int job = lin_tile(a, t, r0, c0);
  const int64_t C = a.cols[job];
  const uint16_t* src = a.src[job] + r0 * C + c0 + 8 * (tid & 15);
  const uint32_t dst = smem_u32(buf + 8 * (tid & 15));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = (tid >> 4) + 16 * i;
    cp_async_16(dst + row * kLinPitch * 2, src + row * C);
  }
}

template <int FMT>
__global__ void __launch_bounds__(256, kLinCtasPerSm) linear_quant_kernel(const LinQuantArgs a) {
  extern __shared__ __align__(16) uint8_t lin_smem[];
  uint16_t* bufs = reinterpret_cast<uint16_t*>(lin_smem);
  uint8_t* atom = lin_smem + 2 * kLinTileBytes;  // [0, 512) transposed operand, [512, 1024) dY row-wise
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int tid = threadIdx.x;
  const int pc = tid & 15;   // 16-byte piece of a row: columns 8 pc .. 8 pc + 7
  const int h = tid & 127;   // transposed phase: source column h
  int64_t t = blockIdx.x;
  if (t < a.total) lin_issue(a, t, bufs, tid);
  cp_async_commit();
  for (int buf = 0; t < a.total; t += gridDim.x, buf ^= 1) {
    // the next tile's copies go into the other buffer (free: every thread passed the barrier after
    // the last reads of it), then this tile's own copies are waited for
    if (t + gridDim.x < a.total) lin_issue(a, t + gridDim.x, bufs + (buf ^ 1) * (kLinTileBytes / 2), tid);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint16_t* tile = bufs + buf * (kLinTileBytes / 2);
    int64_t r0, c0;
    const int job = lin_tile(a, t, r0, c0);
    const int64_t R = a.rows[job], C = a.cols[job];
    if (job == 0) {  // dY row-wise: an aligned quad of lanes holds a row's 32-column group
      uint8_t* qr = a.qr + r0 * C + c0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = (tid >> 4) + 16 * i;
        const uint4 v = *reinterpret_cast<const uint4*>(tile + row * kLinPitch + 8 * pc);
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
        const uint32_t byte = e8m0_byte(__float_as_uint(am), FMT);
        const uint64_t inv2 = f2_splat(e8m0_inv_scale(byte));
        *reinterpret_cast<uint2*>(qr + row * C + 8 * pc) =
            make_uint2(fp8x4_scaled<FMT>(d[0], d[1], d[2], d[3], inv2), fp8x4_scaled<FMT>(d[4], d[5], d[6], d[7], inv2));
        if ((pc & 3) == 0) atom[512 + (row & 31) * 16 + (row >> 5) * 4 + (pc >> 2)] = (uint8_t)byte;
      }
    }
    // transposed: output row c0 + h, contraction columns r0 + 32 g .. (the source rows)
    uint8_t* qt = a.qt[job] + (c0 + h) * R + r0;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const int g = (tid >> 7) + 2 * gi;
      float c32[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) c32[j] = bf16_bits_to_float(tile[(32 * g + j) * kLinPitch + h]);
      uint32_t w[8];
      const uint32_t byte = quantize_group32_t<FMT>(c32, w);
      st_global_32b(qt + 32 * g, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
      atom[(h & 31) * 16 + (h >> 5) * 4 + g] = (uint8_t)byte;
    }
    __syncthreads();  // the atoms are complete; the tile buffer and atoms are free after the writes below
    if (tid < 32) {   // atom of output rows c0.., contraction columns r0.. of the transposed operand
      uint8_t* dst = a.sft[job] + ((c0 >> 7) * (R >> 7) + (r0 >> 7)) * 512;
      reinterpret_cast<uint4*>(dst)[tid] = reinterpret_cast<const uint4*>(atom)[tid];
    } else if (job == 0 && tid < 64) {  // atom of dY rows r0.., columns c0..
      uint8_t* dst = a.sfr + ((r0 >> 7) * (C >> 7) + (c0 >> 7)) * 512;
      reinterpret_cast<uint4*>(dst)[tid - 32] = reinterpret_cast<const uint4*>(atom + 512)[tid - 32];
    }
  }
  cp_async_wait<0>();  // nothing left in flight when the CTA exits
}

}  // namespace

int launch_linear_quant(const uint16_t* dY, const uint16_t* W, const uint16_t* X, int64_t M, int64_t N, int64_t K,
                        int fmt, uint8_t* dY_q, uint8_t* dY_sf, uint8_t* Wt_q, uint8_t* Wt_sf, uint8_t* dYt_q,
                        uint8_t* dYt_sf, uint8_t* Xt_q, uint8_t* Xt_sf, cudaStream_t st) {
  if (M % 128 || N % 128 || K % 128) return fail(MOE_ERR_UNSUPPORTED, "linear quantiser: sizes must be multiples of 128");
  LinQuantArgs a{};
  a.src[0] = dY; a.rows[0] = M; a.cols[0] = N; a.qt[0] = dYt_q; a.sft[0] = dYt_sf;
  a.src[1] = W;  a.rows[1] = N; a.cols[1] = K; a.qt[1] = Wt_q;  a.sft[1] = Wt_sf;
  a.src[2] = X;  a.rows[2] = M; a.cols[2] = K; a.qt[2] = Xt_q;  a.sft[2] = Xt_sf;
  a.qr = dY_q;
  a.sfr = dY_sf;
  a.end0 = (M / 128) * (N / 128);
  a.end1 = a.end0 + (N / 128) * (K / 128);
  a.total = a.end1 + (M / 128) * (K / 128);
  if (a.total > INT32_MAX) return fail(MOE_ERR_UNSUPPORTED, "linear quantiser: too many tiles");
  const int grid = (int)std::min<int64_t>(a.total, (int64_t)kLinCtasPerSm * device_sm_count());
  auto k = fmt == MOE_FP8_E5M2 ? linear_quant_kernel<MOE_FP8_E5M2> : linear_quant_kernel<MOE_FP8_E4M3>;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kLinSmemBytes);
  if (e != cudaSuccess) return cuda_check(e, "linear quantiser attribute");
  return launch_pdl(k, dim3((unsigned)grid), dim3(256), kLinSmemBytes, st, "linear quantiser", a);
}

}  // namespace moebwd
