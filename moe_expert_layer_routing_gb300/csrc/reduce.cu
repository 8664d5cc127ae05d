// Reductions after the grouped GEMMs:
//   dx_scatter_sum   dx[t] = sum_k dx_expanded[row(t,k)]   (sonic-moe _token_broadcast_backward),
//                    fp32 accumulation in ascending k, 16-byte vector loads, one CTA per token row
//   ds_finalize      ds[f] = sum of the dA-epilogue partials of its row + <dout_t, b2_e>
//                    (gemm_dgated colvec_reduce and db2_and_ds_kernel)
//   segment_rowsum   db[e, j] = sum over the tile rows of expert e of buf[j, p] (* w_p)
//                    (db1_kernel and the db2 half of db2_and_ds_kernel), one warp per (e, j)
#include <cuda_runtime.h>

#include "moebwd_internal.h"
#include "mx_device.cuh"

namespace moebwd {

__global__ void __launch_bounds__(256) dx_scatter_sum_kernel(const uint16_t* __restrict__ dx_exp,
                                                             const int32_t* __restrict__ flat_tile_row, int K, int H,
                                                             uint16_t* __restrict__ dx) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int64_t t = blockIdx.x;
  __shared__ int32_t rows[64];
  if (threadIdx.x < K) rows[threadIdx.x] = flat_tile_row[t * K + threadIdx.x];
  __syncthreads();
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < K; ++k) {
      const int p = rows[k];
      if (p < 0) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(dx_exp + (int64_t)p * H + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * j] += __uint_as_float(w[j] << 16);
        acc[2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
    *reinterpret_cast<uint4*>(dx + t * H + c) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
  }
}

int launch_dx_scatter_sum(const uint16_t* dx_exp, const int32_t* flat_tile_row, int T, int K, int H, uint16_t* dx,
                          cudaStream_t st) {
  if (T == 0) return MOE_OK;
  if (K > 64) return fail(MOE_ERR_UNSUPPORTED, "top-K above 64");
  return launch_pdl(dx_scatter_sum_kernel, dim3(T), dim3(256), 0, st, "dx_scatter_sum", dx_exp, flat_tile_row, K, H, dx);
}

__global__ void ds_finalize_kernel(const float* __restrict__ ds_part, int nparts, const float* __restrict__ ds_bias,
                                   const int32_t* __restrict__ flat_tile_row, int64_t TK, float* __restrict__ ds) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int64_t f = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= TK) return;
  const int p = flat_tile_row[f];
  float v = 0.f;
  if (p >= 0) {  // the row's partials in order, read as 16- or 8-byte vectors where nparts allows
    const float* src = ds_part + (int64_t)p * nparts;
    if ((nparts & 3) == 0) {
      for (int n = 0; n < nparts; n += 4) {
        const float4 q = *reinterpret_cast<const float4*>(src + n);
        v += q.x; v += q.y; v += q.z; v += q.w;
      }
    } else if ((nparts & 1) == 0) {
      for (int n = 0; n < nparts; n += 2) {
        const float2 q = *reinterpret_cast<const float2*>(src + n);
        v += q.x; v += q.y;
      }
    } else {
      for (int n = 0; n < nparts; ++n) v += src[n];
    }
    if (ds_bias) v += ds_bias[p];
  }
  ds[f] = v;
}

int launch_ds_finalize(const float* ds_part, int nparts, const float* ds_bias, const int32_t* flat_tile_row,
                       int64_t TK, float* ds, cudaStream_t st) {
  if (TK == 0) return MOE_OK;
  return launch_pdl(ds_finalize_kernel, dim3((unsigned)((TK + 255) / 256)), dim3(256), 0, st, "ds_finalize", ds_part,
                    nparts, ds_bias, flat_tile_row, TK, ds);
}

__global__ void __launch_bounds__(256) segment_rowsum_kernel(const uint16_t* __restrict__ buf, int64_t ld, int R,
                                                             const int32_t* __restrict__ tile_offsets,
                                                             const float* __restrict__ w,
                                                             const int32_t* __restrict__ tile_row_flat,
                                                             float* __restrict__ out, int accumulate) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int e = blockIdx.y;
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= R) return;
  const int64_t beg = tile_offsets[e], end = tile_offsets[e + 1];
  const uint16_t* row = buf + (int64_t)j * ld;
  float acc = 0.f;
  for (int64_t p = beg + lane * 8; p < end; p += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + p);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float lo = __uint_as_float(wv[q] << 16), hi = __uint_as_float(wv[q] & 0xFFFF0000u);
      if (w) {
        const int f0 = tile_row_flat[p + 2 * q], f1 = tile_row_flat[p + 2 * q + 1];
        lo = f0 >= 0 ? lo * w[f0] : 0.f;
        hi = f1 >= 0 ? hi * w[f1] : 0.f;
      }
      acc += lo;
      acc += hi;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) out[(int64_t)e * R + j] = accumulate ? out[(int64_t)e * R + j] + acc : acc;
}

// One thread per (expert, column) of one or two partial arrays: the expert's tile partials summed in a
// fixed order (tiles two at a time into two accumulators, added at the end): deterministic.
struct BiasJob {
  const float* part;
  int64_t F;
  float* out;
  int parts;
  unsigned blocks;  // blocks of 256 columns
};

template <int PARTS>
__device__ __forceinline__ float bias_sum(const float* __restrict__ part, int64_t F, int64_t f, int t0, int t1) {
  float a0 = 0.f, a1 = 0.f;
  int t = t0;
  for (; t + 1 < t1; t += 2) {
#pragma unroll
    for (int k = 0; k < PARTS; ++k) {
      a0 += part[((int64_t)t * PARTS + k) * F + f];
      a1 += part[((int64_t)(t + 1) * PARTS + k) * F + f];
    }
  }
  if (t < t1) {
#pragma unroll
    for (int k = 0; k < PARTS; ++k) a0 += part[((int64_t)t * PARTS + k) * F + f];
  }
  return a0 + a1;
}

__global__ void __launch_bounds__(256) bias_parts_reduce_kernel(BiasJob j0, BiasJob j1,
                                                                const int32_t* __restrict__ tile_offsets,
                                                                int accumulate) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int e = blockIdx.y;
  const bool second = blockIdx.x >= j0.blocks;
  const BiasJob& j = second ? j1 : j0;
  const int64_t f = (int64_t)(blockIdx.x - (second ? j0.blocks : 0u)) * blockDim.x + threadIdx.x;
  if (f >= j.F) return;
  const int t0 = tile_offsets[e] / 128, t1 = tile_offsets[e + 1] / 128;
  float acc;
  if (j.parts == 4)
    acc = bias_sum<4>(j.part, j.F, f, t0, t1);
  else if (j.parts == 2)
    acc = bias_sum<2>(j.part, j.F, f, t0, t1);
  else
    acc = bias_sum<1>(j.part, j.F, f, t0, t1);
  float* o = j.out + (int64_t)e * j.F + f;
  *o = accumulate ? *o + acc : acc;
}

int launch_bias_parts_reduce(const float* part, int parts, int64_t F, const int32_t* tile_offsets, int E, float* out,
                             cudaStream_t st, int accumulate, const float* part2, int parts2, int64_t F2,
                             float* out2) {
  if (E == 0 || (F == 0 && F2 == 0)) return MOE_OK;
  if ((parts != 1 && parts != 2 && parts != 4) || (part2 && parts2 != 1 && parts2 != 2 && parts2 != 4))
    return fail(MOE_ERR_INVALID, "bias_parts_reduce: parts must be 1, 2 or 4");
  BiasJob j0{part, F, out, parts, (unsigned)((F + 255) / 256)};
  BiasJob j1{part2, part2 ? F2 : 0, out2, parts2, part2 ? (unsigned)((F2 + 255) / 256) : 0u};
  dim3 grid(j0.blocks + j1.blocks, (unsigned)E);
  return launch_pdl(bias_parts_reduce_kernel, grid, dim3(256), 0, st, "bias_parts_reduce", j0, j1, tile_offsets,
                    accumulate);
}

int launch_segment_rowsum(const uint16_t* buf, int64_t ld, int R, const int32_t* tile_offsets, int E, const float* w,
                          const int32_t* tile_row_flat, float* out, cudaStream_t st, int accumulate) {
  if (R == 0 || E == 0) return MOE_OK;
  dim3 grid((unsigned)((R + 7) / 8), (unsigned)E);
  segment_rowsum_kernel<<<grid, 256, 0, st>>>(buf, ld, R, tile_offsets, w, tile_row_flat, out, accumulate);
  count_launch();
  return cuda_check(cudaGetLastError(), "segment_rowsum");
}

// [BW] expert_affinities_masked_grad: ds laid out over all E experts of each token (zero where the
// token did not select the expert; repeated selections add).  One thread per token, in slot order.
__global__ void ds_masked_kernel(const float* __restrict__ ds, const int32_t* __restrict__ ids,
                                 const int32_t* __restrict__ num_valid, int T, int K, int E, float* __restrict__ out) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  if (num_valid && t >= *num_valid) return;
  float* row = out + (int64_t)t * E;
  for (int k = 0; k < K; ++k) {
    const int e = ids[(int64_t)t * K + k];
    if (e >= 0 && e < E) row[e] += ds[(int64_t)t * K + k];
  }
}

int launch_ds_masked(const float* ds, const int32_t* ids, const int32_t* num_valid, int T, int K, int E, float* out,
                     cudaStream_t st) {
  int rc = cuda_check(cudaMemsetAsync(out, 0, sizeof(float) * (size_t)T * E, st), "memset ds_masked");
  if (rc || T == 0) return rc;
  ds_masked_kernel<<<(T + 255) / 256, 256, 0, st>>>(ds, ids, num_valid, T, K, E, out);
  count_launch();
  return cuda_check(cudaGetLastError(), "ds_masked");
}

}  // namespace moebwd
