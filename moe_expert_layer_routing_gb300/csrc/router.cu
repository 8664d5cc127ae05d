// Router backward: ds (the gradient of the K routing scores of each token) -> gradient of the E
// router logits (sonic-moe functional/backward.py, `_topk_softmax_bwd` and `_topk_bwd`).
//
//   softmax over top-K   s = softmax(l[idx]):            dl[idx_k] = s_k (g_k - <g, s>), 0 elsewhere
//   top-K over softmax   p = softmax(l) over E, r = p[idx], s = r / sum(r) (renormalised) or r:
//                        dr = (g - <g, s>) / sum(r) (renormalised) or g, dp = scatter(dr),
//                        dl = p (dp - <dr, r>)   for every logit
//   plain top-K          s = l[idx]:                     dl[idx_k] = g_k
//
// fp32.  router_bwd_vec_kernel (E a multiple of 4): one token per 8 lanes (E <= 256, K <= 8), per
// half-warp (E <= 512, K <= 16) or per warp (E <= 1024, K <= 32), one pass over the token's logits
// held in registers as float4 (lane l of a segment of L lanes owns columns 4 L j + 4 l .. + 3), each
// slot's own exponential from its logit re-read, the slot weights scattered once through a
// per-segment shared buffer (repeated ids summed in slot order), the row written as float4.  router_bwd_kernel (any E, K <= 64): lane j owns logits j, j+32, ..., the
// K selected slots broadcast by shuffles per 32 logits.  Ids outside [0, E) are skipped.
#include <cuda_runtime.h>

#include "moebwd_internal.h"

namespace moebwd {

__global__ void __launch_bounds__(256) router_bwd_kernel(int mode, int renorm, const float* __restrict__ logits,
                                                         const float* __restrict__ scores,
                                                         const float* __restrict__ g, const int32_t* __restrict__ ids,
                                                         int T, int K, int E, float* __restrict__ dl) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  // the K selected slots of this token: lane k (and k - 32) holds slot k's id, gradient and score
  int id0 = -1, id1 = -1;
  float g0 = 0.f, g1 = 0.f, s0 = 0.f, s1 = 0.f;
  if (lane < K) {
    id0 = ids[(int64_t)t * K + lane];
    g0 = g[(int64_t)t * K + lane];
    if (scores) s0 = scores[(int64_t)t * K + lane];
  }
  if (lane + 32 < K) {
    id1 = ids[(int64_t)t * K + lane + 32];
    g1 = g[(int64_t)t * K + lane + 32];
    if (scores) s1 = scores[(int64_t)t * K + lane + 32];
  }
  if (id0 >= E) id0 = -1;
  if (id1 >= E) id1 = -1;
  const float* lt = logits ? logits + (int64_t)t * E : nullptr;
  float* out = dl + (int64_t)t * E;
  // per-slot weight w_k scattered to logit id_k, and the shift applied (top-K over softmax) below
  float mx = 0.f, inv = 1.f, dot = 0.f;
  float w0 = 0.f, w1 = 0.f;
  if (mode == MOE_ROUTER_TOPK) {
    w0 = g0;
    w1 = g1;
  } else if (mode == MOE_ROUTER_SOFTMAX_OVER_TOPK) {
    float d = (id0 >= 0 ? g0 * s0 : 0.f) + (id1 >= 0 ? g1 * s1 : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    w0 = s0 * (g0 - d);
    w1 = s1 * (g1 - d);
  } else {
    mx = -INFINITY;
    for (int e = lane; e < E; e += 32) mx = fmaxf(mx, lt[e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int e = lane; e < E; e += 32) sum += __expf(lt[e] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    inv = 1.f / sum;
    const float p0 = id0 >= 0 ? __expf(lt[id0] - mx) * inv : 0.f;
    const float p1 = id1 >= 0 ? __expf(lt[id1] - mx) * inv : 0.f;
    float S = p0 + p1, ds = (id0 >= 0 ? g0 * s0 : 0.f) + (id1 >= 0 ? g1 * s1 : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      S += __shfl_xor_sync(0xffffffffu, S, o);
      ds += __shfl_xor_sync(0xffffffffu, ds, o);
    }
    w0 = renorm ? (g0 - ds) / S : g0;  // dr of each selected slot
    w1 = renorm ? (g1 - ds) / S : g1;
    float d = (id0 >= 0 ? w0 * p0 : 0.f) + (id1 >= 0 ? w1 * p1 : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    dot = d;
  }
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    float dp = 0.f;
    for (int k = 0; k < K; ++k) {  // broadcast slot k; uniform loop, every lane takes part
      const int idk = __shfl_sync(0xffffffffu, k < 32 ? id0 : id1, k & 31);
      const float wk = __shfl_sync(0xffffffffu, k < 32 ? w0 : w1, k & 31);
      if (idk == e) dp += wk;
    }
    if (e < E) out[e] = mode == MOE_ROUTER_TOPK_OVER_SOFTMAX ? __expf(lt[e] - mx) * inv * (dp - dot) : dp;
  }
}

// One token per segment of LANES lanes (a whole warp, or 16 or 8 of its lanes: more rows in flight
// and reductions one or two shuffle steps shorter); NV float4 column groups per lane:
// ceil(E / (4 LANES)).
template <int LANES>
__device__ __forceinline__ float seg_sum(float v, unsigned mask) {
#pragma unroll
  for (int o = LANES / 2; o > 0; o >>= 1) v += __shfl_xor_sync(mask, v, o);
  return v;
}
template <int LANES>
__device__ __forceinline__ float seg_max(float v, unsigned mask) {
#pragma unroll
  for (int o = LANES / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(mask, v, o));
  return v;
}

template <int NV, int LANES>
__global__ void __launch_bounds__(256) router_bwd_vec_kernel(int mode, int renorm, const float* __restrict__ logits,
                                                             const float* __restrict__ scores,
                                                             const float* __restrict__ g,
                                                             const int32_t* __restrict__ ids, int T, int K, int E,
                                                             float* __restrict__ dl) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  constexpr int SEGS = 32 / LANES;  // tokens per warp
  constexpr int COLS = 4 * LANES;   // logits of one float4 column group across the segment
  __shared__ float4 sbuf[8 * SEGS][NV * LANES];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, seg = lane / LANES, sl = lane % LANES;
  const unsigned mask = (0xffffffffu >> (32 - LANES)) << (LANES * seg);  // this segment's lanes
  const int t = (blockIdx.x * 8 + w) * SEGS + seg;
  if (t >= T) return;  // only segment-level synchronisation below
  float4* buf = sbuf[w * SEGS + seg];
  int id = -1;
  float gk = 0.f, sk = 0.f;
  if (sl < K) {
    id = ids[(int64_t)t * K + sl];
    gk = g[(int64_t)t * K + sl];
    if (scores) sk = scores[(int64_t)t * K + sl];
    if (id < 0 || id >= E) id = -1;
  }
  const float* lt = logits ? logits + (int64_t)t * E : nullptr;
  float4 L[NV];
  float mx = 0.f, inv = 1.f, dot = 0.f, wk = 0.f;
  if (mode == MOE_ROUTER_TOPK) {
    wk = gk;
  } else if (mode == MOE_ROUTER_SOFTMAX_OVER_TOPK) {
    const float d = seg_sum<LANES>(id >= 0 ? gk * sk : 0.f, mask);
    wk = sk * (gk - d);
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = j * COLS + 4 * sl;
      L[j] = c < E ? reinterpret_cast<const float4*>(lt)[j * LANES + sl]
                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      m = fmaxf(m, fmaxf(fmaxf(L[j].x, L[j].y), fmaxf(L[j].z, L[j].w)));
    }
    mx = seg_max<LANES>(m, mask);
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {  // L now holds exp(l - max) (0 past E)
      L[j] = make_float4(__expf(L[j].x - mx), __expf(L[j].y - mx), __expf(L[j].z - mx), __expf(L[j].w - mx));
      sum += (L[j].x + L[j].y) + (L[j].z + L[j].w);
    }
    inv = 1.f / seg_sum<LANES>(sum, mask);
    // exp(l[id] - max) of this lane's slot: the same expression as the row's, on the logit re-read
    // from the row just loaded (a cache hit) instead of 4 NV shuffles from the lane that holds it
    const float pk = id >= 0 ? __expf(lt[id] - mx) * inv : 0.f;
    const float S = seg_sum<LANES>(pk, mask), dsum = seg_sum<LANES>(id >= 0 ? gk * sk : 0.f, mask);
    wk = renorm ? (gk - dsum) / S : gk;  // dr of the slot
    dot = seg_sum<LANES>(id >= 0 ? wk * pk : 0.f, mask);
  }
#pragma unroll
  for (int j = 0; j < NV; ++j) buf[j * LANES + sl] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncwarp(mask);
  // the first slot of each distinct id writes the sum of its slots' weights, in slot order
  float tot = 0.f;
  for (int j = 0; j < K; ++j) {
    const int idj = __shfl_sync(mask, id, j, LANES);
    const float wj = __shfl_sync(mask, wk, j, LANES);
    if (idj == id) tot += wj;
  }
  const unsigned same = __match_any_sync(mask, id);
  if (id >= 0 && lane == __ffs(same) - 1) reinterpret_cast<float*>(buf)[id] = tot;
  __syncwarp(mask);
  float4* out = reinterpret_cast<float4*>(dl + (int64_t)t * E);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    if (j * COLS + 4 * sl >= E) continue;
    float4 v = buf[j * LANES + sl];
    if (mode == MOE_ROUTER_TOPK_OVER_SOFTMAX) {
      v.x = L[j].x * inv * (v.x - dot);
      v.y = L[j].y * inv * (v.y - dot);
      v.z = L[j].z * inv * (v.z - dot);
      v.w = L[j].w * inv * (v.w - dot);
    }
    out[j * LANES + sl] = v;
  }
}

template <int NV, int LANES>
static void router_vec_launch(int mode, int renorm, const float* logits, const float* scores, const float* dscores,
                              const int32_t* ids, int T, int K, int E, float* dlogits, cudaStream_t st) {
  constexpr int per_block = 8 * (32 / LANES);  // tokens per 256-thread block
  router_bwd_vec_kernel<NV, LANES><<<(T + per_block - 1) / per_block, 256, 0, st>>>(mode, renorm, logits, scores,
                                                                                  dscores, ids, T, K, E, dlogits);
}

}  // namespace moebwd

using namespace moebwd;

extern "C" int moe_router_bwd(int mode, int renorm, const float* logits, const float* scores, const float* dscores,
                              const int32_t* ids, int T, int K, int E, float* dlogits, moe_stream_t stream) {
  clear_error();
  if (T < 0 || K <= 0 || E <= 0 || K > 64) return fail(MOE_ERR_INVALID, "moe_router_bwd: bad sizes (need K <= 64)");
  if (mode != MOE_ROUTER_SOFTMAX_OVER_TOPK && mode != MOE_ROUTER_TOPK_OVER_SOFTMAX && mode != MOE_ROUTER_TOPK)
    return fail(MOE_ERR_INVALID, "moe_router_bwd: bad mode");
  if (T == 0) return MOE_OK;  // nothing to write (the pointers may be null)
  if (!dscores || !ids || !dlogits) return fail(MOE_ERR_INVALID, "moe_router_bwd: null pointer");
  if (mode == MOE_ROUTER_TOPK_OVER_SOFTMAX && !logits) return fail(MOE_ERR_INVALID, "moe_router_bwd: logits needed");
  if ((mode == MOE_ROUTER_SOFTMAX_OVER_TOPK || (mode == MOE_ROUTER_TOPK_OVER_SOFTMAX && renorm)) && !scores)
    return fail(MOE_ERR_INVALID, "moe_router_bwd: forward scores needed");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool aligned = ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(dlogits)) & 15) == 0;
  if (E % 4 == 0 && E <= 256 && K <= 8 && aligned) {  // one pass, the row in registers, four tokens a warp
    const int nv = (E + 31) / 32;
    switch (nv) {
      case 1: router_vec_launch<1, 8>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      case 2: router_vec_launch<2, 8>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      case 3:
      case 4: router_vec_launch<4, 8>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      default: router_vec_launch<8, 8>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
    }
  } else if (E % 4 == 0 && E <= 512 && K <= 16 && aligned) {  // two tokens a warp
    const int nv = (E + 63) / 64;
    switch (nv) {
      case 1: router_vec_launch<1, 16>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      case 2: router_vec_launch<2, 16>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      case 3:
      case 4: router_vec_launch<4, 16>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      default: router_vec_launch<8, 16>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
    }
  } else if (E % 4 == 0 && E <= 1024 && K <= 32 && aligned) {  // one pass, the row in registers
    const int nv = (E + 127) / 128;
    switch (nv) {
      case 1: router_vec_launch<1, 32>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      case 2: router_vec_launch<2, 32>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      case 3:
      case 4: router_vec_launch<4, 32>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
      default: router_vec_launch<8, 32>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits, st); break;
    }
  } else {
    router_bwd_kernel<<<(T + 7) / 8, 256, 0, st>>>(mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits);
  }
  count_launch();
  return cuda_check(cudaGetLastError(), "router_bwd");
}
