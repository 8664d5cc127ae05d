// Router backward: ds (the gradient of the K routing scores of each token) -> gradient of the E
// router logits (sonic-moe functional/backward.py, `_topk_softmax_bwd` and `_topk_bwd`).
//
//   softmax over top-K   s = softmax(l[idx]):            dl[idx_k] = s_k (g_k - <g, s>), 0 elsewhere
//   top-K over softmax   p = softmax(l) over E, r = p[idx], s = r / sum(r) (renormalised) or r:
//                        dr = (g - <g, s>) / sum(r) (renormalised) or g, dp = scatter(dr),
//                        dl = p (dp - <dr, r>)   for every logit
//   plain top-K          s = l[idx]:                     dl[idx_k] = g_k
//
// One warp per token, fp32; lane j owns logits j, j+32, ...; the K selected slots are read by every
// lane (K <= 64).  Ids outside [0, E) are skipped.
#include <cuda_runtime.h>

#include "moebwd_internal.h"

namespace moebwd {

__global__ void __launch_bounds__(256) router_bwd_kernel(int mode, int renorm, const float* __restrict__ logits,
                                                         const float* __restrict__ scores,
                                                         const float* __restrict__ g, const int32_t* __restrict__ ids,
                                                         int T, int K, int E, float* __restrict__ dl) {
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

}  // namespace moebwd

using namespace moebwd;

extern "C" int moe_router_bwd(int mode, int renorm, const float* logits, const float* scores, const float* dscores,
                              const int32_t* ids, int T, int K, int E, float* dlogits, moe_stream_t stream) {
  clear_error();
  if (T < 0 || K <= 0 || E <= 0 || K > 64) return fail(MOE_ERR_INVALID, "moe_router_bwd: bad sizes (need K <= 64)");
  if (mode != MOE_ROUTER_SOFTMAX_OVER_TOPK && mode != MOE_ROUTER_TOPK_OVER_SOFTMAX && mode != MOE_ROUTER_TOPK)
    return fail(MOE_ERR_INVALID, "moe_router_bwd: bad mode");
  if (!dscores || !ids || !dlogits) return fail(MOE_ERR_INVALID, "moe_router_bwd: null pointer");
  if (mode == MOE_ROUTER_TOPK_OVER_SOFTMAX && !logits) return fail(MOE_ERR_INVALID, "moe_router_bwd: logits needed");
  if ((mode == MOE_ROUTER_SOFTMAX_OVER_TOPK || (mode == MOE_ROUTER_TOPK_OVER_SOFTMAX && renorm)) && !scores)
    return fail(MOE_ERR_INVALID, "moe_router_bwd: forward scores needed");
  if (T == 0) return MOE_OK;
  router_bwd_kernel<<<(T + 7) / 8, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      mode, renorm, logits, scores, dscores, ids, T, K, E, dlogits);
  count_launch();
  return cuda_check(cudaGetLastError(), "router_bwd");
}
