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
  const int32_t* idt = ids + (int64_t)t * K;
  const float* gt = g + (int64_t)t * K;
  float* out = dl + (int64_t)t * E;
  if (mode == MOE_ROUTER_TOPK || mode == MOE_ROUTER_SOFTMAX_OVER_TOPK) {
    float dot = 0.f;
    if (mode == MOE_ROUTER_SOFTMAX_OVER_TOPK)
      for (int k = 0; k < K; ++k) {
        const int e = idt[k];
        if (e >= 0 && e < E) dot = fmaf(gt[k], scores[(int64_t)t * K + k], dot);
      }
    for (int e = lane; e < E; e += 32) {
      float v = 0.f;
      for (int k = 0; k < K; ++k)
        if (idt[k] == e)
          v += mode == MOE_ROUTER_TOPK ? gt[k] : scores[(int64_t)t * K + k] * (gt[k] - dot);
      out[e] = v;
    }
    return;
  }
  // top-K over softmax: recompute p over all E logits
  const float* lt = logits + (int64_t)t * E;
  float mx = -INFINITY;
  for (int e = lane; e < E; e += 32) mx = fmaxf(mx, lt[e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int e = lane; e < E; e += 32) sum += __expf(lt[e] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.f / sum;
  // selected probabilities, optional renormalisation, <dr, r>
  float S = 0.f, dot_s = 0.f;
  for (int k = 0; k < K; ++k) {
    const int e = idt[k];
    if (e < 0 || e >= E) continue;
    S += __expf(lt[e] - mx) * inv;
    if (renorm) dot_s = fmaf(gt[k], scores[(int64_t)t * K + k], dot_s);
  }
  const float rS = renorm ? 1.f / S : 1.f;
  float dot = 0.f;
  for (int k = 0; k < K; ++k) {
    const int e = idt[k];
    if (e < 0 || e >= E) continue;
    const float dr = renorm ? (gt[k] - dot_s) * rS : gt[k];
    dot = fmaf(dr, __expf(lt[e] - mx) * inv, dot);
  }
  for (int e = lane; e < E; e += 32) {
    float dp = 0.f;
    for (int k = 0; k < K; ++k)
      if (idt[k] == e) dp += renorm ? (gt[k] - dot_s) * rS : gt[k];
    out[e] = __expf(lt[e] - mx) * inv * (dp - dot);
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
