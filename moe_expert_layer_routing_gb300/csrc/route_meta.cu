// Routing metadata: expert histogram, prefix offsets, a deterministic stable grouping of the flat
// (t, k) rows by expert, the block layout (token_position_to_id / block_to_expert, blockwise MoE
// backward page) and the 128-row tile layout used by the grouped GEMMs.
//
// Three kernels, no host synchronisation:
//   route_count   one CTA per 4096 flat ids: per-chunk expert histogram (shared-memory atomics)
//   route_scan    one CTA: per-expert totals, exclusive scans (rows, blocks, tiles), per-chunk
//                 bases, block/tile owner tables, experts ordered by load
//   route_scatter one CTA per chunk: warp-level match_any ranks give every row its stable position
#include <cuda_runtime.h>

#include <algorithm>

#include "moebwd_internal.h"

namespace moebwd {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kIdsPerWarp = kRouteChunk / kRouteWarps;  // 128

int route_nchunks(int64_t TK) { return (int)((TK + kRouteChunk - 1) / kRouteChunk); }

// Slots taking part in the routing: flat index f = t*K + k with t below the valid-token count.
// An id of -1 marks an unused slot (variable top-K); any other id outside [0, E) is reported.
__device__ __forceinline__ int64_t live_slots(const int32_t* num_valid, int64_t TK, int K) {
  if (!num_valid) return TK;
  const int64_t nv = *num_valid;
  return nv <= 0 ? 0 : (nv * K < TK ? nv * K : TK);
}

// Tables the later kernels fill sparsely, set to -1 (and, optionally, a few counters to 0) by the
// counting kernel's threads instead of separate memsets.
struct RouteFill {
  int32_t* neg[4];
  int64_t n[4];
  int32_t* zero;
  int nzero;
};

__global__ void __launch_bounds__(kRouteThreads) route_count_kernel(const int32_t* __restrict__ ids, int64_t TK,
                                                                    int K, int E,
                                                                    const int32_t* __restrict__ num_valid,
                                                                    int32_t* __restrict__ chunk_counts,
                                                                    int32_t* status, RouteFill fill) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (int64_t)gridDim.x * blockDim.x;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      for (int64_t i = tid; i < fill.n[j]; i += stride) fill.neg[j][i] = -1;
    if (tid < fill.nzero) fill.zero[tid] = 0;
  }
  __syncthreads();
  const int64_t live = live_slots(num_valid, TK, K);
  const int64_t base = (int64_t)blockIdx.x * kRouteChunk;
  const int64_t end = min(base + (int64_t)kRouteChunk, TK);
  int bad = 0;
  for (int64_t f = base + threadIdx.x; f < end; f += blockDim.x) {
    if (f >= live) break;
    const int e = ids[f];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else if (e != -1)
      bad = 1;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, MOE_STATUS_BAD_EXPERT_ID);
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// Exclusive scan of v[0..n) in place by one CTA of 1024 threads; returns the total.
__device__ int block_exclusive_scan(int32_t* v, int n, int32_t* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (n + 1023) / 1024;
  const int beg = min(tid * per, n), end = min(beg + per, n);
  int local = 0;
  for (int i = beg; i < end; ++i) local += v[i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int t = warp_tot[lane];
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += y;
    }
    warp_tot[lane] = ti - t;  // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = ti;
  }
  __syncthreads();
  int run = warp_tot[w] + incl - local;
  for (int i = beg; i < end; ++i) {
    const int x = v[i];
    v[i] = run;
    run += x;
  }
  const int total = warp_tot[32];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(1024) route_scan_kernel(int nchunks, int E, int B, int32_t* chunk_counts,
                                                          int32_t* expert_offsets, int32_t* block_offsets,
                                                          int32_t* tile_offsets, int32_t* expert_order,
                                                          int32_t* block_to_expert, int32_t* tile_expert,
                                                          int32_t* scalars, int32_t* num_blocks_out,
                                                          int32_t* pair_offsets) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  __shared__ int32_t cnt[kMaxExperts + 1];
  __shared__ int32_t rows[kMaxExperts + 1];
  __shared__ int32_t blks[kMaxExperts + 1];
  __shared__ int32_t tiles[kMaxExperts + 1];
  __shared__ int32_t prs[kMaxExperts + 1];
  __shared__ int32_t wt[33];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int tot = 0;
    for (int c = 0; c < nchunks; ++c) tot += chunk_counts[(int64_t)c * E + e];
    cnt[e] = tot;
    rows[e] = tot;
    blks[e] = (tot + B - 1) / B;
    tiles[e] = (tot + kTileM - 1) / kTileM;
    prs[e] = (tiles[e] + 1) / 2;  // the expert's tiles taken two at a time (CTA-pair GEMMs)
  }
  __syncthreads();
  const int tot_rows = block_exclusive_scan(rows, E, wt);
  const int tot_blks = block_exclusive_scan(blks, E, wt);
  const int tot_tiles = block_exclusive_scan(tiles, E, wt);
  const int tot_pairs = block_exclusive_scan(prs, E, wt);
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    expert_offsets[e] = e < E ? rows[e] : tot_rows;
    block_offsets[e] = e < E ? blks[e] : tot_blks;
    tile_offsets[e] = (e < E ? tiles[e] : tot_tiles) * kTileM;
    if (pair_offsets) pair_offsets[e] = e < E ? prs[e] : tot_pairs;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = rows[e];
    for (int c = 0; c < nchunks; ++c) {
      const int v = chunk_counts[(int64_t)c * E + e];
      chunk_counts[(int64_t)c * E + e] = run;
      run += v;
    }
    const int b_end = (e + 1 < E) ? blks[e + 1] : tot_blks;
    for (int b = blks[e]; b < b_end; ++b) block_to_expert[b] = e;
    const int t_end = (e + 1 < E) ? tiles[e + 1] : tot_tiles;
    for (int t = tiles[e]; t < t_end; ++t) tile_expert[t] = e;
    // experts by descending load, ties by index
    const int me = cnt[e];
    int rank = 0;
    for (int o = 0; o < E; ++o) rank += (cnt[o] > me) || (cnt[o] == me && o < e);
    expert_order[rank] = e;
  }
  if (threadIdx.x == 0) {
    scalars[0] = tot_blks;
    scalars[1] = tot_tiles;
    scalars[2] = tot_pairs;
    if (num_blocks_out) *num_blocks_out = tot_blks;
  }
}

__global__ void __launch_bounds__(kRouteThreads) route_scatter_kernel(
    const int32_t* __restrict__ ids, int64_t TK, int K, int E, int B, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ expert_offsets, const int32_t* __restrict__ block_offsets,
    const int32_t* __restrict__ tile_offsets, int32_t* x_gather_idx, int32_t* s_scatter_idx, int32_t* s_reverse,
    int32_t* token_position_to_id, int32_t* tile_row_flat, int32_t* flat_tile_row,
    const int32_t* __restrict__ num_valid) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  extern __shared__ int32_t sm[];
  int32_t* wbase = sm;                       // [warps][E]
  int32_t* eo = wbase + kRouteWarps * E;     // [E]
  int32_t* bo = eo + E;                      // [E]
  int32_t* to = bo + E;                      // [E]
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kRouteWarps * E; i += blockDim.x) wbase[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    eo[e] = expert_offsets[e];
    bo[e] = block_offsets[e];
    to[e] = tile_offsets[e];
  }
  __syncthreads();
  const int64_t wbeg = (int64_t)blockIdx.x * kRouteChunk + (int64_t)w * kIdsPerWarp;
  const int64_t live = live_slots(num_valid, TK, K);
  // pass 1: rows per expert in this warp's slice
  for (int it = 0; it < kIdsPerWarp / 32; ++it) {
    const int64_t f = wbeg + it * 32 + lane;
    const int e = f < live ? ids[f] : -1;
    const bool valid = e >= 0 && e < E;
    const int key = valid ? e : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    if (valid && lane == __ffs(grp) - 1) wbase[w * E + e] += __popc(grp);
  }
  __syncthreads();
  // per-expert bases of the warps of this chunk, in warp order
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_base[(int64_t)blockIdx.x * E + e];
    for (int ww = 0; ww < kRouteWarps; ++ww) {
      const int v = wbase[ww * E + e];
      wbase[ww * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  // pass 2: stable positions
  const unsigned lt = (1u << lane) - 1u;
  for (int it = 0; it < kIdsPerWarp / 32; ++it) {
    const int64_t f = wbeg + it * 32 + lane;
    const bool in = f < TK;
    const int e = f < live ? ids[f] : -1;
    const bool valid = e >= 0 && e < E;
    const int key = valid ? e : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    if (valid) {
      const int r = wbase[w * E + e] + __popc(grp & lt);
      const int t = (int)(f / K);
      x_gather_idx[r] = t;
      s_scatter_idx[r] = (int)f;
      s_reverse[f] = r;
      const int j = r - eo[e];
      token_position_to_id[(int64_t)bo[e] * B + j] = t;
      const int p = to[e] + j;
      tile_row_flat[p] = (int)f;
      flat_tile_row[f] = p;
    } else if (in) {
      s_reverse[f] = -1;
      flat_tile_row[f] = -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(grp) - 1) wbase[w * E + e] += __popc(grp);
    __syncwarp();
  }
}

// Order of the 128-row tiles by the token of their first row (a counting sort over token buckets,
// one CTA).  A pass that gathers token rows tile by tile in this order keeps the tokens its
// concurrently running tiles read within a narrow window, so the K reads of a token row mostly hit
// L2.  The order inside a bucket is arbitrary; it only changes the processing order.
constexpr int kOrderBuckets = 4096;
__global__ void __launch_bounds__(1024) tile_order_kernel(const int32_t* __restrict__ tile_row_flat,
                                                          const int32_t* __restrict__ num_tiles, int T, int K,
                                                          int32_t* __restrict__ order) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  __shared__ int32_t cnt[kOrderBuckets];
  __shared__ int32_t wt[33];
  const int n = *num_tiles;
  for (int b = threadIdx.x; b < kOrderBuckets; b += blockDim.x) cnt[b] = 0;
  __syncthreads();
  auto bucket = [&](int j) {
    const int f = tile_row_flat[(int64_t)j * kTileM];  // first row of a tile is always routed
    const int64_t t = f >= 0 ? f / K : 0;
    return (int)(t * kOrderBuckets / T);
  };
  for (int j = threadIdx.x; j < n; j += blockDim.x) atomicAdd(&cnt[bucket(j)], 1);
  __syncthreads();
  block_exclusive_scan(cnt, kOrderBuckets, wt);
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += blockDim.x) order[atomicAdd(&cnt[bucket(j)], 1)] = j;
}

// ------------------------------------------------------------------------------------------
// Routing metadata supplied by the caller
// ------------------------------------------------------------------------------------------
// The grouped form (expert_offsets, s_scatter_idx) and the block layout (block_offsets; the
// token_position_to_id / block_to_expert tables when given, which are only checked) are taken as
// they come, e.g. kept from the forward pass; the tables the GEMMs use (tile offsets, tile owners,
// tile row -> flat index and back, processing order) are derived from them.  Every caller value is
// checked before it is used as an index.  Metadata that is not a routing of the ids raises
// MOE_STATUS_BAD_ROUTE_META: bad offsets make every row drop out (an empty routing), a bad row
// (flat index out of range, taken twice, or routed to another expert by the ids) drops that row.

// Owner of grouped row r: the largest e < E with eo[e] <= r (offsets nondecreasing, eo[0] = 0).
__device__ __forceinline__ int owner_of_row(const int32_t* eo, int E, int r) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (eo[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(1024) route_in_scan_kernel(
    const int32_t* __restrict__ eo_in, const int32_t* __restrict__ bo_in, const int32_t* __restrict__ b2e_in,
    int64_t TK, const int32_t* __restrict__ num_valid, int K, int E, int B, int64_t Nb, int32_t* expert_offsets,
    int32_t* block_offsets, int32_t* tile_offsets, int32_t* expert_order, int32_t* tile_expert, int32_t* scalars,
    int32_t* pair_offsets, int32_t* status) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  __shared__ int32_t cnt[kMaxExperts + 1];
  __shared__ int32_t tiles[kMaxExperts + 1];
  __shared__ int32_t prs[kMaxExperts + 1];
  __shared__ int32_t wt[33];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  const int64_t live = live_slots(num_valid, TK, K);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int64_t r0 = eo_in[e], r1 = eo_in[e + 1], b0 = bo_in[e], b1 = bo_in[e + 1];
    bool ok = r1 >= r0 && b1 >= b0 && (b1 - b0) * B >= r1 - r0;  // the expert's blocks hold its rows
    if (e == 0) ok = ok && r0 == 0 && b0 == 0;
    if (e == E - 1) ok = ok && r1 <= live && b1 <= Nb;
    if (!ok) bad = 1;
  }
  __syncthreads();
  const bool ok = bad == 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int n = ok ? eo_in[e + 1] - eo_in[e] : 0;
    cnt[e] = n;
    tiles[e] = (n + kTileM - 1) / kTileM;
    prs[e] = (tiles[e] + 1) / 2;
  }
  __syncthreads();
  // tile_offsets / pair_offsets from exclusive scans of the counts
  const int tot_tiles = block_exclusive_scan(tiles, E, wt);
  const int tot_pairs = block_exclusive_scan(prs, E, wt);
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    expert_offsets[e] = ok ? eo_in[e] : 0;
    block_offsets[e] = ok ? bo_in[e] : 0;
    tile_offsets[e] = (e < E ? tiles[e] : tot_tiles) * kTileM;
    if (pair_offsets) pair_offsets[e] = e < E ? prs[e] : tot_pairs;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int t_end = (e + 1 < E) ? tiles[e + 1] : tot_tiles;
    for (int t = tiles[e]; t < t_end; ++t) tile_expert[t] = e;
    const int me = cnt[e];
    int rank = 0;
    for (int o = 0; o < E; ++o) rank += (cnt[o] > me) || (cnt[o] == me && o < e);
    expert_order[rank] = e;
    // the block table, when given, names e for every block that holds e's rows
    if (ok && b2e_in) {
      const int nb = (me + B - 1) / B;
      for (int j = 0; j < nb; ++j)
        if (b2e_in[bo_in[e] + j] != e) bad = 2;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    scalars[0] = ok ? bo_in[E] : 0;
    scalars[1] = tot_tiles;
    scalars[2] = tot_pairs;
    if (bad) atomicOr(status, MOE_STATUS_BAD_ROUTE_META);
  }
}

__global__ void __launch_bounds__(kRouteThreads) route_in_rows_kernel(
    const int32_t* __restrict__ s_scatter_in, const int32_t* __restrict__ tpid_in, const int32_t* __restrict__ ids,
    int64_t TK, const int32_t* __restrict__ num_valid, int K, int E, int B, const int32_t* __restrict__ expert_offsets,
    const int32_t* __restrict__ block_offsets, const int32_t* __restrict__ tile_offsets, int32_t* tile_row_flat,
    int32_t* flat_tile_row, int32_t* status) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  extern __shared__ int32_t eo[];  // [E+1] checked copy of the expert offsets
  for (int e = threadIdx.x; e <= E; e += blockDim.x) eo[e] = expert_offsets[e];
  __syncthreads();
  const int total = eo[E];  // <= live slots <= TK (checked by the scan)
  const int64_t live = live_slots(num_valid, TK, K);
  int bad = 0;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < total; r += (int64_t)gridDim.x * blockDim.x) {
    const int e = owner_of_row(eo, E, (int)r);
    const int j = (int)r - eo[e];
    const int f = s_scatter_in[r];
    bool ok = f >= 0 && f < live && ids[f] == e;
    if (ok && tpid_in) ok = tpid_in[(int64_t)block_offsets[e] * B + j] == f / K;
    if (ok) {
      const int p = tile_offsets[e] + j;
      if (atomicCAS(&flat_tile_row[f], -1, p) == -1)
        tile_row_flat[p] = f;
      else
        ok = false;  // a flat index taken by two rows: the later one drops out
    }
    if (!ok) bad = 1;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, MOE_STATUS_BAD_ROUTE_META);
}

// Every routed slot must be some row of the metadata; ids outside [0, E) other than -1 are reported
// as by the routing kernels.
__global__ void __launch_bounds__(kRouteThreads) route_in_cover_kernel(const int32_t* __restrict__ ids, int64_t TK,
                                                                       const int32_t* __restrict__ num_valid, int K,
                                                                       int E, const int32_t* __restrict__ flat_tile_row,
                                                                       int32_t* status) {
  pdl_wait();  // results of the previous kernel on the stream
  pdl_trigger();
  const int64_t live = live_slots(num_valid, TK, K);
  int miss = 0, badid = 0;
  for (int64_t f = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; f < live; f += (int64_t)gridDim.x * blockDim.x) {
    const int e = ids[f];
    if (e >= 0 && e < E)
      miss |= flat_tile_row[f] < 0;
    else if (e != -1)
      badid = 1;
  }
  const int m = __syncthreads_or(miss), b = __syncthreads_or(badid);
  if (threadIdx.x == 0) {
    if (m) atomicOr(status, MOE_STATUS_BAD_ROUTE_META);
    if (b) atomicOr(status, MOE_STATUS_BAD_EXPERT_ID);
  }
}

int launch_route_meta_in(const RouteMetaIn& in, const int32_t* ids, int T, int K, int E, int B, int64_t Nb, int64_t P,
                         const RouteBufs& r, cudaStream_t st) {
  const int64_t TK = (int64_t)T * K;
  int rc;
  if (r.zero_counters &&
      (rc = cuda_check(cudaMemsetAsync(r.zero_counters, 0, sizeof(int32_t) * (size_t)r.nzero, st), "memset counters")))
    return rc;
  if ((rc = cuda_check(cudaMemsetAsync(r.tile_row_flat, 0xFF, sizeof(int32_t) * (size_t)P, st), "memset tile rows")))
    return rc;
  if ((rc = cuda_check(cudaMemsetAsync(r.tile_expert, 0xFF, sizeof(int32_t) * (size_t)(P / kTileM + 1), st),
                       "memset tile experts")))
    return rc;
  if ((rc = cuda_check(cudaMemsetAsync(r.flat_tile_row, 0xFF, sizeof(int32_t) * (size_t)(TK > 0 ? TK : 1), st),
                       "memset flat rows")))
    return rc;
  route_in_scan_kernel<<<1, 1024, 0, st>>>(in.expert_offsets, in.block_offsets, in.block_to_expert, TK, r.num_valid,
                                           K, E, B, Nb, r.expert_offsets, r.block_offsets, r.tile_offsets,
                                           r.expert_order, r.tile_expert, r.scalars, r.pair_offsets, r.status);
  count_launch();
  if ((rc = cuda_check(cudaGetLastError(), "route_in_scan"))) return rc;
  if (TK > 0) {
    const int grid = (int)std::min<int64_t>((TK + kRouteThreads - 1) / kRouteThreads, 4 * 152);
    route_in_rows_kernel<<<grid, kRouteThreads, sizeof(int32_t) * (size_t)(E + 1), st>>>(
        in.s_scatter_idx, in.token_position_to_id, ids, TK, r.num_valid, K, E, B, r.expert_offsets, r.block_offsets,
        r.tile_offsets, r.tile_row_flat, r.flat_tile_row, r.status);
    count_launch();
    if ((rc = cuda_check(cudaGetLastError(), "route_in_rows"))) return rc;
    route_in_cover_kernel<<<grid, kRouteThreads, 0, st>>>(ids, TK, r.num_valid, K, E, r.flat_tile_row, r.status);
    count_launch();
    if ((rc = cuda_check(cudaGetLastError(), "route_in_cover"))) return rc;
  }
  return MOE_OK;
}

int launch_tile_order(const int32_t* tile_row_flat, const int32_t* num_tiles, int T, int K, int32_t* order,
                      cudaStream_t st) {
  if (T <= 0) return MOE_OK;
  return launch_pdl(tile_order_kernel, dim3(1), dim3(1024), 0, st, "tile_order", tile_row_flat, num_tiles, T, K, order);
}

int launch_route_meta(const int32_t* ids, int T, int K, int E, int B, int64_t Nb, int64_t P, const RouteBufs& r,
                      cudaStream_t st) {
  const int64_t TK = (int64_t)T * K;
  int rc;
  // padding entries of the block and tile tables are -1: filled by route_count's threads (one extra
  // CTA when there is nothing to count), before route_scatter writes the routed entries
  RouteFill fill{};
  fill.neg[0] = r.token_position_to_id; fill.n[0] = Nb * B;
  fill.neg[1] = r.block_to_expert;      fill.n[1] = Nb > 0 ? Nb : 1;
  fill.neg[2] = r.tile_row_flat;        fill.n[2] = P;
  fill.neg[3] = r.tile_expert;          fill.n[3] = P / kTileM + 1;
  fill.zero = r.zero_counters;          fill.nzero = r.zero_counters ? r.nzero : 0;
  const int nch = route_nchunks(TK);
  if ((rc = launch_pdl(route_count_kernel, dim3(nch > 0 ? nch : 1), dim3(kRouteThreads), sizeof(int32_t) * E, st,
                       "route_count", ids, TK, K, E, r.num_valid, r.chunk_counts, r.status, fill)))
    return rc;
  if ((rc = launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, st, "route_scan", nch, E, B, r.chunk_counts,
                       r.expert_offsets, r.block_offsets, r.tile_offsets, r.expert_order, r.block_to_expert,
                       r.tile_expert, r.scalars, r.num_blocks_out, r.pair_offsets)))
    return rc;
  if (nch > 0) {
    const size_t smem = sizeof(int32_t) * (size_t)(kRouteWarps * E + 3 * E);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if ((rc = cuda_check(e, "route_scatter attribute"))) return rc;
    }
    if ((rc = launch_pdl(route_scatter_kernel, dim3(nch), dim3(kRouteThreads), smem, st, "route_scatter", ids, TK, K,
                         E, B, (const int32_t*)r.chunk_counts, (const int32_t*)r.expert_offsets,
                         (const int32_t*)r.block_offsets, (const int32_t*)r.tile_offsets, r.x_gather_idx,
                         r.s_scatter_idx, r.s_reverse, r.token_position_to_id, r.tile_row_flat, r.flat_tile_row,
                         r.num_valid)))
      return rc;
  }
  return MOE_OK;
}

}  // namespace moebwd
