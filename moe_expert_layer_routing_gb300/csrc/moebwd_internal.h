// Internal declarations shared by the translation units of libmoebwd.
#pragma once
#include <cstddef>
#include <cstdint>
#include <functional>
#include <cuda_runtime.h>

#include "../../include/moebwd.h"

namespace moebwd {

// Default limit of a pipeline wait inside a GEMM kernel before it reports MOE_STATUS_TIMEOUT
// (MOE_OPT_WAIT_LIMIT_NS changes it); the drain waits before a CTA exits always keep this one.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

constexpr int kTileM = 128;       // rows of a GEMM tile = UMMA M = tile-row padding granule
constexpr int kMaxExperts = 1024;
constexpr int kRouteChunk = 4096; // flat ids per CTA in the routing kernels

// ------------------------------------------------------------------------------------------
// host helpers (host.cu)
// ------------------------------------------------------------------------------------------
int fail(int code, const char* fmt, ...);
void clear_error();
int cuda_check(cudaError_t e, const char* what);
int device_sm_count();
size_t align_up(size_t v, size_t a);
void count_launch();   // one kernel launched by this library
int64_t option(int opt);  // current value of a MOE_OPT_* option
// Runs `side` on a library-owned second stream of the current device, ordered after the work already
// enqueued on `st`, and `main` on `st` meanwhile; `st` then waits for the side work.  Returns the first
// nonzero code (main is skipped when side failed).
int fork_join(cudaStream_t st, const std::function<int(cudaStream_t)>& side, const std::function<int()>& main);

// Programmatic dependent launch, device side: wait until the grids this one depends on have completed
// and their memory is visible (a no-op without such a dependency); allow the dependent grid to be
// scheduled (its CTAs then wait in their own pdl_wait).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic dependent launch (unless MOE_OPT_PDL is 0): the kernel's CTAs may be
// scheduled while the previous kernel on the stream finishes; every kernel launched this way calls
// pdl_wait() before it touches memory that earlier work wrote, and pdl_trigger() to let the next
// kernel be scheduled early in turn.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, const char* what,
               Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = option(MOE_OPT_PDL) ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  count_launch();
  if (e != cudaSuccess) return cuda_check(e, what);
  return cuda_check(cudaGetLastError(), what);
}

// 2D tensor map over a row-major [rows, cols] matrix of `elem_bytes`-byte elements with the given
// row pitch, box [box_rows, box_cols], 128-byte swizzle (or none).  Returns false on failure (message set).
bool make_tmap_2d(void* out_tmap /* CUtensorMap* */, const void* base, int elem_bytes, uint64_t rows,
                  uint64_t cols, uint64_t row_pitch_bytes, uint32_t box_rows, uint32_t box_cols,
                  bool swizzle128 = true);

// ------------------------------------------------------------------------------------------
// routing (route_meta.cu)
// ------------------------------------------------------------------------------------------
struct RouteBufs {
  int32_t* chunk_counts;      // [nchunks*E]
  int32_t* expert_offsets;    // [E+1]
  int32_t* block_offsets;     // [E+1]
  int32_t* tile_offsets;      // [E+1]
  int32_t* expert_order;      // [E] experts by descending row count
  int32_t* scalars;           // [4]: num_blocks, num_tiles, num_pairs
  int32_t* pair_offsets;      // nullable [E+1]: prefix of ceil(tiles_e / 2)
  const int32_t* num_valid;   // nullable device count: only tokens t < count are routed
  int32_t* x_gather_idx;      // [TK]
  int32_t* s_scatter_idx;     // [TK]
  int32_t* s_reverse;         // [TK]
  int32_t* token_position_to_id;  // [Nb*B]
  int32_t* block_to_expert;   // [Nb]
  int32_t* tile_row_flat;     // [P]
  int32_t* flat_tile_row;     // [TK]
  int32_t* tile_expert;       // [P/128]
  int32_t* num_blocks_out;    // nullable public copy of scalars[0]
  int32_t* status;
  int32_t* zero_counters;     // nullable: nzero counters set to 0 by the routing kernels
  int nzero;
};
int route_nchunks(int64_t TK);
// size checks shared by moe_route_meta and moe_route_meta_noalloc (same order, same messages)
int check_route_sizes(const char* who, int T, int K, int E, int block_size);
// order[0..num_tiles) = tiles sorted (bucketed) by the token of their first row
int launch_tile_order(const int32_t* tile_row_flat, const int32_t* num_tiles, int T, int K, int32_t* order,
                      cudaStream_t st);
int launch_route_meta(const int32_t* ids, int T, int K, int E, int B, int64_t Nb, int64_t P,
                      const RouteBufs& r, cudaStream_t st);
// routing metadata supplied by the caller (checked; tile tables derived into r)
struct RouteMetaIn {
  const int32_t* expert_offsets;        // [E+1]
  const int32_t* s_scatter_idx;         // [T*K]
  const int32_t* block_offsets;         // [E+1]
  const int32_t* token_position_to_id;  // [Nb*B] or null (checked only)
  const int32_t* block_to_expert;       // [Nb] or null (checked only)
};
int launch_route_meta_in(const RouteMetaIn& in, const int32_t* ids, int T, int K, int E, int B, int64_t Nb, int64_t P,
                         const RouteBufs& r, cudaStream_t st);

// ------------------------------------------------------------------------------------------
// gathers / quantisation (prep.cu)
// ------------------------------------------------------------------------------------------
struct PrepArgs {
  const uint16_t* dout;      // [T,H] bf16
  const uint16_t* x;         // [T,H] bf16
  const float* s;            // [T*K]
  const uint16_t* b2;        // [E,H] bf16 or null
  const int32_t* tile_row_flat;
  const int32_t* tile_expert;
  const int32_t* num_tiles;  // device scalar
  const int32_t* tile_order; // nullable: processing order of the tiles (CTA i takes tile_order[i])
  int H, K;
  int64_t P;                 // tile-row capacity (leading dim of transposed outputs)
  int mx, fmt, scale_t;      // MXFP8 outputs; fp8 format; multiply dout^T by s (affinity on H)
  void* dout_g; uint8_t* dout_g_sf;    // [P,H]
  void* dout_gt; uint8_t* dout_gt_sf;  // [H,P]
  void* x_gt; uint8_t* x_gt_sf;        // [H,P]
  void* x_g; uint8_t* x_g_sf;          // [P,H] row-major (nullable: only when h is recomputed)
  int skip_dout_t;                     // dout_gt is built elsewhere (from a saved s*dout checkpoint)
  float* ds_bias;                      // [P] <dout_t, b2_e> or null
  float* db2_part;                     // with biases: [P/128][4][H] column sums of s*dout per tile
                                       // (four 32-row quarters of its rows; [P/128][H] with no_t), or null
  // BF16 with MN-major weight-gradient operands: no transposed outputs (no_t); dout_b, when not null,
  // gets the rows of the dW2 GEMM's B operand ([P,H]: s*dout with dout_b_s, else dout), and db2's
  // partials are per-tile column sums ([P/128][H]) taken in the row-wise phase
  int no_t;
  void* dout_b;
  int dout_b_s;                        // dout_b rows are s*dout (else dout)
  uint32_t k_mul; int k_shift;         // set by launch_prep: f / K = umulhi(f, k_mul) >> (k_shift - 1)
                                       // for 0 <= f < 2^31 (k_shift = 0: K = 1)
};
int launch_prep(const PrepArgs& a, cudaStream_t st);
// a'^T [I,P] from an [N,I,B] block checkpoint of a (times s when s_or_null) or s*a
int launch_apt_from_ckpt(const uint16_t* ckpt, int I, int B, int64_t P, const int32_t* num_tiles,
                         const int32_t* tile_expert, const int32_t* tile_offsets, const int32_t* block_offsets,
                         const int32_t* tile_row_flat, const float* s_or_null, int mx, int fmt, void* out,
                         uint8_t* out_sf, cudaStream_t st);
// slot[p] = block-layout slot of tile row p, -1 for padding
int launch_tile_row_slot(int64_t P, int B, const int32_t* num_tiles, const int32_t* tile_expert,
                         const int32_t* tile_offsets, const int32_t* block_offsets, const int32_t* tile_row_flat,
                         int32_t* slot, cudaStream_t st);

// scales of an [R, C] MXFP8 B operand re-tiled into ceil(bn / 128) atoms per bn-row tile
// (R % bn == 0, R and C multiples of 128); dst holds (R / bn) * ceil(bn / 128) * (C / 128) * 512 bytes
int launch_sf_retile(const uint8_t* src, int64_t R, int64_t C, int bn, uint8_t* dst, cudaStream_t st);

int launch_quant_rowwise(const uint16_t* in, int64_t src_rows, int64_t rows, int64_t cols, int64_t ld,
                         const int32_t* row_index, int fmt, uint8_t* q, uint8_t* sf, int tiled, cudaStream_t st);
// colwise: out is the transposed [cols, rows] matrix, fp8 (+scales) when mx, else bf16
int launch_quant_colwise(const uint16_t* in, int64_t src_rows, int64_t rows, int64_t cols, int64_t ld,
                         const int32_t* row_index, int mx, int fmt, void* q, uint8_t* sf, int tiled,
                         cudaStream_t st);

// MXFP8 operands of the dense linear backward in one launch (linear.cu): dY row-wise [M,N], and the
// transposed W^T [K,N], dY^T [N,M], X^T [K,M], each with tiled scales; M, N, K multiples of 128
int launch_linear_quant(const uint16_t* dY, const uint16_t* W, const uint16_t* X, int64_t M, int64_t N, int64_t K,
                        int fmt, uint8_t* dY_q, uint8_t* dY_sf, uint8_t* Wt_q, uint8_t* Wt_sf, uint8_t* dYt_q,
                        uint8_t* dYt_sf, uint8_t* Xt_q, uint8_t* Xt_sf, cudaStream_t st);

// ------------------------------------------------------------------------------------------
// tcgen05 grouped GEMM (gemm_*.cu)
// ------------------------------------------------------------------------------------------
enum GemmMode { kMGrouped = 0, kKGrouped = 1 };
// kEpiDSwiGLU2: the dSwiGLU epilogue with two groups of epilogue warps taking alternate 32-feature
// chunks (sixteen warps, three checkpoint buffers, one pipeline stage fewer)
enum EpiKind { kEpiStore = 0, kEpiDSwiGLU = 1, kEpiCkpt = 2, kEpiDSwiGLU2 = 3 };
// dSwiGLU epilogue (G1): warps per TMEM lane quarter; each takes 32 / kG1Subs of every 32 columns
// and writes one ds partial per (row, N tile).
#ifndef MOEBWD_G1_SUBS
#define MOEBWD_G1_SUBS 2
#endif
constexpr int kG1Subs = MOEBWD_G1_SUBS;
static_assert(kG1Subs == 2 || kG1Subs == 4, "G1 epilogue warps per lane quarter");

struct GemmParams {
  int mode;
  int M, N, K;             // M-grouped: K = contraction; K-grouped: M, N per expert
  int m_tiles;             // M-grouped: capacity tiles (used when num_tiles is null); K-grouped: M/128
  int n_tiles;             // N / BN
  int num_experts;
  const int32_t* tile_expert;   // M-grouped: expert of each 128-row tile (null: expert 0)
  const int32_t* num_tiles;     // M-grouped: device count of tiles (null: m_tiles)
  const int32_t* tile_offsets;  // K-grouped: [E+1] tile-row offsets
  const int32_t* expert_order;  // K-grouped: [E] processing order (null: 0..E-1)
  int b_rows_per_expert;        // M-grouped: B rows per expert (0: shared B)
  // block scales (MXFP8)
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sfa_ktiles, sfb_ktiles;   // 128-column tiles along K in the tiled scale layouts
  int fmt_a, fmt_b;
  // epilogue
  int epi;
  void* out;
  int64_t ldo;
  int64_t out_expert_stride;    // K-grouped: elements between experts' outputs
  // dSwiGLU epilogue (G1)
  const float* s;
  const int32_t* tile_row_flat;
  const int32_t* e_tile_offsets;
  const int32_t* block_offsets;
  const uint16_t* ckpt;         // [N,2,I,B]
  const uint16_t* b1;           // G0 (checkpoint epilogue): [E,2I] bias or null
  int I, B, affinity_on_i, fmt_act;
  int glu;                      // MOE_GLU_SWIGLU or MOE_GLU_GEGLU
  int interleaved;              // dh (and W1, dW1, db1) columns: gate_i, up_i at 2i, 2i+1
  const uint16_t* gate_act;     // [N,I,B] saved act(gate) (block layout) or null
  int64_t P;
  void* dh; uint8_t* dh_sf;
  void* dht; uint8_t* dht_sf;
  void* apt; uint8_t* apt_sf;
  float* ds_part;               // [P, kG1Subs*groups*I/BN] (groups: 2 for kEpiDSwiGLU2, else 1)
  float* db1_part;              // BF16 with biases: [P/128][4][2I] column sums of dh per tile and TMEM
                                // lane quarter (W1's gate/up layout), or null
  // CTA-pair kernel, M-grouped: expert e's 128-row tiles form ceil(tiles_e / 2) pairs; pair_offsets
  // [E+1] is their prefix (null: one expert, pairs of consecutive tiles), num_pairs its device total
  const int32_t* pair_offsets;
  const int32_t* num_pairs;
  int32_t* tile_counter;        // zeroed before the launch: dynamic tile claims
  int accumulate;               // store epilogue: add the tile to the output instead of overwriting
  int32_t* status;
  uint64_t wait_ns;             // limit of each pipeline wait (set by launch_gemm from MOE_OPT_WAIT_LIMIT_NS)
  // dSwiGLU GEMM (G1) with a gathered A operand: A row p is row tile_row_flat[p] / a_gather_div of
  // a_gather (row pitch a_gather_ld bytes; padding rows read row 0, whose results are discarded),
  // copied by the producer warp into the swizzled stage; null: A comes through the tensor map
  const void* a_gather;
  int64_t a_gather_ld;
  int a_gather_div;
  // BF16: operand A (B) stored MN-major, i.e. as the [K, M] ([K, N]) matrix with M (N) contiguous,
  // read through 64 x 64 tensor-map boxes and the tensor core's MN-major descriptors
  int a_mn, b_mn;
  int ap_rows;                  // BF16 dSwiGLU GEMM: a' written as rows [P,I] at apt (for an MN-major read)
  int ap_s;                     // a' = s a also for affinity on H (the dW2 GEMM then reads unscaled dout)
};

// A [rows, K] and B [rows, K] K-major operands (bf16 or fp8 bytes), tile counts in p.
// The dSwiGLU epilogue also reads the checkpoint [N*2*I, B] (bf16) through a third tensor map.
int launch_gemm(bool mx, int BN, const GemmParams& p, const void* A, int64_t a_rows, int64_t a_cols,
                const void* B, int64_t b_rows, int64_t b_cols, cudaStream_t st, const void* ckpt = nullptr,
                int64_t ck_rows = 0, int64_t ck_cols = 0);
int launch_gemm_bf16(int BN, const GemmParams& p, const void* tmA, const void* tmB, const void* tmC, int grid,
                     cudaStream_t st);
int launch_gemm_mx(int BN, const GemmParams& p, const void* tmA, const void* tmB, const void* tmC, int grid,
                   cudaStream_t st);
// CTA-pair GEMM (gemm_pair.cu): pair tiles of 256 rows x BN (128 or 256) columns, p.n_tiles = N / BN,
// store or checkpoint epilogue; tmSFA / tmSFB map the tiled scales as rows of 512 bytes (MXFP8).
// max_pairs bounds the pairs launched.
int launch_gemm_pair(bool mx, int BN, const GemmParams& p, const void* tmA, const void* tmB, const void* tmC,
                     const void* tmSFA, const void* tmSFB, int max_pairs, cudaStream_t st);

// ------------------------------------------------------------------------------------------
// reductions (reduce.cu)
// ------------------------------------------------------------------------------------------
int launch_dx_scatter_sum(const uint16_t* dx_exp, const int32_t* flat_tile_row, int T, int K, int H,
                          uint16_t* dx, cudaStream_t st);
// [T*E] masked view of ds: out[t*E + e] = sum of ds[t,k] over the slots k of token t routed to e
int launch_ds_masked(const float* ds, const int32_t* ids, const int32_t* num_valid, int T, int K, int E, float* out,
                     cudaStream_t st);
int launch_ds_finalize(const float* ds_part, int nparts, const float* ds_bias, const int32_t* flat_tile_row,
                       int64_t TK, float* ds, cudaStream_t st);
// out[e, j] = sum over tile rows p of expert e of buf[j, p] (* w[flat(p)] when w != null)
int launch_segment_rowsum(const uint16_t* buf, int64_t ld, int R, const int32_t* tile_offsets, int E,
                          const float* w, const int32_t* tile_row_flat, float* out, cudaStream_t st,
                          int accumulate = 0);
// out[e, f] (+)= sum over expert e's 128-row tiles t and k < parts of part[(t * parts + k) * F + f]
// (in that order: deterministic)
// and, in the same launch when part2 is given, out2[e, f] (+)= the same sums of part2 (parts2, F2)
int launch_bias_parts_reduce(const float* part, int parts, int64_t F, const int32_t* tile_offsets, int E,
                             float* out, cudaStream_t st, int accumulate, const float* part2 = nullptr,
                             int parts2 = 0, int64_t F2 = 0, float* out2 = nullptr);

}  // namespace moebwd
