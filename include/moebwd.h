/*
 * moebwd -- backward pass of a top-K routed SwiGLU Mixture-of-Experts layer on one GB300 GPU
 * (sm_103a), BF16 and MXFP8, plus the dense MXFP8 linear backward.  C ABI.
 *
 * Sources of the operations (pages):
 *   [BW]  "Blockwise MM Backward MXFP8 Kernel API Reference" (blockwise_mm_bwd_mxfp8): parameters
 *         hidden_states, expert_affinities_masked, gate_up_proj_weight [E,H,2,I],
 *         down_proj_weight [E,I,H], token_position_to_id [N*B], block_to_expert [N,1],
 *         output_hidden_states_grad, block_size in {128,256,512,1024},
 *         gate_up_proj_act_checkpoint_T [N,2,I,B], gate_up_weight_scales, down_weight_scales;
 *         the returned gradient tuple; "Dimensions": N = (T*TopK - (E-1))/B + E - 1.
 *   [MM]  "Matmul MXFP8 Backward Kernel API Reference" (matmul_mxfp8_backward): "Forward pass
 *         convention" Y = X @ W^T; dX = dY @ W; dW = dY^T @ X; float8_dtype; output_dtype.
 *   [SM]  sonic-moe functional/backward.py: expert_frequency_offset, x_gather_idx, s_scatter_idx,
 *         s_reverse_scatter_idx; _down_projection_backward_act (gemm_dgated with colvec_scale and
 *         colvec_reduce), db2_and_ds_kernel, _down_projection_backward_weight,
 *         _up_projection_backward_act, db1_kernel, _up_projection_backward_weight,
 *         _token_broadcast_backward.
 *
 * Conventions for every entry point:
 *   - Pointers marked (device) are CUDA device pointers on the current device; (host) are host.
 *     The library never allocates device memory: scratch comes from the caller's workspace,
 *     whose size the matching *_workspace_size() call reports.  Workspace pointers must be
 *     256-byte aligned.
 *   - BF16 tensors are passed as `const void*` / `void*` holding IEEE bfloat16 values; all
 *     matrices are dense row-major with the shapes given.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream) and do
 *     not synchronise the host.  Inputs are never modified; outputs are overwritten.
 *   - Return value: MOE_OK, or a negative MOE_ERR_* code; moe_last_error() then holds a message
 *     (per host thread).  Errors detected on the device (invalid expert ids, a pipeline wait that
 *     ran out of time) are OR-ed into the caller's `status_dev` word, readable after the stream
 *     has been synchronised; a nonzero word means the outputs are not valid.
 */
#ifndef MOEBWD_H
#define MOEBWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same handle as cudaStream_t */

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = -1,     /* null pointer, bad shape, misaligned buffer, workspace too small */
  MOE_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. H not a multiple of 128) */
  MOE_ERR_CUDA = -3,        /* a CUDA launch or driver call failed */
  MOE_ERR_DEVICE = -4       /* reserved: device-side errors are reported through status_dev */
};

/* Bits of the device status word. */
enum {
  MOE_STATUS_BAD_EXPERT_ID = 1, /* some ids[t,k] outside [0,E); those rows are skipped */
  MOE_STATUS_TIMEOUT = 2,       /* a pipeline wait exceeded its time limit; outputs invalid */
  MOE_STATUS_BAD_ROUTE_META = 4 /* caller-supplied routing metadata is not a routing of the ids
                                   (moe_bwd with expert_offsets given); outputs invalid */
};

enum { MOE_PREC_BF16 = 0, MOE_PREC_MXFP8 = 1 };
/* Where the routing affinity multiplies in the forward ([BW] down_proj_act_checkpoint "Affinity H
 * mode", scaled_intermediate_checkpoint_T "Affinity I mode").  The forward value is the same in
 * both; the mode selects which operand of the dW_down GEMM carries the score. */
enum { MOE_AFFINITY_ON_H = 0, MOE_AFFINITY_ON_I = 1 };
enum { MOE_FP8_E4M3 = 0, MOE_FP8_E5M2 = 1 };
/* Quantisation direction of mxfp8_quantize. */
enum { MOE_QUANT_ROWWISE = 0, MOE_QUANT_COLWISE = 1 };
/* Layout of E8M0 scale bytes. */
enum { MOE_SF_PLAIN = 0, MOE_SF_TILED = 1 };
/* Source of the gate/up pre-activations h = x W1_e + b1_e that the dSwiGLU step needs.
 * CHECKPOINT: read from [BW] gate_up_proj_act_checkpoint_T [N,2,I,B] (gate_up_ckpt).
 * RECOMPUTE:  recomputed inside moe_bwd by a forward grouped GEMM over the gathered rows of
 *             hidden_states and the gate/up weights (the pre-activation that checkpoint stores;
 *             its forward is h = x W1_e + b1_e of the routed SwiGLU layer), written to a
 *             checkpoint of the same layout in the workspace, rounded to bf16 like the stored one.
 *             Costs 4*T*K*H*I extra FLOPs and saves the caller the [N,2,I,B] tensor. */
enum { MOE_ACT_CHECKPOINT = 0, MOE_ACT_RECOMPUTE = 1 };
/* Gated activation a = act(gate) * up (sonic-moe `activation_type`): SwiGLU act = SiLU, GeGLU
 * act = GELU with the exact normal CDF, GELU(z) = z * Phi(z). */
enum { MOE_GLU_SWIGLU = 0, MOE_GLU_GEGLU = 1 };
/* Column layout of gate and up in W1 [E,H,2I] (and in dW1, db1): CONCAT gate_i at i, up_i at I + i;
 * INTERLEAVED gate_i at 2i, up_i at 2i + 1 (sonic-moe's interleaved gate/up layout).  The
 * checkpoint [N,2,I,B] and W1t (recomputation) keep gate and up apart in either case. */
enum { MOE_GATE_UP_CONCAT = 0, MOE_GATE_UP_INTERLEAVED = 1 };

/* Message of the last failed call on this host thread ("" if none). */
const char* moe_last_error(void);

/* Library version string. */
const char* moe_version(void);

/* ------------------------------------------------------------------------------------------ */
/* Routing metadata                                                                            */
/* ------------------------------------------------------------------------------------------ */

/* [BW] "Dimensions": N = ceil((T*K - (E-1)) / B) + E - 1, the largest number of blocks any
 * routing of T*K rows over E experts needs (the "/" is read as a ceiling division); T*K when
 * T*K < E - 1; 0 when T*K == 0.  Pure host function. */
int64_t moe_num_blocks_bound(int64_t T, int K, int E, int block_size);

/* Bytes of workspace moe_route_meta needs; 0 for sizes moe_route_meta rejects (block_size outside
 * {128,256,512,1024}, E outside [1, 1024], K <= 0, T < 0). */
size_t moe_route_meta_workspace_size(int T, int K, int E, int block_size);

/* Routing metadata from expert ids ([BW] token_position_to_id, block_to_expert; [SM]
 * expert_frequency_offset, x_gather_idx, s_scatter_idx, s_reverse_scatter_idx).
 *
 * ids (device) int32 [T,K].  Rows are grouped by expert; inside an expert the order is by flat
 * index f = t*K + k (stable).  Outputs (device, int32), with TKv = number of valid ids:
 *   expert_offsets [E+1]        exclusive prefix of per-expert row counts
 *   x_gather_idx [T*K]          grouped row r < TKv -> token t
 *   s_scatter_idx [T*K]         grouped row r < TKv -> flat index f
 *   s_reverse_scatter_idx [T*K] flat f -> grouped row, -1 for an invalid id
 *   token_position_to_id [N*B]  slot -> token, -1 for padding (N = moe_num_blocks_bound)
 *   block_to_expert [N]         block -> expert, -1 for blocks >= *num_blocks
 *   block_offsets [E+1]         exclusive prefix of ceil(n_e / B)
 *   num_blocks [1]              total blocks in use
 * status_dev (device) int32 [1]: MOE_STATUS_BAD_EXPERT_ID is OR-ed in for ids outside [0,E).
 * Entries x_gather_idx / s_scatter_idx [TKv, T*K) are left unchanged.  block_size must be one of
 * 128, 256, 512, 1024; 1 <= E <= 1024; T*K < 2^31.  T = 0: the offsets and num_blocks are zeroed and
 * nothing else is written (ids, the [T*K] and [N*B] arrays, block_to_expert and the workspace may then
 * be null). */
int moe_route_meta(const int32_t* ids, int T, int K, int E, int block_size, int32_t* expert_offsets,
                   int32_t* x_gather_idx, int32_t* s_scatter_idx, int32_t* s_reverse_scatter_idx,
                   int32_t* token_position_to_id, int32_t* block_to_expert, int32_t* block_offsets,
                   int32_t* num_blocks, int32_t* status_dev, void* workspace, size_t workspace_bytes,
                   moe_stream_t stream);

/* moe_route_meta without a workspace, for callers that cannot allocate device memory (code inside
 * a memory pool or arena without raw allocations, hooks that may not call cudaMalloc mid-step,
 * callers that must not allocate after start-up).  None of the source pages has a counterpart: it is
 * an interface addition of this library.  Same arguments, outputs and errors as moe_route_meta, minus
 * the workspace (its size arguments are checked first, in moe_route_meta's order, with the same
 * codes): the scratch is a fixed 4 MiB device array owned by the library (held on every GPU
 * that loads it, until exit), which admits about T*K <= 150k routed rows for E <= 128 (the exact
 * limit is moe_route_meta_workspace_size(T,K,E,B) <= 4 MiB; larger sizes return
 * MOE_ERR_UNSUPPORTED with a message and launch nothing).  The first call on a device looks up the
 * array's device address and should come before any stream capture.  All calls on a device share
 * the array: calls that overlap on the GPU race and must be serialised by the caller.  Allocates
 * no memory. */
int moe_route_meta_noalloc(const int32_t* ids, int T, int K, int E, int block_size, int32_t* expert_offsets,
                           int32_t* x_gather_idx, int32_t* s_scatter_idx, int32_t* s_reverse_scatter_idx,
                           int32_t* token_position_to_id, int32_t* block_to_expert, int32_t* block_offsets,
                           int32_t* num_blocks, int32_t* status_dev, moe_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* MXFP8 quantisation                                                                          */
/* ------------------------------------------------------------------------------------------ */

/* Quantise a BF16 matrix to MXFP8: groups of 32 consecutive elements along one dimension share an
 * E8M0 scale ([BW] first paragraph, gate_up_weight_scales; [MM] float8_dtype).  Scale rule (OCP
 * MX v1.0): byte = clamp(floor(log2(amax)) - emax + 127, 0, 254), emax = 8 (e4m3) / 15 (e5m2),
 * floor(log2) taken from the binary exponent of amax; element = round-to-nearest-even of
 * v * 2^(127 - byte), saturated to +-448 / +-57344, the sign kept: a value that rounds to zero
 * encodes as 0x00 when positive and 0x80 (-0) when negative, as a float8 cast of the scaled value does.
 *
 * in (device) bf16 [src_rows, cols] with row stride `ld` elements (ld >= cols, ld % 8 == 0).
 * row_index (device, nullable) int32 [rows]: output row r reads input row row_index[r], -1 reads
 *   zeros; NULL means row r reads row r (then rows <= src_rows).
 * axis = MOE_QUANT_ROWWISE: groups run along cols; q (device) is [rows, cols];
 *   scales (device) are [rows, cols/32] (PLAIN) or tiled for the [rows, cols] matrix.
 * axis = MOE_QUANT_COLWISE: groups run along rows; q (device) holds the TRANSPOSED matrix
 *   [cols, rows] so that every group is contiguous; scales are [cols, rows/32] (PLAIN) or tiled
 *   for the [cols, rows] matrix.
 * Tiled scale layout (MOE_SF_TILED), the one the block-scaled tensor-core MMA consumes, for a
 * quantised matrix [R, C] (groups along C): 512-byte atoms of 128 rows x 4 groups, atom (R/128 x
 * C/128 grid, row-major) at byte ((r/128)*(C/128) + c/128)*512, inside it byte
 * (r%32)*16 + ((r%128)/32)*4 + (c/32)%4.  It requires R % 128 == 0 and C % 128 == 0.
 * The grouped dimension must be a multiple of 32, the other a multiple of 16 (ROWWISE) or
 * 128 (COLWISE).  rows == 0 or cols == 0: nothing is written (the pointers may be null). */
int mxfp8_quantize(const void* in, int64_t src_rows, int64_t rows, int64_t cols, int64_t ld,
                   const int32_t* row_index, int axis, int fp8_fmt, uint8_t* q, uint8_t* scales,
                   int scale_layout, moe_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* MoE layer backward                                                                          */
/* ------------------------------------------------------------------------------------------ */

/* Arguments of moe_bwd.  Forward being differentiated ([BW] Background; [SM] backward.py): for
 * every token t and slot k with e = ids[t,k], h = x_t W1_e + b1_e (gate = h[:I], up = h[I:]),
 * a = SiLU(gate) * up, y = a W2_e + b2_e, out_t = sum_k s[t,k] y.  The pass returns
 *   dx = d<dout,out>/dx [T,H] (bf16), dW1 [E,H,2I] (bf16), dW2 [E,I,H] (bf16),
 *   ds[t,k] = <dout_t, y> [T,K] (fp32), db1 [E,2I] and db2 [E,H] (fp32, when has_bias).
 * Experts that receive no row get zero gradients. */
typedef struct MoeBwdArgs {
  int T, H, I, E, K;  /* tokens, hidden, intermediate (per half), experts, top-K */
  int block_size;     /* B in {128,256,512,1024}: block layout of the checkpoint */
  int precision;      /* MOE_PREC_BF16 or MOE_PREC_MXFP8 */
  int affinity;       /* MOE_AFFINITY_ON_H or MOE_AFFINITY_ON_I */
  int fp8_act;        /* MXFP8: format of activation-side operands (dout, x, dh, a'), default E5M2 */
  int fp8_w;          /* MXFP8: format of the pre-quantised weights, default E4M3 */
  int has_bias;       /* produce db1/db2 and add <dout_t, b2_e> to ds (from the unquantised values in
                         both precisions; MXFP8 with down_proj_act_ckpt returns MOE_ERR_UNSUPPORTED) */

  const void* x;     /* (device) bf16 [T,H]  hidden_states */
  const void* dout;  /* (device) bf16 [T,H]  output_hidden_states_grad */
  const void* W1;    /* (device) bf16 [E,H,2I] gate|up weights (BF16 precision) */
  const void* W2;    /* (device) bf16 [E,I,H] down weights (BF16 precision) */
  const uint8_t* W1_q;  /* (device) MXFP8: W1 as [E*H, 2I] quantised ROWWISE (groups along 2I) */
  const uint8_t* W1_sf; /*          its scales, MOE_SF_TILED for the [E*H, 2I] matrix */
  const uint8_t* W2_q;  /* (device) MXFP8: W2 as [E*I, H] quantised ROWWISE (groups along H) */
  const uint8_t* W2_sf; /*          its scales, MOE_SF_TILED for the [E*I, H] matrix */
  const void* b2;       /* (device) bf16 [E,H] down bias (has_bias) */
  const float* s;       /* (device) fp32 [T,K] routing scores */
  const int32_t* ids;   /* (device) int32 [T,K] expert ids; -1 marks an unused slot (a token routed to
                           fewer than K experts: variable top-K); any other id outside [0,E) is
                           reported in status_dev (MOE_STATUS_BAD_EXPERT_ID) and skipped */
  const void* gate_up_ckpt; /* (device) bf16 [N,2,I,B] gate/up pre-activation checkpoint in the
                               block layout of moe_route_meta (N = moe_num_blocks_bound):
                               gate of the j-th row of expert e at [blk,0,:,b], up at [blk,1,:,b],
                               slot blk*B + b = block_offsets[e]*B + j. */

  void* dx;     /* (device) bf16 [T,H] */
  void* dW1;    /* (device) bf16 [E,H,2I] */
  void* dW2;    /* (device) bf16 [E,I,H] */
  float* ds;    /* (device) fp32 [T,K] */
  float* db1;   /* (device) fp32 [E,2I] (has_bias) */
  float* db2;   /* (device) fp32 [E,H] (has_bias) */

  int32_t* status_dev;    /* (device) int32 [1]; reset to 0 by the call, then OR-ed with MOE_STATUS_* */
  void* workspace;        /* (device) scratch, 256-byte aligned */
  size_t workspace_bytes; /* >= moe_bwd_workspace_size(args) */
  int accumulate;         /* [BW] accumulation / grad-init: 0 overwrites dW1, dW2, db1, db2; 1 adds this
                             pass's gradients to their current contents (bf16 adds for dW, fp32 for db).
                             dx and ds are always overwritten. */
  int act_src;            /* MOE_ACT_CHECKPOINT (gate_up_ckpt read) or MOE_ACT_RECOMPUTE (gate_up_ckpt
                             unused, may be NULL; the fields below are read) */
  const void* W1t;        /* (device) RECOMPUTE, BF16: bf16 [E,2I,H], W1 with each expert's block
                             transposed, rows [gate | up] (row j of expert e = column j of the
                             concat-layout W1[e], whatever gate_up_layout) */
  const uint8_t* W1t_q;   /* (device) RECOMPUTE, MXFP8: W1t as [E*2I, H] quantised ROWWISE (groups
                             along H) with fp8_w */
  const uint8_t* W1t_sf;  /*          its scales, MOE_SF_TILED for the [E*2I, H] matrix */
  const void* b1;         /* (device) RECOMPUTE: bf16 [E,2I] gate/up bias added to h ([gate | up]), or NULL */
  float* ds_masked;       /* (device) fp32 [T*E] or NULL: [BW] expert_affinities_masked_grad, ds laid out
                             over all experts of each token: [t*E + e] = ds of the slot of token t
                             routed to e (repeated selections add), 0 where e was not selected */
  const int32_t* num_valid_tokens; /* (device) int32 [1] or NULL: [BW] num_valid_tokens, only the
                             leading min(n, T) tokens are routed (values <= 0 route none); later
                             tokens take no part and get zero dx rows and ds / ds_masked entries */
  int glu;                /* MOE_GLU_SWIGLU (default 0) or MOE_GLU_GEGLU */
  int gate_up_layout;     /* MOE_GATE_UP_CONCAT (default 0) or MOE_GATE_UP_INTERLEAVED */
  /* [BW] optional checkpoints: forward values that replace recomputed ones in the dW_down product
   * (dW2_e = sum a'^T (s dout)); each (device) bf16 in the block layout of gate_up_ckpt, or NULL.
   * With one given, moe_bwd builds that operand from it and does not compute it itself. */
  const void* intermediate_ckpt;        /* [N,I,B] a = act(gate)*up (intermediate_checkpoint_T); with
                                           the affinity on I, dW_down uses s * this */
  const void* scaled_intermediate_ckpt; /* [N,I,B] s*a (scaled_intermediate_checkpoint_T), affinity on I
                                           only; preferred over intermediate_ckpt */
  const void* down_proj_act_ckpt;       /* [N,B,H] s*dout per slot (down_proj_act_checkpoint), affinity
                                           on H only; also the rows summed into db2 */
  /* [BW] gate_act_checkpoint_T: (device) bf16 [N,I,B] act(gate) saved by the forward (SiLU, or GELU
   * with MOE_GLU_GEGLU), in the block layout of gate_up_ckpt, or NULL.  Given, the dSwiGLU step takes
   * act(gate) from it wherever the activation's value enters (a = act(gate)*up for ds and the dW_down
   * factor, dup = dA*act(gate)); act'(gate) in dgate still needs the pre-activation, so gate_up_ckpt
   * (or the recomputation) stays required.  16-byte aligned. */
  const void* gate_act_ckpt;
  /* Routing metadata from the caller ([BW] token_position_to_id, block_to_expert, "Dimensions";
   * [SM] expert_frequency_offset, s_scatter_idx), e.g. kept from the forward pass, in the layout
   * moe_route_meta writes (all (device) int32).  All NULL: moe_bwd computes it from ids.  Given,
   * expert_offsets, s_scatter_idx and block_offsets are required and moe_bwd takes from them which
   * grouped row is which (token, slot), the rows of each expert in the given order (the MXFP8
   * token-direction groups are 32 consecutive rows in that order), and where each row's checkpoint
   * column sits: row j of expert e at block-layout slot block_offsets[e]*B + j.  ids stay required
   * and must agree.  Everything is checked on the device before use: offsets that do not start at 0,
   * decrease, exceed the routed slots or give an expert fewer blocks than ceil(rows/B) (or blocks
   * beyond N) make every row drop out; a row whose flat index is out of range, repeated, or routed to
   * another expert by ids drops out; a routed slot that no row names, or a given token_position_to_id
   * / block_to_expert entry that disagrees, is reported too -- each case OR-s
   * MOE_STATUS_BAD_ROUTE_META into status_dev (outputs then invalid, but no access goes out of
   * bounds).  With num_valid_tokens, rows may name only the leading valid tokens' slots. */
  const int32_t* expert_offsets;       /* [E+1] [SM] expert_frequency_offset: rows of expert e are the
                                          grouped rows expert_offsets[e] .. expert_offsets[e+1]-1 */
  const int32_t* s_scatter_idx;        /* [T*K] grouped row -> flat slot t*K + k */
  const int32_t* block_offsets;        /* [E+1] first block of each expert in the block layout */
  const int32_t* token_position_to_id; /* [N*B] or NULL: [BW] slot -> token (checked only) */
  const int32_t* block_to_expert;      /* [N] or NULL: [BW] block -> expert (checked only) */
} MoeBwdArgs;

/* Bytes of workspace moe_bwd needs for these shapes and options (pointers are not read). */
size_t moe_bwd_workspace_size(const MoeBwdArgs* args);

/* The whole backward on `stream`: routing metadata, gathers/quantisation, the four grouped GEMMs
 * (dA with the fused dSwiGLU/ds epilogue, dW_down, dx_expanded, dW_gate_up), the top-K
 * scatter-sum into dx, ds and the bias gradients.  Requirements: H % 128 == 0, I % 128 == 0,
 * 1 <= K <= E <= 1024, K <= 64, T*K < 2^31, x/dout/weights 16-byte aligned; other sizes return
 * MOE_ERR_INVALID or MOE_ERR_UNSUPPORTED before any launch.  T = 0: dW1, dW2 (and db1, db2) are
 * zeroed, or left as they are with accumulate; the token-sized pointers may then be null. */
int moe_bwd(const MoeBwdArgs* args, moe_stream_t stream);

/* Regions of the moe_bwd workspace (for inspection of intermediates in tests and debugging).
 * Rows of the grouped operands are "tile rows": the rows of expert e occupy
 * [tile_offsets[e], tile_offsets[e] + n_e) with tile_offsets[e] a multiple of 128 and padding rows
 * zero; P = capacity of the tile-row space. */
enum {
  MOE_WS_EXPERT_OFFSETS = 0, /* int32 [E+1] */
  MOE_WS_TILE_OFFSETS,       /* int32 [E+1] */
  MOE_WS_BLOCK_OFFSETS,      /* int32 [E+1] */
  MOE_WS_TILE_ROW_FLAT,      /* int32 [P]   tile row -> flat t*K+k, -1 padding */
  MOE_WS_FLAT_TILE_ROW,      /* int32 [T*K] flat -> tile row, -1 invalid id */
  MOE_WS_DOUT_G,             /* G1 A operand: dout rows [P,H] (bf16 | fp8); empty with MOE_OPT_G1_GATHER = 1 */
  MOE_WS_DOUT_G_SF,          /*   its tiled scales (MXFP8) */
  MOE_WS_DOUT_GT,            /* G3 B operand: [H,P] (bf16 | fp8), s-scaled for affinity on H; BF16 under
                                MOE_OPT_MN_OPERANDS: rows [P,H] of dout when G1 gathers its own, of s*dout
                                when a' comes from a saved intermediate (affinity on H), else unused (G3
                                reads DOUT_G; for affinity on H, G1 writes a' = s*a) */
  MOE_WS_DOUT_GT_SF,
  MOE_WS_X_GT,               /* G4 A operand: [H,P]; BF16 under MOE_OPT_MN_OPERANDS: x's gathered rows [P,H]
                                (unused when h is recomputed: G4 reads X_G) */
  MOE_WS_X_GT_SF,
  MOE_WS_DH,                 /* G2 A operand: dh [P,2I] */
  MOE_WS_DH_SF,
  MOE_WS_DH_T,               /* G4 B operand: dh^T [2I,P] (empty for BF16 under MOE_OPT_MN_OPERANDS, the default) */
  MOE_WS_DH_T_SF,
  MOE_WS_AP_T,               /* G3 A operand: a'^T [I,P] (s*a for affinity on I, a on H); BF16 under
                                MOE_OPT_MN_OPERANDS: a' rows [P,I], s*a for both affinities */
  MOE_WS_AP_T_SF,
  MOE_WS_DX_EXP,             /* G2 output: dx_expanded [P,H] bf16 */
  MOE_WS_X_G,                /* RECOMPUTE: G0 A operand, gathered x rows [P,H] (bf16 | fp8) */
  MOE_WS_X_G_SF,
  MOE_WS_GATE_UP_CKPT,       /* RECOMPUTE: G0 output, bf16 [Nb,2,I,B] in the checkpoint layout
                                (Nb = moe_num_blocks_bound; only the slots of routed tile rows are
                                written) */
  MOE_WS_DOUT_Q,             /* MXFP8 with MOE_OPT_G1_GATHER = 1: dout quantised once per token [T,H] fp8
                                (groups along H), the rows G1 gathers; DOUT_G then holds no codes, only
                                its tiled scales DOUT_G_SF (gathered) */
  MOE_WS_NUM_REGIONS
};
/* Offset and size in bytes of one region inside the workspace (0 bytes when unused). */
int moe_bwd_workspace_region(const MoeBwdArgs* args, int region, size_t* offset, size_t* bytes);

/* Capacity P of the tile-row space for these shapes. */
int64_t moe_tile_rows_capacity(int T, int K, int E);

/* ------------------------------------------------------------------------------------------ */
/* Router backward (the consumer of ds)                                                        */
/* ------------------------------------------------------------------------------------------ */

/* Forms of the router forward ([SM] `_topk_softmax_bwd`, `_topk_bwd`). */
enum {
  MOE_ROUTER_SOFTMAX_OVER_TOPK = 0, /* s = softmax over the K selected logits */
  MOE_ROUTER_TOPK_OVER_SOFTMAX = 1, /* s = top-K of softmax over all E logits (renorm: / their sum) */
  MOE_ROUTER_TOPK = 2               /* s = the K selected logits */
};

/* Gradient of the router logits from the gradient of the routing scores (dscores = moe_bwd's ds).
 *   SOFTMAX_OVER_TOPK: dlogits[idx_k] = s_k (g_k - <g, s>), 0 elsewhere; needs `scores` (forward s).
 *   TOPK_OVER_SOFTMAX: p = softmax(logits) recomputed over all E; dr = (g - <g, s>) / sum(p[idx])
 *                      when `renorm` (needs `scores`), else g; dlogits = p (scatter(dr) - <dr, p[idx]>)
 *                      for every logit; needs `logits`.
 *   TOPK:              dlogits[idx_k] = g_k, 0 elsewhere.
 * logits (device) fp32 [T,E]; scores, dscores (device) fp32 [T,K]; ids (device) int32 [T,K];
 * dlogits (device) fp32 [T,E], fully written.  K <= 64.  Repeated ids accumulate; ids outside [0,E)
 * are skipped.  fp32 arithmetic.  T = 0: nothing is written (the pointers may be null). */
int moe_router_bwd(int mode, int renorm, const float* logits, const float* scores, const float* dscores,
                   const int32_t* ids, int T, int K, int E, float* dlogits, moe_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* Instrumentation                                                                             */
/* ------------------------------------------------------------------------------------------ */

/* Stages of moe_bwd.  Launch order: ROUTE, PREP, G0 (RECOMPUTE only), G1, G3, G2, G4, REDUCE. */
enum {
  MOE_STAGE_ROUTE = 0, /* routing metadata */
  MOE_STAGE_PREP,      /* gathered / transposed / quantised activation operands */
  MOE_STAGE_G1,        /* dA = dout_g W2_e^T with the dSwiGLU + ds epilogue */
  MOE_STAGE_G3,        /* dW2_e = a'^T dout_g */
  MOE_STAGE_G2,        /* dx_expanded = dh W1_e */
  MOE_STAGE_G4,        /* dW1_e = x_g^T dh */
  MOE_STAGE_REDUCE,    /* dx scatter-sum, ds, bias sums */
  MOE_STAGE_G0,        /* RECOMPUTE only: h = x_g W1_e + b1_e (runs between PREP and G1) */
  MOE_NUM_STAGES
};

/* Stage timing.  While enabled, every moe_bwd call records CUDA events on its own stream at the
 * stage boundaries (no host synchronisation; up to 1024 calls are kept).  moe_profile_read waits
 * for the recorded events and returns, per stage, the total milliseconds over the profiled calls
 * (stage_ms[MOE_NUM_STAGES]) and the number of calls.  Enabling (or disabling) discards what was
 * recorded.  Process-global host state; not thread-safe. */
int moe_profile_enable(int enable);
int moe_profile_read(double* stage_ms, int max_stages, int* calls);

/* Number of kernels this library has launched in this process. */
uint64_t moe_kernel_launches(void);

/* ------------------------------------------------------------------------------------------ */
/* Options                                                                                     */
/* ------------------------------------------------------------------------------------------ */

/* Process-wide options, read by every later call on any host thread (set them while no call is
 * running).  None is needed for correct results: the defaults are the measured-fastest choices, and
 * every choice computes the same gradients (tile widths only change the order of fp32 additions
 * inside a GEMM).  They exist for tests, tuning runs and diagnosis.  A tile width that does not
 * divide the GEMM's N dimension falls back to the default; options that change a tile width change
 * moe_bwd_workspace_size, so query it after setting them. */
enum {
  MOE_OPT_WAIT_LIMIT_NS = 0, /* limit of each pipeline wait inside the GEMM kernels before the kernel
                                reports MOE_STATUS_TIMEOUT, drains what it has in flight and returns;
                                1 .. 6e10 ns, default 2e9 (2 s).  A short limit on a real workload makes
                                the kernels give up (a way to exercise that path without a fault); the
                                waits that drain copies and tensor-core work before a CTA exits keep 2 s */
  MOE_OPT_PAIR_GEMMS,        /* CTA-pair GEMMs: 0 never, 1 the BF16 store/recompute GEMMs where they
                                apply (default), 2 also MXFP8 */
  MOE_OPT_PAIR_TILE_N,       /* N width of the pair tile: 256 (default) or 128 */
  MOE_OPT_G1_TILE_N,         /* N tile of the dA/dSwiGLU GEMM: 0 automatic (default: MXFP8 192 where it
                                divides I, BF16 256 where it divides I, else 128), 128, 192 (MXFP8), 256 */
  MOE_OPT_G2_TILE_N,         /* N tile of dx_expanded: 0 automatic (256 where it divides H), 128, 256 */
  MOE_OPT_G3_TILE_N,         /* N tile of dW_down: 0 automatic (256 where it divides H), 128, 256 */
  MOE_OPT_G4_TILE_N,         /* N tile of dW_gate_up: 0 automatic (256), 128, 256 */
  MOE_OPT_PREP_TILE_ORDER,   /* 1 (default): the gather pass walks tiles in token order; 0: in index order */
  MOE_OPT_G1_GATHER,         /* 0 (default): the dA/dSwiGLU GEMM reads a gathered copy of dout written by
                                the gather pass (MOE_WS_DOUT_G); 1: it gathers the rows itself (from dout,
                                or for MXFP8 from dout quantised once per token, MOE_WS_DOUT_Q) with 16-byte
                                asynchronous copies -- same results, less memory, but slower (the copies of
                                one producer warp keep fewer bytes in flight than tensor-map loads) */
  MOE_OPT_G1_WARPS,          /* epilogue warps of the MXFP8 dA/dSwiGLU GEMM: 0 automatic (8), 8, or 16 (two
                                groups taking alternate 32-feature chunks, three checkpoint buffers, one
                                pipeline stage fewer: measured no faster -- the epilogue is bound by the
                                load/store unit's wavefronts, not by warps to hide latency); BF16 uses 8 */
  MOE_OPT_PDL,               /* 1 (default): the kernels of a call are launched with programmatic dependent
                                launch (each may be scheduled while the previous one finishes and waits on
                                the device for its results); 0: plain stream order */
  MOE_OPT_MN_OPERANDS,       /* BF16: 1 (default) the weight-gradient GEMMs read their token-major operands
                                as row-major [tokens, features] matrices through the tensor core's MN-major
                                layout: dW1 reads x's gathered rows and dh itself, dW2 reads a' rows and
                                dout (s*dout for affinity on H) rows, so prep builds no transposed copies
                                and the dA GEMM no dh^T or a'^T (the DH_T region is empty; X_GT, DOUT_GT
                                and AP_T hold rows; operands made from saved checkpoints stay transposed);
                                linear_bwd's BF16 GEMMs read dY, W and X themselves (no workspace copies);
                                0: transposed copies as for MXFP8 */
  MOE_OPT_LINEAR_CONCURRENT, /* linear_bwd: 1 (default) the dW GEMM runs on a second stream owned by the
                                library, concurrently with the dX GEMM on the caller's stream (ordered
                                after the quantised operands, joined back before the call returns, so
                                the caller's stream sees both results as before); the persistent CTAs of
                                one GEMM fill the SMs the other's last wave leaves idle.  0: both on the
                                caller's stream, one after the other */
  MOE_NUM_OPTIONS
};
/* Set an option; value -1 restores its default.  MOE_ERR_INVALID for an unknown option or value. */
int moe_set_option(int option, int64_t value);
/* Current value of an option (-1 for an unknown option). */
int64_t moe_get_option(int option);

/* ------------------------------------------------------------------------------------------ */
/* Dense linear backward (the E=1, K=1 degenerate case)                                        */
/* ------------------------------------------------------------------------------------------ */

/* [MM] "Forward pass convention": Y = X @ W^T with X [M,K], W [N,K]; returns dX = dY @ W [M,K]
 * and dW = dY^T @ X [N,K] in bf16.  precision MOE_PREC_MXFP8 quantises every operand in 32-groups
 * along its GEMM's contraction dimension (dY and W along N for dX; dY and X along M for dW) with
 * `fp8_fmt` (the page's default is e5m2); MOE_PREC_BF16 multiplies the BF16 values directly.
 * dY, W, X, dX, dW (device) bf16; M, N, K multiples of 128.  The workspace holds the quantised or
 * transposed operand copies (none for BF16 under MOE_OPT_MN_OPERANDS, the default: its size is taken
 * with the option as it stands, which must not change between the size query and the call).
 * M, N or K = 0 (multiples of 128 too): an empty contraction gives zeros -- dX is zeroed when N = 0,
 * dW when M = 0 -- and empty outputs need no pointer.
 * Stream: everything is ordered on `stream` as seen by the caller.  Under MOE_OPT_LINEAR_CONCURRENT
 * (the default) the dW GEMM runs on a stream the library creates on first use (one per device, with
 * two events), forked from `stream` and joined back to it inside the call; the call may be captured
 * into a CUDA graph once that stream exists (any earlier call on the device creates it).  That stream
 * belongs to the device's primary context: a process that resets the device (cudaDeviceReset) sets
 * MOE_OPT_LINEAR_CONCURRENT to 0 before calling again. */
size_t linear_bwd_workspace_size(int64_t M, int64_t N, int64_t K, int precision);
int linear_bwd(const void* dY, const void* W, const void* X, int64_t M, int64_t N, int64_t K, int precision,
               int fp8_fmt, void* dX, void* dW, void* workspace, size_t workspace_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOEBWD_H */
