// Host side of the MoE backward and of the dense linear backward: argument checks, workspace
// layout, and the launch sequence on one stream (no host synchronisation):
//
//   route meta -> prep (gather, transpose, quantise) -> [G0 h = x_g W1_e + b1_e, when the
//   pre-activations are recomputed] -> [W2's scales re-tiled, for 192-column MXFP8 G1 tiles] ->
//   G1 dA + dSwiGLU epilogue ->
//   G3 dW2 (K-grouped) -> G2 dx_expanded (M-grouped) -> G4 dW1 (K-grouped) ->
//   dx scatter-sum, ds finalize, bias column sums
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <vector>

#include "moebwd_internal.h"

namespace moebwd {

// CTA-pair GEMMs replace the single-CTA kernel for BF16 where they apply: a store or checkpoint
// epilogue, N a multiple of 256, and M-grouped schedules that know their expert pairs (or have one
// expert) / K-grouped M a multiple of 256.  For MXFP8 the single-CTA kernel is kept (its pair tile
// has a single TMEM accumulator and measured slower).  MOE_OPT_PAIR_GEMMS = 0 disables pairs, 2 also
// uses them for MXFP8.
static bool use_pair(bool mx, int BN, const GemmParams& p) {
  const int64_t mode = option(MOE_OPT_PAIR_GEMMS);
  if (mode == 0 || (mx && mode != 2)) return false;
  if (BN != 256 || (p.epi != kEpiStore && p.epi != kEpiCkpt)) return false;
  if (p.mode == kMGrouped) return p.pair_offsets != nullptr || p.tile_expert == nullptr;
  return p.m_tiles % 2 == 0;
}

// Width of the pair tile: 256, or 128 (MOE_OPT_PAIR_TILE_N).
static int pair_bn() { return option(MOE_OPT_PAIR_TILE_N) == 128 ? 128 : 256; }

int launch_gemm(bool mx, int BN, const GemmParams& p_in, const void* A, int64_t a_rows, int64_t a_cols,
                const void* B, int64_t b_rows, int64_t b_cols, cudaStream_t st, const void* ckpt, int64_t ck_rows,
                int64_t ck_cols) {
  GemmParams p = p_in;
  p.wait_ns = (uint64_t)option(MOE_OPT_WAIT_LIMIT_NS);
  alignas(64) CUtensorMap ta, tb, tc, tsa, tsb;
  const int es = mx ? 1 : 2;
  const uint32_t bke = mx ? 128 : 64;
  const bool pair = use_pair(mx, BN, p);
  const int pbn = pair ? pair_bn() : BN;
  if (mx && (p.a_mn || p.b_mn)) return fail(MOE_ERR_UNSUPPORTED, "MN-major operands are BF16-only");
  // K-major operand: [rows, K] boxes of the tile's rows x one K stage; MN-major ([K, M] / [K, N]):
  // 64 x 64 boxes (a K stage of rows, 64 columns)
  if (!make_tmap_2d(&ta, A, es, (uint64_t)a_rows, (uint64_t)a_cols, (uint64_t)a_cols * es, p.a_mn ? 64 : 128,
                    p.a_mn ? 64 : bke))
    return MOE_ERR_INVALID;
  if (!make_tmap_2d(&tb, B, es, (uint64_t)b_rows, (uint64_t)b_cols, (uint64_t)b_cols * es,
                    p.b_mn ? 64 : pair ? (uint32_t)pbn / 2 : (uint32_t)BN, p.b_mn ? 64 : bke))
    return MOE_ERR_INVALID;
  if (ckpt) {  // checkpoint chunks: 32 features x 128 rows of the [N*2*I, B] view, unswizzled
    if (!make_tmap_2d(&tc, ckpt, 2, (uint64_t)ck_rows, (uint64_t)ck_cols, (uint64_t)ck_cols * 2, 32, 128, false))
      return MOE_ERR_INVALID;
  } else if (p.epi == kEpiStore) {  // output [rows, N] bf16, 64-column x 128-row boxes, 128B swizzle
    const int64_t out_rows = p.mode == kMGrouped ? (int64_t)p.m_tiles * 128 : (int64_t)p.num_experts * p.M;
    if (!make_tmap_2d(&tc, p.out, 2, (uint64_t)out_rows, (uint64_t)p.N, (uint64_t)p.ldo * 2, 128, 64, true))
      return MOE_ERR_INVALID;
  } else {
    tc = ta;
  }
  if (pair) {
    if (mx) {  // tiled scales as rows of 512 bytes (128 x uint32): one row per (128-row block, K tile)
      if (!make_tmap_2d(&tsa, p.sfa, 4, (uint64_t)(a_rows / 128) * p.sfa_ktiles, 128, 512, 1, 128, false))
        return MOE_ERR_INVALID;
      if (!make_tmap_2d(&tsb, p.sfb, 4, (uint64_t)(b_rows / 128) * p.sfb_ktiles, 128, 512, 1, 128, false))
        return MOE_ERR_INVALID;
    } else {
      tsa = ta;
      tsb = ta;
    }
    GemmParams pp = p;
    pp.n_tiles = p.N / pbn;
    // upper bound of the pair tiles: sum_e ceil(tiles_e / 2) <= (tiles + E) / 2
    const int64_t pairs = p.mode == kMGrouped
                              ? (int64_t)((p.m_tiles + (p.pair_offsets ? p.num_experts : 0) + 1) / 2) * pp.n_tiles
                              : (int64_t)p.num_experts * (p.m_tiles / 2) * pp.n_tiles;
    const int max_pairs = (int)std::min<int64_t>(pairs, device_sm_count() / 2);
    if (max_pairs <= 0) return MOE_OK;
    return launch_gemm_pair(mx, pbn, pp, &ta, &tb, &tc, &tsa, &tsb, max_pairs, st);
  }
  const int64_t tiles = (int64_t)(p.mode == kMGrouped ? p.m_tiles : p.num_experts * p.m_tiles) * p.n_tiles;
  const int grid = (int)std::min<int64_t>(tiles, device_sm_count());
  if (grid <= 0) return MOE_OK;
  return mx ? launch_gemm_mx(BN, p, &ta, &tb, &tc, grid, st) : launch_gemm_bf16(BN, p, &ta, &tb, &tc, grid, st);
}

// ------------------------------------------------------------------------------------------
// workspace layout
// ------------------------------------------------------------------------------------------
enum Region {
  R_CHUNK_COUNTS, R_EXPERT_OFFSETS, R_BLOCK_OFFSETS, R_TILE_OFFSETS, R_EXPERT_ORDER, R_SCALARS,
  R_X_GATHER, R_S_SCATTER, R_S_REV, R_TPID, R_B2E, R_TILE_ROW_FLAT, R_FLAT_TILE_ROW, R_TILE_EXPERT,
  R_DOUT_G, R_DOUT_G_SF, R_DOUT_GT, R_DOUT_GT_SF, R_X_GT, R_X_GT_SF, R_DH, R_DH_SF, R_DH_T, R_DH_T_SF,
  R_AP_T, R_AP_T_SF, R_DX_EXP, R_DS_PART, R_DS_BIAS, R_COUNTERS, R_X_G, R_X_G_SF, R_CKPT, R_PAIR_OFFSETS, R_TILE_ORDER, R_TILE_ROW_SLOT, R_W2_SF_T, R_DB1_PART, R_DB2_PART, R_DOUT_Q, R_COUNT
};

struct Layout {
  size_t off[R_COUNT];
  size_t bytes[R_COUNT];
  size_t total;
  int64_t P, Nb, TK;
  int BN1, BN2, BN3, BN4;
  bool gather;  // G1 gathers its dout rows (MOE_OPT_G1_GATHER)
  bool mn;      // BF16: the weight-gradient GEMMs read row-major operands MN-major (MOE_OPT_MN_OPERANDS)
  int g1_groups; // G1 epilogue warp groups: 2 (sixteen warps) or 1 (MOE_OPT_G1_WARPS)
};

static int64_t tile_capacity(int64_t TK, int E) {
  if (TK <= 0) return 0;
  const int64_t ne = std::min<int64_t>(E, TK);
  return (TK + ne * (kTileM - 1) + kTileM - 1) / kTileM * kTileM;
}

static int64_t blocks_bound(int64_t T, int K, int E, int B) {
  const int64_t TK = T * K;
  if (TK <= 0) return 0;
  const int64_t num = TK - (E - 1);
  if (num <= 0) return TK;
  return (num + B - 1) / B + E - 1;
}

// Tile width chosen by an option (MOE_OPT_G*_TILE_N): a nonzero value that divides n (192 only
// where allowed) replaces the default.
static int bn_option(int opt, int dflt, int64_t n, bool allow192 = false) {
  const int bn = (int)option(opt);
  return (bn == 128 || bn == 256 || (allow192 && bn == 192)) && n % bn == 0 ? bn : dflt;
}

static Layout make_layout(const MoeBwdArgs& a) {
  Layout L{};
  const bool mx = a.precision == MOE_PREC_MXFP8;
  const int64_t es = mx ? 1 : 2;
  L.TK = (int64_t)a.T * a.K;
  L.P = tile_capacity(L.TK, a.E);
  L.Nb = blocks_bound(a.T, a.K, a.E, a.block_size);
  // N-tile widths: G1 carries the heavy dSwiGLU epilogue, so it keeps a double-buffered TMEM
  // accumulator: for MXFP8 192 columns where I allows (two 192-column accumulators and the scales fit
  // TMEM; 256 would leave room for one), for BF16 256 where I allows (three stages with one shared
  // transpose buffer), else 128; the store-epilogue GEMMs take 256 where N allows.
  L.BN1 = mx ? (a.I % 192 == 0 ? 192 : 128) : (a.I % 256 == 0 ? 256 : 128);
  L.BN2 = a.H % 256 == 0 ? 256 : 128;
  L.BN3 = L.BN2;
  L.BN4 = 256;
  L.BN1 = bn_option(MOE_OPT_G1_TILE_N, L.BN1, a.I, mx);
  L.BN2 = bn_option(MOE_OPT_G2_TILE_N, L.BN2, a.H);
  L.BN3 = bn_option(MOE_OPT_G3_TILE_N, L.BN3, a.H);
  L.BN4 = bn_option(MOE_OPT_G4_TILE_N, L.BN4, 2 * a.I);
  {  // sixteen G1 epilogue warps (MXFP8, 128- or 192-column tiles) only on request: measured no faster
    const int64_t w = option(MOE_OPT_G1_WARPS);
    const bool two = w == 16;
    L.g1_groups = (mx && two && (L.BN1 == 128 || L.BN1 == 192)) ? 2 : 1;
  }
  const int64_t P = L.P, H = a.H, I = a.I, E = a.E;
  size_t b[R_COUNT] = {};
  b[R_CHUNK_COUNTS] = sizeof(int32_t) * (size_t)std::max<int64_t>(1, route_nchunks(L.TK)) * E;
  b[R_EXPERT_OFFSETS] = b[R_BLOCK_OFFSETS] = b[R_TILE_OFFSETS] = sizeof(int32_t) * (E + 1);
  b[R_EXPERT_ORDER] = sizeof(int32_t) * E;
  b[R_SCALARS] = 16;
  b[R_X_GATHER] = b[R_S_SCATTER] = b[R_S_REV] = b[R_FLAT_TILE_ROW] = sizeof(int32_t) * (size_t)std::max<int64_t>(1, L.TK);
  b[R_TPID] = sizeof(int32_t) * (size_t)std::max<int64_t>(1, L.Nb * a.block_size);
  b[R_B2E] = sizeof(int32_t) * (size_t)std::max<int64_t>(1, L.Nb);
  b[R_TILE_ROW_FLAT] = sizeof(int32_t) * (size_t)std::max<int64_t>(1, P);
  b[R_TILE_EXPERT] = sizeof(int32_t) * (size_t)(P / kTileM + 1);
  L.gather = option(MOE_OPT_G1_GATHER) != 0;
  L.mn = !mx && option(MOE_OPT_MN_OPERANDS) != 0;
  b[R_DOUT_G] = L.gather ? 0 : (size_t)(P * H * es);
  b[R_DOUT_Q] = (L.gather && mx) ? (size_t)((int64_t)a.T * H) : 0;  // dout codes per token
  b[R_DOUT_GT] = (size_t)(H * P * es);
  b[R_X_GT] = (size_t)(H * P * es);
  b[R_DH] = (size_t)(P * 2 * I * es);
  b[R_DH_T] = L.mn ? 0 : (size_t)(2 * I * P * es);  // BF16: G4 reads dh itself (MN-major)
  b[R_AP_T] = (size_t)(I * P * es);
  if (mx) {
    b[R_DOUT_G_SF] = (size_t)(P * H / 32);
    b[R_DOUT_GT_SF] = (size_t)(H * P / 32);
    b[R_X_GT_SF] = (size_t)(H * P / 32);
    b[R_DH_SF] = (size_t)(P * 2 * I / 32);
    b[R_DH_T_SF] = (size_t)(2 * I * P / 32);
    b[R_AP_T_SF] = (size_t)(I * P / 32);
  }
  b[R_DX_EXP] = (size_t)(P * H * 2);
  // one partial per column slice, warp group and N tile
  b[R_DS_PART] = sizeof(float) * (size_t)(P * kG1Subs * L.g1_groups * (I / L.BN1));
  b[R_DS_BIAS] = a.has_bias ? sizeof(float) * (size_t)P : 0;
  b[R_COUNTERS] = 64;  // one tile counter per grouped GEMM
  b[R_PAIR_OFFSETS] = sizeof(int32_t) * (E + 1);
  b[R_TILE_ORDER] = sizeof(int32_t) * (size_t)(P / kTileM + 1);
  b[R_TILE_ROW_SLOT] = sizeof(int32_t) * (size_t)std::max<int64_t>(1, P);  // saved s*dout rows (pointers not read)
  // W2's scales re-tiled for 192-column G1 tiles: two atoms per tile
  if (mx && L.BN1 % 128) b[R_W2_SF_T] = (size_t)(E * I / L.BN1) * ((L.BN1 + 127) / 128) * (size_t)(H / 128) * 512;
  // bias gradients: per-tile column sums from G1's transposes (four lane quarters) and prep (four row quarters)
  if (a.has_bias) {
    b[R_DB1_PART] = sizeof(float) * (size_t)(P / kTileM) * 4 * (size_t)(2 * I);
    b[R_DB2_PART] = sizeof(float) * (size_t)(P / kTileM) * 4 * (size_t)H;
  }
  if (a.act_src == MOE_ACT_RECOMPUTE) {
    b[R_X_G] = (size_t)(P * H * es);
    b[R_X_G_SF] = mx ? (size_t)(P * H / 32) : 0;
    b[R_CKPT] = (size_t)(L.Nb * 2 * I * a.block_size * 2);
  }
  size_t off = 0;
  for (int r = 0; r < R_COUNT; ++r) {
    L.off[r] = off;
    L.bytes[r] = b[r];
    off = align_up(off + b[r], 256);
  }
  L.total = off;
  return L;
}

static int check_args(const MoeBwdArgs* a, bool need_ptrs) {
  if (!a) return fail(MOE_ERR_INVALID, "moe_bwd: null args");
  if (a->T < 0 || a->H <= 0 || a->I <= 0 || a->E <= 0 || a->K <= 0)
    return fail(MOE_ERR_INVALID, "moe_bwd: sizes must be positive (T >= 0)");
  if (a->E > kMaxExperts) return fail(MOE_ERR_UNSUPPORTED, "moe_bwd: E above %d", kMaxExperts);
  if (a->K > a->E || a->K > 64) return fail(MOE_ERR_INVALID, "moe_bwd: need K <= E and K <= 64");
  if (a->H % 128 || a->I % 128) return fail(MOE_ERR_UNSUPPORTED, "moe_bwd: H and I must be multiples of 128");
  if (a->block_size != 128 && a->block_size != 256 && a->block_size != 512 && a->block_size != 1024)
    return fail(MOE_ERR_UNSUPPORTED, "moe_bwd: block_size must be 128, 256, 512 or 1024");
  if ((int64_t)a->T * a->K >= (int64_t)1 << 31) return fail(MOE_ERR_UNSUPPORTED, "moe_bwd: T*K too large");
  if (a->accumulate != 0 && a->accumulate != 1) return fail(MOE_ERR_INVALID, "moe_bwd: accumulate must be 0 or 1");
  if (a->precision != MOE_PREC_BF16 && a->precision != MOE_PREC_MXFP8)
    return fail(MOE_ERR_INVALID, "moe_bwd: bad precision");
  if (a->affinity != MOE_AFFINITY_ON_H && a->affinity != MOE_AFFINITY_ON_I)
    return fail(MOE_ERR_INVALID, "moe_bwd: bad affinity");
  const bool mx = a->precision == MOE_PREC_MXFP8;
  if (mx && ((a->fp8_act != MOE_FP8_E4M3 && a->fp8_act != MOE_FP8_E5M2) ||
             (a->fp8_w != MOE_FP8_E4M3 && a->fp8_w != MOE_FP8_E5M2)))
    return fail(MOE_ERR_INVALID, "moe_bwd: bad fp8 format");
  if (mx && a->has_bias && a->down_proj_act_ckpt)
    return fail(MOE_ERR_UNSUPPORTED, "moe_bwd: MXFP8 bias gradients with a saved down_proj_act_ckpt are not implemented");
  if (a->act_src != MOE_ACT_CHECKPOINT && a->act_src != MOE_ACT_RECOMPUTE)
    return fail(MOE_ERR_INVALID, "moe_bwd: bad act_src");
  if (a->glu != MOE_GLU_SWIGLU && a->glu != MOE_GLU_GEGLU) return fail(MOE_ERR_INVALID, "moe_bwd: bad glu");
  if (a->gate_up_layout != MOE_GATE_UP_CONCAT && a->gate_up_layout != MOE_GATE_UP_INTERLEAVED)
    return fail(MOE_ERR_INVALID, "moe_bwd: bad gate_up_layout");
  if (a->scaled_intermediate_ckpt && a->affinity != MOE_AFFINITY_ON_I)
    return fail(MOE_ERR_INVALID, "moe_bwd: scaled_intermediate_ckpt needs the affinity on I");
  if (a->down_proj_act_ckpt && a->affinity != MOE_AFFINITY_ON_H)
    return fail(MOE_ERR_INVALID, "moe_bwd: down_proj_act_ckpt needs the affinity on H");
  {
    const void* al[] = {a->intermediate_ckpt, a->scaled_intermediate_ckpt, a->down_proj_act_ckpt, a->gate_act_ckpt};
    for (const void* q : al)
      if (reinterpret_cast<uintptr_t>(q) & 15) return fail(MOE_ERR_INVALID, "moe_bwd: checkpoints must be 16-byte aligned");
  }
  if (a->gate_up_layout == MOE_GATE_UP_INTERLEAVED && kG1Subs != 2)
    return fail(MOE_ERR_UNSUPPORTED, "moe_bwd: the interleaved layout needs 16 columns per G1 epilogue warp");
  const bool rec = a->act_src == MOE_ACT_RECOMPUTE;
  if (!need_ptrs) return MOE_OK;
  // token-sized arrays may be null when there are no tokens (T = 0: only the weight gradients, zeroed)
  const void* req_tok[] = {a->x, a->dout, a->s, a->ids, a->dx, a->ds};
  const void* req[] = {a->dW1, a->dW2, a->status_dev};
  if (reinterpret_cast<uintptr_t>(a->num_valid_tokens) & 3)
    return fail(MOE_ERR_INVALID, "moe_bwd: num_valid_tokens must be 4-byte aligned");
  for (const void* q : req)
    if (!q) return fail(MOE_ERR_INVALID, "moe_bwd: required pointer is null");
  for (const void* q : req_tok)
    if (!q && a->T > 0) return fail(MOE_ERR_INVALID, "moe_bwd: required pointer is null");
  if (!rec && !a->gate_up_ckpt && a->T > 0) return fail(MOE_ERR_INVALID, "moe_bwd: gate_up_ckpt is null");
  {
    const int given = (a->expert_offsets != nullptr) + (a->s_scatter_idx != nullptr) + (a->block_offsets != nullptr);
    if (given != 0 && given != 3)
      return fail(MOE_ERR_INVALID, "moe_bwd: routing metadata needs expert_offsets, s_scatter_idx and block_offsets");
    if (given == 0 && (a->token_position_to_id || a->block_to_expert))
      return fail(MOE_ERR_INVALID, "moe_bwd: token_position_to_id / block_to_expert come with expert_offsets");
    const void* m[] = {a->expert_offsets, a->s_scatter_idx, a->block_offsets, a->token_position_to_id,
                       a->block_to_expert};
    for (const void* q : m)
      if (reinterpret_cast<uintptr_t>(q) & 3) return fail(MOE_ERR_INVALID, "moe_bwd: routing metadata must be 4-byte aligned");
  }
  if (rec && (mx ? (!a->W1t_q || !a->W1t_sf) : !a->W1t))
    return fail(MOE_ERR_INVALID, "moe_bwd: recomputing the pre-activations needs W1t (or W1t_q, W1t_sf)");
  const void* al16r[] = {a->W1t, a->W1t_q, a->W1t_sf, a->b1};
  for (const void* q : al16r)
    if (rec && (reinterpret_cast<uintptr_t>(q) & 15))
      return fail(MOE_ERR_INVALID, "moe_bwd: W1t and b1 must be 16-byte aligned");
  if (mx ? (!a->W1_q || !a->W1_sf || !a->W2_q || !a->W2_sf) : (!a->W1 || !a->W2))
    return fail(MOE_ERR_INVALID, "moe_bwd: weights are null");
  if (a->has_bias && (!a->b2 || !a->db1 || !a->db2)) return fail(MOE_ERR_INVALID, "moe_bwd: bias pointers are null");
  const void* al16[] = {a->x, a->dout, mx ? (const void*)a->W1_q : a->W1, mx ? (const void*)a->W2_q : a->W2,
                        a->W1_sf, a->W2_sf, a->dx, a->dW1, a->dW2, a->b2};
  for (const void* q : al16)
    if (reinterpret_cast<uintptr_t>(q) & 15) return fail(MOE_ERR_INVALID, "moe_bwd: tensors must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255)
    return fail(MOE_ERR_INVALID, "moe_bwd: workspace must be 256-byte aligned");
  return MOE_OK;
}

// ------------------------------------------------------------------------------------------
// stage profiler: a ring of event sets recorded on the call's stream, read on demand
// ------------------------------------------------------------------------------------------
struct Profiler {
  static constexpr int kRing = 1024;
  bool on = false;
  int calls = 0;
  std::vector<cudaEvent_t> ev;  // kRing * (MOE_NUM_STAGES + 1)
};
static Profiler g_prof;

static void prof_mark(cudaStream_t st, int slot, int boundary) {
  if (!g_prof.on || slot < 0) return;
  cudaEventRecord(g_prof.ev[(size_t)slot * (MOE_NUM_STAGES + 1) + boundary], st);
}

static int prof_slot() {
  if (!g_prof.on || g_prof.calls >= Profiler::kRing) return -1;
  return g_prof.calls++;
}

template <typename T>
static T* reg(const Layout& L, void* ws, int r) {
  return L.bytes[r] ? reinterpret_cast<T*>(static_cast<char*>(ws) + L.off[r]) : nullptr;
}

}  // namespace moebwd

using namespace moebwd;

extern "C" int64_t moe_num_blocks_bound(int64_t T, int K, int E, int block_size) {
  if (block_size <= 0 || E <= 0 || K <= 0 || T < 0) return 0;
  return blocks_bound(T, K, E, block_size);
}

extern "C" int64_t moe_tile_rows_capacity(int T, int K, int E) { return tile_capacity((int64_t)T * K, E); }

extern "C" size_t moe_bwd_workspace_size(const MoeBwdArgs* args) {
  if (check_args(args, false) != MOE_OK) return 0;
  return make_layout(*args).total;
}

extern "C" int moe_bwd_workspace_region(const MoeBwdArgs* args, int region, size_t* offset, size_t* bytes) {
  clear_error();
  int rc = check_args(args, false);
  if (rc) return rc;
  if (!offset || !bytes) return fail(MOE_ERR_INVALID, "moe_bwd_workspace_region: null output");
  static const int map[MOE_WS_NUM_REGIONS] = {R_EXPERT_OFFSETS, R_TILE_OFFSETS, R_BLOCK_OFFSETS, R_TILE_ROW_FLAT,
                                              R_FLAT_TILE_ROW,  R_DOUT_G,       R_DOUT_G_SF,     R_DOUT_GT,
                                              R_DOUT_GT_SF,     R_X_GT,         R_X_GT_SF,       R_DH,
                                              R_DH_SF,          R_DH_T,         R_DH_T_SF,       R_AP_T,
                                              R_AP_T_SF,        R_DX_EXP,         R_X_G,           R_X_G_SF,
                                              R_CKPT,           R_DOUT_Q};
  if (region < 0 || region >= MOE_WS_NUM_REGIONS) return fail(MOE_ERR_INVALID, "bad region");
  const Layout L = make_layout(*args);
  *offset = L.off[map[region]];
  *bytes = L.bytes[map[region]];
  return MOE_OK;
}

// Size arguments of the routing-metadata entry points, checked in one order so that every entry
// point reports the same error for the same input.
int moebwd::check_route_sizes(const char* who, int T, int K, int E, int block_size) {
  if (T < 0 || K <= 0 || E <= 0 || K > E) return fail(MOE_ERR_INVALID, "%s: bad sizes", who);
  if (E > kMaxExperts) return fail(MOE_ERR_UNSUPPORTED, "%s: E above %d", who, kMaxExperts);
  if (block_size != 128 && block_size != 256 && block_size != 512 && block_size != 1024)
    return fail(MOE_ERR_UNSUPPORTED, "%s: block_size must be 128, 256, 512 or 1024", who);
  if ((int64_t)T * K >= (int64_t)1 << 31) return fail(MOE_ERR_UNSUPPORTED, "%s: T*K too large", who);
  return MOE_OK;
}

extern "C" size_t moe_route_meta_workspace_size(int T, int K, int E, int block_size) {
  if (T < 0 || K <= 0 || E <= 0 || E > kMaxExperts) return 0;
  if (block_size != 128 && block_size != 256 && block_size != 512 && block_size != 1024) return 0;
  MoeBwdArgs a{};
  a.T = T; a.K = K; a.E = E; a.block_size = block_size; a.H = 128; a.I = 128;
  const Layout L = make_layout(a);
  // the routing regions come first in the layout
  return L.off[R_DOUT_G];
}

extern "C" int moe_route_meta(const int32_t* ids, int T, int K, int E, int block_size, int32_t* expert_offsets,
                              int32_t* x_gather_idx, int32_t* s_scatter_idx, int32_t* s_reverse_scatter_idx,
                              int32_t* token_position_to_id, int32_t* block_to_expert, int32_t* block_offsets,
                              int32_t* num_blocks, int32_t* status_dev, void* workspace, size_t workspace_bytes,
                              moe_stream_t stream) {
  clear_error();
  int rc0 = check_route_sizes("moe_route_meta", T, K, E, block_size);
  if (rc0) return rc0;
  if (T == 0) {  // no routed rows: zero offsets and block count; the per-row arrays are empty (may be null)
    if (!expert_offsets || !block_offsets || !num_blocks || !status_dev)
      return fail(MOE_ERR_INVALID, "moe_route_meta: null pointer");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int rc = cuda_check(cudaMemsetAsync(status_dev, 0, sizeof(int32_t), st), "memset status");
    if (!rc) rc = cuda_check(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st), "memset offsets");
    if (!rc) rc = cuda_check(cudaMemsetAsync(block_offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st), "memset offsets");
    if (!rc) rc = cuda_check(cudaMemsetAsync(num_blocks, 0, sizeof(int32_t), st), "memset num_blocks");
    return rc;
  }
  if (!ids || !expert_offsets || !x_gather_idx || !s_scatter_idx || !s_reverse_scatter_idx || !token_position_to_id ||
      !block_to_expert || !block_offsets || !num_blocks || !status_dev || !workspace)
    return fail(MOE_ERR_INVALID, "moe_route_meta: null pointer");
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(MOE_ERR_INVALID, "moe_route_meta: workspace must be 256-byte aligned");
  const size_t need = moe_route_meta_workspace_size(T, K, E, block_size);
  if (workspace_bytes < need) return fail(MOE_ERR_INVALID, "moe_route_meta: workspace too small (%zu < %zu)", workspace_bytes, need);
  MoeBwdArgs a{};
  a.T = T; a.K = K; a.E = E; a.block_size = block_size; a.H = 128; a.I = 128;
  const Layout L = make_layout(a);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc = cuda_check(cudaMemsetAsync(status_dev, 0, sizeof(int32_t), st), "memset status");
  if (rc) return rc;
  RouteBufs r{};
  r.chunk_counts = reg<int32_t>(L, workspace, R_CHUNK_COUNTS);
  r.expert_offsets = expert_offsets;
  r.block_offsets = block_offsets;
  r.tile_offsets = reg<int32_t>(L, workspace, R_TILE_OFFSETS);
  r.expert_order = reg<int32_t>(L, workspace, R_EXPERT_ORDER);
  r.scalars = reg<int32_t>(L, workspace, R_SCALARS);
  r.x_gather_idx = x_gather_idx;
  r.s_scatter_idx = s_scatter_idx;
  r.s_reverse = s_reverse_scatter_idx;
  r.token_position_to_id = token_position_to_id;
  r.block_to_expert = block_to_expert;
  r.tile_row_flat = reg<int32_t>(L, workspace, R_TILE_ROW_FLAT);
  r.flat_tile_row = reg<int32_t>(L, workspace, R_FLAT_TILE_ROW);
  r.tile_expert = reg<int32_t>(L, workspace, R_TILE_EXPERT);
  r.num_blocks_out = num_blocks;
  r.status = status_dev;
  return launch_route_meta(ids, T, K, E, block_size, L.Nb, L.P, r, st);
}

extern "C" int moe_bwd(const MoeBwdArgs* args, moe_stream_t stream) {
  clear_error();
  int rc = check_args(args, true);
  if (rc) return rc;
  const MoeBwdArgs& a = *args;
  const Layout L = make_layout(a);
  if (a.workspace_bytes < L.total)
    return fail(MOE_ERR_INVALID, "moe_bwd: workspace too small (%zu < %zu)", a.workspace_bytes, L.total);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* ws = a.workspace;
  const bool mx = a.precision == MOE_PREC_MXFP8;
  const int64_t H = a.H, I = a.I, E = a.E, P = L.P, TK = L.TK;
  if ((rc = cuda_check(cudaMemsetAsync(a.status_dev, 0, sizeof(int32_t), st), "memset status"))) return rc;
  if (TK == 0 && a.accumulate) return MOE_OK;  // nothing to add
  if (TK == 0) {  // no routed rows: every gradient is zero
    if ((rc = cuda_check(cudaMemsetAsync(a.dW1, 0, (size_t)(E * H * 2 * I * 2), st), "memset dW1"))) return rc;
    if ((rc = cuda_check(cudaMemsetAsync(a.dW2, 0, (size_t)(E * I * H * 2), st), "memset dW2"))) return rc;
    if (a.has_bias) {
      if ((rc = cuda_check(cudaMemsetAsync(a.db1, 0, (size_t)(E * 2 * I * 4), st), "memset db1"))) return rc;
      if ((rc = cuda_check(cudaMemsetAsync(a.db2, 0, (size_t)(E * H * 4), st), "memset db2"))) return rc;
    }
    if (a.ds_masked && a.T > 0 &&
        (rc = cuda_check(cudaMemsetAsync(a.ds_masked, 0, sizeof(float) * (size_t)a.T * E, st), "memset ds_masked")))
      return rc;
    return MOE_OK;
  }

  const int slot = prof_slot();
  prof_mark(st, slot, 0);
  int32_t* counters = reg<int32_t>(L, ws, R_COUNTERS);  // zeroed by the routing kernels
  int32_t* tile_offsets = reg<int32_t>(L, ws, R_TILE_OFFSETS);
  int32_t* expert_order = reg<int32_t>(L, ws, R_EXPERT_ORDER);
  int32_t* scalars = reg<int32_t>(L, ws, R_SCALARS);
  int32_t* tile_row_flat = reg<int32_t>(L, ws, R_TILE_ROW_FLAT);
  int32_t* flat_tile_row = reg<int32_t>(L, ws, R_FLAT_TILE_ROW);
  int32_t* tile_expert = reg<int32_t>(L, ws, R_TILE_EXPERT);
  int32_t* block_offsets = reg<int32_t>(L, ws, R_BLOCK_OFFSETS);

  // 1. routing metadata
  RouteBufs r{};
  r.chunk_counts = reg<int32_t>(L, ws, R_CHUNK_COUNTS);
  r.expert_offsets = reg<int32_t>(L, ws, R_EXPERT_OFFSETS);
  r.block_offsets = block_offsets;
  r.tile_offsets = tile_offsets;
  r.expert_order = expert_order;
  r.scalars = scalars;
  r.x_gather_idx = reg<int32_t>(L, ws, R_X_GATHER);
  r.s_scatter_idx = reg<int32_t>(L, ws, R_S_SCATTER);
  r.s_reverse = reg<int32_t>(L, ws, R_S_REV);
  r.token_position_to_id = reg<int32_t>(L, ws, R_TPID);
  r.block_to_expert = reg<int32_t>(L, ws, R_B2E);
  r.tile_row_flat = tile_row_flat;
  r.flat_tile_row = flat_tile_row;
  r.tile_expert = tile_expert;
  r.num_blocks_out = nullptr;
  r.pair_offsets = reg<int32_t>(L, ws, R_PAIR_OFFSETS);
  r.num_valid = a.num_valid_tokens;
  r.status = a.status_dev;
  r.zero_counters = counters;
  r.nzero = (int)(L.bytes[R_COUNTERS] / sizeof(int32_t));
  if (a.expert_offsets) {  // the caller's metadata, checked; tile tables derived from it
    RouteMetaIn in{a.expert_offsets, a.s_scatter_idx, a.block_offsets, a.token_position_to_id, a.block_to_expert};
    if ((rc = launch_route_meta_in(in, a.ids, a.T, a.K, a.E, a.block_size, L.Nb, P, r, st))) return rc;
  } else if ((rc = launch_route_meta(a.ids, a.T, a.K, a.E, a.block_size, L.Nb, P, r, st))) {
    return rc;
  }
  int32_t* tile_order = reg<int32_t>(L, ws, R_TILE_ORDER);
  if ((rc = launch_tile_order(tile_row_flat, scalars + 1, a.T, a.K, tile_order, st))) return rc;
  prof_mark(st, slot, 1);

  // 2. gathered / transposed / quantised activation operands
  PrepArgs pa{};
  pa.dout = static_cast<const uint16_t*>(a.dout);
  pa.x = static_cast<const uint16_t*>(a.x);
  pa.s = a.s;
  pa.b2 = a.has_bias ? static_cast<const uint16_t*>(a.b2) : nullptr;
  pa.tile_row_flat = tile_row_flat;
  pa.tile_expert = tile_expert;
  pa.num_tiles = scalars + 1;
  pa.tile_order = option(MOE_OPT_PREP_TILE_ORDER) ? tile_order : nullptr;
  pa.H = a.H;
  pa.K = a.K;
  pa.P = P;
  pa.mx = mx;
  pa.fmt = a.fp8_act;
  pa.scale_t = a.affinity == MOE_AFFINITY_ON_H;
  pa.dout_g = reg<void>(L, ws, R_DOUT_G);  // null when G1 gathers its rows
  pa.dout_g_sf = reg<uint8_t>(L, ws, R_DOUT_G_SF);
  pa.dout_gt = reg<void>(L, ws, R_DOUT_GT);
  pa.dout_gt_sf = reg<uint8_t>(L, ws, R_DOUT_GT_SF);
  pa.x_gt = reg<void>(L, ws, R_X_GT);
  pa.x_gt_sf = reg<uint8_t>(L, ws, R_X_GT_SF);
  pa.ds_bias = a.has_bias ? reg<float>(L, ws, R_DS_BIAS) : nullptr;
  const bool rec = a.act_src == MOE_ACT_RECOMPUTE;
  pa.x_g = rec ? reg<void>(L, ws, R_X_G) : nullptr;
  pa.x_g_sf = rec ? reg<uint8_t>(L, ws, R_X_G_SF) : nullptr;
  pa.skip_dout_t = a.down_proj_act_ckpt != nullptr;
  pa.db2_part = (a.has_bias && !pa.skip_dout_t) ? reg<float>(L, ws, R_DB2_PART) : nullptr;
  // BF16 with MN-major weight-gradient operands: no transposed copies; x rows for the dW1 GEMM (the
  // recomputation's copy when there is one, else in the X_GT region), the dW2 GEMM's B rows (s*dout
  // for affinity on H, or dout when G1 gathers its rows and writes no dout_g) in the DOUT_GT region
  // For affinity on H the factor s goes to a' (G1 writes s*a) unless a' comes from a saved intermediate;
  // the dW2 GEMM then reads dout_g itself, and an s*dout copy is made only in that saved case.
  const void* inter = a.scaled_intermediate_ckpt ? a.scaled_intermediate_ckpt : a.intermediate_ckpt;
  const bool g3_b_scaled = a.affinity == MOE_AFFINITY_ON_H && inter != nullptr;
  void* x_rows = L.mn ? (rec ? reg<void>(L, ws, R_X_G) : reg<void>(L, ws, R_X_GT)) : nullptr;
  void* g3_b_rows = nullptr;
  if (L.mn && !pa.skip_dout_t)
    g3_b_rows = (g3_b_scaled || L.gather) ? reg<void>(L, ws, R_DOUT_GT) : reg<void>(L, ws, R_DOUT_G);
  if (L.mn) {
    pa.no_t = 1;
    pa.x_g = x_rows;
    pa.dout_b = g3_b_rows == reg<void>(L, ws, R_DOUT_GT) ? g3_b_rows : nullptr;
    pa.dout_b_s = g3_b_scaled;
  }
  if ((rc = launch_prep(pa, st))) return rc;
  if (L.gather && mx &&  // the rows G1 gathers: dout quantised once per token (the scales come from prep)
      (rc = launch_quant_rowwise(pa.dout, a.T, a.T, H, H, nullptr, a.fp8_act, reg<uint8_t>(L, ws, R_DOUT_Q), nullptr,
                                 1, st)))
    return rc;
  // dW_down operands from saved forward values ([BW] optional checkpoints)
  if (inter && (rc = launch_apt_from_ckpt(static_cast<const uint16_t*>(inter), a.I, a.block_size, P, scalars + 1,
                                         tile_expert, tile_offsets, block_offsets, tile_row_flat,
                                         (!a.scaled_intermediate_ckpt && a.affinity == MOE_AFFINITY_ON_I) ? a.s
                                                                                                         : nullptr,
                                         mx, a.fp8_act, reg<void>(L, ws, R_AP_T), reg<uint8_t>(L, ws, R_AP_T_SF), st)))
    return rc;
  if (a.down_proj_act_ckpt) {
    int32_t* slot = reg<int32_t>(L, ws, R_TILE_ROW_SLOT);
    if ((rc = launch_tile_row_slot(P, a.block_size, scalars + 1, tile_expert, tile_offsets, block_offsets,
                                   tile_row_flat, slot, st)))
      return rc;
    if ((rc = launch_quant_colwise(static_cast<const uint16_t*>(a.down_proj_act_ckpt), L.Nb * a.block_size, P, H, H,
                                   slot, mx, a.fp8_act, reg<void>(L, ws, R_DOUT_GT), reg<uint8_t>(L, ws, R_DOUT_GT_SF),
                                   1, st)))
      return rc;
  }
  prof_mark(st, slot, 2);

  // 2b. G0 (recompute): h = x_g W1_e + b1_e written into a block checkpoint in the workspace
  const void* ckpt = a.gate_up_ckpt;
  if (rec) {
    GemmParams p{};
    p.mode = kMGrouped;
    p.M = (int)P; p.N = (int)(2 * I); p.K = (int)H;
    p.m_tiles = (int)(P / kTileM);
    p.n_tiles = (int)(2 * I / 256);
    p.num_experts = (int)E;
    p.tile_expert = tile_expert;
    p.num_tiles = scalars + 1;
    p.b_rows_per_expert = (int)(2 * I);
    p.sfa = reg<uint8_t>(L, ws, R_X_G_SF);
    p.sfb = a.W1t_sf;
    p.sfa_ktiles = p.sfb_ktiles = (int)(H / 128);
    p.fmt_a = a.fp8_act; p.fmt_b = a.fp8_w;
    p.epi = kEpiCkpt;
    p.e_tile_offsets = tile_offsets;
    p.pair_offsets = reg<int32_t>(L, ws, R_PAIR_OFFSETS);
    p.num_pairs = scalars + 2;
    p.block_offsets = block_offsets;
    p.b1 = static_cast<const uint16_t*>(a.b1);
    p.I = a.I; p.B = a.block_size;
    p.P = P;
    p.tile_counter = counters + 4;
    p.status = a.status_dev;
    ckpt = reg<void>(L, ws, R_CKPT);
    if ((rc = launch_gemm(mx, 256, p, reg<void>(L, ws, R_X_G), P, H, mx ? static_cast<const void*>(a.W1t_q) : a.W1t,
                          E * 2 * I, H, st, ckpt, L.Nb * 2 * I, a.block_size)))
      return rc;
  }
  prof_mark(st, slot, 3);

  const void* W1 = mx ? static_cast<const void*>(a.W1_q) : a.W1;
  const void* W2 = mx ? static_cast<const void*>(a.W2_q) : a.W2;

  // 3. G1: dA_raw = dout_g W2_e^T with the dSwiGLU / ds epilogue
  {
    GemmParams p{};
    p.mode = kMGrouped;
    p.M = (int)P; p.N = (int)I; p.K = (int)H;
    p.m_tiles = (int)(P / kTileM);
    p.n_tiles = (int)(I / L.BN1);
    p.num_experts = (int)E;
    p.tile_expert = tile_expert;
    p.num_tiles = scalars + 1;
    p.b_rows_per_expert = (int)I;
    p.sfa = reg<uint8_t>(L, ws, R_DOUT_G_SF);
    p.sfb = a.W2_sf;
    if (mx && L.BN1 % 128) {  // W2's scales in whole atoms per 192-row tile
      uint8_t* t = reg<uint8_t>(L, ws, R_W2_SF_T);
      if ((rc = launch_sf_retile(a.W2_sf, E * I, H, L.BN1, t, st))) return rc;
      p.sfb = t;
    }
    p.sfa_ktiles = p.sfb_ktiles = (int)(H / 128);
    p.fmt_a = a.fp8_act; p.fmt_b = a.fp8_w;
    p.epi = L.g1_groups == 2 ? kEpiDSwiGLU2 : kEpiDSwiGLU;
    p.s = a.s;
    p.tile_row_flat = tile_row_flat;
    p.e_tile_offsets = tile_offsets;
    p.block_offsets = block_offsets;
    p.ckpt = static_cast<const uint16_t*>(ckpt);
    p.I = a.I; p.B = a.block_size;
    p.affinity_on_i = a.affinity == MOE_AFFINITY_ON_I;
    p.fmt_act = a.fp8_act;
    p.glu = a.glu;
    p.interleaved = a.gate_up_layout == MOE_GATE_UP_INTERLEAVED;
    p.gate_act = static_cast<const uint16_t*>(a.gate_act_ckpt);
    p.P = P;
    p.dh = reg<void>(L, ws, R_DH); p.dh_sf = reg<uint8_t>(L, ws, R_DH_SF);
    p.dht = reg<void>(L, ws, R_DH_T); p.dht_sf = reg<uint8_t>(L, ws, R_DH_T_SF);
    p.apt = inter ? nullptr : reg<void>(L, ws, R_AP_T);
    p.ap_rows = L.mn;  // BF16: a' rows [P,I] for the dW2 GEMM's MN-major read
    // ... scaled by s for affinity on H when the dW2 GEMM reads unscaled dout rows (not with a saved s*dout)
    p.ap_s = L.mn && a.affinity == MOE_AFFINITY_ON_H && !pa.skip_dout_t;
    p.apt_sf = inter ? nullptr : reg<uint8_t>(L, ws, R_AP_T_SF);
    p.ds_part = reg<float>(L, ws, R_DS_PART);
    p.db1_part = a.has_bias ? reg<float>(L, ws, R_DB1_PART) : nullptr;
    p.tile_counter = counters + 0;
    p.status = a.status_dev;
    const void* A = reg<void>(L, ws, R_DOUT_G);
    int64_t a_rows = P;
    if (L.gather) {  // A rows gathered from dout (BF16) or its per-token codes (MXFP8): row = flat / K
      p.a_gather = mx ? static_cast<const void*>(reg<uint8_t>(L, ws, R_DOUT_Q)) : a.dout;
      p.a_gather_ld = H * (mx ? 1 : 2);
      p.a_gather_div = a.K;
      A = p.a_gather;
      a_rows = a.T;
    }
    if ((rc = launch_gemm(mx, L.BN1, p, A, a_rows, H, W2, E * I, H, st, ckpt, L.Nb * 2 * I, a.block_size)))
      return rc;
  }
  prof_mark(st, slot, 4);
  // 4. G3: dW2_e = a'^T dout_g over the expert's tile rows
  {
    GemmParams p{};
    p.mode = kKGrouped;
    p.M = (int)I; p.N = (int)H;
    p.m_tiles = (int)(I / kTileM);
    p.n_tiles = (int)(H / L.BN3);
    p.num_experts = (int)E;
    p.tile_offsets = tile_offsets;
    p.expert_order = expert_order;
    p.sfa = reg<uint8_t>(L, ws, R_AP_T_SF);
    p.sfb = reg<uint8_t>(L, ws, R_DOUT_GT_SF);
    p.sfa_ktiles = p.sfb_ktiles = (int)(P / 128);
    p.fmt_a = a.fp8_act; p.fmt_b = a.fp8_act;
    p.epi = kEpiStore;
    p.out = a.dW2; p.ldo = H; p.out_expert_stride = I * H;
    p.accumulate = a.accumulate;
    p.tile_counter = counters + 1;
    p.status = a.status_dev;
    // BF16 (MN_OPERANDS): a' rows and the dout rows read MN-major, except operands built from saved
    // checkpoints (a'^T from the intermediate, dout^T from down_proj_act), which stay transposed
    p.a_mn = L.mn && !inter;
    p.b_mn = g3_b_rows != nullptr;
    if ((rc = launch_gemm(mx, L.BN3, p, reg<void>(L, ws, R_AP_T), p.a_mn ? P : I, p.a_mn ? I : P,
                          p.b_mn ? g3_b_rows : reg<void>(L, ws, R_DOUT_GT), p.b_mn ? P : H, p.b_mn ? H : P, st)))
      return rc;
  }
  prof_mark(st, slot, 5);
  // 5. G2: dx_expanded = dh W1_e^T
  {
    GemmParams p{};
    p.mode = kMGrouped;
    p.M = (int)P; p.N = (int)H; p.K = (int)(2 * I);
    p.m_tiles = (int)(P / kTileM);
    p.n_tiles = (int)(H / L.BN2);
    p.num_experts = (int)E;
    p.tile_expert = tile_expert;
    p.num_tiles = scalars + 1;
    p.b_rows_per_expert = (int)H;
    p.sfa = reg<uint8_t>(L, ws, R_DH_SF);
    p.sfb = a.W1_sf;
    p.sfa_ktiles = p.sfb_ktiles = (int)(2 * I / 128);
    p.fmt_a = a.fp8_act; p.fmt_b = a.fp8_w;
    p.epi = kEpiStore;
    p.out = reg<void>(L, ws, R_DX_EXP); p.ldo = H;
    p.e_tile_offsets = tile_offsets;
    p.pair_offsets = reg<int32_t>(L, ws, R_PAIR_OFFSETS);
    p.num_pairs = scalars + 2;
    p.tile_counter = counters + 2;
    p.status = a.status_dev;
    if ((rc = launch_gemm(mx, L.BN2, p, reg<void>(L, ws, R_DH), P, 2 * I, W1, E * H, 2 * I, st))) return rc;
  }
  prof_mark(st, slot, 6);
  // 6. G4: dW1_e = x_g^T dh over the expert's tile rows
  {
    GemmParams p{};
    p.mode = kKGrouped;
    p.M = (int)H; p.N = (int)(2 * I);
    p.m_tiles = (int)(H / kTileM);
    p.n_tiles = (int)(2 * I / L.BN4);
    p.num_experts = (int)E;
    p.tile_offsets = tile_offsets;
    p.expert_order = expert_order;
    p.sfa = reg<uint8_t>(L, ws, R_X_GT_SF);
    p.sfb = reg<uint8_t>(L, ws, R_DH_T_SF);
    p.sfa_ktiles = p.sfb_ktiles = (int)(P / 128);
    p.fmt_a = a.fp8_act; p.fmt_b = a.fp8_act;
    p.epi = kEpiStore;
    p.out = a.dW1; p.ldo = 2 * I; p.out_expert_stride = H * 2 * I;
    p.accumulate = a.accumulate;
    p.tile_counter = counters + 3;
    p.status = a.status_dev;
    // BF16 (MN_OPERANDS): B is dh itself, [P, 2I] read MN-major (no transposed copy); else dh^T (for
    // MXFP8 quantised along tokens)
    p.a_mn = p.b_mn = L.mn;  // BF16: x rows and dh, both read MN-major
    if ((rc = L.mn ? launch_gemm(mx, L.BN4, p, x_rows, P, H, reg<void>(L, ws, R_DH), P, 2 * I, st)
                   : launch_gemm(mx, L.BN4, p, reg<void>(L, ws, R_X_GT), H, P, reg<void>(L, ws, R_DH_T), 2 * I, P, st)))
      return rc;
  }
  prof_mark(st, slot, 7);
  // 7. reductions
  if ((rc = launch_dx_scatter_sum(reg<uint16_t>(L, ws, R_DX_EXP), flat_tile_row, a.T, a.K, a.H,
                                  static_cast<uint16_t*>(a.dx), st)))
    return rc;
  if ((rc = launch_ds_finalize(reg<float>(L, ws, R_DS_PART), (int)(kG1Subs * L.g1_groups * (I / L.BN1)),
                               a.has_bias ? reg<float>(L, ws, R_DS_BIAS) : nullptr,
                               flat_tile_row, TK, a.ds, st)))
    return rc;
  if (a.ds_masked && (rc = launch_ds_masked(a.ds, a.ids, a.num_valid_tokens, a.T, a.K, a.E, a.ds_masked, st)))
    return rc;
  if (a.has_bias) {  // per-expert sums of the per-tile partials (dout_gt read again only when it was not built here)
    if (pa.db2_part) {  // db1 and db2 from their per-tile partials in one launch
      rc = launch_bias_parts_reduce(reg<float>(L, ws, R_DB1_PART), 4, 2 * I, tile_offsets, (int)E, a.db1, st,
                                    a.accumulate, pa.db2_part, L.mn ? 1 : 4, H, a.db2);
    } else {
      if ((rc = launch_bias_parts_reduce(reg<float>(L, ws, R_DB1_PART), 4, 2 * I, tile_offsets, (int)E, a.db1, st,
                                         a.accumulate)))
        return rc;
      rc = launch_segment_rowsum(reg<uint16_t>(L, ws, R_DOUT_GT), P, (int)H, tile_offsets, (int)E,
                                 a.affinity == MOE_AFFINITY_ON_I ? a.s : nullptr, tile_row_flat, a.db2, st,
                                 a.accumulate);
    }
    if (rc) return rc;
  }
  prof_mark(st, slot, 8);
  return MOE_OK;
}

extern "C" int moe_profile_enable(int enable) {
  clear_error();
  if (g_prof.ev.empty() && enable) {
    g_prof.ev.resize((size_t)Profiler::kRing * (MOE_NUM_STAGES + 1));
    for (auto& e : g_prof.ev) {
      int rc = cuda_check(cudaEventCreate(&e), "cudaEventCreate");
      if (rc) {
        g_prof.ev.clear();
        return rc;
      }
    }
  }
  g_prof.on = enable != 0;
  g_prof.calls = 0;
  return MOE_OK;
}

// Event boundaries are recorded in launch order; stage of the interval between boundary i and i+1.
static const int kStageOfInterval[MOE_NUM_STAGES] = {MOE_STAGE_ROUTE, MOE_STAGE_PREP, MOE_STAGE_G0, MOE_STAGE_G1,
                                                     MOE_STAGE_G3,    MOE_STAGE_G2,   MOE_STAGE_G4, MOE_STAGE_REDUCE};

extern "C" int moe_profile_read(double* stage_ms, int max_stages, int* calls) {
  clear_error();
  if (!stage_ms || max_stages < 0) return fail(MOE_ERR_INVALID, "moe_profile_read: null output");
  for (int i = 0; i < max_stages; ++i) stage_ms[i] = 0.0;
  if (calls) *calls = g_prof.calls;
  for (int c = 0; c < g_prof.calls; ++c) {
    cudaEvent_t* e = &g_prof.ev[(size_t)c * (MOE_NUM_STAGES + 1)];
    int rc = cuda_check(cudaEventSynchronize(e[MOE_NUM_STAGES]), "cudaEventSynchronize");
    if (rc) return rc;
    for (int i = 0; i < MOE_NUM_STAGES; ++i) {
      if (kStageOfInterval[i] >= max_stages) continue;
      float ms = 0.f;
      if ((rc = cuda_check(cudaEventElapsedTime(&ms, e[i], e[i + 1]), "cudaEventElapsedTime"))) return rc;
      stage_ms[kStageOfInterval[i]] += ms;
    }
  }
  return MOE_OK;
}

// ------------------------------------------------------------------------------------------
// dense linear backward
// ------------------------------------------------------------------------------------------
namespace {
struct LinLayout {
  size_t off[9], bytes[9], total;
};
LinLayout lin_layout(int64_t M, int64_t N, int64_t K, int precision) {
  LinLayout L{};
  const bool mx = precision == MOE_PREC_MXFP8;
  const int64_t es = mx ? 1 : 2;
  // BF16 with MN-major operands (MOE_OPT_MN_OPERANDS): both GEMMs read dY, W and X themselves, no copies
  const int64_t tc = (mx || option(MOE_OPT_MN_OPERANDS) == 0) ? 1 : 0;
  // 0 dY (rowwise, mx only) 1 its sf | 2 W^T [K,N] 3 sf | 4 dY^T [N,M] 5 sf | 6 X^T [K,M] 7 sf | 8 counters
  size_t b[9] = {mx ? (size_t)(M * N) : 0, mx ? (size_t)(M * N / 32) : 0, (size_t)(K * N * es * tc),
                 mx ? (size_t)(K * N / 32) : 0, (size_t)(N * M * es * tc), mx ? (size_t)(N * M / 32) : 0,
                 (size_t)(K * M * es * tc), mx ? (size_t)(K * M / 32) : 0, 64 /* tile counters */};
  size_t off = 0;
  for (int i = 0; i < 9; ++i) {
    L.off[i] = off;
    L.bytes[i] = b[i];
    off = align_up(off + b[i], 256);
  }
  L.total = off;
  return L;
}
}  // namespace

extern "C" size_t linear_bwd_workspace_size(int64_t M, int64_t N, int64_t K, int precision) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return lin_layout(M, N, K, precision).total;
}

extern "C" int linear_bwd(const void* dY, const void* W, const void* X, int64_t M, int64_t N, int64_t K, int precision,
                          int fp8_fmt, void* dX, void* dW, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  clear_error();
  if (M < 0 || N < 0 || K < 0) return fail(MOE_ERR_INVALID, "linear_bwd: negative size");
  if (M % 128 || N % 128 || K % 128) return fail(MOE_ERR_UNSUPPORTED, "linear_bwd: M, N, K must be multiples of 128");
  if (precision != MOE_PREC_BF16 && precision != MOE_PREC_MXFP8) return fail(MOE_ERR_INVALID, "linear_bwd: bad precision");
  if (M == 0 || N == 0 || K == 0) {  // an empty contraction gives zeros; empty outputs need no pointer
    cudaStream_t st0 = reinterpret_cast<cudaStream_t>(stream);
    if (M * K > 0 && !dX) return fail(MOE_ERR_INVALID, "linear_bwd: null pointer");
    if (N * K > 0 && !dW) return fail(MOE_ERR_INVALID, "linear_bwd: null pointer");
    int rc0 = M * K > 0 ? cuda_check(cudaMemsetAsync(dX, 0, (size_t)(M * K * 2), st0), "memset dX") : MOE_OK;
    if (!rc0 && N * K > 0) rc0 = cuda_check(cudaMemsetAsync(dW, 0, (size_t)(N * K * 2), st0), "memset dW");
    return rc0;
  }
  if (!dY || !W || !X || !dX || !dW || !workspace) return fail(MOE_ERR_INVALID, "linear_bwd: null pointer");
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return fail(MOE_ERR_UNSUPPORTED, "linear_bwd: too large");
  if (precision == MOE_PREC_MXFP8 && fp8_fmt != MOE_FP8_E4M3 && fp8_fmt != MOE_FP8_E5M2)
    return fail(MOE_ERR_INVALID, "linear_bwd: bad fp8 format");
  const void* al[] = {dY, W, X, dX, dW};
  for (const void* q : al)
    if (reinterpret_cast<uintptr_t>(q) & 15) return fail(MOE_ERR_INVALID, "linear_bwd: tensors must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(MOE_ERR_INVALID, "linear_bwd: workspace must be 256-byte aligned");
  const LinLayout L = lin_layout(M, N, K, precision);
  if (workspace_bytes < L.total) return fail(MOE_ERR_INVALID, "linear_bwd: workspace too small (%zu < %zu)", workspace_bytes, L.total);
  const bool mx = precision == MOE_PREC_MXFP8;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  auto R = [&](int i) { return L.bytes[i] ? static_cast<void*>(ws + L.off[i]) : nullptr; };
  const uint16_t* dYb = static_cast<const uint16_t*>(dY);
  int32_t* counters = static_cast<int32_t*>(R(8));
  int rc = cuda_check(cudaMemsetAsync(counters, 0, L.bytes[8], st), "memset tile counters");
  if (rc) return rc;
  // operands: dX = dY @ W contracts over N, dW = dY^T @ X contracts over M; BF16 with MN-major operands
  // reads W (dX's B), dY (dW's A) and X (dW's B) row-major, so only MXFP8 (or transposed BF16) copies
  const bool mn = !mx && L.bytes[2] == 0;
  if (mx) {  // dY row-wise and the three transposed operands, one launch
    if ((rc = launch_linear_quant(dYb, static_cast<const uint16_t*>(W), static_cast<const uint16_t*>(X), M, N, K, fp8_fmt,
                                  static_cast<uint8_t*>(R(0)), static_cast<uint8_t*>(R(1)), static_cast<uint8_t*>(R(2)),
                                  static_cast<uint8_t*>(R(3)), static_cast<uint8_t*>(R(4)), static_cast<uint8_t*>(R(5)),
                                  static_cast<uint8_t*>(R(6)), static_cast<uint8_t*>(R(7)), st)))
      return rc;
  } else if (!mn) {  // BF16 with transposed copies
    if ((rc = launch_quant_colwise(static_cast<const uint16_t*>(W), N, N, K, K, nullptr, 0, fp8_fmt, R(2), nullptr, 1,
                                   st)) ||
        (rc = launch_quant_colwise(dYb, M, M, N, N, nullptr, 0, fp8_fmt, R(4), nullptr, 1, st)) ||
        (rc = launch_quant_colwise(static_cast<const uint16_t*>(X), M, M, K, K, nullptr, 0, fp8_fmt, R(6), nullptr, 1,
                                   st)))
      return rc;
  }
  const int BN = K % 256 == 0 ? 256 : 128;
  auto gemm_dx = [&](cudaStream_t s) {
    GemmParams p{};
    p.mode = kMGrouped;
    p.M = (int)M; p.N = (int)K; p.K = (int)N;
    p.m_tiles = (int)(M / 128);
    p.n_tiles = (int)(K / BN);
    p.num_experts = 1;
    p.sfa = static_cast<const uint8_t*>(R(1));
    p.sfb = static_cast<const uint8_t*>(R(3));
    p.sfa_ktiles = p.sfb_ktiles = (int)(N / 128);
    p.fmt_a = p.fmt_b = fp8_fmt;
    p.epi = kEpiStore;
    p.out = dX; p.ldo = K;
    p.tile_counter = counters + 0;
    p.b_mn = mn;  // W itself: [N, K] = [contraction, output columns]
    return mn ? launch_gemm(mx, BN, p, dY, M, N, W, N, K, s) : launch_gemm(mx, BN, p, mx ? R(0) : dY, M, N, R(2), K, N, s);
  };
  auto gemm_dw = [&](cudaStream_t s) {
    GemmParams p{};
    p.mode = kMGrouped;
    p.M = (int)N; p.N = (int)K; p.K = (int)M;
    p.m_tiles = (int)(N / 128);
    p.n_tiles = (int)(K / BN);
    p.num_experts = 1;
    p.sfa = static_cast<const uint8_t*>(R(5));
    p.sfb = static_cast<const uint8_t*>(R(7));
    p.sfa_ktiles = p.sfb_ktiles = (int)(M / 128);
    p.fmt_a = p.fmt_b = fp8_fmt;
    p.epi = kEpiStore;
    p.out = dW; p.ldo = K;
    p.tile_counter = counters + 1;
    p.a_mn = p.b_mn = mn;  // dY [M, N] and X [M, K]: both [contraction, output] row-major
    return mn ? launch_gemm(mx, BN, p, dY, M, N, X, M, K, s) : launch_gemm(mx, BN, p, R(4), N, M, R(6), K, M, s);
  };
  // the two GEMMs are independent: dW on the library's second stream beside dX (MOE_OPT_LINEAR_CONCURRENT)
  if (option(MOE_OPT_LINEAR_CONCURRENT)) return fork_join(st, gemm_dw, [&] { return gemm_dx(st); });
  if ((rc = gemm_dx(st))) return rc;
  return gemm_dw(st);
}
