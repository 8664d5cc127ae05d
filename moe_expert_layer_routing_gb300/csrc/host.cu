// Host utilities: per-thread error text, CUDA error mapping, SM count, TMA descriptor encoding.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <functional>
#include <mutex>

#include "moebwd_internal.h"

namespace moebwd {

static thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_err[0] = 0; }

int cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MOE_OK;
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Library options (moe_set_option): process-wide, read by every later call.
static std::atomic<int64_t> g_opt[MOE_NUM_OPTIONS];
static const int64_t kOptDefault[MOE_NUM_OPTIONS] = {
    (int64_t)kWaitLimitNs,  // MOE_OPT_WAIT_LIMIT_NS
    1,                      // MOE_OPT_PAIR_GEMMS
    256,                    // MOE_OPT_PAIR_TILE_N
    0, 0, 0, 0,             // MOE_OPT_G1_TILE_N .. MOE_OPT_G4_TILE_N (automatic)
    1,                      // MOE_OPT_PREP_TILE_ORDER
    0,                      // MOE_OPT_G1_GATHER (measured slower: see the option's comment)
    0,                      // MOE_OPT_G1_WARPS (automatic)
    1,                      // MOE_OPT_PDL
    1,                      // MOE_OPT_MN_OPERANDS
    1,                      // MOE_OPT_LINEAR_CONCURRENT
};
static std::once_flag g_opt_once;
static void opt_init() {
  std::call_once(g_opt_once, [] {
    for (int i = 0; i < MOE_NUM_OPTIONS; ++i) g_opt[i].store(kOptDefault[i]);
  });
}

int64_t option(int o) {
  opt_init();
  return g_opt[o].load(std::memory_order_relaxed);
}

static bool option_value_ok(int o, int64_t v) {
  switch (o) {
    case MOE_OPT_WAIT_LIMIT_NS: return v >= 1 && v <= 60000000000ll;
    case MOE_OPT_PAIR_GEMMS: return v >= 0 && v <= 2;
    case MOE_OPT_PAIR_TILE_N: return v == 128 || v == 256;
    case MOE_OPT_G1_TILE_N: return v == 0 || v == 128 || v == 192 || v == 256;
    case MOE_OPT_G2_TILE_N:
    case MOE_OPT_G3_TILE_N:
    case MOE_OPT_G4_TILE_N: return v == 0 || v == 128 || v == 256;
    case MOE_OPT_PREP_TILE_ORDER:
    case MOE_OPT_G1_GATHER:
    case MOE_OPT_PDL:
    case MOE_OPT_MN_OPERANDS:
    case MOE_OPT_LINEAR_CONCURRENT: return v == 0 || v == 1;
    case MOE_OPT_G1_WARPS: return v == 0 || v == 8 || v == 16;
    default: return false;
  }
}

// A second stream and a fork / join event pair per device, created on first use.  Enqueueing on it
// holds g_aux_mu from the fork to the join, so concurrent callers never re-record an event between
// another caller's record and the wait on it.
namespace {
constexpr int kMaxDevices = 64;
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
AuxStream g_aux[kMaxDevices];
std::mutex g_aux_mu;
}  // namespace

int fork_join(cudaStream_t st, const std::function<int(cudaStream_t)>& side, const std::function<int()>& main) {
  int dev = 0;
  int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device index %d above the library's limit", dev);
  std::lock_guard<std::mutex> lock(g_aux_mu);
  AuxStream& a = g_aux[dev];
  if (!a.s) {
    if ((rc = cuda_check(cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking), "second stream"))) return rc;
    if ((rc = cuda_check(cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming), "fork event")) ||
        (rc = cuda_check(cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming), "join event"))) {
      if (a.fork) cudaEventDestroy(a.fork);
      cudaStreamDestroy(a.s);
      a = AuxStream{};
      return rc;
    }
  }
  if ((rc = cuda_check(cudaEventRecord(a.fork, st), "fork record")) ||
      (rc = cuda_check(cudaStreamWaitEvent(a.s, a.fork, 0), "fork wait")))
    return rc;
  const int rc_side = side(a.s);
  // the join is enqueued whatever the side work returned, so the caller's stream never runs ahead of it
  if ((rc = cuda_check(cudaEventRecord(a.join, a.s), "join record"))) return rc;
  const int rc_main = rc_side ? MOE_OK : main();
  if ((rc = cuda_check(cudaStreamWaitEvent(st, a.join, 0), "join wait"))) return rc;
  return rc_side ? rc_side : rc_main;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_tmap_2d(void* out_tmap, const void* base, int elem_bytes, uint64_t rows, uint64_t cols,
                  uint64_t row_pitch_bytes, uint32_t box_rows, uint32_t box_cols, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
    return false;
  }
  CUtensorMap* m = static_cast<CUtensorMap*>(out_tmap);
  std::memset(m, 0, sizeof(*m));
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_pitch_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT32;
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fail(MOE_ERR_INVALID, "cuTensorMapEncodeTiled failed (%d): rows=%llu cols=%llu pitch=%llu box=%ux%u", (int)r,
         (unsigned long long)rows, (unsigned long long)cols, (unsigned long long)row_pitch_bytes, box_rows, box_cols);
    return false;
  }
  return true;
}

}  // namespace moebwd

extern "C" const char* moe_last_error(void) { return moebwd::g_err; }
extern "C" uint64_t moe_kernel_launches(void) { return moebwd::g_launches.load(); }
extern "C" const char* moe_version(void) { return "moebwd 0.1 (sm_103a tcgen05)"; }

extern "C" int moe_set_option(int opt, int64_t value) {
  moebwd::clear_error();
  if (opt < 0 || opt >= MOE_NUM_OPTIONS) return moebwd::fail(MOE_ERR_INVALID, "moe_set_option: unknown option %d", opt);
  if (value == -1) value = moebwd::kOptDefault[opt];
  if (!moebwd::option_value_ok(opt, value))
    return moebwd::fail(MOE_ERR_INVALID, "moe_set_option: value %lld not allowed for option %d", (long long)value, opt);
  moebwd::opt_init();
  moebwd::g_opt[opt].store(value);
  return MOE_OK;
}

extern "C" int64_t moe_get_option(int opt) {
  if (opt < 0 || opt >= MOE_NUM_OPTIONS) return -1;
  return moebwd::option(opt);
}
