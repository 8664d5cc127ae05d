// moe_route_meta_noalloc: routing metadata for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code running inside a memory pool or
// arena that does not expose raw allocations, framework hooks that are not allowed to call
// cudaMalloc (it synchronises the device and can fail mid-step), and embedded or real-time callers
// that must not allocate after start-up.  For them this entry point runs the same routing kernels as
// moe_route_meta, but its scratch lives in a fixed, library-owned device array instead of a
// caller-provided workspace.
//
// The scratch is a file-scope `static __device__` array of kNoAllocScratchBytes.  Every GPU that
// loads the library holds it until the process exits.  In host code the array's name is only a
// host-side stand-in, so the device address is looked up once per device with cudaGetSymbolAddress
// (with that device current) on the first call made on that device; that first call should
// therefore come before any stream capture.  All calls on a device share the one array, which keeps
// the last call's contents: calls whose executions overlap on the GPU (different streams, or a call
// not yet finished on one stream while another stream starts) race on it and must be serialised by
// the caller.  The routing kernels write every scratch byte they later read within the same call
// (including the -1 fills of the padding tables), so nothing has to be cleared between calls.
#include <cuda_runtime.h>

#include <mutex>

#include "moebwd_internal.h"

namespace moebwd {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mutex;
static void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
static int noalloc_scratch(void** out) {
  int dev = 0;
  int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    rc = cuda_check(cudaGetSymbolAddress(&p, g_route_scratch), "cudaGetSymbolAddress(route scratch)");
    if (rc) return rc;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

}  // namespace moebwd

using namespace moebwd;

extern "C" int moe_route_meta_noalloc(const int32_t* ids, int T, int K, int E, int block_size,
                                      int32_t* expert_offsets, int32_t* x_gather_idx, int32_t* s_scatter_idx,
                                      int32_t* s_reverse_scatter_idx, int32_t* token_position_to_id,
                                      int32_t* block_to_expert, int32_t* block_offsets, int32_t* num_blocks,
                                      int32_t* status_dev, moe_stream_t stream) {
  clear_error();
  // the size checks of moe_route_meta, in its order and with its messages, before the scratch size
  // is computed from them
  int rc = check_route_sizes("moe_route_meta_noalloc", T, K, E, block_size);
  if (rc) return rc;
  const size_t need = moe_route_meta_workspace_size(T, K, E, block_size);
  if (need > kNoAllocScratchBytes)
    return fail(MOE_ERR_UNSUPPORTED,
                "moe_route_meta_noalloc: T=%d K=%d E=%d need %zu bytes of scratch, above the fixed %zu; "
                "use moe_route_meta with a workspace",
                T, K, E, need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  return moe_route_meta(ids, T, K, E, block_size, expert_offsets, x_gather_idx, s_scatter_idx, s_reverse_scatter_idx,
                        token_position_to_id, block_to_expert, block_offsets, num_blocks, status_dev, scratch,
                        kNoAllocScratchBytes, stream);
}
