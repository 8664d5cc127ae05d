// MXFP8 instantiations of the tcgen05 grouped GEMM (kind::mxf8f6f4 block-scaled, E8M0 scales per
// 32 K-elements staged into TMEM with tcgen05.cp, FP32 accumulation in TMEM).
#include "gemm_kernel.cuh"

namespace moebwd {

int launch_gemm_mx(int BN, const GemmParams& p, const void* tmA, const void* tmB, const void* tmC, int grid,
                     cudaStream_t st) {
  if (p.epi == kEpiCkpt)  // G0 (recomputed pre-activations): 2I is a multiple of 256
    return gemm_launch_instance<true, 256, kEpiCkpt>(p, tmA, tmB, tmC, grid, st);
  if (p.epi == kEpiStore)
    return BN == 256 ? gemm_launch_instance<true, 256, kEpiStore>(p, tmA, tmB, tmC, grid, st)
                     : gemm_launch_instance<true, 128, kEpiStore>(p, tmA, tmB, tmC, grid, st);
  // G1 with two groups of epilogue warps (128- or 192-column tiles)
  if (p.epi == kEpiDSwiGLU2)
    return BN == 192 ? gemm_launch_instance<true, 192, kEpiDSwiGLU2>(p, tmA, tmB, tmC, grid, st)
                     : gemm_launch_instance<true, 128, kEpiDSwiGLU2>(p, tmA, tmB, tmC, grid, st);
  // G1: 192 columns (two TMEM accumulators, scales of W2 re-tiled per tile) where I allows
  if (BN == 192) return gemm_launch_instance<true, 192, kEpiDSwiGLU>(p, tmA, tmB, tmC, grid, st);
  return BN == 256 ? gemm_launch_instance<true, 256, kEpiDSwiGLU>(p, tmA, tmB, tmC, grid, st)
                   : gemm_launch_instance<true, 128, kEpiDSwiGLU>(p, tmA, tmB, tmC, grid, st);
}

}  // namespace moebwd
