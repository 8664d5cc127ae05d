// Instantiations of the CTA-pair grouped GEMM (cta_group::2 tcgen05 MMA, 256 rows x BN per pair):
// BF16 and MXFP8, pair tiles 128 or 256 wide, store and checkpoint epilogues.
#include "gemm_pair_kernel.cuh"

namespace moebwd {

template <bool MX, int BN>
static int launch_bn(const GemmParams& p, const void* tmA, const void* tmB, const void* tmC, const void* tmSFA,
                     const void* tmSFB, int max_pairs, cudaStream_t st) {
  return p.epi == kEpiCkpt
             ? gemm_pair_launch_instance<MX, BN, kEpiCkpt>(p, tmA, tmB, tmC, tmSFA, tmSFB, max_pairs, st)
             : gemm_pair_launch_instance<MX, BN, kEpiStore>(p, tmA, tmB, tmC, tmSFA, tmSFB, max_pairs, st);
}

int launch_gemm_pair(bool mx, int BN, const GemmParams& p, const void* tmA, const void* tmB, const void* tmC,
                     const void* tmSFA, const void* tmSFB, int max_pairs, cudaStream_t st) {
  if (mx)
    return BN == 256 ? launch_bn<true, 256>(p, tmA, tmB, tmC, tmSFA, tmSFB, max_pairs, st)
                     : launch_bn<true, 128>(p, tmA, tmB, tmC, tmSFA, tmSFB, max_pairs, st);
  return BN == 256 ? launch_bn<false, 256>(p, tmA, tmB, tmC, tmSFA, tmSFB, max_pairs, st)
                   : launch_bn<false, 128>(p, tmA, tmB, tmC, tmSFA, tmSFB, max_pairs, st);
}

}  // namespace moebwd
