// Instantiations of the tcgen05 GEMMs (one-CTA, and CTA pairs with 256- and
// 512-column tiles) for the kFwd contraction; one translation unit per
// contraction so the four compile in parallel.
#include "tc_gemm.cuh"
#include "tc_gemm2.cuh"

namespace lmhead {
template cudaError_t launch_tc_gemm<kFwd>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                       const TcGemmParams&, int, cudaStream_t);
template cudaError_t launch_tc_gemm_pair<kFwd, 1>(const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const TcGemmParams&, int,
                                               cudaStream_t);
template cudaError_t launch_tc_gemm_pair<kFwd, 2>(const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const TcGemmParams&, int,
                                               cudaStream_t);
}  // namespace lmhead
