// Instantiations of the tcgen05 GEMMs (one-CTA and CTA-pair) for the kDh
// contraction; one translation unit per contraction so the four compile in
// parallel.
#include "tc_gemm.cuh"
#include "tc_gemm2.cuh"
#include "tc_gemm4.cuh"

namespace lmhead {
template cudaError_t launch_tc_gemm<kDh>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                           const TcGemmParams&, int, cudaStream_t);
template cudaError_t launch_tc_gemm_pair<kDh>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const TcGemmParams&, int, cudaStream_t);
template cudaError_t launch_tc_gemm_quad<kDh>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const TcGemmParams&, int64_t, cudaStream_t, int*);
}  // namespace lmhead
