// Instantiations of the tcgen05 GEMMs (one-CTA and CTA-pair) for the kFwd
// contraction; one translation unit per contraction so the four compile in
// parallel.
#include "tc_gemm.cuh"
#include "tc_gemm2.cuh"
#include "tc_gemm4.cuh"

namespace lmhead {
template cudaError_t launch_tc_gemm<kFwd>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                           const TcGemmParams&, int, cudaStream_t);
template cudaError_t launch_tc_gemm_pair<kFwd>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const TcGemmParams&, int, cudaStream_t);
template cudaError_t launch_tc_gemm_quad<kFwd>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const TcGemmParams&, int64_t, cudaStream_t, int*);
}  // namespace lmhead
