// Instantiation of the tcgen05 GEMM for the kDh contraction (one
// translation unit per contraction so the four compile in parallel).
#include "tc_gemm.cuh"

namespace lmhead {
template cudaError_t launch_tc_gemm<kDh>(const CUtensorMap&, const CUtensorMap&,
                                           const TcGemmParams&, int, cudaStream_t);
}  // namespace lmhead
