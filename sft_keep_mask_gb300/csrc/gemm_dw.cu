// Instantiation of the tcgen05 GEMM for the kDw contraction (one
// translation unit per contraction so the four compile in parallel).
#include "tc_gemm.cuh"

namespace lmhead {
template cudaError_t launch_tc_gemm<kDw>(const CUtensorMap&, const CUtensorMap&,
                                           const TcGemmParams&, int, cudaStream_t);
}  // namespace lmhead
