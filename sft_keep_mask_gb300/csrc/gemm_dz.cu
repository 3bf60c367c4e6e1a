// Instantiation of the tcgen05 GEMM for the kDz contraction (one
// translation unit per contraction so the four compile in parallel).
#include "tc_gemm.cuh"

namespace lmhead {
template cudaError_t launch_tc_gemm<kDz>(const CUtensorMap&, const CUtensorMap&,
                                           const TcGemmParams&, int, cudaStream_t);
}  // namespace lmhead
