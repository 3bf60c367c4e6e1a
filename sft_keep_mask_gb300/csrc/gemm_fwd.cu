// Instantiation of the tcgen05 GEMM for the kFwd contraction (one
// translation unit per contraction so the four compile in parallel).
#include "tc_gemm.cuh"

namespace lmhead {
template cudaError_t launch_tc_gemm<kFwd>(const CUtensorMap&, const CUtensorMap&,
                                           const TcGemmParams&, int, cudaStream_t);
}  // namespace lmhead
