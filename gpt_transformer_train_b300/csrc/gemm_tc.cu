// tcgen05 tensor-core GEMM (placeholder until the TMA/TMEM kernel lands).
#include "kernels.cuh"
bool gemm_tc_supported(const GemmArgs&) { return false; }
cudaError_t gemm_tc(const GemmArgs&, int*, cudaStream_t) { return cudaErrorNotSupported; }
