// Check of the bounded waits that every tensor-core kernel relies on.
//
// The tensor-core kernels never spin without a limit: each mbarrier wait
// gives up after a fixed time, raises the CTA's abort flag so the CTA's other
// warps stop waiting too, frees the CTA's tensor memory and reports
// FLAG_TIMEOUT to the host, which then returns GPT2_ERR_TIMEOUT with the
// context still usable.  gpt2_op_wait_probe runs that path on purpose: one
// CTA allocates tensor memory like the GEMM and attention kernels do, and its
// two warps wait on an mbarrier that nothing ever arrives on, one warp with
// the caller's short limit and one with the kernels' default limit (it ends
// when the first warp raises the abort flag).
#include "../../include/gpt2_ops.h"
#include "kernels.cuh"
#include "tc_common.cuh"

extern void gpt2_count_launches(int n);

namespace {

__global__ void __launch_bounds__(64) wait_probe_kernel(int* flags, uint64_t limit_ns) {
  using namespace tc;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_holder), 32);
  fence_before();
  __syncthreads();
  fence_after();
  pdl_enter();
  volatile int* ab = &abort_flag;
  // nothing arrives on `bar`: both waits end by the limit or the abort flag
  if (warp == 1) mbar_wait(smem_u32(&bar), 0, ab, limit_ns);
  else mbar_wait(smem_u32(&bar), 0, ab);
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tmem_holder, 32);
  if (threadIdx.x == 0 && *ab) atomicOr(flags, FLAG_TIMEOUT);
}

}  // namespace

extern "C" int gpt2_op_wait_probe(int limit_us, int* flags_dev, void* stream) {
  if (limit_us <= 0 || limit_us > 1000000 || !flags_dev) return GPT2_ERR_INVALID_ARG;
  if (!tc_available()) return GPT2_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  gpt2_count_launches(1);
  launch_k(wait_probe_kernel, dim3(1), dim3(64), 0, st, flags_dev, (uint64_t)limit_us * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return GPT2_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GPT2_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, flags_dev, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GPT2_ERR_CUDA;
  return (h & FLAG_TIMEOUT) ? GPT2_ERR_TIMEOUT : GPT2_OK;
}
