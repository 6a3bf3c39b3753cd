// Shared device helpers: element types, 128-bit vector access, warp/block
// reductions.  The "one 16-byte load per access" discipline follows the
// Packed128 idea of the CUDA MODE talk ([13:50] Avengers Assemble): every
// bandwidth kernel moves whole 128-bit words.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;

// ---- programmatic dependent launch ---------------------------------------
// Every kernel of the library is launched with launch_k(), which lets it
// start while the kernel before it on the stream is still finishing (its
// CTAs set up shared memory, barriers and TMEM meanwhile).  Each kernel calls
// pdl_wait() before its first access to global memory, in every CTA: that
// returns once the previous kernel has completed and its writes are visible,
// so the stream order of the results is unchanged (and, as every kernel
// waits, a kernel's completion still implies that of all kernels before it).
// pdl_trigger() right after it lets the next kernel be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_trigger();
}

// cudaLaunchKernelEx with the programmatic-serialisation attribute (plus an
// optional cluster size)
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  Function attributes are per device, so the library keeps
// one record per (kernel, device) under a lock and calls
// cudaFuncSetAttribute once for each; the first failure is returned (and
// retried on the next call).
cudaError_t kernel_smem_attr(const void* kernel, int bytes);
template <typename... KArgs>
inline cudaError_t kernel_smem_attr(void (*kernel)(KArgs...), int bytes) {
  return kernel_smem_attr(reinterpret_cast<const void*>(kernel), bytes);
}

// elements per 16-byte word
template <typename T> struct VecN;
template <> struct VecN<float> { static constexpr int n = 4; };
template <> struct VecN<bf16> { static constexpr int n = 8; };

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }
// value after a round trip through T (identity for float)
template <typename T> __device__ __forceinline__ float round_to(float x) { return to_f(from_f<T>(x)); }

// GELU in its tanh form, 0.5 x (1 + tanh u) with u = sqrt(2/pi) (x + 0.044715 x^3),
// evaluated as x * sigmoid(2u): the same function, since 0.5 (1 + tanh u) =
// 1 / (1 + exp(-2u)) = 1 / (1 + 2^(-2u log2 e)).  One base-2 exponential and
// one reciprocal, no branch, and no cancellation for negative x.  Every GELU
// of the library (the GEMM epilogues, the standalone and recompute kernels)
// goes through these two functions, so a recomputed GELU reproduces the
// forward's bits.
constexpr float GELU_2U = 1.5957691216057308f;    // 2 sqrt(2/pi)
constexpr float GELU_2U3 = 0.07135481627260025f;  // 2 sqrt(2/pi) * 0.044715
constexpr float GELU_E1 = -2.302208198144325f;    // -2 sqrt(2/pi) log2(e)
constexpr float GELU_E3 = -0.1029432395800235f;   // -2 sqrt(2/pi) * 0.044715 * log2(e)
__device__ __forceinline__ float gelu_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float gelu_fwd(float x) {
  const float e = gelu_exp2(x * fmaf(GELU_E3, x * x, GELU_E1));  // exp(-2u)
  return __fdividef(x, 1.f + e);
}
// its derivative: s + x s (1 - s) d(2u)/dx with s = sigmoid(2u)
__device__ __forceinline__ float gelu_bwd(float x) {
  const float x2 = x * x;
  const float e = gelu_exp2(x * fmaf(GELU_E3, x2, GELU_E1));
  const float du2 = fmaf(3.f * GELU_2U3, x2, GELU_2U);
  const float s = __fdividef(1.f, 1.f + e);
  return s * fmaf(x * du2, 1.f - s, 1.f);
}

// 16-byte load/store of VecN<T> elements as floats
__device__ __forceinline__ void ld16(const float* p, float (&f)[4]) {
  float4 v = *reinterpret_cast<const float4*>(p);
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
__device__ __forceinline__ void ld16(const bf16* p, float (&f)[8]) {
  uint4 v = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; i++) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x; f[2 * i + 1] = t.y;
  }
}
// streaming (evict-first) variants for data read exactly once
__device__ __forceinline__ void ld16_cs(const float* p, float (&f)[4]) {
  float4 v = __ldcs(reinterpret_cast<const float4*>(p));
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
__device__ __forceinline__ void ld16_cs(const bf16* p, float (&f)[8]) {
  uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; i++) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x; f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void st16(float* p, const float (&f)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
}
__device__ __forceinline__ void st16(bf16* p, const float (&f)[8]) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = v;
}
__device__ __forceinline__ void st16_cs(float* p, const float (&f)[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(f[0], f[1], f[2], f[3]));
}
__device__ __forceinline__ void st16_cs(bf16* p, const float (&f)[8]) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  __stcs(reinterpret_cast<uint4*>(p), v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum; every thread gets the result.  blockDim.x multiple of 32.
__device__ __forceinline__ float block_sum(float v, float* smem32) {
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) smem32[w] = v;
  __syncthreads();
  v = lane < nw ? smem32[lane] : 0.f;
  return warp_sum(v);
}

// flag bits raised by kernels, read back by the host at sync points
enum : int { FLAG_TOKEN_RANGE = 1, FLAG_TARGET_RANGE = 2, FLAG_TIMEOUT = 4 };

__host__ __device__ inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }
