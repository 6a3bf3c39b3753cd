// Encoder backward for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: code embedded in a
// host program that owns every byte of device memory (a framework's caching
// allocator, or a fixed memory budget planned up front), and code on a
// latency-critical path where cudaMalloc's implicit device-wide
// synchronisation is not acceptable.  gpt2_op_encoder_backward_noalloc gives
// them the deterministic encoder backward without a scratch argument: its
// sort keys live in a file-scope device array that the library itself owns.
//
// The array holds GPT2_NOALLOC_MAX_TOKENS 32-bit keys (128 KiB) on every GPU
// that loads the library, until the process exits.  Host code only sees a
// host-side stand-in under the array's name, so its device address is looked
// up once per device (cudaGetSymbolAddress, with that device current) on the
// first call made on that device.  The sort kernel writes every key slot it
// later reads, so nothing needs clearing between calls; calls that overlap
// on the GPU (two streams, or two threads) share the array and race.
// Tokens outside [0, V) are sorted past every real token and never scattered
// (dwte is indexed only by checked tokens); they raise FLAG_TOKEN_RANGE.
#include <mutex>

#include "../../include/gpt2_ops.h"
#include "kernels.cuh"

static __device__ __align__(256) uint32_t noalloc_keys[GPT2_NOALLOC_MAX_TOKENS];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_keys[kMaxDevices] = {};

// device address of noalloc_keys on the current device (nullptr on failure)
uint32_t* keys_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_keys[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, noalloc_keys) != cudaSuccess) return nullptr;
    g_keys[dev] = (uint32_t*)p;
  }
  return g_keys[dev];
}
}  // namespace

extern "C" int gpt2_op_encoder_backward_noalloc(float* dwte, float* dwpe, const float* dres, const int32_t* tokens,
                                                int B, int T, int C, int V, int* flags_dev, void* stream) {
  if (!dwte || !dwpe || !dres || !tokens || B <= 0 || T <= 0 || C <= 0 || C % 4) return GPT2_ERR_INVALID_ARG;
  if (V <= 0 || V > 65535) return GPT2_ERR_INVALID_ARG;
  // the keys of B*T positions, padded to a power of two, must fit the array
  if ((long long)B * T > GPT2_NOALLOC_MAX_TOKENS) return GPT2_ERR_BUFFER_TOO_SMALL;
  uint32_t* keys = keys_on_current_device();
  if (!keys) return GPT2_ERR_CUDA;
  cudaError_t e = encoder_backward(dwte, dwpe, dres, tokens, B, T, C, V, flags_dev, keys, (cudaStream_t)stream);
  return e == cudaSuccess ? GPT2_OK : (e == cudaErrorInvalidValue ? GPT2_ERR_INVALID_ARG : GPT2_ERR_CUDA);
}
