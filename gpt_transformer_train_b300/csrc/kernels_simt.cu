// Bandwidth-bound kernels of the training step plus the SIMT GEMM and SIMT
// attention used by the fp32 exact-check mode.
//
// Layer semantics follow "llm.c: GPT-2 training in plain C, with every
// gradient written by hand", §2 How the code works (encoder, layernorm,
// matmul, attention, gelu, residual, softmax + crossentropy, each with a
// hand-written backward), and the talk "llm.c's Origin and the Future of LLM
// Compilers", [13:50] Avengers Assemble (fused residual+LayerNorm, fused
// classifier, full determinism: no floating-point atomics anywhere here).
#include "kernels.cuh"
#include "tc_common.cuh"
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>

#define LN_EPS 1e-5f

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

cudaError_t kernel_smem_attr(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;  // (kernel, device) -> bytes set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({kernel, dev});
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[{kernel, dev}] = bytes;
  return e;
}

static std::atomic<unsigned long long> g_launches{0};
void gpt2_count_launches(int n) { g_launches += (unsigned long long)(long long)n; }
unsigned long long gpt2_total_launches() { return g_launches.load(); }
// status of the kernels just enqueued; n = how many were launched
static inline cudaError_t launch_status(int n) {
  gpt2_count_launches(n);
  return cudaGetLastError();
}

// ============================================================================
// encoder: out[b,t,:] = wte[tok[b,t]] + wpe[t]
// ============================================================================
template <typename T>
__global__ void encoder_forward_kernel(T* __restrict__ out, const int* __restrict__ tok,
                                       const T* __restrict__ wte, const T* __restrict__ wpe, int BT,
                                       int T_, int C, int V, int* flags) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  const int nvec = C / N;
  long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)BT * nvec) return;
  int bt = (int)(idx / nvec), cv = (int)(idx % nvec);
  int t = bt % T_;
  int v = tok[bt];
  if (v < 0 || v >= V) {  // out-of-range token: flag it, read row 0 instead
    if (cv == 0) atomicOr(flags, FLAG_TOKEN_RANGE);
    v = 0;
  }
  float a[N], b[N];
  ld16(wte + (size_t)v * C + cv * N, a);
  ld16(wpe + (size_t)t * C + cv * N, b);
#pragma unroll
  for (int i = 0; i < N; i++) a[i] += b[i];
  st16(out + (size_t)bt * C + cv * N, a);
}

template <typename T>
cudaError_t encoder_forward(T* out, const int* tok, const T* wte, const T* wpe, int B, int T_, int C,
                            int V, int* flags, cudaStream_t st) {
  long long n = (long long)B * T_ * (C / VecN<T>::n);
  launch_k(encoder_forward_kernel<T>, dim3((unsigned)cdiv(n, 256)), dim3(256), 0, st, out, tok, wte, wpe, B * T_, T_, C, V, flags);
  return launch_status(1);
}

// ----------------------------------------------------------------------------
// encoder backward, deterministic (no atomics):
//   dwpe[t] += sum_b dres[b,t]
//   dwte[v] += sum over positions with token v, in increasing position order.
// Positions are bucketed by a single-CTA bitonic sort of (token << 16 | pos).
// ----------------------------------------------------------------------------
__global__ void wpe_grad_kernel(float* __restrict__ dwpe, const float* __restrict__ dres, int B, int T_, int C,
                                int accumulate) {
  pdl_enter();
  int nvec = C / 4;
  long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)T_ * nvec) return;
  int t = (int)(idx / nvec), cv = (int)(idx % nvec);
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  for (int b = 0; b < B; b++) {
    float x[4];
    ld16(dres + ((size_t)b * T_ + t) * C + cv * 4, x);
#pragma unroll
    for (int i = 0; i < 4; i++) s[i] += x[i];
  }
  float* dst = dwpe + (size_t)t * C + cv * 4;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  if (accumulate) ld16(dst, o);
#pragma unroll
  for (int i = 0; i < 4; i++) o[i] += s[i];
  st16(dst, o);
}

static inline int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}
size_t encoder_backward_scratch_bytes(int BT) { return (size_t)pow2_at_least(BT) * sizeof(uint32_t); }

// The sort key of position i: (token << 16) | i.  A token outside [0, V)
// (V <= 65535) gets the token field BAD_TOKEN, which sorts after every real
// token and is never scattered into dwte; it raises FLAG_TOKEN_RANGE.
constexpr uint32_t BAD_TOKEN = 0xFFFFu;
__device__ __forceinline__ uint32_t sort_key(const int* tok, int i, int V, int* flags) {
  const int v = tok[i];
  if (v < 0 || v >= V) {
    if (flags) atomicOr(flags, FLAG_TOKEN_RANGE);
    return (BAD_TOKEN << 16) | (uint32_t)i;
  }
  return ((uint32_t)v << 16) | (uint32_t)i;
}

// one CTA sorts n (power of two, <= 32768) keys in shared memory
__global__ void bitonic_sort_keys_kernel(uint32_t* keys_out, const int* __restrict__ tok, int BT, int n, int V,
                                         int* flags) {
  pdl_enter();
  extern __shared__ uint32_t sk[];
  for (int i = threadIdx.x; i < n; i += blockDim.x) sk[i] = i < BT ? sort_key(tok, i, V, flags) : 0xFFFFFFFFu;
  __syncthreads();
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int ixj = i ^ j;
        if (ixj > i) {
          uint32_t a = sk[i], b = sk[ixj];
          bool up = (i & k) == 0;
          if ((a > b) == up) { sk[i] = b; sk[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) keys_out[i] = sk[i];
}

// Block (i, column chunk of 128): if sorted key i starts a token run, sum that
// run's rows.  The run is cut at the multiples of WTE_CH in sorted order (the
// chunks of the large-scratch form below); warp w sums segments w, w+8, ...,
// each in entry order, and warp 0 adds the segment sums in order: the same
// additions in the same order as the large-scratch form, so both forms give
// identical bits.
constexpr int WTE_CH = 32;  // sorted entries per chunk
constexpr int RUNS_WARPS = 8;
__global__ void __launch_bounds__(32 * RUNS_WARPS) wte_grad_runs_kernel(float* __restrict__ dwte,
                                                                        const float* __restrict__ dres,
                                                                        const uint32_t* __restrict__ keys, int BT,
                                                                        int C) {
  pdl_enter();
  __shared__ float4 part[RUNS_WARPS][32];
  const int i = blockIdx.x;
  const uint32_t tk = keys[i] >> 16;
  if (tk == BAD_TOKEN || (i > 0 && (keys[i - 1] >> 16) == tk)) return;
  int lo = i + 1, hi = BT;  // first entry past the run
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((keys[mid] >> 16) <= tk) lo = mid + 1;
    else hi = mid;
  }
  const int j = lo, c0 = i / WTE_CH, nseg = (j - 1) / WTE_CH - c0 + 1;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int cv = blockIdx.y * 32 + lane;  // float4 column
  const bool on = cv < C / 4;
  float4 total = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < nseg; base += RUNS_WARPS) {
    const int k = base + w;
    float4 sg = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k < nseg) {
      const int a = max(i, (c0 + k) * WTE_CH), b = min(j, (c0 + k + 1) * WTE_CH);
      const uint32_t mykey = a + lane < b ? keys[a + lane] : 0u;  // the segment's keys, one per lane
      for (int e = 0; e < b - a; e += 8) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
          const uint32_t ku = __shfl_sync(0xffffffffu, mykey, (e + u) & 31);
          x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (on && e + u < b - a) x[u] = __ldcs(reinterpret_cast<const float4*>(dres + (size_t)(ku & 0xFFFFu) * C) + cv);
        }
#pragma unroll
        for (int u = 0; u < 8; u++)
          if (e + u < b - a) {
            sg.x += x[u].x; sg.y += x[u].y; sg.z += x[u].z; sg.w += x[u].w;
          }
      }
    }
    part[w][lane] = sg;
    __syncthreads();
    if (w == 0) {
      const int nq = min(RUNS_WARPS, nseg - base);
      for (int q = 0; q < nq; q++) {
        const float4 y = part[q][lane];
        if (base == 0 && q == 0) total = y;
        else {
          total.x += y.x; total.y += y.y; total.z += y.z; total.w += y.w;
        }
      }
    }
    __syncthreads();
  }
  if (w == 0 && on) {
    float4* dst = reinterpret_cast<float4*>(dwte + (size_t)tk * C) + cv;
    float4 o = *dst;
    o.x += total.x; o.y += total.y; o.z += total.z; o.w += total.w;
    *dst = o;
  }
}

cudaError_t encoder_backward(float* dwte, float* dwpe, const float* dres, const int* tok, int B, int T_,
                             int C, int V, int* flags, uint32_t* keys, cudaStream_t st,
                             int accumulate_wpe) {  // the small-scratch form
  int BT = B * T_;
  int n = pow2_at_least(BT);
  if (n > 32768 || V <= 0 || V > (int)BAD_TOKEN) return cudaErrorInvalidValue;
  long long nv = (long long)T_ * (C / 4);
  launch_k(wpe_grad_kernel, dim3((unsigned)cdiv(nv, 256)), dim3(256), 0, st, dwpe, dres, B, T_, C,
           accumulate_wpe);
  size_t smem = (size_t)n * sizeof(uint32_t);
  cudaError_t ea = kernel_smem_attr(bitonic_sort_keys_kernel, 32768 * 4);
  if (ea != cudaSuccess) return ea;
  launch_k(bitonic_sort_keys_kernel, dim3(1), dim3(1024), smem, st, keys, tok, BT, n, V, flags);
  launch_k(wte_grad_runs_kernel, dim3((unsigned)BT, (unsigned)cdiv(C / 4, 32)), dim3(256), 0, st, dwte, dres, keys, BT, C);
  return launch_status(3);
}

// ----------------------------------------------------------------------------
// The same encoder backward with a larger scratch (encoder_backward_fast_*):
// the keys are sorted by one CTA with a two-pass least-significant-digit
// radix sort on the token (8 bits a pass; positions start in order and every
// pass is stable, so equal tokens stay in position order), and the dwte sums
// go over fixed chunks of WTE_CH sorted entries, so that no CTA waits on a
// long run of one frequent token:
//   - a run of one token that starts and ends inside a chunk is summed there
//     and added into dwte;
//   - a run crossing chunk boundaries leaves one partial sum per chunk it
//     touches (slot 0: the chunk's first segment, slot 1: its last), and the
//     chunk where the run starts adds those partials into dwte in chunk order.
// Every dwte row is written by exactly one CTA and every sum has a fixed
// order: the result is deterministic.
// ----------------------------------------------------------------------------
constexpr int RADIX_MAX = 16384;  // keys the one-CTA radix sort holds in shared memory (twice)
static size_t fast_keys_bytes(int BT) { return ((size_t)BT * 4 + 255) & ~(size_t)255; }
size_t encoder_backward_fast_scratch_bytes(int BT, int C) {
  return fast_keys_bytes(BT) + (size_t)cdiv(BT, WTE_CH) * 2 * C * sizeof(float);
}
bool encoder_backward_fast_supported(int BT, int C) { return BT > 0 && BT <= RADIX_MAX && C % 4 == 0; }

__global__ void __launch_bounds__(1024) radix_sort_tokens_kernel(uint32_t* __restrict__ keys_out,
                                                                 const int* __restrict__ tok, int BT, int V,
                                                                 int* flags) {
  pdl_enter();
  extern __shared__ uint32_t rs_sh[];
  uint32_t* bufA = rs_sh;
  uint32_t* bufB = rs_sh + BT;
  uint32_t* cur = rs_sh + 2 * BT;  // [32 warps][256 digits]: counts, then scatter cursors
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int seg = ((BT + 31) / 32 + 31) & ~31;  // keys per warp, a multiple of 32
  const unsigned lt = (1u << lane) - 1u;
  for (int i = threadIdx.x; i < BT; i += blockDim.x) bufA[i] = sort_key(tok, i, V, flags);
  for (int pass = 0; pass < 2; pass++) {
    const int shift = 16 + 8 * pass;
    const uint32_t* src = pass == 0 ? bufA : bufB;
    uint32_t* dst = pass == 0 ? bufB : bufA;
    for (int i = threadIdx.x; i < 32 * 256; i += blockDim.x) cur[i] = 0;
    __syncthreads();
    for (int i = w * seg + lane; i < min(BT, (w + 1) * seg); i += 32) atomicAdd(&cur[w * 256 + ((src[i] >> shift) & 255)], 1u);
    __syncthreads();
    // exclusive scan in (digit, warp) order: thread t owns entries 8t .. 8t+7
    // of that order (digit = e / 32, warp = e % 32)
    uint32_t v[8], tsum = 0;
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const int e = 8 * threadIdx.x + q;
      v[q] = cur[(e & 31) * 256 + (e >> 5)];
      tsum += v[q];
    }
    uint32_t incl = tsum;  // inclusive scan of the thread sums: within the warp, then over the warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __shared__ uint32_t wsum[32];
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    uint32_t wpre = 0;
    for (int q = 0; q < w; q++) wpre += wsum[q];
    uint32_t run = wpre + incl - tsum;  // exclusive prefix of this thread's first entry
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const int e = 8 * threadIdx.x + q;
      cur[(e & 31) * 256 + (e >> 5)] = run;
      run += v[q];
    }
    __syncthreads();
    // stable scatter: each warp walks its keys in order, 32 at a time
    for (int base = w * seg; base < (w + 1) * seg; base += 32) {
      const int i = base + lane;
      const bool valid = i < BT;
      const uint32_t key = valid ? src[i] : 0u;
      const uint32_t d = valid ? (key >> shift) & 255 : 256u + lane;  // invalid lanes match nobody
      const unsigned peers = __match_any_sync(0xffffffffu, d);
      uint32_t pos = 0;
      if (valid) pos = cur[w * 256 + d] + __popc(peers & lt);
      __syncwarp();
      if (valid) {
        dst[pos] = key;
        if (lane == 31 - __clz(peers)) cur[w * 256 + d] += __popc(peers);
      }
      __syncwarp();
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < BT; i += blockDim.x) keys_out[i] = bufA[i];
}

// Block (chunk c, 128 float4 columns): the segments of equal tokens among
// sorted entries [c*WTE_CH, (c+1)*WTE_CH), each summed in entry order
__global__ void __launch_bounds__(128) wte_chunk_kernel(float* __restrict__ dwte, const float* __restrict__ dres,
                                                        const uint32_t* __restrict__ keys,
                                                        float* __restrict__ slots, int BT, int C) {
  pdl_enter();
  __shared__ uint32_t sk[WTE_CH + 2];  // tokens of entries e0-1 .. e1 (0xFFFFFFFF outside 0..BT-1)
  const int c = blockIdx.x, e0 = c * WTE_CH, e1 = min(BT, e0 + WTE_CH), ne = e1 - e0;
  if (threadIdx.x < ne + 2) {
    const int e = e0 - 1 + (int)threadIdx.x;
    sk[threadIdx.x] = (e >= 0 && e < BT) ? keys[e] : 0xFFFFFFFFu;
  }
  __syncthreads();
  auto tok_at = [&](int e) { return sk[e - e0 + 1] >> 16; };  // e in e0-1 .. e1
  const int cv = blockIdx.y * 128 + threadIdx.x;
  const bool on = cv < C / 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int seg_first = e0;
  for (int b = e0; b < e1; b += 8) {
    float4 x[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (on && b + u < e1)
        x[u] = __ldcs(reinterpret_cast<const float4*>(dres + (size_t)(sk[b + u - e0 + 1] & 0xFFFFu) * C) + cv);
    }
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int e = b + u;
      if (e >= e1) break;
      acc.x += x[u].x; acc.y += x[u].y; acc.z += x[u].z; acc.w += x[u].w;
      const uint32_t t = tok_at(e);
      if (e == e1 - 1 || tok_at(e + 1) != t) {  // end of a segment
        const bool run_start = seg_first > e0 || tok_at(e0 - 1) != t;
        const bool run_end = tok_at(e + 1) != t;
        if (on && t != BAD_TOKEN) {
          if (run_start && run_end) {
            float4* dst = reinterpret_cast<float4*>(dwte + (size_t)t * C) + cv;
            float4 o = *dst;
            o.x += acc.x; o.y += acc.y; o.z += acc.z; o.w += acc.w;
            *dst = o;
          } else {
            reinterpret_cast<float4*>(slots + ((size_t)c * 2 + (seg_first == e0 ? 0 : 1)) * C)[cv] = acc;
          }
        }
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        seg_first = e + 1;
      }
    }
  }
}

// Block (chunk c, 128 float4 columns): if a run that crosses into the next
// chunk starts in chunk c, add its partial sums into dwte in chunk order
__global__ void __launch_bounds__(128) wte_span_kernel(float* __restrict__ dwte, const uint32_t* __restrict__ keys,
                                                       const float* __restrict__ slots, int BT, int C) {
  pdl_enter();
  const int c = blockIdx.x, e0 = c * WTE_CH, e1 = min(BT, e0 + WTE_CH);
  const uint32_t tk = keys[e1 - 1] >> 16;
  if (tk == BAD_TOKEN || e1 >= BT || (keys[e1] >> 16) != tk) return;  // the chunk's last run ends here
  int s = e1 - 1;
  while (s > e0 && (keys[s - 1] >> 16) == tk) s--;
  if (s == e0 && e0 > 0 && (keys[e0 - 1] >> 16) == tk) return;  // the run started in an earlier chunk
  int lo = e1, hi = BT;  // first entry past the run
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((keys[mid] >> 16) <= tk) lo = mid + 1;
    else hi = mid;
  }
  const int c1 = (lo - 1) / WTE_CH;
  const int cv = blockIdx.y * 128 + threadIdx.x;
  if (cv >= C / 4) return;
  float4 sum = reinterpret_cast<const float4*>(slots + ((size_t)c * 2 + (s == e0 ? 0 : 1)) * C)[cv];
  for (int cc = c + 1; cc <= c1; cc++) {
    const float4 x = reinterpret_cast<const float4*>(slots + (size_t)cc * 2 * C)[cv];
    sum.x += x.x; sum.y += x.y; sum.z += x.z; sum.w += x.w;
  }
  float4* dst = reinterpret_cast<float4*>(dwte + (size_t)tk * C) + cv;
  float4 o = *dst;
  o.x += sum.x; o.y += sum.y; o.z += sum.z; o.w += sum.w;
  *dst = o;
}

cudaError_t encoder_backward_fast(float* dwte, float* dwpe, const float* dres, const int* tok, int B, int T_, int C,
                                  int V, int* flags, void* scratch, cudaStream_t st, int accumulate_wpe) {
  const int BT = B * T_;
  if (!encoder_backward_fast_supported(BT, C) || V <= 0 || V > (int)BAD_TOKEN) return cudaErrorInvalidValue;
  uint32_t* keys = (uint32_t*)scratch;
  float* slots = (float*)((char*)scratch + fast_keys_bytes(BT));
  const long long nv = (long long)T_ * (C / 4);
  launch_k(wpe_grad_kernel, dim3((unsigned)cdiv(nv, 256)), dim3(256), 0, st, dwpe, dres, B, T_, C,
           accumulate_wpe);
  const size_t smem = ((size_t)2 * BT + 32 * 256) * sizeof(uint32_t);
  {
    cudaError_t e = kernel_smem_attr(radix_sort_tokens_kernel, (int)(((size_t)2 * RADIX_MAX + 32 * 256) * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
  }
  launch_k(radix_sort_tokens_kernel, dim3(1), dim3(1024), smem, st, keys, tok, BT, V, flags);
  const dim3 grid((unsigned)cdiv(BT, WTE_CH), (unsigned)cdiv(C / 4, 128));
  launch_k(wte_chunk_kernel, grid, dim3(128), 0, st, dwte, dres, keys, slots, BT, C);
  launch_k(wte_span_kernel, grid, dim3(128), 0, st, dwte, keys, slots, BT, C);
  return launch_status(4);
}

// ============================================================================
// fused residual + LayerNorm forward: r = a (+ b); y = (r - mean) * rstd * w + bias
// one warp per row; the row lives in registers.  In bf16 the stored residual
// is rounded first and the statistics are taken from the rounded values.
// ============================================================================
template <typename T, int NV, int R>
__global__ void __launch_bounds__(256) residual_layernorm_forward_kernel(
    T* __restrict__ resid_out, T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd,
    const T* __restrict__ a, const T* __restrict__ b, const T* __restrict__ w, const T* __restrict__ bias, int rows,
    int C) {
  pdl_enter();
  // R rows per warp, all of their loads issued before any reduction (R = 1
  // measured fastest at GPT-2 widths)
  constexpr int N = VecN<T>::n;
  const int lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * R;
  const int nvec = C / N;
  float x[R][NV][N];
#pragma unroll
  for (int q = 0; q < R; q++) {
    const int row = row0 + q;
    if (row >= rows) break;
#pragma unroll
    for (int i = 0; i < NV; i++) {
      const int vi = lane + i * 32;
      if (vi < nvec) {
        ld16_cs(a + (size_t)row * C + vi * N, x[q][i]);
        if (b) {
          float xb[N];
          ld16_cs(b + (size_t)row * C + vi * N, xb);
#pragma unroll
          for (int k = 0; k < N; k++) x[q][i][k] = round_to<T>(x[q][i][k] + xb[k]);
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < R; q++) {
    const int row = row0 + q;
    if (row >= rows) break;
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
      const int vi = lane + i * 32;
      if (vi < nvec) {
        if (b) st16(resid_out + (size_t)row * C + vi * N, x[q][i]);
#pragma unroll
        for (int k = 0; k < N; k++) sum += x[q][i][k];
      }
    }
    const float mu = warp_sum(sum) / (float)C;
    float var = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
      if (lane + i * 32 < nvec) {
#pragma unroll
        for (int k = 0; k < N; k++) {
          const float d = x[q][i][k] - mu;
          var += d * d;
        }
      }
    }
    var = warp_sum(var) / (float)C;
    const float rs = 1.0f / sqrtf(var + LN_EPS);
    if (y) {  // (no y: only the statistics, for a product that folds the LayerNorm in)
#pragma unroll
      for (int i = 0; i < NV; i++) {
        const int vi = lane + i * 32;
        if (vi < nvec) {
          float wv[N], bv[N], o[N];
          ld16(w + vi * N, wv);
          ld16(bias + vi * N, bv);
#pragma unroll
          for (int k = 0; k < N; k++) o[k] = (x[q][i][k] - mu) * rs * wv[k] + bv[k];
          st16(y + (size_t)row * C + vi * N, o);
        }
      }
    }
    if (lane == 0) {
      mean[row] = mu;
      rstd[row] = rs;
    }
  }
}

template <typename T>
cudaError_t residual_layernorm_forward(T* resid_out, T* y, float* mean, float* rstd, const T* a,
                                       const T* b, const T* w, const T* bias, int rows, int C,
                                       cudaStream_t st) {
  constexpr int N = VecN<T>::n;
  const int nvec = C / N;
#define LNF(NVv, Rv)                                                                                      \
  launch_k(residual_layernorm_forward_kernel<T, NVv, Rv>, dim3((unsigned)cdiv(rows, 8 * Rv)), dim3(256), 0, st, resid_out, y, mean, \
                                                                                             rstd, a, b, w, bias, \
                                                                                             rows, C)
  if (nvec <= 32) LNF(1, 1);
  else if (nvec <= 64) LNF(2, 1);
  else if (nvec <= 96) LNF(3, 1);
  else if (nvec <= 128) LNF(4, 1);
  else if (nvec <= 256) LNF(8, 1);
  else if (nvec <= 512) LNF(16, 1);
  else return cudaErrorInvalidValue;
#undef LNF
  return launch_status(1);
}

// y = (r - mean) * rstd * w + bias from a stored residual row and its stored
// statistics: the forward's last step, on the same stored values, for
// activation recompute (same expression, same bits as the forward's y)
template <typename T>
__global__ void __launch_bounds__(256) layernorm_apply_kernel(T* __restrict__ y, const T* __restrict__ r,
                                                              const float* __restrict__ mean,
                                                              const float* __restrict__ rstd,
                                                              const T* __restrict__ w, const T* __restrict__ bias,
                                                              int rows, int C) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  const int nvec = C / N;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)rows * nvec) return;
  const int row = (int)(i / nvec), vi = (int)(i % nvec);
  const float mu = mean[row], rs = rstd[row];
  float x[N], wv[N], bv[N], o[N];
  ld16_cs(r + (size_t)row * C + vi * N, x);
  ld16(w + vi * N, wv);
  ld16(bias + vi * N, bv);
#pragma unroll
  for (int k = 0; k < N; k++) o[k] = (x[k] - mu) * rs * wv[k] + bv[k];
  st16(y + (size_t)row * C + vi * N, o);
}

template <typename T>
cudaError_t layernorm_apply(T* y, const T* r, const float* mean, const float* rstd, const T* w, const T* bias,
                            int rows, int C, cudaStream_t st) {
  constexpr int N = VecN<T>::n;
  if (C % N || rows <= 0) return cudaErrorInvalidValue;
  const long long n = (long long)rows * (C / N);
  launch_k(layernorm_apply_kernel<T>, dim3((unsigned)cdiv(n, 256)), dim3(256), 0, st, y, r, mean, rstd, w, bias,
           rows, C);
  return launch_status(1);
}

// ============================================================================
// Deterministic column reductions.  Producers write per-chunk partial sums
// (a chunk = a fixed block of rows, summed in a fixed order); reduce_partials
// then adds the chunks into the outputs in a fixed order.  No atomics, so
// every gradient below is bitwise repeatable.
// ============================================================================
constexpr int RED_ROWS = 64;  // rows per chunk
constexpr int CS_ROWS = 512;  // rows per chunk of the column sums (a multiple of RED_ROWS)
int reduce_chunks(int rows) {
  int c = (int)cdiv(rows, RED_ROWS);
  return c < 1 ? 1 : c;
}
size_t ln_backward_partial_floats(int rows, int C) { return (size_t)reduce_chunks(rows) * 3 * C; }
size_t colsum_partial_floats(int rows, int cols) { return (size_t)reduce_chunks(rows) * cols; }

// out_o[c] += sum_k partial[k][o][c] for o < nout (out_o may be null: skipped).
// Block (column group of 32, output o, batch item z: partial and out_o
// advance by sPart and sOut per item); warp w sums chunks w, w+8, ... in
// order, then the eight warp sums are added in warp order.
__global__ void __launch_bounds__(256) reduce_partials_kernel(float* __restrict__ out0, float* __restrict__ out1,
                                                              float* __restrict__ out2,
                                                              const float* __restrict__ partial, int nchunks,
                                                              int C, int nout, long long sOut, long long sPart,
                                                              int accumulate) {
  pdl_enter();
  __shared__ float sh[8][32];
  const int o = blockIdx.y;
  float* out = o == 0 ? out0 : (o == 1 ? out1 : out2);
  if (!out) return;
  out += blockIdx.z * sOut;
  partial += blockIdx.z * sPart;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  // chunks w, w+8, w+16, ... in increasing order; eight loads in flight, added in that order
  float s = 0.f;
  if (c < C) {
    const float* src = partial + (size_t)o * C + c;
    const size_t stride = (size_t)nout * C;
    int k = w;
    for (; k + 56 < nchunks; k += 64) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; u++) v[u] = src[(size_t)(k + 8 * u) * stride];
#pragma unroll
      for (int u = 0; u < 8; u++) s += v[u];
    }
    for (; k < nchunks; k += 8) s += src[(size_t)k * stride];
  }
  sh[w][lane] = s;
  __syncthreads();
  if (w == 0 && c < C) {
    float t = sh[0][lane];
#pragma unroll
    for (int i = 1; i < 8; i++) t += sh[i][lane];
    out[c] = accumulate ? out[c] + t : t;
  }
}

cudaError_t reduce_partials(float* out0, float* out1, float* out2, const float* partial, int nchunks, int C,
                            int nout, cudaStream_t st, int nbatch, long long sOut, long long sPart, int accumulate) {
  if (nbatch < 1 || nbatch > 65535) return cudaErrorInvalidValue;
  if (sPart == 0) sPart = (long long)nchunks * nout * C;
  dim3 grid((unsigned)cdiv(C, 32), nout, nbatch);
  launch_k(reduce_partials_kernel, dim3(grid), dim3(256), 0, st, out0, out1, out2, partial, nchunks, C, nout, sOut,
           sPart, accumulate);
  return launch_status(1);
}

// Partial sums of the eight warps' per-lane column accumulators, added in warp
// order through shared memory; acc[i][k] is column (lane + 32 i) * N + k.
template <int NV, int N>
__device__ __forceinline__ void block_column_sum(float (&acc)[NV][N], float* sh, int nvec, float* dst) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int turn = 0; turn < 8; turn++) {
    if (w == turn) {
#pragma unroll
      for (int i = 0; i < NV; i++) {
        const int vi = lane + i * 32;
        if (vi < nvec)
#pragma unroll
          for (int k = 0; k < N; k++) sh[vi * N + k] = turn == 0 ? acc[i][k] : sh[vi * N + k] + acc[i][k];
      }
    }
    __syncthreads();
  }
  for (int c = threadIdx.x; c < nvec * N; c += blockDim.x) dst[c] = sh[c];
  __syncthreads();
}

// ============================================================================
// LayerNorm backward, one warp per row (RPW rows per warp, 8 warps a block):
//   dnorm = dy * w; dx = rstd * (dnorm - mean(dnorm) - xhat * mean(dnorm * xhat))
//   dres = (accumulate ? dres : 0) + dx   (fp32; optional copy in T)
// With partial: each warp accumulates, in its own shared-memory slice, the
// column sums over its rows of dy * xhat, dy and (if want_rsum) the new dres;
// the block adds the eight slices in warp order into partial[block][3][C] for
// dw, db and the bias gradient of the projection whose output gradient dres is.
// ============================================================================
// The residual gradient passes from rin to rout in its own type RT (float,
// or the activation type: the training step's bf16 form):
//   rout = (rin ? rin : 0) + dx, rcopy (optional, T) and rf32 (optional,
//   float) receive the same new value; rout may be null when rf32 is given,
//   and rin may equal rout (in place).
constexpr int LNB_RPW = 8;
// 8 consecutive values of a residual-gradient row, as floats
__device__ __forceinline__ void ld8(const float* p, float (&f)[8]) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p)), b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void ld8(const bf16* p, float (&f)[8]) { ld16_cs(p, f); }
__device__ __forceinline__ void st8(float* p, const float (&f)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ void st8(bf16* p, const float (&f)[8]) { st16(p, f); }
template <typename T, typename RT, int NV>
__global__ void __launch_bounds__(256, NV <= 4 ? 2 : 1) layernorm_backward_kernel(
    RT* rout, const RT* rin, T* __restrict__ rcopy, float* __restrict__ rf32, const T* __restrict__ dy,
    const T* __restrict__ x, const float* __restrict__ mean, const float* __restrict__ rstd, const T* __restrict__ w,
    int rows, int C, float* __restrict__ partial, int want_rsum) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  extern __shared__ float lnb_sh[];  // [8 warps][3][N][nvec] when partial
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = C / N;
  // this warp's accumulators, element-major ([array][k][vector]) so that the
  // 32 lanes of a warp touch 32 consecutive floats: no bank conflicts
  float* acc = lnb_sh + (size_t)warp * 3 * C;
  if (partial)
    for (int c = lane; c < 3 * C; c += 32) acc[c] = 0.f;
  const int r0 = (blockIdx.x * 8 + warp) * LNB_RPW;
  for (int rr = 0; rr < LNB_RPW; rr++) {
    const int row = r0 + rr;
    if (row >= rows) break;
    const float mu = mean[row], rs = rstd[row];
    float dn[NV][N], xh[NV][N], acc_in[NV][N];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
      const int vi = lane + i * 32;
      if (vi < nvec) {
        float xv[N], dv[N], wv[N];
        ld16_cs(dy + (size_t)row * C + vi * N, dv);
        ld16_cs(x + (size_t)row * C + vi * N, xv);
        ld16(w + vi * N, wv);
        // the incoming residual gradient, fetched with the row rather than after the reductions
#pragma unroll
        for (int k = 0; k < N; k++) acc_in[i][k] = 0.f;
        if (rin) {
          if constexpr (sizeof(RT) == 4) {
#pragma unroll
            for (int k = 0; k < N; k += 4) {
              float a4[4];
              ld16_cs(reinterpret_cast<const float*>(rin) + (size_t)row * C + vi * N + k, a4);
#pragma unroll
              for (int u = 0; u < 4; u++) acc_in[i][k + u] = a4[u];
            }
          } else {
            static_assert(sizeof(RT) == 4 || N == 8, "a bf16 residual gradient goes with bf16 rows");
            ld16_cs(reinterpret_cast<const bf16*>(rin) + (size_t)row * C + vi * N,
                    *reinterpret_cast<float(*)[8]>(acc_in[i]));
          }
        }
#pragma unroll
        for (int k = 0; k < N; k++) {
          xh[i][k] = (xv[k] - mu) * rs;
          dn[i][k] = dv[k] * wv[k];
          s1 += dn[i][k];
          s2 += dn[i][k] * xh[i][k];
        }
        if (partial) {
#pragma unroll
          for (int k = 0; k < N; k++) {
            acc[k * nvec + vi] += dv[k] * xh[i][k];
            acc[(N + k) * nvec + vi] += dv[k];
          }
        }
      }
    }
    s1 = warp_sum(s1) / (float)C;
    s2 = warp_sum(s2) / (float)C;
#pragma unroll
    for (int i = 0; i < NV; i++) {
      const int vi = lane + i * 32;
      if (vi < nvec) {
        float o[N];
#pragma unroll
        for (int k = 0; k < N; k++) o[k] = acc_in[i][k] + (dn[i][k] - s1 - xh[i][k] * s2) * rs;
        if (rout) {
          if constexpr (sizeof(RT) == 4) {
            float* dst = reinterpret_cast<float*>(rout) + (size_t)row * C + vi * N;
#pragma unroll
            for (int k = 0; k < N; k += 4) {
              float r4[4] = {o[k], o[k + 1], o[k + 2], o[k + 3]};
              st16(dst + k, r4);
            }
          } else {
            st16(reinterpret_cast<T*>(rout) + (size_t)row * C + vi * N, o);
          }
        }
        if (rcopy) st16(rcopy + (size_t)row * C + vi * N, o);
        if (rf32) {
#pragma unroll
          for (int k = 0; k < N; k += 4) {
            float r4[4] = {o[k], o[k + 1], o[k + 2], o[k + 3]};
            st16(rf32 + (size_t)row * C + vi * N + k, r4);
          }
        }
        if (partial && want_rsum) {
#pragma unroll
          for (int k = 0; k < N; k++) acc[(2 * N + k) * nvec + vi] += o[k];
        }
      }
    }
  }
  if (!partial) return;  // uniform over the block
  __syncthreads();
  // sum the eight warps' slices in warp order; column c = vi * N + k
  float* dst = partial + (size_t)blockIdx.x * 3 * C;
  const int nc = want_rsum ? 3 * C : 2 * C;
  for (int idx = threadIdx.x; idx < nc; idx += blockDim.x) {  // shared-memory order: no bank conflicts
    const int a = idx / C, rem = idx - a * C, k = rem / nvec, vi = rem - k * nvec;
    float t = lnb_sh[idx];
#pragma unroll
    for (int q = 1; q < 8; q++) t += lnb_sh[(size_t)q * 3 * C + idx];
    dst[a * C + vi * N + k] = t;
  }
}

// bf16 rows of at most 1024 columns: one CTA of LNBP_WARPS warps per SM, each
// warp owning a contiguous range of rpw rows and keeping the next row's dy,
// x, mean, rstd and (bf16, up to 768 columns) incoming residual gradient in
// flight (registers) while it computes the current one; a wider or fp32
// incoming residual gradient is fetched before the row's reductions.  Same
// arithmetic, per-warp shared-memory accumulators and partial layout
// (partial[block][3][C]) as layernorm_backward_kernel.
constexpr int LNBP_WARPS = 16;
template <int NV>
__device__ __forceinline__ void lnbp_fetch(uint4 (&vdy)[NV], uint4 (&vx)[NV], const bf16* dy, const bf16* x, size_t off,
                                           int lane, int nvec) {
#pragma unroll
  for (int i = 0; i < NV; i++) {
    const int vi = lane + i * 32;
    if (vi < nvec) {
      vdy[i] = __ldcs(reinterpret_cast<const uint4*>(dy + off) + vi);
      vx[i] = __ldcs(reinterpret_cast<const uint4*>(x + off) + vi);
    }
  }
}
__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
// packed fp32 pairs (one instruction for two values)
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 x, y, z, w;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%6, %7};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 x, y, w;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 x, y, w;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "add.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// 8 bf16 values of a 16-byte word as four float pairs
__device__ __forceinline__ void unpack_bf16x8_2(const uint4& v, float2 (&f)[4]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; i++) f[i] = __bfloat1622float2(h[i]);
}
// The per-warp column sums live in shared memory as [3][C] (dw, db, new
// residual gradient), each lane updating its own 8 columns with two 16-byte
// read-modify-writes per array, laid out so that those of a warp hit
// consecutive addresses (acc_slot; with the columns in order, lanes 32 bytes
// apart made every update an 8-way bank conflict, which cost more than the
// rest of the kernel); the CTA's sum over its warps goes out in column order.
// All arithmetic on packed fp32 pairs.
template <typename RT, int NV>
__global__ void __launch_bounds__(32 * LNBP_WARPS, 1) layernorm_backward_pipe_kernel(
    RT* rout, const RT* rin, bf16* __restrict__ rcopy, float* __restrict__ rf32, const bf16* __restrict__ dy,
    const bf16* __restrict__ x, const float* __restrict__ mean, const float* __restrict__ rstd,
    const bf16* __restrict__ w, int rows, int C, float* __restrict__ partial, int want_rsum, int rpw) {
  pdl_enter();
  constexpr int N = 8;
  extern __shared__ float lnb_sh[];  // [LNBP_WARPS][3][C] when partial
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = C / N;
  float* acc = lnb_sh + (size_t)warp * 3 * C;
  // columns 8 vi + 4 h .. + 3 of array a at acc + a C + h C/2 + 4 vi: a warp's
  // 16-byte updates of one half fall on consecutive addresses (no bank conflicts)
  auto acc_slot = [&](int a, int h, int vi) {
    return reinterpret_cast<float4*>(acc + (size_t)a * C + (size_t)h * (C / 2) + 4 * vi);
  };
  if (partial)
    for (int c = 4 * lane; c < 3 * C; c += 128) *reinterpret_cast<float4*>(acc + c) = make_float4(0.f, 0.f, 0.f, 0.f);
  uint4 wv[NV];
#pragma unroll
  for (int i = 0; i < NV; i++)
    if (lane + i * 32 < nvec) wv[i] = reinterpret_cast<const uint4*>(w)[lane + i * 32];
  const int r0 = (blockIdx.x * LNBP_WARPS + warp) * rpw;
  const int r1 = min(rows, r0 + rpw);
  uint4 ndy[NV], nx[NV];
  float nmu = 0.f, nrs = 0.f;  // the next row's statistics, fetched with its dy and x
  // a bf16 incoming residual gradient is fetched a row ahead as well
  constexpr bool PRE_DIN = sizeof(RT) == 2 && NV < 4;
  uint4 ndin[PRE_DIN ? NV : 1];
  auto fetch_next = [&](int rr) {
    lnbp_fetch<NV>(ndy, nx, dy, x, (size_t)rr * C, lane, nvec);
    nmu = mean[rr];
    nrs = rstd[rr];
    if constexpr (PRE_DIN) {
#pragma unroll
      for (int i = 0; i < NV; i++) {
        const int vi = lane + i * 32;
        ndin[i] = make_uint4(0u, 0u, 0u, 0u);
        if (rin && vi < nvec) ndin[i] = __ldcs(reinterpret_cast<const uint4*>(rin + (size_t)rr * C) + vi);
      }
    }
  };
  if (r0 < r1) fetch_next(r0);
  for (int row = r0; row < r1; row++) {
    uint4 cdy[NV], cx[NV], cdin[PRE_DIN ? NV : 1];
#pragma unroll
    for (int i = 0; i < NV; i++) {
      cdy[i] = ndy[i];
      cx[i] = nx[i];
      if constexpr (PRE_DIN) cdin[i] = ndin[i];
    }
    const float mu = nmu, rs = nrs;
    if (row + 1 < r1) fetch_next(row + 1);
    const float2 rs2 = make_float2(rs, rs), nmr = make_float2(-mu * rs, -mu * rs);
    // the incoming residual gradient: fetched with the row, or (the widest
    // rows, to keep registers free) after the first pass
    float din[NV][N];
    auto load_din = [&]() {
#pragma unroll
      for (int i = 0; i < NV; i++) {
        if constexpr (PRE_DIN) {
          unpack_bf16x8(cdin[i], din[i]);
        } else {
          const int vi = lane + i * 32;
#pragma unroll
          for (int k = 0; k < N; k++) din[i][k] = 0.f;
          if (rin && vi < nvec) ld8(rin + (size_t)row * C + vi * N, din[i]);
        }
      }
    };
    if constexpr (NV < 4) load_din();
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NV; i++) {
      const int vi = lane + i * 32;
      if (vi < nvec) {
        float2 dv[4], xv[4], ww[4];
        unpack_bf16x8_2(cdy[i], dv);
        unpack_bf16x8_2(cx[i], xv);
        unpack_bf16x8_2(wv[i], ww);
        float2 xh[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
          xh[k] = f2_fma(xv[k], rs2, nmr);
          const float2 dn = f2_mul(dv[k], ww[k]);
          s1 = f2_add(s1, dn);
          s2 = f2_fma(dn, xh[k], s2);
        }
        if (partial) {
#pragma unroll
          for (int h = 0; h < 2; h++) {
            float4* aw = acc_slot(0, h, vi);
            float4* ab = acc_slot(1, h, vi);
            float4 a = *aw, b = *ab;
            const float2 lo = f2_fma(dv[2 * h], xh[2 * h], make_float2(a.x, a.y));
            const float2 hi = f2_fma(dv[2 * h + 1], xh[2 * h + 1], make_float2(a.z, a.w));
            const float2 blo = f2_add(dv[2 * h], make_float2(b.x, b.y));
            const float2 bhi = f2_add(dv[2 * h + 1], make_float2(b.z, b.w));
            *aw = make_float4(lo.x, lo.y, hi.x, hi.y);
            *ab = make_float4(blo.x, blo.y, bhi.x, bhi.y);
          }
        }
      }
    }
    if constexpr (NV >= 4) load_din();
    const float m1 = -warp_sum(s1.x + s1.y) / (float)C;
    const float m2 = -warp_sum(s2.x + s2.y) / (float)C;
    const float2 m1v = make_float2(m1, m1), m2v = make_float2(m2, m2);
#pragma unroll
    for (int i = 0; i < NV; i++) {
      const int vi = lane + i * 32;
      if (vi < nvec) {
        float2 dv[4], xv[4], ww[4];
        unpack_bf16x8_2(cdy[i], dv);
        unpack_bf16x8_2(cx[i], xv);
        unpack_bf16x8_2(wv[i], ww);
        float o[N];
#pragma unroll
        for (int k = 0; k < 4; k++) {
          // o = din + (dn - mean(dn) - xhat * mean(dn xhat)) * rstd
          const float2 xh = f2_fma(xv[k], rs2, nmr);
          const float2 t = f2_fma(xh, m2v, f2_add(f2_mul(dv[k], ww[k]), m1v));
          const float2 ov = f2_fma(t, rs2, make_float2(din[i][2 * k], din[i][2 * k + 1]));
          o[2 * k] = ov.x;
          o[2 * k + 1] = ov.y;
        }
        if (rout) st8(rout + (size_t)row * C + vi * N, o);
        if (rcopy) st16(rcopy + (size_t)row * C + vi * N, o);
        if (rf32) st8(rf32 + (size_t)row * C + vi * N, o);
        if (partial && want_rsum) {
#pragma unroll
          for (int h = 0; h < 2; h++) {
            float4* ar = acc_slot(2, h, vi);
            const float4 a = *ar;
            const float2 lo = f2_add(make_float2(o[4 * h], o[4 * h + 1]), make_float2(a.x, a.y));
            const float2 hi = f2_add(make_float2(o[4 * h + 2], o[4 * h + 3]), make_float2(a.z, a.w));
            *ar = make_float4(lo.x, lo.y, hi.x, hi.y);
          }
        }
      }
    }
  }
  if (!partial) return;  // uniform over the block
  __syncthreads();
  float* dst = partial + (size_t)blockIdx.x * 3 * C;
  const int nc = want_rsum ? 3 * C : 2 * C;
  for (int idx = 4 * threadIdx.x; idx < nc; idx += 4 * blockDim.x) {
    float4 t = *reinterpret_cast<const float4*>(lnb_sh + idx);
#pragma unroll
    for (int q = 1; q < LNBP_WARPS; q++) {
      const float4 u = *reinterpret_cast<const float4*>(lnb_sh + (size_t)q * 3 * C + idx);
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    // back to the partial buffer's column order (see acc_slot)
    const int a = idx / C, f = idx % C, h = f / (C / 2), vi = (f % (C / 2)) / 4;
    *reinterpret_cast<float4*>(dst + (size_t)a * C + 8 * vi + 4 * h) = t;
  }
}

template <typename T, typename RT>
cudaError_t layernorm_backward_rg(RT* rout, const RT* rin, T* rcopy, float* rf32, const T* dy, const T* x,
                                  const float* mean, const float* rstd, const T* w, int rows, int C, float* dw,
                                  float* db, float* dres_sum, float* partial, cudaStream_t st, int* deferred_chunks) {
  static_assert(sizeof(RT) == 4 || sizeof(T) == 2, "a bf16 residual gradient goes with bf16 rows");
  if (!rout && !rf32) return cudaErrorInvalidValue;
  constexpr int N = VecN<T>::n;
  const int nvec = C / N;
  const bool sums = dw || db || dres_sum;
  if (sums && (!dw || !db || !partial)) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)cdiv(rows, 8 * LNB_RPW);
  const size_t smem = sums ? (size_t)8 * 3 * C * sizeof(float) : 0;
  if (sums) {
    const int mx = 8 * 3 * 2048 * (int)sizeof(float);
    for (auto k : {layernorm_backward_kernel<T, RT, 1>, layernorm_backward_kernel<T, RT, 2>,
                   layernorm_backward_kernel<T, RT, 3>, layernorm_backward_kernel<T, RT, 4>,
                   layernorm_backward_kernel<T, RT, 6>, layernorm_backward_kernel<T, RT, 8>,
                   layernorm_backward_kernel<T, RT, 12>, layernorm_backward_kernel<T, RT, 16>}) {
      cudaError_t e = kernel_smem_attr(k, mx);
      if (e != cudaSuccess) return e;
    }
  }
  float* part = sums ? partial : nullptr;
  const int rsum = dres_sum != nullptr;
  if constexpr (sizeof(T) == 2) {
    if (nvec <= 128 && ((uintptr_t)rout & 15) == 0 && ((uintptr_t)rin & 15) == 0 && ((uintptr_t)rf32 & 15) == 0 &&
        ((uintptr_t)w & 15) == 0) {
      // one CTA per SM, never more CTAs than the partial buffer has chunks
      const int pgrid = std::min(tc_num_sms(), reduce_chunks(rows));
      const int rpw = (int)cdiv(rows, (long long)pgrid * LNBP_WARPS);
      const size_t psmem = sums ? (size_t)LNBP_WARPS * 3 * C * sizeof(float) : 0;
      {
        const int mx = LNBP_WARPS * 3 * 1024 * (int)sizeof(float);
        for (auto k : {layernorm_backward_pipe_kernel<RT, 1>, layernorm_backward_pipe_kernel<RT, 2>,
                       layernorm_backward_pipe_kernel<RT, 3>, layernorm_backward_pipe_kernel<RT, 4>}) {
          cudaError_t e = kernel_smem_attr(k, mx);
          if (e != cudaSuccess) return e;
        }
      }
#define LNBP(NVv)                                                                                            \
  launch_k(layernorm_backward_pipe_kernel<RT, NVv>, dim3(pgrid), dim3(32 * LNBP_WARPS), psmem, st, rout, rin,     \
           (bf16*)rcopy, rf32, (const bf16*)dy, (const bf16*)x, mean, rstd, (const bf16*)w, rows, C, part, rsum, \
           rpw)
      if (nvec <= 32) LNBP(1);
      else if (nvec <= 64) LNBP(2);
      else if (nvec <= 96) LNBP(3);
      else LNBP(4);
#undef LNBP
      cudaError_t e = launch_status(1);
      if (e != cudaSuccess || !sums) return e;
      if (deferred_chunks) {
        *deferred_chunks = pgrid;
        return cudaSuccess;
      }
      return reduce_partials(dw, db, dres_sum, partial, pgrid, C, 3, st);
    }
  }
#define LNB(NVv)                                                                                              \
  launch_k(layernorm_backward_kernel<T, RT, NVv>, dim3(grid), dim3(256), smem, st, rout, rin, rcopy, rf32, dy, x, \
           mean, rstd, w, rows, C, part, rsum)
  if (nvec <= 32) LNB(1);
  else if (nvec <= 64) LNB(2);
  else if (nvec <= 96) LNB(3);
  else if (nvec <= 128) LNB(4);
  else if (nvec <= 192) LNB(6);
  else if (nvec <= 256) LNB(8);
  else if (nvec <= 384) LNB(12);
  else if (nvec <= 512) LNB(16);
  else return cudaErrorInvalidValue;
#undef LNB
  cudaError_t e = launch_status(1);
  if (e != cudaSuccess || !sums) return e;
  // rows of 64 per chunk = 8 warps x LNB_RPW rows per block
  if (deferred_chunks) {
    *deferred_chunks = (int)grid;
    return cudaSuccess;
  }
  return reduce_partials(dw, db, dres_sum, partial, (int)grid, C, 3, st);
}

template <typename T>
cudaError_t layernorm_backward(float* dres, T* dres_c, const T* dy, const T* x, const float* mean,
                               const float* rstd, const T* w, int rows, int C, int accumulate, float* dw,
                               float* db, float* dres_sum, float* partial, cudaStream_t st, int* deferred_chunks) {
  return layernorm_backward_rg<T, float>(dres, accumulate ? dres : nullptr, dres_c, nullptr, dy, x, mean, rstd, w,
                                         rows, C, dw, db, dres_sum, partial, st, deferred_chunks);
}

// ============================================================================
// column sums: out[c] += sum_r X[r*ldx + c], chunks of RED_ROWS rows
// ============================================================================
template <typename T>
__global__ void __launch_bounds__(256) colsum_partial_kernel(float* __restrict__ partial, const T* __restrict__ X,
                                                             int rows, int cols, long long ldx, long long sX,
                                                             int chunk_rows) {
  pdl_enter();
  X += blockIdx.z * sX;  // batch item z: its own matrix and partial rows
  partial += (size_t)blockIdx.z * gridDim.y * cols;
  constexpr int N = VecN<T>::n;
  extern __shared__ float cs_sh[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v0 = blockIdx.x * 32;  // first vector column of this block
  const int nvec = cols / N;
  const int vi = v0 + lane;
  float acc[1][N];
#pragma unroll
  for (int k = 0; k < N; k++) acc[0][k] = 0.f;
  const int r0 = blockIdx.y * chunk_rows, r1 = min(rows, r0 + chunk_rows);
  if (vi < nvec) {
    // rows warp, warp+8, ... in order; four loads in flight, added in that order
    int r = r0 + warp;
    for (; r + 24 < r1; r += 32) {
      float v[4][N];
#pragma unroll
      for (int u = 0; u < 4; u++) ld16_cs(X + (size_t)(r + 8 * u) * ldx + (size_t)vi * N, v[u]);
#pragma unroll
      for (int u = 0; u < 4; u++)
#pragma unroll
        for (int k = 0; k < N; k++) acc[0][k] += v[u][k];
    }
    for (; r < r1; r += 8) {
      float v[N];
      ld16_cs(X + (size_t)r * ldx + (size_t)vi * N, v);
#pragma unroll
      for (int k = 0; k < N; k++) acc[0][k] += v[k];
    }
  }
  // warp-ordered combine of this block's 32 vector columns
  for (int turn = 0; turn < 8; turn++) {
    if (warp == turn && vi < nvec)
#pragma unroll
      for (int k = 0; k < N; k++) cs_sh[lane * N + k] = turn == 0 ? acc[0][k] : cs_sh[lane * N + k] + acc[0][k];
    __syncthreads();
  }
  float* dst = partial + (size_t)blockIdx.y * cols + (size_t)v0 * N;
  for (int c = threadIdx.x; c < 32 * N; c += blockDim.x)
    if (v0 * N + c < cols) dst[c] = cs_sh[c];
}

template <typename T>
cudaError_t colsum(float* out, const T* X, int rows, int cols, long long ldx, float* partial, cudaStream_t st,
                   int nbatch, long long sOut, long long sX, int accumulate) {
  constexpr int N = VecN<T>::n;
  if (cols % N || ldx % N || nbatch < 1 || nbatch > 65535) return cudaErrorInvalidValue;
  // chunks of CS_ROWS rows (a block's fixed setup and its ordered warp combine
  // are paid once per 512 rows, not per 64; at most reduce_chunks(rows) chunks,
  // which the partial buffer is sized for)
  const int nch = std::max(1, (int)cdiv(rows, CS_ROWS));
  dim3 grid((unsigned)cdiv(cols / N, 32), nch, nbatch);
  launch_k(colsum_partial_kernel<T>, dim3(grid), dim3(256), 32 * N * sizeof(float), st, partial, X, rows, cols, ldx,
           sX, (int)CS_ROWS);
  cudaError_t e = launch_status(1);
  if (e != cudaSuccess) return e;
  return reduce_partials(out, nullptr, nullptr, partial, nch, cols, 1, st, nbatch, sOut, 0, accumulate);
}

// ============================================================================
// SIMT GEMM (fp32 mode, and any shape the tensor-core path does not take)
// 64x64 tile, BK 16, 256 threads, 4x4 per thread, fp32 accumulate.
// ============================================================================
template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
  pdl_enter();
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const T* A = (const T*)g.A;
  const T* B = (const T*)g.B;
  int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < g.K; k0 += 16) {
    // 64x16 tiles of A and B: 1024 elements each, 4 per thread
#pragma unroll
    for (int r = 0; r < 4; r++) {
      int e = threadIdx.x + r * 256;
      int mm, kk;
      if (g.a_kmajor) { mm = e / 16; kk = e % 16; } else { kk = e / 64; mm = e % 64; }
      int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < g.M && gk < g.K)
        v = to_f(g.a_kmajor ? A[(size_t)gm * g.lda + gk] : A[(size_t)gk * g.lda + gm]);
      As[kk][mm] = v;
      int nn;
      if (g.b_kmajor) { nn = e / 16; kk = e % 16; } else { kk = e / 64; nn = e % 64; }
      int gn = n0 + nn;
      gk = k0 + kk;
      v = 0.f;
      if (gn < g.N && gk < g.K)
        v = to_f(g.b_kmajor ? B[(size_t)gn * g.ldb + gk] : B[(size_t)gk * g.ldb + gn]);
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; kk++) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; i++) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; j++) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; i++) {
    int m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      float v = acc[i][j];
      if (g.epi == EPI_ACC_F32) {
        float* D = (float*)g.D;
        D[(size_t)m * g.ldd + n] = g.acc_store ? v : D[(size_t)m * g.ldd + n] + v;
      } else if (g.epi == EPI_GELU_BWD) {
        float h = to_f(((const T*)g.aux)[(size_t)m * g.ldaux + n]);
        ((T*)g.D)[(size_t)m * g.ldd + n] = from_f<T>(v * gelu_bwd(h));
      } else {
        if (g.bias) v += to_f(((const T*)g.bias)[n]);
        if (g.epi == EPI_GELU) {
          // GELU of the pre-activation as stored, so a later recompute from aux gives the same bits
          ((T*)g.aux)[(size_t)m * g.ldaux + n] = from_f<T>(v);
          v = gelu_fwd(round_to<T>(v));
        }
        ((T*)g.D)[(size_t)m * g.ldd + n] = from_f<T>(v);
      }
    }
  }
}

template <typename T>
cudaError_t gemm_simt(const GemmArgs& a, cudaStream_t st) {
  if (a.M <= 0 || a.N <= 0 || a.K <= 0) return cudaErrorInvalidValue;
  if (a.ln_mean) return cudaErrorNotSupported;  // the folded LayerNorm is a tensor-core epilogue
  dim3 grid((unsigned)cdiv(a.N, 64), (unsigned)cdiv(a.M, 64));
  const int nb = a.batch > 1 ? a.batch : 1;
  if (nb > 1 && a.bias) return cudaErrorInvalidValue;
  const size_t dsz = a.epi == EPI_ACC_F32 ? sizeof(float) : sizeof(T);
  for (int z = 0; z < nb; z++) {  // a batch is launched item by item
    GemmArgs b = a;
    b.batch = 1;
    b.A = (const T*)a.A + z * a.sA;
    b.B = (const T*)a.B + z * a.sB;
    b.D = (char*)a.D + z * a.sD * dsz;
    if (a.aux) b.aux = (T*)a.aux + z * a.sAux;
    launch_k(gemm_simt_kernel<T>, dim3(grid), dim3(256), 0, st, b);
  }
  return launch_status(nb);
}

// ============================================================================
// Products with few rows (M <= 32: one position per sequence when decoding):
// D[m][n] = sum_k A[m][k] B[n][k] (+ bias, optionally GELU with aux), both
// operands K-major.  Bound by the stream of B: A is copied to shared memory
// once per CTA; each warp owns NC output columns and issues every 16-byte load
// of those rows of B at once (lane l takes elements 8l.. of each of the KCH
// 256-wide chunks; KCH = K / 256 for bf16), so one round trip serves the whole
// row, then walks the rows m one at a time (a short loop body that stays in
// the instruction cache), one fp32 sum per column, and adds the 32 lanes'
// sums by a shuffle tree.
// ============================================================================
constexpr int SKINNY_WARPS = 8;
template <typename T, int KCH, int NC>
__global__ void __launch_bounds__(32 * SKINNY_WARPS) gemm_skinny_kernel(GemmArgs g) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  extern __shared__ __align__(16) unsigned char sk_raw[];
  T* xs = reinterpret_cast<T*>(sk_raw);  // [M][K]
  const int M = g.M, K = g.K, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const T* A = (const T*)g.A;
  const T* Bw = (const T*)g.B;
  const int ngroups = (g.N + NC - 1) / NC;
  uint4 wr[NC][KCH];  // this warp's rows of B, all in flight at once
  auto fetch = [&](int grp) {
    const int n0 = grp * NC;
#pragma unroll
    for (int c = 0; c < NC; c++)
#pragma unroll
      for (int j = 0; j < KCH; j++)
        wr[c][j] = n0 + c < g.N ? __ldcs(reinterpret_cast<const uint4*>(Bw + (size_t)(n0 + c) * g.ldb) + j * 32 + lane)
                                : make_uint4(0u, 0u, 0u, 0u);
  };
  // the first group's B rows are requested before A is copied, so both round trips overlap
  int grp = blockIdx.x * SKINNY_WARPS + w;
  if (grp < ngroups) fetch(grp);
  for (int i0 = threadIdx.x; i0 < M * (K / N); i0 += 4 * blockDim.x) {
    uint4 t[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int i = i0 + u * blockDim.x;
      if (i < M * (K / N)) t[u] = reinterpret_cast<const uint4*>(A + (size_t)(i / (K / N)) * g.lda)[i % (K / N)];
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int i = i0 + u * blockDim.x;
      if (i < M * (K / N)) reinterpret_cast<uint4*>(xs + (size_t)(i / (K / N)) * K)[i % (K / N)] = t[u];
    }
  }
  __syncthreads();
  for (; grp < ngroups; grp += gridDim.x * SKINNY_WARPS) {
    const int n0 = grp * NC;
    if (grp != (int)(blockIdx.x * SKINNY_WARPS + w)) fetch(grp);
    for (int m = 0; m < M; m++) {
      float acc[NC];
#pragma unroll
      for (int c = 0; c < NC; c++) acc[c] = 0.f;
#pragma unroll
      for (int j = 0; j < KCH; j++) {
        float xv[N];
        ld16(xs + (size_t)m * K + (j * 32 + lane) * N, xv);
#pragma unroll
        for (int c = 0; c < NC; c++) {
          float wv[N];
          if constexpr (N == 8) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&wr[c][j]);
#pragma unroll
            for (int e = 0; e < 4; e++) {
              const float2 t = __bfloat1622float2(h[e]);
              wv[2 * e] = t.x;
              wv[2 * e + 1] = t.y;
            }
          } else {
            const float* q = reinterpret_cast<const float*>(&wr[c][j]);
#pragma unroll
            for (int e = 0; e < N; e++) wv[e] = q[e];
          }
#pragma unroll
          for (int e = 0; e < N; e++) acc[c] = fmaf(xv[e], wv[e], acc[c]);
        }
      }
#pragma unroll
      for (int c = 0; c < NC; c++) {
        const int n = n0 + c;
        float v = warp_sum(acc[c]);
        if (lane == c && n < g.N) {
          if (g.bias) v += to_f(((const T*)g.bias)[n]);
          if (g.epi == EPI_GELU) {
            ((T*)g.aux)[(size_t)m * g.ldaux + n] = from_f<T>(v);
            v = gelu_fwd(round_to<T>(v));
          }
          ((T*)g.D)[(size_t)m * g.ldd + n] = from_f<T>(v);
        }
      }
    }
  }
}

template <typename T>
static int skinny_chunks(int K) {
  constexpr int N = VecN<T>::n;
  return K % (32 * N) ? 0 : K / (32 * N);
}

template <typename T>
bool gemm_skinny_supported(const GemmArgs& a) {
  auto al16 = [](const void* q) { return ((uintptr_t)q & 15) == 0; };
  const int kch = skinny_chunks<T>(a.K);
  return a.M >= 1 && a.M <= 32 && a.N >= 1 && kch >= 1 && kch <= 12 && a.a_kmajor && a.b_kmajor && !a.ln_mean &&
         a.batch <= 1 && (a.epi == EPI_STORE || (a.epi == EPI_GELU && a.aux)) && a.lda % VecN<T>::n == 0 &&
         a.ldb % VecN<T>::n == 0 && al16(a.A) && al16(a.B) && (size_t)a.M * a.K * sizeof(T) <= 200 * 1024;
}

template <typename T, int KCH, int NC>
static cudaError_t skinny_launch(const GemmArgs& a, size_t smem, cudaStream_t st) {
  {
    cudaError_t e = kernel_smem_attr(gemm_skinny_kernel<T, KCH, NC>, 200 * 1024);
    if (e != cudaSuccess) return e;
  }
  const int grid = (int)std::min<long long>(cdiv(cdiv(a.N, NC), SKINNY_WARPS), 8LL * tc_num_sms());
  launch_k(gemm_skinny_kernel<T, KCH, NC>, dim3(grid), dim3(32 * SKINNY_WARPS), smem, st, a);
  return cudaSuccess;
}

template <typename T>
static cudaError_t skinny_by_k(const GemmArgs& a, size_t smem, cudaStream_t st) {
  switch (skinny_chunks<T>(a.K)) {  // two columns per warp while the registers allow
    case 1: return skinny_launch<T, 1, 2>(a, smem, st);
    case 2: return skinny_launch<T, 2, 2>(a, smem, st);
    case 3: return skinny_launch<T, 3, 2>(a, smem, st);
    case 4: return skinny_launch<T, 4, 2>(a, smem, st);
    case 5: return skinny_launch<T, 5, 1>(a, smem, st);
    case 6: return skinny_launch<T, 6, 1>(a, smem, st);
    case 7: return skinny_launch<T, 7, 1>(a, smem, st);
    case 8: return skinny_launch<T, 8, 1>(a, smem, st);
    case 9: return skinny_launch<T, 9, 1>(a, smem, st);
    case 10: return skinny_launch<T, 10, 1>(a, smem, st);
    case 11: return skinny_launch<T, 11, 1>(a, smem, st);
    default: return skinny_launch<T, 12, 1>(a, smem, st);
  }
}

template <typename T>
cudaError_t gemm_skinny(const GemmArgs& a, cudaStream_t st) {
  if (!gemm_skinny_supported<T>(a)) return cudaErrorInvalidValue;
  const size_t smem = (size_t)a.M * a.K * sizeof(T);
  const cudaError_t e = skinny_by_k<T>(a, smem, st);
  if (e != cudaSuccess) return e;
  return launch_status(1);
}

// ============================================================================
// SIMT causal attention (any head size <= 128).  Forward: one warp per query
// row, keys in chunks of 32 (one key per lane), online max/sum, LSE saved.
// Backward: D = rowsum(dO*O); a dQ pass per query row and a dK/dV pass per
// key row recompute P from the LSE (no atomics).
// ============================================================================
#define ATT_WARPS 8
template <typename T>
__global__ void __launch_bounds__(256) attention_forward_simt_kernel(T* __restrict__ out, float* __restrict__ lse,
                                                                     const T* __restrict__ qkv, int B, int T_, int C,
                                                                     int H, float scale) {
  pdl_enter();
  __shared__ float qs[ATT_WARPS][128];
  int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long gq = (long long)blockIdx.x * ATT_WARPS + warp;
  if (gq >= (long long)B * H * T_) return;
  int hd = C / H;
  int t = (int)(gq % T_);
  int h = (int)((gq / T_) % H);
  int b = (int)(gq / ((long long)T_ * H));
  const size_t rs = 3 * (size_t)C;
  const T* base = qkv + (size_t)b * T_ * rs;
  for (int d = lane; d < hd; d += 32) qs[warp][d] = to_f(base[(size_t)t * rs + h * hd + d]) * scale;
  __syncwarp();
  float m = -INFINITY, l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 <= t; k0 += 32) {
    int t2 = k0 + lane;
    float s = -INFINITY;
    if (t2 <= t) {
      const T* kr = base + (size_t)t2 * rs + C + h * hd;
      s = 0.f;
      for (int d = 0; d < hd; d++) s = fmaf(qs[warp][d], to_f(kr[d]), s);
    }
    float mn = fmaxf(m, warp_max(s));
    float p = t2 <= t ? expf(s - mn) : 0.f;
    float alpha = expf(m - mn);
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int i = 0; i < 4; i++) o[i] *= alpha;
    int jn = min(32, t - k0 + 1);
    for (int j = 0; j < jn; j++) {
      float pj = __shfl_sync(0xffffffffu, p, j);
      const T* vr = base + (size_t)(k0 + j) * rs + 2 * C + h * hd;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        int d = lane + 32 * i;
        if (d < hd) o[i] = fmaf(pj, to_f(vr[d]), o[i]);
      }
    }
    m = mn;
  }
  float inv = 1.f / l;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    int d = lane + 32 * i;
    if (d < hd) out[((size_t)b * T_ + t) * C + h * hd + d] = from_f<T>(o[i] * inv);
  }
  if (lane == 0) lse[((size_t)b * H + h) * T_ + t] = m + logf(l);
}

template <typename T>
cudaError_t attention_forward_simt(T* out, float* lse, const T* qkv, int B, int T_, int C, int H,
                                   cudaStream_t st) {
  int hd = C / H;
  if (hd > 128 || C % H) return cudaErrorInvalidValue;
  long long rows = (long long)B * H * T_;
  launch_k(attention_forward_simt_kernel<T>, dim3((unsigned)cdiv(rows, ATT_WARPS)), dim3(32 * ATT_WARPS), 0, st, out, lse, qkv, B, T_, C, H, 1.0f / sqrtf((float)hd));
  return launch_status(1);
}

// D[b,h,t] = sum_d dO[b,t,h,d] * O[b,t,h,d]
template <typename T>
__global__ void attention_bwd_dot_kernel(float* __restrict__ Dbuf, const T* __restrict__ dout,
                                         const T* __restrict__ out, int B, int T_, int C, int H) {
  pdl_enter();
  int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long gq = (long long)blockIdx.x * ATT_WARPS + warp;
  if (gq >= (long long)B * H * T_) return;
  int hd = C / H;
  int t = (int)(gq % T_), h = (int)((gq / T_) % H), b = (int)(gq / ((long long)T_ * H));
  size_t o = ((size_t)b * T_ + t) * C + h * hd;
  float s = 0.f;
  for (int d = lane; d < hd; d += 32) s += to_f(dout[o + d]) * to_f(out[o + d]);
  s = warp_sum(s);
  if (lane == 0) Dbuf[((size_t)b * H + h) * T_ + t] = s;
}

// dQ[t] = scale * sum_{t2<=t} dS[t,t2] K[t2],  dS = P (dP - D), dP = dO . V
template <typename T>
__global__ void __launch_bounds__(256) attention_bwd_dq_kernel(T* __restrict__ dqkv, const T* __restrict__ dout,
                                                               const T* __restrict__ qkv, const float* __restrict__ lse,
                                                               const float* __restrict__ Dbuf, int B, int T_, int C,
                                                               int H, float scale) {
  pdl_enter();
  __shared__ float qs[ATT_WARPS][128];
  __shared__ float dos[ATT_WARPS][128];
  int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long gq = (long long)blockIdx.x * ATT_WARPS + warp;
  if (gq >= (long long)B * H * T_) return;
  int hd = C / H;
  int t = (int)(gq % T_), h = (int)((gq / T_) % H), b = (int)(gq / ((long long)T_ * H));
  const size_t rs = 3 * (size_t)C;
  const T* base = qkv + (size_t)b * T_ * rs;
  for (int d = lane; d < hd; d += 32) {
    qs[warp][d] = to_f(base[(size_t)t * rs + h * hd + d]) * scale;
    dos[warp][d] = to_f(dout[((size_t)b * T_ + t) * C + h * hd + d]);
  }
  __syncwarp();
  float L = lse[((size_t)b * H + h) * T_ + t];
  float Dv = Dbuf[((size_t)b * H + h) * T_ + t];
  float dq[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 <= t; k0 += 32) {
    int t2 = k0 + lane;
    float ds = 0.f;
    if (t2 <= t) {
      const T* kr = base + (size_t)t2 * rs + C + h * hd;
      const T* vr = base + (size_t)t2 * rs + 2 * C + h * hd;
      float s = 0.f, dp = 0.f;
      for (int d = 0; d < hd; d++) {
        s = fmaf(qs[warp][d], to_f(kr[d]), s);
        dp = fmaf(dos[warp][d], to_f(vr[d]), dp);
      }
      float p = expf(s - L);
      ds = p * (dp - Dv);
    }
    int jn = min(32, t - k0 + 1);
    for (int j = 0; j < jn; j++) {
      float dsj = __shfl_sync(0xffffffffu, ds, j);
      const T* kr = base + (size_t)(k0 + j) * rs + C + h * hd;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        int d = lane + 32 * i;
        if (d < hd) dq[i] = fmaf(dsj, to_f(kr[d]), dq[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; i++) {
    int d = lane + 32 * i;
    if (d < hd) dqkv[((size_t)b * T_ + t) * rs + h * hd + d] = from_f<T>(dq[i] * scale);
  }
}

// dV[t2] = sum_{t>=t2} P[t,t2] dO[t];  dK[t2] = scale * sum_{t>=t2} dS[t,t2] Q[t]
template <typename T>
__global__ void __launch_bounds__(256) attention_bwd_dkv_kernel(T* __restrict__ dqkv, const T* __restrict__ dout,
                                                                const T* __restrict__ qkv, const float* __restrict__ lse,
                                                                const float* __restrict__ Dbuf, int B, int T_, int C,
                                                                int H, float scale) {
  pdl_enter();
  __shared__ float ks[ATT_WARPS][128];
  __shared__ float vs[ATT_WARPS][128];
  int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long gk = (long long)blockIdx.x * ATT_WARPS + warp;
  if (gk >= (long long)B * H * T_) return;
  int hd = C / H;
  int t2 = (int)(gk % T_), h = (int)((gk / T_) % H), b = (int)(gk / ((long long)T_ * H));
  const size_t rs = 3 * (size_t)C;
  const T* base = qkv + (size_t)b * T_ * rs;
  for (int d = lane; d < hd; d += 32) {
    ks[warp][d] = to_f(base[(size_t)t2 * rs + C + h * hd + d]) * scale;
    vs[warp][d] = to_f(base[(size_t)t2 * rs + 2 * C + h * hd + d]);
  }
  __syncwarp();
  const float* L = lse + ((size_t)b * H + h) * T_;
  const float* Dv = Dbuf + ((size_t)b * H + h) * T_;
  float dk[4] = {0.f, 0.f, 0.f, 0.f}, dv[4] = {0.f, 0.f, 0.f, 0.f};
  for (int q0 = t2; q0 < T_; q0 += 32) {
    int t = q0 + lane;
    float p = 0.f, ds = 0.f;
    if (t < T_) {
      const T* qr = base + (size_t)t * rs + h * hd;
      const T* dor = dout + ((size_t)b * T_ + t) * C + h * hd;
      float s = 0.f, dp = 0.f;
      for (int d = 0; d < hd; d++) {
        s = fmaf(ks[warp][d], to_f(qr[d]), s);
        dp = fmaf(vs[warp][d], to_f(dor[d]), dp);
      }
      p = expf(s - L[t]);
      ds = p * (dp - Dv[t]);
    }
    int jn = min(32, T_ - q0);
    for (int j = 0; j < jn; j++) {
      float pj = __shfl_sync(0xffffffffu, p, j);
      float dsj = __shfl_sync(0xffffffffu, ds, j);
      const T* qr = base + (size_t)(q0 + j) * rs + h * hd;
      const T* dor = dout + ((size_t)b * T_ + q0 + j) * C + h * hd;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        int d = lane + 32 * i;
        if (d < hd) {
          dv[i] = fmaf(pj, to_f(dor[d]), dv[i]);
          dk[i] = fmaf(dsj, to_f(qr[d]), dk[i]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; i++) {
    int d = lane + 32 * i;
    if (d < hd) {
      dqkv[((size_t)b * T_ + t2) * rs + C + h * hd + d] = from_f<T>(dk[i] * scale);
      dqkv[((size_t)b * T_ + t2) * rs + 2 * C + h * hd + d] = from_f<T>(dv[i]);
    }
  }
}

template <typename T>
cudaError_t attention_backward_simt(T* dqkv, float* Dbuf, const T* dout, const T* qkv, const T* out,
                                    const float* lse, int B, int T_, int C, int H, cudaStream_t st) {
  int hd = C / H;
  if (hd > 128 || C % H) return cudaErrorInvalidValue;
  long long rows = (long long)B * H * T_;
  unsigned grid = (unsigned)cdiv(rows, ATT_WARPS);
  float scale = 1.0f / sqrtf((float)hd);
  launch_k(attention_bwd_dot_kernel<T>, dim3(grid), dim3(32 * ATT_WARPS), 0, st, Dbuf, dout, out, B, T_, C, H);
  launch_k(attention_bwd_dq_kernel<T>, dim3(grid), dim3(32 * ATT_WARPS), 0, st, dqkv, dout, qkv, lse, Dbuf, B, T_, C, H, scale);
  launch_k(attention_bwd_dkv_kernel<T>, dim3(grid), dim3(32 * ATT_WARPS), 0, st, dqkv, dout, qkv, lse, Dbuf, B, T_, C, H, scale);
  return launch_status(3);
}

// ============================================================================
// fused softmax + cross-entropy over the first V of Vp columns, one CTA per
// row.  Pass 1: online (max, sum) with 128-bit loads; loss = lse - z[target].
// Pass 2 (write_grad): dlogits = (softmax - onehot) * dloss written in place,
// pad columns 0.  The row (<= 100 KB in bf16) is re-read from L2.
// ============================================================================
template <typename T>
__global__ void __launch_bounds__(1024) softmax_ce_kernel(T* __restrict__ logits, float* __restrict__ losses,
                                                          const int* __restrict__ targets, int V, int Vp,
                                                          float dloss, int write_grad, int* flags) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  __shared__ float sm[32], ss[32];
  __shared__ float s_lse;
  __shared__ int s_tg;
  int row = blockIdx.x;
  T* z = logits + (size_t)row * Vp;
  const int nvec = Vp / N;
  float m = -INFINITY, s = 0.f;
  for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
    float f[N];
    ld16(z + (size_t)vi * N, f);
#pragma unroll
    for (int k = 0; k < N; k++) {
      if (vi * N + k < V) {
        float x = f[k];
        if (x > m) { s = s * expf(m - x) + 1.f; m = x; }
        else s += expf(x - m);
      }
    }
  }
  // combine (m, s) across the warp, then across warps
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    float mm = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * expf(m2 - mm));
    m = mm;
  }
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) { sm[w] = m; ss[w] = s; }
  __syncthreads();
  if (w == 0) {
    m = lane < nw ? sm[lane] : -INFINITY;
    s = lane < nw ? ss[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      float mm = fmaxf(m, m2);
      s = (m == -INFINITY ? 0.f : s * expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * expf(m2 - mm));
      m = mm;
    }
    if (lane == 0) {
      int tg = targets[row];
      if (tg < 0 || tg >= V) {
        atomicOr(flags, FLAG_TARGET_RANGE);
        tg = 0;
      }
      float lse = m + logf(s);
      s_lse = lse;
      s_tg = tg;
      losses[row] = lse - to_f(z[tg]);
    }
  }
  __syncthreads();
  if (!write_grad) return;
  float lse = s_lse;
  int tg = s_tg;
  for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
    float f[N];
    ld16(z + (size_t)vi * N, f);
#pragma unroll
    for (int k = 0; k < N; k++) {
      int idx = vi * N + k;
      f[k] = idx < V ? (expf(f[k] - lse) - (idx == tg ? 1.f : 0.f)) * dloss : 0.f;
    }
    st16(z + (size_t)vi * N, f);
  }
}

// Register-resident variant: the row is read from HBM once into registers
// (VPT 16-byte words per thread), max and sum are block reductions over the
// registers, and dlogits is written from them: one read and one write of the
// row.  exp2 of pre-scaled arguments (ex2.approx).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <typename T, int VPT>
__global__ void __launch_bounds__(1024) softmax_ce_reg_kernel(T* __restrict__ logits, float* __restrict__ losses,
                                                              const int* __restrict__ targets, int V, int Vp,
                                                              float dloss, int write_grad, int* flags) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  constexpr float L2E = 1.4426950408889634f;
  __shared__ float red[32];
  __shared__ float s_bcast[2];
  T* z = logits + (size_t)blockIdx.x * Vp;
  const int nvec = Vp / N;
  uint4 raw[VPT];
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * 1024;
    if (vi < nvec) raw[k] = __ldcs(reinterpret_cast<const uint4*>(z) + vi);
  }
  auto unpack = [&](int k, float (&f)[N]) {
    if constexpr (N == 8) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[k]);
#pragma unroll
      for (int i = 0; i < 4; i++) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x; f[2 * i + 1] = t.y;
      }
    } else {
      const float* q = reinterpret_cast<const float*>(&raw[k]);
#pragma unroll
      for (int i = 0; i < N; i++) f[i] = q[i];
    }
  };
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // row max over the first V columns (only a vector reaching past V needs the mask)
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * 1024;
    if (vi < nvec) {
      float f[N];
      unpack(k, f);
      if (vi * N + N <= V) {
#pragma unroll
        for (int i = 0; i < N; i++) m = fmaxf(m, f[i]);
      } else {
#pragma unroll
        for (int i = 0; i < N; i++)
          if (vi * N + i < V) m = fmaxf(m, f[i]);
      }
    }
  }
  m = warp_max(m);
  if (lane == 0) red[w] = m;
  __syncthreads();
  if (w == 0) {
    float t = red[lane];
    t = warp_max(t);
    if (lane == 0) s_bcast[0] = t;
  }
  __syncthreads();
  m = s_bcast[0];
  const float ml = m * L2E;
  // exp(z - max) of every element; in bf16 the values are kept, as fp16
  // (2^-11 relative, more than the bf16 output needs), in the registers that
  // held the logits, so the gradient pass needs no second exponential
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * 1024;
    if (vi < nvec) {
      float f[N];
      unpack(k, f);
      if (vi * N + N <= V) {
#pragma unroll
        for (int i = 0; i < N; i++) f[i] = fast_exp2(fmaf(f[i], L2E, -ml));
      } else {
#pragma unroll
        for (int i = 0; i < N; i++) f[i] = vi * N + i < V ? fast_exp2(fmaf(f[i], L2E, -ml)) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < N; i++) s += f[i];
      if constexpr (N == 8) {
        __half2* hp = reinterpret_cast<__half2*>(&raw[k]);
#pragma unroll
        for (int i = 0; i < 4; i++) hp[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      } else {
        float* q = reinterpret_cast<float*>(&raw[k]);
#pragma unroll
        for (int i = 0; i < N; i++) q[i] = f[i];
      }
    }
  }
  s = block_sum(s, red);
  if (threadIdx.x == 0) {
    int tg = targets[blockIdx.x];
    if (tg < 0 || tg >= V) {
      atomicOr(flags, FLAG_TARGET_RANGE);
      tg = 0;
    }
    const float zt = to_f(z[tg]);
    const float lse = m + logf(s);
    losses[blockIdx.x] = lse - zt;
    s_bcast[1] = (float)tg;
    // the target's probability in fp32: p - 1 loses everything when p is near 1
    s_bcast[0] = (fast_exp2(fmaf(zt, L2E, -ml)) / s - 1.f) * dloss;
  }
  if (!write_grad) return;
  __syncthreads();
  const int tg = (int)s_bcast[1];
  const float g_tg = s_bcast[0];
  const float scale = dloss / s;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * 1024;
    if (vi < nvec) {
      float f[N];
      if constexpr (N == 8) {
        const __half2* hp = reinterpret_cast<const __half2*>(&raw[k]);
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const float2 t = __half22float2(hp[i]);
          f[2 * i] = t.x;
          f[2 * i + 1] = t.y;
        }
      } else {
        const float* q = reinterpret_cast<const float*>(&raw[k]);
#pragma unroll
        for (int i = 0; i < N; i++) f[i] = q[i];
      }
#pragma unroll
      for (int i = 0; i < N; i++) f[i] *= scale;  // pads hold exp = 0
      if (tg >= vi * N && tg < vi * N + N) f[tg - vi * N] = g_tg;
      st16_cs(z + (size_t)vi * N, f);
    }
  }
}

// bf16 rows that fit in shared memory (Vp * 2 <= 110 KB): one CTA of 512
// threads per row, two CTAs per SM.  The row is copied into shared memory with
// cp.async (16 bytes a request, all in flight at once) and the three passes
// (maximum, exp and sum, dlogits) read it there, so one CTA's copy overlaps the
// other's passes.  exp(z - max) is kept in place as fp16, as in the register
// kernel; same arithmetic, the reductions over 512 threads.
constexpr int SCE_SMEM_THREADS = 512;
__global__ void __launch_bounds__(SCE_SMEM_THREADS, 2)
    softmax_ce_smem_kernel(bf16* __restrict__ logits, float* __restrict__ losses, const int* __restrict__ targets,
                           int V, int Vp, float dloss, int write_grad, int* flags) {
  pdl_enter();
  constexpr int N = 8;
  constexpr float L2E = 1.4426950408889634f;
  constexpr int W = SCE_SMEM_THREADS / 32;
  extern __shared__ __align__(16) unsigned char sce_row[];
  __shared__ float red[2][W];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  // rows from the last: the classifier GEMM wrote the last rows last (they are
  // still in L2), and the input-gradient GEMM after this kernel starts from row 0
  const int rowi = gridDim.x - 1 - blockIdx.x;
  bf16* z = logits + (size_t)rowi * Vp;
  const int nvec = Vp / N;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sce_row);
  for (int vi = tid; vi < nvec; vi += SCE_SMEM_THREADS)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sbase + vi * 16), "l"(z + (size_t)vi * N)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  int tg = targets[rowi];
  const bool bad = tg < 0 || tg >= V;
  if (bad) tg = 0;
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  uint4* row = reinterpret_cast<uint4*>(sce_row);
  // row max over the first V columns
  float m = -INFINITY;
  for (int vi = tid; vi < nvec; vi += SCE_SMEM_THREADS) {
    float f[N];
    ld16(reinterpret_cast<const bf16*>(row + vi), f);
    if (vi * N + N <= V) {
#pragma unroll
      for (int j = 0; j < N; j++) m = fmaxf(m, f[j]);
    } else {
#pragma unroll
      for (int j = 0; j < N; j++)
        if (vi * N + j < V) m = fmaxf(m, f[j]);
    }
  }
  const float zt = to_f(reinterpret_cast<const bf16*>(sce_row)[tg]);
  m = warp_max(m);
  if (lane == 0) red[0][w] = m;
  __syncthreads();
  m = red[0][0];
#pragma unroll
  for (int j = 1; j < W; j++) m = fmaxf(m, red[0][j]);
  const float ml = m * L2E;
  // exp(z - max) in place as fp16, and its sum
  float s = 0.f;
  for (int vi = tid; vi < nvec; vi += SCE_SMEM_THREADS) {
    float f[N];
    ld16(reinterpret_cast<const bf16*>(row + vi), f);
    if (vi * N + N <= V) {
#pragma unroll
      for (int j = 0; j < N; j++) f[j] = fast_exp2(fmaf(f[j], L2E, -ml));
    } else {
#pragma unroll
      for (int j = 0; j < N; j++) f[j] = vi * N + j < V ? fast_exp2(fmaf(f[j], L2E, -ml)) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < N; j++) s += f[j];
    uint4 h;
    __half2* hp = reinterpret_cast<__half2*>(&h);
#pragma unroll
    for (int j = 0; j < 4; j++) hp[j] = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
    row[vi] = h;
  }
  s = warp_sum(s);
  if (lane == 0) red[1][w] = s;
  __syncthreads();
  s = red[1][0];
#pragma unroll
  for (int j = 1; j < W; j++) s += red[1][j];
  if (tid == 0) {
    if (bad) atomicOr(flags, FLAG_TARGET_RANGE);
    losses[rowi] = m + logf(s) - zt;
  }
  if (!write_grad) return;
  // the target's probability in fp32: p - 1 loses everything when p is near 1
  const float g_tg = (fast_exp2(fmaf(zt, L2E, -ml)) / s - 1.f) * dloss;
  const float scale = dloss / s;
  for (int vi = tid; vi < nvec; vi += SCE_SMEM_THREADS) {
    const uint4 h = row[vi];
    const __half2* hp = reinterpret_cast<const __half2*>(&h);
    float f[N];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float2 t = __half22float2(hp[j]);
      f[2 * j] = t.x * scale;
      f[2 * j + 1] = t.y * scale;
    }
    if (tg >= vi * N && tg < vi * N + N) f[tg - vi * N] = g_tg;
    st16_cs(z + (size_t)vi * N, f);
  }
}

// Softmax + cross-entropy from the classifier product's per-tile row
// statistics (m_n, s_n) = (max, sum of exp(z - max)) over each 256-column
// tile: M = max_n m_n, S = sum_n s_n exp(m_n - M) give the row's
// log-sum-exp M + ln S, so the row itself is read once and written once
// (dlogits in place), a plain stream at 256 threads per row.  Same outputs as
// softmax_ce: loss = lse - z[target], dlogits = (softmax - onehot) * dloss
// over the first V columns, 0 on the pads; the target's probability in fp32.
constexpr int SCS_THREADS = 256;
__global__ void __launch_bounds__(SCS_THREADS) softmax_ce_stats_kernel(
    bf16* __restrict__ logits, float* __restrict__ losses, const int* __restrict__ targets,
    const float* __restrict__ rowstats, int tiles, int V, int Vp, float dloss, int* flags) {
  pdl_enter();
  constexpr int N = 8;
  constexpr float L2E = 1.4426950408889634f;
  __shared__ float sh[3];
  const int tid = threadIdx.x, lane = tid & 31;
  // rows from the last: the classifier product wrote the last rows last (they
  // are still in L2), and the input-gradient product after this kernel starts
  // from row 0, which is then the most recently written
  const int row = gridDim.x - 1 - blockIdx.x;
  bf16* z = logits + (size_t)row * Vp;
  int tg = targets[row];
  const bool bad = tg < 0 || tg >= V;
  if (bad) tg = 0;
  if (tid < 32) {
    // the tiles' statistics, combined in a fixed order (lane-strided, then a shuffle tree)
    const float2* st = reinterpret_cast<const float2*>(rowstats) + (size_t)row * tiles;
    float m = -INFINITY, sm = 0.f;
    for (int i = lane; i < tiles; i += 32) {
      const float2 t = st[i];
      const float mn = fmaxf(m, t.x);
      if (mn > -INFINITY) {
        sm = sm * tc::ex2((m - mn) * L2E) + t.y * tc::ex2((t.x - mn) * L2E);
        m = mn;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off), s2 = __shfl_xor_sync(0xffffffffu, sm, off);
      const float mn = fmaxf(m, m2);
      if (mn > -INFINITY) {
        sm = sm * tc::ex2((m - mn) * L2E) + s2 * tc::ex2((m2 - mn) * L2E);
        m = mn;
      }
    }
    if (lane == 0) {
      sh[0] = m;
      sh[1] = sm;
      sh[2] = __bfloat162float(z[tg]);  // read before any thread overwrites the row
    }
  }
  __syncthreads();
  const float m = sh[0], sm = sh[1], zt = sh[2];
  if (tid == 0) {
    if (bad) atomicOr(flags, FLAG_TARGET_RANGE);
    losses[row] = m + logf(sm) - zt;
  }
  const float ml = m * L2E, scale = dloss / sm;
  // the target's probability in fp32: p - 1 loses everything when p is near 1
  const float g_tg = (tc::ex2(fmaf(zt, L2E, -ml)) / sm - 1.f) * dloss;
  const int nvec = Vp / N;
  for (int v0 = tid; v0 < nvec; v0 += 4 * SCS_THREADS) {
    uint4 r[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int vi = v0 + u * SCS_THREADS;
      if (vi < nvec) r[u] = __ldcs(reinterpret_cast<const uint4*>(z) + vi);
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int vi = v0 + u * SCS_THREADS;
      if (vi >= nvec) break;
      float f[N];
      unpack_bf16x8(r[u], f);
#pragma unroll
      for (int j = 0; j < N; j++) f[j] = vi * N + j < V ? tc::ex2(fmaf(f[j], L2E, -ml)) * scale : 0.f;
      if (tg >= vi * N && tg < vi * N + N) f[tg - vi * N] = g_tg;
      st16_cs(z + (size_t)vi * N, f);
    }
  }
}

cudaError_t softmax_ce_from_stats(bf16* logits, float* losses, const int* targets, const float* rowstats, int tiles,
                                  int rows, int V, int Vp, float dloss, int* flags, cudaStream_t st) {
  if (rows <= 0 || tiles <= 0 || V <= 0 || Vp < V || Vp % 8 || ((uintptr_t)logits & 15) || ((uintptr_t)rowstats & 7))
    return cudaErrorInvalidValue;
  launch_k(softmax_ce_stats_kernel, dim3(rows), dim3(SCS_THREADS), 0, st, logits, losses, targets, rowstats, tiles, V,
           Vp, dloss, flags);
  return launch_status(1);
}

template <typename T>
cudaError_t softmax_ce(T* logits, float* losses, const int* targets, int rows, int V, int Vp,
                       float dloss, int write_grad, int* flags, cudaStream_t st) {
  constexpr int N = VecN<T>::n;
  if (Vp % N) return cudaErrorInvalidValue;
  if constexpr (sizeof(T) == 2) {
    const size_t smem = (size_t)Vp * 2;
    if (smem <= 110 * 1024 && Vp >= 16384 && ((uintptr_t)logits & 15) == 0 && rows > 0) {
      {
        cudaError_t e = kernel_smem_attr(softmax_ce_smem_kernel, 110 * 1024);
        if (e != cudaSuccess) return e;
      }
      launch_k(softmax_ce_smem_kernel, dim3(rows), dim3(SCE_SMEM_THREADS), smem, st, (bf16*)logits, losses, targets,
               V, Vp, dloss, write_grad, flags);
      return launch_status(1);
    }
  }
  const int vpt = (int)cdiv(Vp / N, 1024);
#define SCE(K) launch_k(softmax_ce_reg_kernel<T, K>, dim3(rows), dim3(1024), 0, st, logits, losses, targets, V, Vp, dloss, write_grad, flags)
  switch (vpt) {
    case 1: SCE(1); break;
    case 2: SCE(2); break;
    case 3: SCE(3); break;
    case 4: SCE(4); break;
    case 5: SCE(5); break;
    case 6: SCE(6); break;
    case 7: SCE(7); break;
    case 8: SCE(8); break;
    default:
      launch_k(softmax_ce_kernel<T>, dim3(rows), dim3(1024), 0, st, logits, losses, targets, V, Vp, dloss, write_grad, flags);
  }
#undef SCE
  return launch_status(1);
}

// ============================================================================
// inference with a KV cache: attention of one new position per sequence and
// the sampler.  The cache is the qkv activation buffer [B*Tmax][3C]: row
// b*Tmax + t holds q | k | v of position t of sequence b.
// ============================================================================
// One CTA per (b, h): scores q.k_t * scale for t = 0..pos (keys from the
// cache), softmax, then the probability-weighted sum of v_t.  Threads take
// keys t = tid, tid+256, ...; for P.V, group g = tid / hd of the 256 / hd
// groups sums keys t = g, g+G, ... for dimension tid % hd, and the groups are
// added in group order.  fp32 throughout.
template <typename T>
__global__ void __launch_bounds__(256) decode_attention_kernel(T* __restrict__ out, const T* __restrict__ qkv,
                                                               int Tmax, int pos, int C, int H, float scale) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  extern __shared__ float da_sh[];  // q[128] | red[32] | s[Tmax] | part[256]
  float* q = da_sh;
  float* red = q + 128;
  float* s = red + 32;
  float* part = s + Tmax;
  const int b = blockIdx.x / H, h = blockIdx.x % H, hd = C / H, tid = threadIdx.x;
  const size_t row0 = (size_t)b * Tmax;
  for (int d = tid; d < hd; d += blockDim.x) q[d] = to_f(qkv[(row0 + pos) * 3 * C + h * hd + d]);
  __syncthreads();
  float mx = -INFINITY;
  for (int t = tid; t <= pos; t += blockDim.x) {
    const T* kp = qkv + (row0 + t) * 3 * C + C + h * hd;
    float a = 0.f;
    for (int d = 0; d < hd; d += N) {
      float k[N];
      ld16(kp + d, k);
#pragma unroll
      for (int e = 0; e < N; e++) a = fmaf(q[d + e], k[e], a);
    }
    a *= scale;
    s[t] = a;
    mx = fmaxf(mx, a);
  }
  mx = warp_max(mx);
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); w++) mx = fmaxf(mx, red[w]);
  __syncthreads();
  float sum = 0.f;
  for (int t = tid; t <= pos; t += blockDim.x) {
    const float e = expf(s[t] - mx);
    s[t] = e;
    sum += e;
  }
  sum = warp_sum(sum);
  if ((tid & 31) == 0) red[tid >> 5] = sum;
  __syncthreads();  // (also: every s[t] written)
  float l = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); w++) l += red[w];
  const int G = blockDim.x / hd, g = tid / hd, d = tid % hd;
  float acc = 0.f;
  if (g < G) {
    const T* vcol = qkv + row0 * 3 * C + 2 * C + h * hd + d;  // v_t[d] at vcol + t*3C
    int t = g;
    for (; t + 7 * G <= pos; t += 8 * G) {  // eight loads in flight, added in key order
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; u++) v[u] = to_f(vcol[(size_t)(t + u * G) * 3 * C]);
#pragma unroll
      for (int u = 0; u < 8; u++) acc = fmaf(s[t + u * G], v[u], acc);
    }
    for (; t <= pos; t += G) acc = fmaf(s[t], to_f(vcol[(size_t)t * 3 * C]), acc);
  }
  part[tid] = acc;
  __syncthreads();
  if (tid < hd) {
    float o = 0.f;
    for (int gg = 0; gg < G; gg++) o += part[gg * hd + tid];
    out[(size_t)b * C + h * hd + tid] = from_f<T>(o / l);
  }
}

template <typename T>
cudaError_t decode_attention(T* out, const T* qkv, int B, int Tmax, int pos, int C, int H, cudaStream_t st) {
  constexpr int N = VecN<T>::n;
  const int hd = C / H;
  if (B <= 0 || H <= 0 || C % H || hd > 128 || hd % N || pos < 0 || pos >= Tmax) return cudaErrorInvalidValue;
  const size_t smem = (size_t)(128 + 32 + Tmax + 256) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = kernel_smem_attr(decode_attention_kernel<T>, (int)smem);
    if (e != cudaSuccess) return e;
  }
  launch_k(decode_attention_kernel<T>, dim3((unsigned)(B * H)), dim3(256), smem, st, out, qkv, Tmax, pos, C, H,
           1.0f / sqrtf((float)hd));
  return launch_status(1);
}

// One CTA per row b: temperature 0 -> the index of the largest of the first V
// logits (lowest index on ties); else the sampler's inverse CDF of
// softmax(z / temperature) at coins[b]: thread t sums exp((z_i - max)/temp)
// over its contiguous chunk of indices in order, the chunk sums are scanned
// in thread order, and the thread whose chunk holds coin * total walks it to
// the first index whose running sum exceeds that (V - 1 if none does).
template <typename T>
__global__ void __launch_bounds__(1024) sample_kernel(int* __restrict__ out_tok, const T* __restrict__ logits,
                                                      long long ld, int V, float temperature,
                                                      const float* __restrict__ coins) {
  pdl_enter();
  __shared__ float sv[32];
  __shared__ int si[32];
  __shared__ float scan[1024];
  __shared__ int found;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const T* z = logits + (size_t)b * ld;
  // maximum (value, lowest index)
  float best = -INFINITY;
  int bi = V;
  for (int i0 = tid; i0 < V; i0 += 8 * blockDim.x) {  // eight loads in flight, compared in index order
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int i = i0 + u * blockDim.x;
      v[u] = i < V ? to_f(z[i]) : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < 8; u++)
      if (v[u] > best) best = v[u], bi = i0 + u * blockDim.x;  // increasing index: the first maximum
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) best = ov, bi = oi;
  }
  if (lane == 0) sv[w] = best, si[w] = bi;
  __syncthreads();
  best = sv[0];
  bi = si[0];
  for (int q = 1; q < (int)(blockDim.x >> 5); q++)
    if (sv[q] > best || (sv[q] == best && si[q] < bi)) best = sv[q], bi = si[q];
  if (temperature == 0.f) {
    if (tid == 0) out_tok[b] = bi;
    return;
  }
  const float inv_t = 1.0f / temperature;
  const int chunk = (V + blockDim.x - 1) / blockDim.x;
  const int c0 = tid * chunk, c1 = min(V, c0 + chunk);
  float cs = 0.f;
  for (int i = c0; i < c1; i++) cs += expf((to_f(z[i]) - best) * inv_t);
  scan[tid] = cs;
  __syncthreads();
  // inclusive scan of the chunk sums in thread order (Hillis-Steele on shared memory)
  for (int o = 1; o < (int)blockDim.x; o <<= 1) {
    const float y = tid >= o ? scan[tid - o] : 0.f;
    __syncthreads();
    scan[tid] += y;
    __syncthreads();
  }
  const float total = scan[blockDim.x - 1];
  const float target = coins[b] * total;
  const float before = tid > 0 ? scan[tid - 1] : 0.f;
  // the chunk whose [start, end) holds the target; should rounding let two
  // chunks claim it, the lower one wins
  if (tid == 0) found = (int)blockDim.x;
  __syncthreads();
  if (c0 < c1 && target >= before && target < scan[tid]) atomicMin(&found, tid);
  __syncthreads();
  if (tid == found) {
    float run = before;
    int pick = c1 - 1;
    for (int i = c0; i < c1; i++) {
      run += expf((to_f(z[i]) - best) * inv_t);
      if (target < run) {
        pick = i;
        break;
      }
    }
    out_tok[b] = pick;
  }
  if (tid == 0 && found == (int)blockDim.x) out_tok[b] = V - 1;
}

template <typename T>
cudaError_t sample_tokens(int* out_tok, const T* logits, long long ld, int rows, int V, float temperature,
                          const float* coins, cudaStream_t st) {
  if (rows <= 0 || V <= 0 || temperature < 0.f || (temperature > 0.f && !coins)) return cudaErrorInvalidValue;
  launch_k(sample_kernel<T>, dim3((unsigned)rows), dim3(1024), 0, st, out_tok, logits, ld, V, temperature, coins);
  return launch_status(1);
}

// mean of n per-position losses, one CTA, fixed summation order
__global__ void mean_loss_kernel(float* loss, const float* __restrict__ losses, int n) {
  pdl_enter();
  __shared__ float sh[32];
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += losses[i];
  s = block_sum(s, sh);
  if (threadIdx.x == 0) *loss = s / (float)n;
}
cudaError_t mean_loss(float* loss, const float* losses, int n, cudaStream_t st) {
  launch_k(mean_loss_kernel, dim3(1), dim3(1024), 0, st, loss, losses, n);
  return launch_status(1);
}

// ============================================================================
// AdamW over the whole buffer, 4 params per thread, per-tensor weight decay
// from a segment table; also writes the bf16 compute copy when pc != nullptr.
// ============================================================================
__global__ void adamw_kernel(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
                             float* __restrict__ v, bf16* __restrict__ pc, long long nvec, float lr, float b1,
                             float b2, float eps, float bc1, float bc2, AdamSegments seg,
                             const float* __restrict__ gscale) {
  pdl_enter();
  // gscale (optional): the clip factor the gradient-norm kernels left on the device
  const float gs = gscale ? *gscale : 1.f;
  long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    long long e = i * 4;
    int s = 0;
    while (s + 1 < seg.n && e >= seg.off[s + 1]) s++;
    float wd = seg.wd[s];
    float pv[4], gv[4], mv[4], vv[4];
    ld16_cs(p + e, pv);
    ld16_cs(g + e, gv);
    ld16_cs(m + e, mv);
    ld16_cs(v + e, vv);
#pragma unroll
    for (int k = 0; k < 4; k++) {
      gv[k] *= gs;
      mv[k] = b1 * mv[k] + (1.f - b1) * gv[k];
      vv[k] = b2 * vv[k] + (1.f - b2) * gv[k] * gv[k];
      float mh = mv[k] / bc1, vh = vv[k] / bc2;
      pv[k] -= lr * (mh / (sqrtf(vh) + eps) + wd * pv[k]);
    }
    st16_cs(p + e, pv);
    st16_cs(m + e, mv);
    st16_cs(v + e, vv);
    if (pc) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(pv[0], pv[1]), hi = __floats2bfloat162_rn(pv[2], pv[3]);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(pc + e) = u;
    }
  }
}

cudaError_t adamw(float* p, const float* g, float* m, float* v, bf16* pc, long long n, float lr,
                  float b1, float b2, float eps, float bc1, float bc2, const AdamSegments& seg,
                  const float* gscale, cudaStream_t st) {
  if (n % 4) return cudaErrorInvalidValue;
  long long nvec = n / 4;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = cdiv(nvec, 256);
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  launch_k(adamw_kernel, dim3((unsigned)blocks), dim3(256), 0, st, p, g, m, v, pc, nvec, lr, b1, b2, eps, bc1, bc2, seg, gscale);
  return launch_status(1);
}

// ============================================================================
// global gradient norm (the pages' global_norm component) and the clip factor
// min(1, max_norm / (norm + 1e-6)): GN_CHUNKS fixed chunks of the vector (the
// partition does not depend on the GPU), each summed by one block in a fixed
// order, then one block adds the chunk sums in order, in double.
// ============================================================================
constexpr int GN_CHUNKS = 1024;
size_t grad_norm_scratch_floats() { return GN_CHUNKS; }

__global__ void __launch_bounds__(256) grad_sq_partial_kernel(const float* __restrict__ g, long long n,
                                                              long long chunk, float* __restrict__ partial) {
  pdl_enter();
  __shared__ float red[32];
  const long long b0 = (long long)blockIdx.x * chunk, b1 = min(n, b0 + chunk);
  float s = 0.f;
  for (long long i = b0 + 4LL * threadIdx.x; i < b1; i += 4LL * blockDim.x) {
    if (i + 4 <= b1) {
      float x[4];
      ld16_cs(g + i, x);
      s = fmaf(x[0], x[0], s);
      s = fmaf(x[1], x[1], s);
      s = fmaf(x[2], x[2], s);
      s = fmaf(x[3], x[3], s);
    } else {
      for (long long j = i; j < b1; j++) s = fmaf(g[j], g[j], s);
    }
  }
  s = block_sum(s, red);
  if (threadIdx.x == 0) partial[blockIdx.x] = s;
}

__global__ void __launch_bounds__(256) grad_norm_finalize_kernel(const float* __restrict__ partial, float max_norm,
                                                                 float* __restrict__ out) {
  pdl_enter();
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < GN_CHUNKS; i += 256) s += (double)partial[i];  // 4 per thread, in order
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {  // fixed tree
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double norm = sqrt(red[0]);
    out[0] = (float)norm;
    const double coef = (double)max_norm / (norm + 1e-6);
    out[1] = coef < 1.0 ? (float)coef : 1.f;
  }
}

cudaError_t grad_norm(const float* g, long long n, float max_norm, float* out2, float* partial, cudaStream_t st) {
  if (n < 0 || (n > 0 && ((uintptr_t)g & 15))) return cudaErrorInvalidValue;
  const long long chunk = ((cdiv(n, GN_CHUNKS) + 3) / 4) * 4;  // chunks start 16-byte aligned
  launch_k(grad_sq_partial_kernel, dim3(GN_CHUNKS), dim3(256), 0, st, g, n, chunk > 0 ? chunk : 4, partial);
  launch_k(grad_norm_finalize_kernel, dim3(1), dim3(256), 0, st, partial, max_norm, out2);
  return launch_status(2);
}

__global__ void convert_f32_bf16_kernel(bf16* __restrict__ out, const float* __restrict__ in, long long n) {
  pdl_enter();
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = __float2bfloat16_rn(in[i]);
}
cudaError_t convert_f32_bf16(bf16* out, const float* in, long long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  launch_k(convert_f32_bf16_kernel, dim3((unsigned)cdiv(n, 256)), dim3(256), 0, st, out, in, n);
  return launch_status(1);
}

// ============================================================================
// standalone GELU forward/backward (128-bit streaming)
// ============================================================================
// GELU over a flat array: a block covers 256 * GELU_U consecutive 16-byte
// words, each thread GELU_U of them 256 words apart, and every thread issues
// all its loads before any arithmetic, so that enough bytes are in flight per
// SM to stream at the copy rate.
constexpr int GELU_U = 4;
template <typename T>
__global__ void __launch_bounds__(256) gelu_forward_kernel(T* __restrict__ out, const T* __restrict__ in,
                                                           long long nvec) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  const long long base = (long long)blockIdx.x * 256 * GELU_U + threadIdx.x;
  float f[GELU_U][N];
#pragma unroll
  for (int u = 0; u < GELU_U; u++)
    if (base + u * 256 < nvec) ld16_cs(in + (base + u * 256) * N, f[u]);
#pragma unroll
  for (int u = 0; u < GELU_U; u++) {
    if (base + u * 256 >= nvec) break;
#pragma unroll
    for (int k = 0; k < N; k++) f[u][k] = gelu_fwd(f[u][k]);
    st16_cs(out + (base + u * 256) * N, f[u]);
  }
}
template <typename T>
__global__ void __launch_bounds__(256) gelu_backward_kernel(T* __restrict__ dinp, const T* __restrict__ inp,
                                                            const T* __restrict__ dout, long long nvec) {
  pdl_enter();
  constexpr int N = VecN<T>::n;
  const long long base = (long long)blockIdx.x * 256 * GELU_U + threadIdx.x;
  float x[GELU_U][N], d[GELU_U][N];
#pragma unroll
  for (int u = 0; u < GELU_U; u++)
    if (base + u * 256 < nvec) {
      ld16_cs(inp + (base + u * 256) * N, x[u]);
      ld16_cs(dout + (base + u * 256) * N, d[u]);
    }
#pragma unroll
  for (int u = 0; u < GELU_U; u++) {
    if (base + u * 256 >= nvec) break;
#pragma unroll
    for (int k = 0; k < N; k++) d[u][k] *= gelu_bwd(x[u][k]);
    st16_cs(dinp + (base + u * 256) * N, d[u]);
  }
}
template <typename T>
cudaError_t gelu_forward(T* out, const T* in, long long n, cudaStream_t st) {
  constexpr int N = VecN<T>::n;
  if (n % N) return cudaErrorInvalidValue;
  launch_k(gelu_forward_kernel<T>, dim3((unsigned)cdiv(n / N, 256 * GELU_U)), dim3(256), 0, st, out, in, n / N);
  return launch_status(1);
}
template <typename T>
cudaError_t gelu_backward(T* dinp, const T* inp, const T* dout, long long n, cudaStream_t st) {
  constexpr int N = VecN<T>::n;
  if (n % N) return cudaErrorInvalidValue;
  launch_k(gelu_backward_kernel<T>, dim3((unsigned)cdiv(n / N, 256 * GELU_U)), dim3(256), 0, st, dinp, inp, dout,
           n / N);
  return launch_status(1);
}

// ============================================================================
// LayerNorm folded into the next product: one warp per weight row n of one
// stacked item; Wf[n][k] = bf16(W[n][k] gamma[k]), s[n] = sum of Wf[n][k] (as
// stored), c[n] = bias[n] + sum_k beta[k] W[n][k], lanes over k in 8-wide
// groups, the sums added by a fixed shuffle tree (deterministic).
// ============================================================================
__global__ void __launch_bounds__(256) lnfold_weights_kernel(bf16* __restrict__ Wf, float* __restrict__ s,
                                                             float* __restrict__ c, const float* __restrict__ W,
                                                             const float* __restrict__ gamma,
                                                             const float* __restrict__ beta,
                                                             const float* __restrict__ bias, int items, int N, int K,
                                                             long long out_rows) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= (long long)items * N) return;
  const int z = (int)(row / N), n = (int)(row % N);
  const long long orow = (long long)z * out_rows + n;  // the row in Wf, s, c
  const float* w = W + (size_t)row * K;
  const float* g = gamma + (size_t)z * K;
  const float* be = beta + (size_t)z * K;
  float ss = 0.f, cc = 0.f;
  for (int k = 8 * lane; k < K; k += 256) {
    float wv[8], gv[8], bv[8];
    ld16(w + k, *reinterpret_cast<float(*)[4]>(wv));
    ld16(w + k + 4, *reinterpret_cast<float(*)[4]>(wv + 4));
    ld16(g + k, *reinterpret_cast<float(*)[4]>(gv));
    ld16(g + k + 4, *reinterpret_cast<float(*)[4]>(gv + 4));
    ld16(be + k, *reinterpret_cast<float(*)[4]>(bv));
    ld16(be + k + 4, *reinterpret_cast<float(*)[4]>(bv + 4));
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; e++) {
      o[e] = round_to<bf16>(wv[e] * gv[e]);
      ss += o[e];
      cc = fmaf(bv[e], wv[e], cc);
    }
    st16(Wf + (size_t)orow * K + k, o);
  }
  ss = warp_sum(ss);
  cc = warp_sum(cc);
  if (lane == 0) {
    s[orow] = ss;
    c[orow] = (bias ? bias[(size_t)z * N + n] : 0.f) + cc;
  }
}

cudaError_t lnfold_weights(bf16* Wf, float* s, float* c, const float* W, const float* gamma, const float* beta,
                           const float* bias, int items, int N, int K, cudaStream_t st, long long out_rows) {
  if (items <= 0 || N <= 0 || K <= 0 || K % 8) return cudaErrorInvalidValue;
  if (out_rows <= 0) out_rows = N;
  launch_k(lnfold_weights_kernel, dim3((unsigned)cdiv((long long)items * N, 8)), dim3(256), 0, st, Wf, s, c, W, gamma,
           beta, bias, items, N, K, out_rows);
  return launch_status(1);
}

// ---- explicit instantiations ----------------------------------------------
#define INST(T)                                                                                           \
  template cudaError_t encoder_forward<T>(T*, const int*, const T*, const T*, int, int, int, int, int*,  \
                                          cudaStream_t);                                                  \
  template cudaError_t residual_layernorm_forward<T>(T*, T*, float*, float*, const T*, const T*, const T*, \
                                                     const T*, int, int, cudaStream_t);                  \
  template cudaError_t layernorm_backward<T>(float*, T*, const T*, const T*, const float*, const float*,  \
                                             const T*, int, int, int, float*, float*, float*, float*,     \
                                             cudaStream_t, int*);                                         \
  template cudaError_t layernorm_apply<T>(T*, const T*, const float*, const float*, const T*, const T*, int,   \
                                          int, cudaStream_t);                                                \
  template cudaError_t decode_attention<T>(T*, const T*, int, int, int, int, int, cudaStream_t);             \
  template cudaError_t sample_tokens<T>(int*, const T*, long long, int, int, float, const float*,            \
                                        cudaStream_t);                                                       \
  template cudaError_t colsum<T>(float*, const T*, int, int, long long, float*, cudaStream_t, int, long long,  \
                                 long long, int);                                                         \
  template cudaError_t gemm_simt<T>(const GemmArgs&, cudaStream_t);                                       \
  template bool gemm_skinny_supported<T>(const GemmArgs&);                                                 \
  template cudaError_t gemm_skinny<T>(const GemmArgs&, cudaStream_t);                                      \
  template cudaError_t attention_forward_simt<T>(T*, float*, const T*, int, int, int, int, cudaStream_t); \
  template cudaError_t attention_backward_simt<T>(T*, float*, const T*, const T*, const T*, const float*, \
                                                  int, int, int, int, cudaStream_t);                     \
  template cudaError_t softmax_ce<T>(T*, float*, const int*, int, int, int, float, int, int*,             \
                                     cudaStream_t);                                                       \
  template cudaError_t gelu_forward<T>(T*, const T*, long long, cudaStream_t);                            \
  template cudaError_t gelu_backward<T>(T*, const T*, const T*, long long, cudaStream_t);
INST(float)
INST(bf16)
template cudaError_t layernorm_backward_rg<float, float>(float*, const float*, float*, float*, const float*,
                                                         const float*, const float*, const float*, const float*, int,
                                                         int, float*, float*, float*, float*, cudaStream_t, int*);
template cudaError_t layernorm_backward_rg<bf16, bf16>(bf16*, const bf16*, bf16*, float*, const bf16*, const bf16*,
                                                       const float*, const float*, const bf16*, int, int, float*,
                                                       float*, float*, float*, cudaStream_t, int*);
