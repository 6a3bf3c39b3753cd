// One decoding step of every transformer block in one persistent launch
// (bf16): the work of one new position per sequence, reading keys and values
// of the earlier positions from the KV cache ("llm.c: GPT-2 training in plain
// C, with every gradient written by hand", §6 Reality check: the pages'
// sampler reruns the whole forward for every token; here the keys and values
// are cached and one position is computed).
//
// A step moves every weight once (about 14 MB per GPT-2 124M layer) and the
// cached keys and values of every sequence; launched as ~7 dependent kernels
// per layer it was bound by launch and ramp latency.  Here one cooperative
// grid of one CTA per SM walks all layers; the phases of a layer are
// separated by a grid barrier (a counter in global memory, every wait
// bounded):
//   A  LN1 of the B residual rows (every CTA, into shared memory), then this
//      CTA's columns of q | k | v = LN1 . Wqkv^T + b, written into the cache
//      at position pos
//   B  attention of position pos over keys 0..pos, one (sequence, head) per
//      CTA at a time
//   C  this CTA's columns of the attention projection, plus the residual
//   D  LN2 of the new residual rows, this CTA's columns of fc + GELU
//   E  this CTA's columns of the fc projection, plus the residual
// A CTA owns a fixed range of output columns in each product; each warp
// takes one column at a time: its lanes split the reduction dimension and
// hold one partial sum per sequence, added by a fixed shuffle tree.
#include "../../include/gpt2.h"
#include "kernels.cuh"
#include "tc_common.cuh"

extern void gpt2_count_launches(int n);

namespace {

constexpr int DEC_THREADS = 512;
constexpr int DEC_WARPS = DEC_THREADS / 32;
constexpr int DEC_MAXB = 32;  // sequences a step handles (B * C bf16 rows in shared memory)

struct DecodeParams {
  const bf16* ln1w; const bf16* ln1b; const bf16* qkvw; const bf16* qkvb;
  const bf16* apw; const bf16* apb; const bf16* ln2w; const bf16* ln2b;
  const bf16* fcw; const bf16* fcb; const bf16* fpw; const bf16* fpb;
  bf16* qkv;          // [L][B*Tmax][3C]: the KV cache (and this position's q)
  bf16* x0;           // [B][C] residual: in (embedded rows) and out; x1 the other half of a ping-pong
  bf16* x1;
  bf16* att;          // [B][C]
  bf16* h;            // [B][4C]
  unsigned* bar;      // grid barrier counter (zero at launch)
  int* flags;
  int L, B, C, H, Tmax, pos;
  float scale;        // 1/sqrt(hd)
};

// 8 bf16 values as floats through L2 only: data written by other CTAs of
// this launch must not come from a stale line of this SM's L1
__device__ __forceinline__ void ld16_cg(const bf16* p, float (&f)[8]) {
  const uint4 v = __ldcg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float2 t = __bfloat1622float2(h2[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ float ldcg_bf16(const bf16* p) {
  const unsigned short u = __ldcg(reinterpret_cast<const unsigned short*>(p));
  return __uint_as_float((unsigned)u << 16);
}
// shared memory at the start of the kernel's dynamic area: the staged operand
// rows of the products ([NB][4C] bf16) and, in the attention phase of a head
// of size 64, the values of every cached position ([Tmax][64] bf16)
__host__ __device__ inline size_t decode_region0(int NB, int C, int Tmax) {
  const size_t a = (size_t)NB * 4 * C * sizeof(bf16), b = (size_t)Tmax * 64 * sizeof(bf16);
  return a > b ? a : b;
}
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Grid-wide barrier number k (1-based) of this launch: every CTA adds one to
// the counter and waits until all gridDim.x CTAs of this phase have.  The
// wait gives up after about 2 s (FLAG_TIMEOUT; every CTA then stops).
__device__ __forceinline__ bool grid_barrier(unsigned* bar, unsigned k, int* flags, int* sh_abort) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const unsigned target = k * gridDim.x;
    const uint64_t t0 = tc::gtimer();
    while (ld_acquire(bar) < target) {
      if (tc::gtimer() - t0 > tc::WAIT_NS || *(volatile int*)flags & FLAG_TIMEOUT) {
        atomicOr(flags, FLAG_TIMEOUT);
        *sh_abort = 1;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
  return *(volatile int*)sh_abort == 0;
}

// LayerNorm of the B rows x [B][C] into shared memory (fp32 math, rounded to
// bf16 as the LayerNorm kernels store it): warp w takes rows w, w + 16, ...;
// a row is copied from global memory once (all its loads in flight) into its
// output slot, and the statistics and the normalisation work from there.
__device__ void ln_rows(bf16* out, const bf16* x, const bf16* w, const bf16* b, int B, int C) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int row = warp; row < B; row += DEC_WARPS) {
    const bf16* xr = x + (size_t)row * C;
    bf16* orow = out + (size_t)row * C;
    for (int c = 8 * lane; c < C; c += 256)
      *reinterpret_cast<uint4*>(orow + c) = __ldcg(reinterpret_cast<const uint4*>(xr + c));
    __syncwarp();
    float sum = 0.f;
    for (int c = 8 * lane; c < C; c += 256) {
      float v[8];
      ld16(orow + c, v);
#pragma unroll
      for (int k = 0; k < 8; k++) sum += v[k];
    }
    const float mu = warp_sum(sum) / (float)C;
    float var = 0.f;
    for (int c = 8 * lane; c < C; c += 256) {
      float v[8];
      ld16(orow + c, v);
#pragma unroll
      for (int k = 0; k < 8; k++) var += (v[k] - mu) * (v[k] - mu);
    }
    const float rs = 1.0f / sqrtf(warp_sum(var) / (float)C + 1e-5f);
    for (int c = 8 * lane; c < C; c += 256) {
      float v[8], wv[8], bv[8];
      ld16(orow + c, v);
      ld16(w + c, wv);
      ld16(b + c, bv);
#pragma unroll
      for (int k = 0; k < 8; k++) v[k] = (v[k] - mu) * rs * wv[k] + bv[k];
      st16(orow + c, v);
    }
  }
}

// y[b][n] = sum_k X[b][k] W[n][k] for the columns n of this CTA's range
// [n0, n1): X [B][K] in shared memory (bf16; rows B..NB-1 are not used), W
// [N][K] row-major bf16.  The work is cut into units of one column and one
// part of its k range: when the CTA has fewer columns than warps, each
// column's k range is split into S parts so that every warp streams weights
// (the weights come from HBM: enough bytes must be in flight).  In a unit,
// lane l takes k = 8 l + 256 j over the part's chunks j, issuing the loads
// of up to DOT_VEC of its 16-byte words before any arithmetic, and keeps one
// partial sum per sequence of a group of DOT_GROUP; each sequence's partials
// are added by a fixed shuffle tree into `red` (S * (n1 - n0) * B floats of
// shared memory); then the parts of each column are added in part order and
// each sum goes out through epi(b, n, value).  Called by every thread of the
// CTA (it synchronises the CTA).
constexpr int DOT_VEC = 3;
constexpr int DOT_GROUP = 8;  // sequences whose partial sums are live at once
template <int NB, typename Epi>
__device__ void dot_columns(const bf16* X, const bf16* W, int K, int n0, int n1, int B, float* red, Epi epi) {
  constexpr int G = NB < DOT_GROUP ? NB : DOT_GROUP;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ncol = n1 - n0, nch = (K + 255) / 256;
  int S = ncol > 0 ? DEC_WARPS / ncol : 1;
  S = S < 1 ? 1 : (S > nch ? nch : S);
  for (int u = warp; u < ncol * S; u += DEC_WARPS) {
    const int n = n0 + u / S, part = u % S;
    const int j0 = part * nch / S, j1 = (part + 1) * nch / S;
    const bf16* wr = W + (size_t)n * K;
    for (int b0 = 0; b0 < B; b0 += G) {  // (a second group re-reads the row from L1)
      float acc[G];
#pragma unroll
      for (int b = 0; b < G; b++) acc[b] = 0.f;
      for (int jb = j0; jb < j1; jb += DOT_VEC) {
        uint4 wq[DOT_VEC];
#pragma unroll
        for (int v = 0; v < DOT_VEC; v++) {
          const int k = 256 * (jb + v) + 8 * lane;
          if (jb + v < j1 && k < K) wq[v] = __ldg(reinterpret_cast<const uint4*>(wr + k));
        }
#pragma unroll
        for (int v = 0; v < DOT_VEC; v++) {
          const int k = 256 * (jb + v) + 8 * lane;
          if (jb + v < j1 && k < K) {
            float wv[8];
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&wq[v]);
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const float2 t = __bfloat1622float2(h2[i]);
              wv[2 * i] = t.x;
              wv[2 * i + 1] = t.y;
            }
#pragma unroll
            for (int b = 0; b < G; b++) {
              float xv[8];
              ld16(X + (size_t)(b0 + b) * K + k, xv);
#pragma unroll
              for (int e = 0; e < 8; e++) acc[b] = fmaf(wv[e], xv[e], acc[b]);
            }
          }
        }
      }
      // each sequence's partial sums across the lanes by a fixed tree
#pragma unroll
      for (int b = 0; b < G; b++) acc[b] = warp_sum(acc[b]);
#pragma unroll
      for (int b = 0; b < G; b++)
        if (lane == b && b0 + b < B) red[((size_t)part * ncol + (n - n0)) * B + b0 + b] = acc[b];
    }
  }
  __syncthreads();
  // the parts of each column, added in part order
  for (int e = threadIdx.x; e < ncol * B; e += DEC_THREADS) {
    float v = red[e];
    for (int q = 1; q < S; q++) v += red[(size_t)q * ncol * B + e];
    epi(e % B, n0 + e / B, v);
  }
}

template <int NB>
__global__ void __launch_bounds__(DEC_THREADS, 1) decode_layers_kernel(DecodeParams p) {
  extern __shared__ __align__(16) uint8_t dec_sh[];
  __shared__ int sh_abort;
  __shared__ float red[DEC_WARPS];
  bf16* xs = reinterpret_cast<bf16*>(dec_sh);  // [B][max(C, 4C)] staged operand rows
  float* sc = reinterpret_cast<float*>(dec_sh + decode_region0(NB, p.C, p.Tmax));  // attention scores [Tmax]
  if (threadIdx.x == 0) sh_abort = 0;
  __syncthreads();
  const int C = p.C, B = p.B, hd = C / p.H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cta = blockIdx.x, ncta = gridDim.x;
  auto range = [&](int N, int& a, int& b) {  // this CTA's columns of an N-wide product
    const int per = (N + ncta - 1) / ncta;
    a = min(N, cta * per);
    b = min(N, a + per);
  };
  float* red_dot = sc + p.Tmax;  // part sums of dot_columns (the attention's partial rows otherwise)
  unsigned nbar = 0;
  bf16 *x = p.x0, *xn = p.x1;
  for (int l = 0; l < p.L; l++) {
    const size_t C3 = 3 * (size_t)C;
    bf16* cache = p.qkv + (size_t)l * B * p.Tmax * C3;
    // ---- A: q | k | v of position pos
    ln_rows(xs, x, p.ln1w + (size_t)l * C, p.ln1b + (size_t)l * C, B, C);
    __syncthreads();
    {
      int n0, n1;
      range(3 * C, n0, n1);
      const bf16* bias = p.qkvb + (size_t)l * C3;
      dot_columns<NB>(xs, p.qkvw + (size_t)l * C3 * C, C, n0, n1, B, red_dot, [&](int b, int n, float v) {
        cache[((size_t)b * p.Tmax + p.pos) * C3 + n] = __float2bfloat16_rn(v + __bfloat162float(bias[n]));
      });
    }
    if (!grid_barrier(p.bar, ++nbar, p.flags, &sh_abort)) return;
    // ---- B: attention of position pos, one (sequence, head) per CTA at a time
    // Head size 64 (every GPT-2 size): the values of keys 0..pos are copied
    // into shared memory (cp.async) while the scores are formed, eight
    // threads per key (one 16-byte piece of the key each, the loads of four
    // keys in flight at once); P V then reads the values from shared memory.
    for (int bh = cta; hd == 64 && bh < B * p.H; bh += ncta) {
      const int b = bh / p.H, hh = bh % p.H, nk = p.pos + 1;
      const bf16* base = cache + (size_t)b * p.Tmax * C3 + hh * 64;
      bf16* vs = reinterpret_cast<bf16*>(dec_sh);  // [nk][64]
      float* part = sc + p.Tmax;                   // [8][64] partial output rows, then q [64]
      float* qf = part + DEC_THREADS * 8 - 64;
      for (int c = threadIdx.x; c < nk * 8; c += DEC_THREADS)
        cp_async16(vs + 8 * c, base + 2 * C + (size_t)(c >> 3) * C3 + 8 * (c & 7));
      if (threadIdx.x < 64) qf[threadIdx.x] = ldcg_bf16(base + (size_t)p.pos * C3 + threadIdx.x) * p.scale;
      __syncthreads();
      const int cc = threadIdx.x & 7, kg = threadIdx.x >> 3;  // piece of the key, first key
      float qv[8];
#pragma unroll
      for (int e = 0; e < 8; e++) qv[e] = qf[8 * cc + e];
      float mx = -INFINITY;
      constexpr int KB = 4;  // keys of a thread whose loads are in flight at once
      // the batch loop is the same for every lane (the shuffles below need the
      // whole warp): lane groups past the last key compute nothing
      for (int tb = 0; tb < nk; tb += KB * (DEC_THREADS / 8)) {
        const int t0 = tb + kg;
        uint4 kw[KB];
#pragma unroll
        for (int u = 0; u < KB; u++) {
          const int t = t0 + u * (DEC_THREADS / 8);
          if (t < nk) kw[u] = __ldcg(reinterpret_cast<const uint4*>(base + (size_t)t * C3 + C) + cc);
        }
#pragma unroll
        for (int u = 0; u < KB; u++) {
          const int t = t0 + u * (DEC_THREADS / 8);
          float a = 0.f;
          if (t < nk) {
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&kw[u]);
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const float2 f = __bfloat1622float2(h2[i]);
              a = fmaf(qv[2 * i], f.x, a);
              a = fmaf(qv[2 * i + 1], f.y, a);
            }
          }
          // the eight pieces of key t: lanes 8m .. 8m+7 of the warp
          a += __shfl_xor_sync(0xffffffffu, a, 1);
          a += __shfl_xor_sync(0xffffffffu, a, 2);
          a += __shfl_xor_sync(0xffffffffu, a, 4);
          if (t < nk) {
            if (cc == 0) sc[t] = a;
            mx = fmaxf(mx, a);
          }
        }
      }
      mx = warp_max(mx);
      if (lane == 0) red[warp] = mx;
      __syncthreads();
      mx = red[0];
#pragma unroll
      for (int w = 1; w < DEC_WARPS; w++) mx = fmaxf(mx, red[w]);
      __syncthreads();
      float sum = 0.f;
      for (int t = threadIdx.x; t < nk; t += DEC_THREADS) {
        const float e = expf(sc[t] - mx);
        sc[t] = e;
        sum += e;
      }
      sum = warp_sum(sum);
      if (lane == 0) red[warp] = sum;
      cp_async_wait_all();
      __syncthreads();
      float lsum = 0.f;
#pragma unroll
      for (int w = 0; w < DEC_WARPS; w++) lsum += red[w];
      // out[d] = sum_t p_t v_t[d]: thread (s, d) takes keys s, s + 8, ...; the
      // eight partial rows are then added in s order
      {
        const int d = threadIdx.x & 63, sl = threadIdx.x >> 6;
        float acc = 0.f;
        for (int t = sl; t < nk; t += DEC_THREADS / 64) acc = fmaf(sc[t], __bfloat162float(vs[t * 64 + d]), acc);
        part[sl * 64 + d] = acc;
      }
      __syncthreads();
      if (threadIdx.x < 64) {
        float o = 0.f;
#pragma unroll
        for (int sl = 0; sl < DEC_THREADS / 64; sl++) o += part[sl * 64 + threadIdx.x];
        p.att[(size_t)b * C + hh * 64 + threadIdx.x] = __float2bfloat16_rn(o / lsum);
      }
      __syncthreads();
    }
    for (int bh = cta; hd != 64 && bh < B * p.H; bh += ncta) {
      const int b = bh / p.H, hh = bh % p.H;
      const bf16* base = cache + (size_t)b * p.Tmax * C3 + hh * hd;
      float* q = reinterpret_cast<float*>(xs);  // hd floats
      for (int d = threadIdx.x; d < hd; d += DEC_THREADS) q[d] = ldcg_bf16(base + (size_t)p.pos * C3 + d);
      __syncthreads();
      float mx = -INFINITY;
      for (int t = threadIdx.x; t <= p.pos; t += DEC_THREADS) {
        const bf16* kp = base + (size_t)t * C3 + C;
        float a = 0.f;
        if (hd == 64) {  // the GPT-2 head size: the key's eight 16-byte loads all in flight at once
          uint4 kw[8];
#pragma unroll
          for (int u = 0; u < 8; u++) kw[u] = __ldcg(reinterpret_cast<const uint4*>(kp) + u);
#pragma unroll
          for (int u = 0; u < 8; u++) {
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&kw[u]);
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const float2 f = __bfloat1622float2(h2[i]);
              a = fmaf(q[8 * u + 2 * i], f.x, a);
              a = fmaf(q[8 * u + 2 * i + 1], f.y, a);
            }
          }
        } else {
          for (int d = 0; d < hd; d += 8) {
            float kv[8];
            ld16_cg(kp + d, kv);
#pragma unroll
            for (int e = 0; e < 8; e++) a = fmaf(q[d + e], kv[e], a);
          }
        }
        a *= p.scale;
        sc[t] = a;
        mx = fmaxf(mx, a);
      }
      mx = warp_max(mx);
      if (lane == 0) red[warp] = mx;
      __syncthreads();
      mx = red[0];
#pragma unroll
      for (int w = 1; w < DEC_WARPS; w++) mx = fmaxf(mx, red[w]);
      __syncthreads();
      float sum = 0.f;
      for (int t = threadIdx.x; t <= p.pos; t += DEC_THREADS) {
        const float e = expf(sc[t] - mx);
        sc[t] = e;
        sum += e;
      }
      sum = warp_sum(sum);
      if (lane == 0) red[warp] = sum;
      __syncthreads();
      float lsum = 0.f;
#pragma unroll
      for (int w = 0; w < DEC_WARPS; w++) lsum += red[w];
      // out[d] = sum_t p_t v_t[d]: thread (g, c) takes 8 dimensions 8c..8c+7
      // (one 16-byte load per key) of keys g, g + KG, ... (four loads in
      // flight); the KG partial rows are then added in g order
      const int DC = hd / 8, KG = DEC_THREADS / DC, g = threadIdx.x / DC, cc = threadIdx.x % DC;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      {
        const bf16* vb = base + 2 * C + 8 * cc;
        int t = g;
        for (; t + 3 * KG <= p.pos; t += 4 * KG) {
          float vv[4][8];
#pragma unroll
          for (int u = 0; u < 4; u++) ld16_cg(vb + (size_t)(t + u * KG) * C3, vv[u]);
#pragma unroll
          for (int u = 0; u < 4; u++)
#pragma unroll
            for (int e = 0; e < 8; e++) acc[e] = fmaf(sc[t + u * KG], vv[u][e], acc[e]);
        }
        for (; t <= p.pos; t += KG) {
          float vv[8];
          ld16_cg(vb + (size_t)t * C3, vv);
#pragma unroll
          for (int e = 0; e < 8; e++) acc[e] = fmaf(sc[t], vv[e], acc[e]);
        }
      }
      float* part = sc + p.Tmax;  // [KG][hd] = DEC_THREADS * 8 floats
#pragma unroll
      for (int e = 0; e < 8; e++) part[g * hd + 8 * cc + e] = acc[e];
      __syncthreads();
      if (threadIdx.x < hd) {
        float o = 0.f;
        for (int gg = 0; gg < KG; gg++) o += part[gg * hd + threadIdx.x];
        p.att[(size_t)b * C + hh * hd + threadIdx.x] = __float2bfloat16_rn(o / lsum);
      }
      __syncthreads();
    }
    if (!grid_barrier(p.bar, ++nbar, p.flags, &sh_abort)) return;
    // ---- C: attention projection + residual
    for (int i = threadIdx.x; i < B * C / 8; i += DEC_THREADS)
      reinterpret_cast<uint4*>(xs)[i] = __ldcg(reinterpret_cast<const uint4*>(p.att) + i);
    __syncthreads();
    {
      int n0, n1;
      range(C, n0, n1);
      const bf16* bias = p.apb + (size_t)l * C;
      dot_columns<NB>(xs, p.apw + (size_t)l * C * C, C, n0, n1, B, red_dot, [&](int b, int n, float v) {
        const float pr = __bfloat162float(__float2bfloat16_rn(v + __bfloat162float(bias[n])));
        xn[(size_t)b * C + n] = __float2bfloat16_rn(ldcg_bf16(x + (size_t)b * C + n) + pr);
      });
    }
    if (!grid_barrier(p.bar, ++nbar, p.flags, &sh_abort)) return;
    { bf16* tmp = x; x = xn; xn = tmp; }
    // ---- D: LN2, fc + GELU
    ln_rows(xs, x, p.ln2w + (size_t)l * C, p.ln2b + (size_t)l * C, B, C);
    __syncthreads();
    {
      int n0, n1;
      range(4 * C, n0, n1);
      const bf16* bias = p.fcb + (size_t)l * 4 * C;
      dot_columns<NB>(xs, p.fcw + (size_t)l * 4 * C * C, C, n0, n1, B, red_dot, [&](int b, int n, float v) {
        // the pre-activation is rounded to bf16 first, as the training forward stores it
        const float pre = __bfloat162float(__float2bfloat16_rn(v + __bfloat162float(bias[n])));
        p.h[(size_t)b * 4 * C + n] = __float2bfloat16_rn(gelu_fwd(pre));
      });
    }
    if (!grid_barrier(p.bar, ++nbar, p.flags, &sh_abort)) return;
    // ---- E: fc projection + residual
    for (int i = threadIdx.x; i < B * 4 * C / 8; i += DEC_THREADS)
      reinterpret_cast<uint4*>(xs)[i] = __ldcg(reinterpret_cast<const uint4*>(p.h) + i);
    __syncthreads();
    {
      int n0, n1;
      range(C, n0, n1);
      const bf16* bias = p.fpb + (size_t)l * C;
      dot_columns<NB>(xs, p.fpw + (size_t)l * 4 * C * C, 4 * C, n0, n1, B, red_dot, [&](int b, int n, float v) {
        const float pr = __bfloat162float(__float2bfloat16_rn(v + __bfloat162float(bias[n])));
        xn[(size_t)b * C + n] = __float2bfloat16_rn(ldcg_bf16(x + (size_t)b * C + n) + pr);
      });
    }
    if (!grid_barrier(p.bar, ++nbar, p.flags, &sh_abort)) return;
    { bf16* tmp = x; x = xn; xn = tmp; }
  }
}

template <int NB>
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st, int sms) {
  const size_t smem = decode_region0(NB, p.C, p.Tmax) + (size_t)p.Tmax * sizeof(float) +
                      (size_t)DEC_THREADS * 8 * sizeof(float);
  static_assert(NB <= DEC_MAXB, "one partial sum per sequence in each lane");
  cudaError_t e = kernel_smem_attr(decode_layers_kernel<NB>, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(DEC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: the grid barriers need it
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layers_kernel<NB>, p);
}

}  // namespace

// the template width (sequences per step, rounded up to a power of two)
static int decode_nb(int B) {
  int nb = 1;
  while (nb < B) nb <<= 1;
  return nb;
}
static size_t decode_layers_smem_bytes(int B, int C, int Tmax) {
  return decode_region0(decode_nb(B), C, Tmax) + (size_t)Tmax * sizeof(float) + (size_t)DEC_THREADS * 8 * sizeof(float);
}

bool decode_layers_supported(int B, int C, int H, int Tmax) {
  if (B < 1 || B > DEC_MAXB || C % 8 || H <= 0 || C % H || (C / H) % 8 || C / H > DEC_THREADS) return false;
  return decode_layers_smem_bytes(B, C, Tmax) <= 200 * 1024;
}

// x0: the B embedded rows of position pos on entry, the residual after the
// last block on return (two exchanges per block); x1, att, h: scratch.
// bar: 4 bytes of device memory, zeroed here.
cudaError_t decode_layers(const bf16* const* w, bf16* qkv, bf16* x0, bf16* x1, bf16* att, bf16* h, unsigned* bar,
                          int* flags, int L, int B, int C, int H, int Tmax, int pos, cudaStream_t st) {
  if (!decode_layers_supported(B, C, H, Tmax) || pos < 0 || pos >= Tmax) return cudaErrorInvalidValue;
  DecodeParams p{w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7], w[8], w[9], w[10], w[11],
                 qkv, x0, x1, att, h, bar, flags, L, B, C, H, Tmax, pos, 1.0f / sqrtf((float)(C / H))};
  cudaError_t e = cudaMemsetAsync(bar, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  gpt2_count_launches(1);
#define DEC_CASE(NBv) \
  if (B <= NBv) return launch_decode<NBv>(p, st, sms);
  DEC_CASE(1) DEC_CASE(2) DEC_CASE(4) DEC_CASE(8) DEC_CASE(16) DEC_CASE(32)
#undef DEC_CASE
  return cudaErrorInvalidValue;
}
