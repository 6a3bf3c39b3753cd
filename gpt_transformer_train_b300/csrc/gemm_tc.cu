// Tensor-core GEMM for sm_103a: TMA -> shared-memory ring -> tcgen05.mma into
// TMEM -> tcgen05.ld epilogue.  Used for every matmul of the bf16 training
// step: the six forward matmuls (qkv, attention projection, fc + GELU, fc
// projection, tied classifier) and their input- and weight-gradient matmuls.
//
// D(m, n) = sum_k A(m, k) B(n, k); A and B are bf16, either K-major
// (row-major [rows][K]) or MN-major ([K][rows]), which covers y = x W^T
// (both K-major), dx = dy W (B MN-major) and dW = dy^T x (both MN-major)
// without any transpose pass.  Accumulation is fp32 in TMEM.
//
// Structure (one CTA per SM, persistent over output tiles, 192 threads):
//   warp 0      TMA producer: per k-block one 128x64 A box (or two 64x64
//               boxes when MN-major) and the matching B boxes, 128-byte
//               swizzle, into a STAGES-deep ring guarded by mbarriers.
//   warp 1      allocates 2*BN TMEM columns (two accumulators) and one
//               thread issues tcgen05.mma (M=128, N=BN, K=16) per 16-wide
//               k step; tcgen05.commit frees ring stages and, at the end
//               of a tile, signals the epilogue.
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time from the TMEM
//               lane quarter each warp may access, bias / GELU / GELU' /
//               fp32 accumulate, 128-bit stores.  The two accumulators let
//               the epilogue of tile i overlap the MMAs of tile i+1.
// Every mbarrier wait is bounded (about 2 s of %globaltimer); on expiry the
// CTA raises FLAG_TIMEOUT, stops issuing work, frees its TMEM and returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace {

using namespace tc;
constexpr int BM = 128, BK = 64;

__device__ __forceinline__ float gelu_tanh(float x) {
  float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
  return 0.5f * x * (1.f + tanhf(u));
}
__device__ __forceinline__ float gelu_tanh_grad(float x) {
  float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
  float th = tanhf(u);
  float du = 0.7978845608028654f * (1.f + 3.f * 0.044715f * x * x);
  return 0.5f * (1.f + th) + 0.5f * x * (1.f - th * th) * du;
}

struct TcParams {
  int M, N, K;
  int a_mn, b_mn;
  int epi;
  void* D;
  long long ldd;
  const bf16* bias;
  void* aux;
  long long ldaux;
  int* flags;
};

// epilogue for 32 consecutive columns [col0, col0+32) of one row
__device__ __forceinline__ void epilogue32(const TcParams& p, int row, int col0, float (&v)[32]) {
  if (p.epi == EPI_ACC_F32) {
    float* d = (float*)p.D + (size_t)row * p.ldd + col0;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      if (col0 + 4 * j < p.N) {
        float o[4];
        ld16(d + 4 * j, o);
        float r[4] = {o[0] + v[4 * j], o[1] + v[4 * j + 1], o[2] + v[4 * j + 2], o[3] + v[4 * j + 3]};
        st16(d + 4 * j, r);
      }
    }
    return;
  }
  bf16* d = (bf16*)p.D + (size_t)row * p.ldd + col0;
  if (p.epi == EPI_GELU_BWD) {
    const bf16* h = (const bf16*)p.aux + (size_t)row * p.ldaux + col0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      if (col0 + 8 * j < p.N) {
        float hv[8], o[8];
        ld16(h + 8 * j, hv);
#pragma unroll
        for (int k = 0; k < 8; k++) o[k] = v[8 * j + k] * gelu_tanh_grad(hv[k]);
        st16(d + 8 * j, o);
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; j++) {
    if (col0 + 8 * j < p.N) {
      float o[8];
      if (p.bias) {
        float bv[8];
        ld16(p.bias + col0 + 8 * j, bv);
#pragma unroll
        for (int k = 0; k < 8; k++) o[k] = v[8 * j + k] + bv[k];
      } else {
#pragma unroll
        for (int k = 0; k < 8; k++) o[k] = v[8 * j + k];
      }
      if (p.epi == EPI_GELU) {
        st16((bf16*)p.aux + (size_t)row * p.ldaux + col0 + 8 * j, o);
#pragma unroll
        for (int k = 0; k < 8; k++) o[k] = gelu_tanh(o[k]);
      }
      st16(d + 8 * j, o);
    }
  }
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, TcParams p) {
  constexpr uint32_t A_BYTES = BM * BK * 2;
  constexpr uint32_t B_BYTES = BN * BK * 2;
  constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint64_t* bars = (uint64_t*)(smem + STAGES * STAGE);
  uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 * STAGES + 4);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);
  const uint32_t ring = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; s++) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; a++) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 2 * BN);
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&ta) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tb) : "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;

  const int num_n = (p.N + BN - 1) / BN;
  const int tiles = ((p.M + BM - 1) / BM) * num_n;
  const int nk = (p.K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      uint32_t it = 0;
      for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int m0 = (t / num_n) * BM, n0 = (t % num_n) * BN;
        bool ok = true;
        for (int kb = 0; kb < nk; kb++, it++) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t fb = full0 + 8 * s;
          mbar_expect_tx(fb, STAGE);
          const uint32_t a_dst = ring + s * STAGE, b_dst = a_dst + A_BYTES;
          const int k0 = kb * BK;
          if (!p.a_mn) {
            tma_load_2d(a_dst, &ta, k0, m0, fb);
          } else {
            tma_load_2d(a_dst, &ta, m0, k0, fb);
            tma_load_2d(a_dst + 8192, &ta, m0 + 64, k0, fb);
          }
          if (!p.b_mn) {
            tma_load_2d(b_dst, &tb, k0, n0, fb);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; j++) tma_load_2d(b_dst + 8192 * j, &tb, n0 + 64 * j, k0, fb);
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      // instruction descriptor: D f32, A/B bf16, A/B major, N>>3, M>>4
      const uint32_t idesc = idesc_bf16(BM, BN, p.a_mn, p.b_mn);
      // K-major: advance 32 bytes per 16-wide k step inside the swizzled row,
      // SBO = 1024 (8 rows of 128 B).  MN-major: 16 k-rows of 128 B per step,
      // LBO = 8192 between 64-element MN blocks, SBO = 1024 between 8-row k groups.
      const uint32_t a_step = p.a_mn ? 2048u : 32u, b_step = p.b_mn ? 2048u : 32u;
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, b_lbo = p.b_mn ? 8192u : 16u;
      uint32_t it = 0, j = 0;
      for (int t = blockIdx.x; t < tiles; t += gridDim.x, j++) {
        const uint32_t a = j & 1, aph = (j >> 1) & 1;
        if (!mbar_wait(tempty0 + 8 * a, aph ^ 1, abort_flag)) break;
        fence_after();
        const uint32_t d = tmem + a * BN;
        bool ok = true;
        for (int kb = 0; kb < nk; kb++, it++) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(full0 + 8 * s, ph, abort_flag)) { ok = false; break; }
          fence_after();
          const uint32_t a_base = ring + s * STAGE, b_base = a_base + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; kk++) {
            const uint64_t ad = sdesc(a_base + kk * a_step, a_lbo, 1024);
            const uint64_t bd = sdesc(b_base + kk * b_step, b_lbo, 1024);
            mma_bf16(d, ad, bd, idesc, (kb | kk) != 0);
          }
          mma_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * a);
      }
    }
  } else {  // ---- epilogue warps 2..5
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t j = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, j++) {
      const int m0 = (t / num_n) * BM, n0 = (t % num_n) * BN;
      const uint32_t a = j & 1, aph = (j >> 1) & 1;
      // warp-uniform wait: tcgen05.ld below needs the whole warp converged
      const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * a, aph, abort_flag));
      if (!ok) break;
      fence_after();
      const int row = m0 + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < BN / 32; c++) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + a * BN + c * 32, v);
        const int col0 = n0 + c * 32;
        if (row < p.M && col0 < p.N) epilogue32(p, row, col0, v);
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * a);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.flags, FLAG_TIMEOUT);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int BN, int STAGES>
cudaError_t launch(const GemmArgs& g, int* flags, cudaStream_t st) {
  constexpr size_t smem = (size_t)STAGES * (BM * BK * 2 + BN * BK * 2) + 1024 + 256;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap ta, tb;
  bool ok = g.a_kmajor ? tc_make_map(&ta, g.A, g.K, g.M, g.lda, 64, BM) : tc_make_map(&ta, g.A, g.M, g.K, g.lda, 64, 64);
  ok = ok && (g.b_kmajor ? tc_make_map(&tb, g.B, g.K, g.N, g.ldb, 64, BN) : tc_make_map(&tb, g.B, g.N, g.K, g.ldb, 64, 64));
  if (!ok) return cudaErrorInvalidValue;
  TcParams p{g.M, g.N, g.K, g.a_kmajor ? 0 : 1, g.b_kmajor ? 0 : 1, g.epi, g.D, g.ldd, (const bf16*)g.bias,
             g.aux, g.ldaux, flags};
  const int sms = tc_num_sms();
  long long tiles = ((g.M + BM - 1) / BM) * (long long)((g.N + BN - 1) / BN);
  unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  gemm_tc_kernel<BN, STAGES><<<grid, 192, smem, st>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace

// ---------------------------------------------------------------------------
// host helpers shared by the tensor-core kernels (declared in tc_common.cuh)
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
  }
  return fn;
}

bool tc_available() { return encode_fn() != nullptr; }

bool tc_make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                 uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_num_sms() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  return sms;
}

extern void gpt2_count_launches(int n);

bool gemm_tc_supported(const GemmArgs& g) {
  auto al16 = [](const void* q) { return ((uintptr_t)q & 15) == 0; };
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return false;
  if (g.N % 8 || g.lda % 8 || g.ldb % 8 || !al16(g.A) || !al16(g.B) || !al16(g.D)) return false;
  if (g.epi == EPI_ACC_F32 ? (g.ldd % 4) : (g.ldd % 8)) return false;
  if ((g.epi == EPI_GELU || g.epi == EPI_GELU_BWD) && (!g.aux || g.ldaux % 8 || !al16(g.aux))) return false;
  if (g.bias && !al16(g.bias)) return false;
  if (g.a_kmajor ? g.lda < g.K : g.lda < g.M) return false;
  if (g.b_kmajor ? g.ldb < g.K : g.ldb < g.N) return false;
  return tc_available();
}

cudaError_t gemm_tc(const GemmArgs& g, int* flags, cudaStream_t st) {
  if (!gemm_tc_supported(g)) return cudaErrorNotSupported;
  gpt2_count_launches(1);
  if (g.N % 256 == 0) return launch<256, 4>(g, flags, st);
  return launch<128, 6>(g, flags, st);
}
