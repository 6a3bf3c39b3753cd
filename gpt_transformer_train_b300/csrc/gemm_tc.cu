// Tensor-core GEMM for sm_103a: TMA -> shared-memory ring -> tcgen05.mma into
// TMEM -> tcgen05.ld epilogue -> shared-memory staging -> TMA store.  Used for
// every matmul of the bf16 training step: the six forward matmuls (qkv,
// attention projection, fc + GELU, fc projection, tied classifier) and their
// input- and weight-gradient matmuls.
//
// D(m, n) = sum_k A(m, k) B(n, k); A and B are bf16, either K-major
// (row-major [rows][K]) or MN-major ([K][rows]), which covers y = x W^T
// (both K-major), dx = dy W (B MN-major) and dW = dy^T x (both MN-major)
// without any transpose pass.  Accumulation is fp32 in TMEM.
//
// Structure (one CTA per SM, persistent over work units, 64 + 32 * EPI_WARPS
// threads):
//   warp 0      TMA producer: per k-block one 128x64 A box (or two 64x64
//               boxes when MN-major) and the matching B boxes, 128-byte
//               swizzle, into a STAGES-deep ring guarded by mbarriers.
//   warp 1      allocates 2*BN TMEM columns (two accumulators) and one
//               thread issues tcgen05.mma (M=128, N=BN, K=16) per 16-wide
//               k step; tcgen05.commit frees ring stages and, at the end
//               of a unit, signals the epilogue.
//   warps 2..   EPI_WARPS = 4 or 8 epilogue warps: warp w takes the 32-row
//               slab of the TMEM lane quarter it may access (w mod 4) and,
//               with 8 warps, one half of the tile's columns, so two
//               epilogue warps share each SM sub-partition and hide each
//               other's latencies: tcgen05.ld 32 columns at a time, bias /
//               GELU / GELU' in registers, the slab's 32 x 64 bf16 (or
//               32 x 32 fp32) piece written to a 128-byte-swizzled staging
//               buffer and sent out by one TMA store per piece; the fp32
//               weight-gradient epilogue uses a TMA reduce-add into D, so D
//               is never read back by the SM.  The GELU' input tile comes in
//               by TMA as well.  The two accumulators let the epilogue of
//               one unit overlap the MMAs of the next.
// CTA pairs (CL = 2, tcgen05 cta_group::2): the two CTAs of a cluster
// compute one 256 x BN tile together.  Each CTA loads its own 128 rows of A
// and one half (BN/2 rows) of the B tile; one thread of the even CTA issues
// M=256 MMAs that read A and B from both CTAs' shared memory and write each
// CTA's 128 rows into its own TMEM.  Every SM then receives 32 KB of operands
// per 64-deep k-block instead of 48 KB for the same work, which is what
// bounds this kernel (operand delivery into the SM, not the tensor pipe),
// and the ring gets 6 stages (5 with eight epilogue warps, whose staging
// buffers take the room of one).  The odd CTA's TMA loads signal the even
// CTA's "full" barrier; the MMA commit arrives on both CTAs' "empty" and
// "accumulator full" barriers; both CTAs' epilogues arrive on the even CTA's
// "accumulator empty" barrier.
// Weight gradients have few output tiles and a long K = B*T, so K is split
// into ranges handled by different CTAs.  Split 0 adds its fp32 partial tile
// into D (TMA reduce-add; no other CTA touches that tile in this kernel);
// split s > 0 stores its tile into slot s-1 of a workspace (TMA store, no
// waiting on other CTAs); splitk_reduce then adds the slots into D in split
// order, so the result, (D + P0) + (P1 + P2 + ...), is deterministic.
// Every wait is bounded (about 2 s of %globaltimer); on expiry the CTA
// raises FLAG_TIMEOUT, stops issuing work, frees its TMEM and returns.
#include <algorithm>

#include "kernels.cuh"
#include "tc_common.cuh"

namespace {

using namespace tc;
constexpr int BM = 128, BK = 64;
constexpr uint32_t STG = 4096;  // one staging buffer: 32 rows x 128 B

struct TcParams {
  int M, N, K;
  int a_mn, b_mn;
  int epi;
  const bf16* bias;
  int* flags;
  int splits;  // K split into this many ranges (EPI_ACC_F32 only)
  int batch;   // independent products, item z at depth z of every tensor map
  float* dvec;  // EPI_ROWDOT: the per-row, per-head dot products
  int dT, dH;
  int acc_store;  // EPI_ACC_F32: split 0 stores its tile into D instead of adding it
  float* rowstats;  // EPI_STORE: per row and column tile, (max, sum of exp) of the stored values
  int stats_cols;   // columns counted in rowstats
  // a grouped launch (EPI_ACC_F32, no K split): after the first product's
  // units come batch2 items of a second product with M2 rows and the same N
  // and K, through the maps ta2, tb2, td2 (batch2 = 0: one product)
  int M2, batch2;
  // EPI_STORE / EPI_GELU: the LayerNorm of A folded in (GemmArgs::ln_*)
  const float* ln_mean; const float* ln_rstd; const float* ln_s; const float* ln_c;
};


// shared::cluster address of the same shared variable in the even CTA of the pair
__device__ __forceinline__ uint32_t leader_addr(uint32_t a) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(a));
  return r;
}
// TMA load of box (x, y) of batch item z into this CTA's shared memory
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// the same with completion signalled on a barrier of either CTA of the pair
// (cluster address)
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// arrive once on the barrier at this offset in both CTAs of the pair when the
// pair's MMAs issued so far have completed
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t holder_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder_smem), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// TMA store / reduce-add of a staged box, and bulk-group bookkeeping (per thread)
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"((uint64_t)map),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, int x, int y, int z, uint32_t src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          (uint64_t)map),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// 32 bf16 values (64 B) into 16-byte chunks ch0..ch0+3 of row r of a staging buffer
__device__ __forceinline__ void stage_bf16(uint32_t buf, uint32_t r, uint32_t ch0, const float (&v)[32]) {
#pragma unroll
  for (int u = 0; u < 4; u++)
    st_shared_v4(buf + swz(r, ch0 + u), pack_bf16(v[8 * u], v[8 * u + 1]), pack_bf16(v[8 * u + 2], v[8 * u + 3]),
                 pack_bf16(v[8 * u + 4], v[8 * u + 5]), pack_bf16(v[8 * u + 6], v[8 * u + 7]));
}
// v rounded to bf16 in place; its packed pairs (16 words) staged into chunks
// ch0..ch0+3 of row r of a staging buffer, as stage_bf16 would
__device__ __forceinline__ void round_stage_bf16(uint32_t buf, uint32_t r, uint32_t ch0, float (&v)[32]) {
#pragma unroll
  for (int u = 0; u < 4; u++) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      w[i] = pack_bf16(v[8 * u + 2 * i], v[8 * u + 2 * i + 1]);
      v[8 * u + 2 * i] = __uint_as_float(w[i] << 16);
      v[8 * u + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    st_shared_v4(buf + swz(r, ch0 + u), w[0], w[1], w[2], w[3]);
  }
}
// online row statistics over one 64-column chunk (v0: columns 0..31, v1:
// 32..63; the first nval count): m = running maximum, s = sum of exp(x - m)
__device__ __forceinline__ void chunk_stats(const float (&v0)[32], const float (&v1)[32], int nval, float& m,
                                            float& s) {
  constexpr float L2E = 1.4426950408889634f;
  if (nval <= 0) return;
  float c4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if (nval >= 64) {
#pragma unroll
    for (int k = 0; k < 32; k++) {
      c4[k & 3] = fmaxf(c4[k & 3], v0[k]);
      c4[(k + 2) & 3] = fmaxf(c4[(k + 2) & 3], v1[k]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; k++) {
      if (k < nval) c4[k & 3] = fmaxf(c4[k & 3], v0[k]);
      if (32 + k < nval) c4[(k + 2) & 3] = fmaxf(c4[(k + 2) & 3], v1[k]);
    }
  }
  const float mn = fmaxf(m, fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3])));
  const float ml = mn * L2E;
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  if (nval >= 64) {
#pragma unroll
    for (int k = 0; k < 32; k++) {
      s4[k & 3] += ex2(fmaf(v0[k], L2E, -ml));
      s4[(k + 2) & 3] += ex2(fmaf(v1[k], L2E, -ml));
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; k++) {
      if (k < nval) s4[k & 3] += ex2(fmaf(v0[k], L2E, -ml));
      if (32 + k < nval) s4[(k + 2) & 3] += ex2(fmaf(v1[k], L2E, -ml));
    }
  }
  // the earlier chunks' sum moves to the new maximum (m = -inf at the first: factor 0)
  s = s * ex2((m - mn) * L2E) + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
  m = mn;
}
// 32 fp32 values (128 B) into row r of a staging buffer
__device__ __forceinline__ void stage_f32(uint32_t buf, uint32_t r, const float (&v)[32]) {
#pragma unroll
  for (int u = 0; u < 8; u++)
    st_shared_v4(buf + swz(r, u), __float_as_uint(v[4 * u]), __float_as_uint(v[4 * u + 1]),
                 __float_as_uint(v[4 * u + 2]), __float_as_uint(v[4 * u + 3]));
}
// 32 bf16 values from chunks ch0..ch0+3 of row r of a staging buffer
__device__ __forceinline__ void unstage_bf16(const uint8_t* buf, uint32_t r, uint32_t ch0, float (&v)[32]) {
#pragma unroll
  for (int u = 0; u < 4; u++) {
    float f[8];
    ld16(reinterpret_cast<const bf16*>(buf + swz(r, ch0 + u)), f);
#pragma unroll
    for (int k = 0; k < 8; k++) v[8 * u + k] = f[k];
  }
}

template <int BN, int STAGES, int CL, int EPI_WARPS>
__global__ void __launch_bounds__(64 + 32 * EPI_WARPS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                   const __grid_constant__ CUtensorMap td, const __grid_constant__ CUtensorMap tx,
                   const __grid_constant__ CUtensorMap ta2, const __grid_constant__ CUtensorMap tb2,
                   const __grid_constant__ CUtensorMap td2, TcParams p) {
  constexpr uint32_t A_BYTES = BM * BK * 2;
  constexpr uint32_t B_BYTES = (BN / CL) * BK * 2;  // this CTA's share of the B tile
  constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* stg_gen = smem + STAGES * STAGE;  // EPI_WARPS warps x 2 staging buffers
  uint64_t* bars = (uint64_t*)(stg_gen + 2 * EPI_WARPS * STG);
  uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
  uint32_t auxbar0 = smem_u32(bars + 2 * STAGES + 4);  // aux tile loads, two per epilogue warp
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 * STAGES + 4 + 2 * EPI_WARPS);
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
      mbar_init(tempty0 + 8 * a, EPI_WARPS * CL);  // the epilogue warps of both CTAs of a pair
    }
    for (int w = 0; w < 2 * EPI_WARPS; w++) mbar_init(auxbar0 + 8 * w, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the peer's loads, commits and arrivals target this CTA's barriers: they must exist first
  if (CL > 1) cluster_sync();
  if (warp == 1) {
    if (CL == 1) tmem_alloc(smem_u32(tmem_holder), 2 * BN);
    else tmem_alloc_pair(smem_u32(tmem_holder), 2 * BN);
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&ta) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tb) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&td) : "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_enter();  // global memory only from here on

  const int num_n = (p.N + BN - 1) / BN;
  // a "tile" here is CL vertically adjacent 128-row tiles (one per CTA of the pair)
  const int tiles = ((p.M + CL * BM - 1) / (CL * BM)) * num_n;
  const int nk = (p.K + BK - 1) / BK;
  // unit u < units1: batch item u / (splits * tiles), split (u / tiles) % splits,
  // tile u % tiles; the second product's units (grouped launch) follow
  const int units1 = tiles * p.splits * p.batch;
  const int tiles2 = ((p.M2 + CL * BM - 1) / (CL * BM)) * num_n;
  const int units = units1 + tiles2 * p.batch2;
  auto decode = [&](int u, int& pr, int& t, int& sp, int& z) {
    if (u < units1) {
      pr = 0;
      t = u % tiles;
      sp = (u / tiles) % p.splits;
      z = u / (tiles * p.splits);
    } else {
      const int v = u - units1;
      pr = 1;
      t = v % tiles2;
      sp = 0;
      z = v / tiles2;
    }
  };
  auto kb_begin = [&](int sp) { return (int)((long long)nk * sp / p.splits); };
  const uint32_t crank = CL > 1 ? cluster_rank() : 0;
  const int ustart = (int)(blockIdx.x / CL), ustep = (int)(gridDim.x / CL);
  auto tile_m0 = [&](int t) { return ((t / num_n) * CL + (int)crank) * BM; };

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      uint32_t it = 0;
      for (int u = ustart; u < units; u += ustep) {
        int pr, t, sp, z;
        decode(u, pr, t, sp, z);
        const CUtensorMap* mA = pr ? &ta2 : &ta;
        const CUtensorMap* mB = pr ? &tb2 : &tb;
        const int m0 = tile_m0(t), n0 = (t % num_n) * BN;
        bool ok = true;
        for (int kb = kb_begin(sp), kb1 = kb_begin(sp + 1); kb < kb1; kb++, it++) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t a_dst = ring + s * STAGE, b_dst = a_dst + A_BYTES;
          const int k0 = kb * BK;
          if (CL == 1) {
            const uint32_t fb = full0 + 8 * s;
            mbar_expect_tx(fb, STAGE);
            if (!p.a_mn) {
              tma_load_3d(a_dst, mA, k0, m0, z, fb);
            } else {
              tma_load_3d(a_dst, mA, m0, k0, z, fb);
              tma_load_3d(a_dst + 8192, mA, m0 + 64, k0, z, fb);
            }
            if (!p.b_mn) {
              tma_load_3d(b_dst, mB, k0, n0, z, fb);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; j++) tma_load_3d(b_dst + 8192 * j, mB, n0 + 64 * j, k0, z, fb);
            }
          } else {
            // both CTAs' loads complete on the even CTA's barrier, which expects all of them
            const uint32_t fb = leader_addr(full0 + 8 * s);
            if (crank == 0) mbar_expect_tx(full0 + 8 * s, 2 * STAGE);
            if (!p.a_mn) {
              tma_load_3d_pair(a_dst, mA, k0, m0, z, fb);
            } else {
              tma_load_3d_pair(a_dst, mA, m0, k0, z, fb);
              tma_load_3d_pair(a_dst + 8192, mA, m0 + 64, k0, z, fb);
            }
            const int nb = n0 + (int)crank * (BN / 2);  // this CTA's half of the B tile
            if (!p.b_mn) {
              tma_load_3d_pair(b_dst, mB, k0, nb, z, fb);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 128; j++) tma_load_3d_pair(b_dst + 8192 * j, mB, nb + 64 * j, k0, z, fb);
            }
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && crank == 0) {  // ---- MMA issuer (the even CTA of a pair)
      const uint32_t idesc = idesc_bf16(CL * BM, BN, p.a_mn, p.b_mn);
      // K-major: advance 32 bytes per 16-wide k step inside the swizzled row,
      // SBO = 1024 (8 rows of 128 B).  MN-major: 16 k-rows of 128 B per step,
      // LBO = 8192 between 64-element MN blocks, SBO = 1024 between 8-row k groups.
      const uint32_t a_step = p.a_mn ? 2048u : 32u, b_step = p.b_mn ? 2048u : 32u;
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, b_lbo = p.b_mn ? 8192u : 16u;
      uint32_t it = 0, j = 0;
      for (int u = ustart; u < units; u += ustep, j++) {
        const uint32_t a = j & 1, aph = (j >> 1) & 1;
        if (!mbar_wait(tempty0 + 8 * a, aph ^ 1, abort_flag)) break;
        fence_after();
        const uint32_t d = tmem + a * BN;
        bool ok = true;
        int pr, t, sp, z;
        decode(u, pr, t, sp, z);
        const int kb0 = kb_begin(sp);
        for (int kb = kb0, kb1 = kb_begin(sp + 1); kb < kb1; kb++, it++) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(full0 + 8 * s, ph, abort_flag)) { ok = false; break; }
          fence_after();
          const uint32_t a_base = ring + s * STAGE, b_base = a_base + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; kk++) {
            const uint64_t ad = sdesc(a_base + kk * a_step, a_lbo, 1024);
            const uint64_t bd = sdesc(b_base + kk * b_step, b_lbo, 1024);
            if (CL == 1) mma_bf16(d, ad, bd, idesc, (kb != kb0) || kk != 0);
            else mma_bf16_pair(d, ad, bd, idesc, (kb != kb0) || kk != 0);
          }
          if (CL == 1) mma_commit(empty0 + 8 * s);
          else mma_commit_pair(empty0 + 8 * s);
        }
        if (!ok) break;
        if (CL == 1) mma_commit(tfull0 + 8 * a);
        else mma_commit_pair(tfull0 + 8 * a);
      }
    }
  } else {  // ---- epilogue warps 2 .. 1 + EPI_WARPS
    constexpr int HALF = BN * 4 / EPI_WARPS;  // columns of the tile per epilogue warp
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int e = warp - 2;  // this warp's staging buffers and aux barriers
    const int hc = (e >> 2) * HALF;  // first tile column of this warp's half
    const uint32_t stg = smem_u32(stg_gen) + e * 2 * STG;
    const uint8_t* stg_g = stg_gen + e * 2 * STG;
    const uint32_t auxbar = auxbar0 + 16 * e;  // buffer b's loads complete on auxbar + 8 b
    // epilogues that read an aux tile (GELU', ROWDOT): live chunk ci of this
    // warp uses buffer ci & 1 (its aux tile in, its output written over it and
    // stored from there); the next chunk's load is issued before this chunk's math
    const bool aux_epi = p.epi == EPI_GELU_BWD || p.epi == EPI_ROWDOT;
    // live chunk ci (of any epilogue but GELU) is staged in buffer ci & 1, so
    // the store two chunks back is the last one that read it
    uint32_t ci = 0;
    int pending = -1;  // buffer with an aux load issued and not yet waited for
    uint32_t pending_par = 0;
    auto aux_issue = [&](int col, int row, int zz, uint32_t b) {  // lane 0
      mbar_expect_tx(auxbar + 8 * b, STG);
      tma_load_3d(stg + b * STG, &tx, col, row, zz, auxbar + 8 * b);
    };
    // the tile's bias: lane l holds columns 8l..8l+7 of it (16 bytes), the next
    // tile's slice is loaded while this tile is processed
    auto bias_slice = [&](int uu) {
      uint4 r = make_uint4(0u, 0u, 0u, 0u);
      if (p.bias && uu < units) {
        const int col = ((uu % tiles) % num_n) * BN + 8 * lane;
        if (8 * lane < BN && col < p.N) r = __ldg(reinterpret_cast<const uint4*>(p.bias + col));
      }
      return r;
    };
    uint4 bias_next = bias_slice(ustart);
    // 32 bias values of columns c0..c0+31 of the tile into v
    auto add_bias = [&](const uint4& bs, int c0, float (&v)[32]) {
#pragma unroll
      for (int g = 0; g < 4; g++) {
        uint4 w;
        w.x = __shfl_sync(0xffffffffu, bs.x, c0 / 8 + g);
        w.y = __shfl_sync(0xffffffffu, bs.y, c0 / 8 + g);
        w.z = __shfl_sync(0xffffffffu, bs.z, c0 / 8 + g);
        w.w = __shfl_sync(0xffffffffu, bs.w, c0 / 8 + g);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const float2 f = __bfloat1622float2(h[k]);
          v[8 * g + 2 * k] += f.x;
          v[8 * g + 2 * k + 1] += f.y;
        }
      }
    };
    // LayerNorm folded into the product: 32 accumulator columns c0.. (tile
    // columns, global column col0) of this lane's row to
    // rstd * (acc - mean * s[n]) + c[n]; s and c are read as broadcast float4s
    auto apply_fold = [&](float (&v)[32], int col0, float mu, float rs) {
#pragma unroll
      for (int g = 0; g < 8; g++) {
        if (col0 + 4 * g < p.N) {
          const float4 sv = __ldg(reinterpret_cast<const float4*>(p.ln_s + col0) + g);
          const float4 cv = __ldg(reinterpret_cast<const float4*>(p.ln_c + col0) + g);
          v[4 * g] = fmaf(rs, fmaf(-mu, sv.x, v[4 * g]), cv.x);
          v[4 * g + 1] = fmaf(rs, fmaf(-mu, sv.y, v[4 * g + 1]), cv.y);
          v[4 * g + 2] = fmaf(rs, fmaf(-mu, sv.z, v[4 * g + 2]), cv.z);
          v[4 * g + 3] = fmaf(rs, fmaf(-mu, sv.w, v[4 * g + 3]), cv.w);
        }
      }
    };
    bool prefetched = false;  // the next tile's first aux chunk is already on its way
    // the accumulator is free again: tell the CTA whose thread issues the MMAs
    auto release_acc = [&](uint32_t bar) {
      if (CL == 1) mbar_arrive(bar);
      else mbar_arrive_cluster(leader_addr(bar));
    };
    uint32_t j = 0;
    for (int u = ustart; u < units; u += ustep, j++) {
      int pr, t, sp, z;
      decode(u, pr, t, sp, z);
      const int m0 = tile_m0(t), n0 = (t % num_n) * BN;
      const int rbase = m0 + q * 32;  // first row of this warp's slab
      const bool rows_in = rbase < (pr ? p.M2 : p.M);
      const uint32_t a = j & 1, aph = (j >> 1) & 1;
      // live 64-column chunks of this warp's half
      const int nlive = rows_in && n0 + hc < p.N ? min(HALF / 64, (p.N - n0 - hc + 63) / 64) : 0;
      if (aux_epi && nlive > 0 && !prefetched) {  // the first chunk's aux tile, before the accumulator is ready
        if (lane == 0) {
          bulk_wait_read<1>();
          aux_issue(n0 + hc, rbase, z, ci & 1);
        }
        pending = (int)(ci & 1);
        pending_par = (ci >> 1) & 1;
      }
      prefetched = false;
      const uint4 bias_cur = bias_next;
      bias_next = bias_slice(u + ustep);
      // warp-uniform wait: tcgen05.ld below needs the whole warp converged
      if (!mbar_wait_warp(tfull0 + 8 * a, aph, abort_flag)) break;
      fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + a * BN;
      float st_m = -INFINITY, st_s = 0.f;  // rowstats of this lane's row over the tile
      // this lane's row statistics when the LayerNorm is folded in
      float ln_mu = 0.f, ln_rs = 0.f;
      if (p.ln_mean && rows_in && rbase + lane < p.M) {
        ln_mu = __ldg(p.ln_mean + rbase + lane);
        ln_rs = __ldg(p.ln_rstd + rbase + lane);
      }
      if (p.epi == EPI_ACC_F32) {
        // split 0: D += tile (TMA reduce-add); split s > 0: workspace slot s - 1
#pragma unroll 1
        for (int c = 0; c < HALF / 32; c++) {
          float v[32];
          tmem_ld32(tacc + hc + c * 32, v);
          const int col0 = n0 + hc + c * 32;
          if (rows_in && col0 < p.N) {
            const uint32_t buf = stg + (ci & 1) * STG;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            stage_f32(buf, lane, v);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (sp == 0) {
                const CUtensorMap* mD = pr ? &td2 : &td;
                if (p.acc_store) tma_store_3d(mD, col0, rbase, z, buf);
                else tma_reduce_add_3d(mD, col0, rbase, z, buf);
              }
              else tma_store_3d(&tx, col0, rbase, sp - 1, buf);  // workspace slot sp - 1
              bulk_commit();
            }
            ci++;
          }
        }
        fence_before();
        __syncwarp();
        if (lane == 0) release_acc(tempty0 + 8 * a);
        continue;
      }
      bool ok = true;
#pragma unroll 1
      for (int cp = 0; cp < HALF / 64; cp++) {
        const int tc0 = hc + cp * 64;  // first column of the chunk within the tile
        const int col0 = n0 + tc0;
        const bool live = rows_in && col0 < p.N;
        float v0[32], v1[32];
        tmem_ld32_async(tacc + tc0, v0);
        tmem_ld32_async(tacc + tc0 + 32, v1);
        tmem_wait_ld();
        if (!live) continue;
        const uint32_t bo = stg + (ci & 1) * STG;  // output piece
        if (p.epi == EPI_STORE) {
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          if (p.bias) {
            add_bias(bias_cur, tc0, v0);
            add_bias(bias_cur, tc0 + 32, v1);
          } else if (p.ln_mean) {
            apply_fold(v0, col0, ln_mu, ln_rs);
            apply_fold(v1, col0 + 32, ln_mu, ln_rs);
          }
          if (p.rowstats) {
            // the values as stored (bf16) enter the statistics
            round_stage_bf16(bo, lane, 0, v0);
            round_stage_bf16(bo, lane, 4, v1);
            chunk_stats(v0, v1, p.stats_cols - col0, st_m, st_s);
          } else {
            stage_bf16(bo, lane, 0, v0);
            stage_bf16(bo, lane, 4, v1);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&td, col0, rbase, z, bo);
            bulk_commit();
          }
          ci++;
        } else if (p.epi == EPI_GELU) {
          // pre-activation (aux) from buffer 0 and GELU output from buffer 1,
          // each store its own bulk group, so each buffer waits only for its
          // own last store (the pre-activation goes out before the GELU math:
          // one proxy fence for both came out slower, 86 against 80 us)
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          if (p.bias) {
            add_bias(bias_cur, tc0, v0);
            add_bias(bias_cur, tc0 + 32, v1);
          } else if (p.ln_mean) {
            apply_fold(v0, col0, ln_mu, ln_rs);
            apply_fold(v1, col0 + 32, ln_mu, ln_rs);
          }
          // the pre-activation as stored (bf16) is what GELU takes, so a later
          // recompute from it gives the same bits
          round_stage_bf16(stg, lane, 0, v0);
          round_stage_bf16(stg, lane, 4, v1);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tx, col0, rbase, z, stg);
            bulk_commit();
          }
#pragma unroll
          for (int k = 0; k < 32; k++) {
            v0[k] = gelu_fwd(v0[k]);
            v1[k] = gelu_fwd(v1[k]);
          }
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          stage_bf16(stg + STG, lane, 0, v0);
          stage_bf16(stg + STG, lane, 4, v1);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&td, col0, rbase, z, stg + STG);
            bulk_commit();
          }
        } else {  // EPI_GELU_BWD: D = acc * GELU'(aux); EPI_ROWDOT: D = acc and its dot with aux
          const uint32_t b = ci & 1, buf = stg + b * STG;
          const uint8_t* buf_g = stg_g + b * STG;
          // the next live chunk's aux tile: this tile's next chunk, else the next tile's first
          bool has_next = false;
          int nx = col0 + 64, ny = rbase, nz = z;
          if (cp + 1 < nlive) {
            has_next = true;
          } else if (u + ustep < units) {
            const int u2 = u + ustep, t2 = u2 % tiles;
            ny = tile_m0(t2) + q * 32;
            nx = (t2 % num_n) * BN + hc;
            nz = u2 / (tiles * p.splits);
            has_next = prefetched = ny < p.M && nx < p.N;
          }
          if (has_next && lane == 0) {
            bulk_wait_read<0>();  // the previous chunk's store has read the other buffer
            aux_issue(nx, ny, nz, b ^ 1);
          }
          __syncwarp();
          if (!mbar_wait_warp(auxbar + 8 * b, (ci >> 1) & 1, abort_flag)) {
            if (has_next) mbar_settle(auxbar + 8 * (b ^ 1), ((ci + 1) >> 1) & 1);
            pending = (int)b;
            pending_par = (ci >> 1) & 1;
            ok = false;
            break;
          }
          pending = has_next ? (int)(b ^ 1) : -1;
          pending_par = ((ci + 1) >> 1) & 1;
          // each lane reads its row's aux values and writes its outputs over them
          float hv[32];
          if (p.epi == EPI_GELU_BWD) {
            unstage_bf16(buf_g, lane, 0, hv);
#pragma unroll
            for (int k = 0; k < 32; k++) v0[k] *= gelu_bwd(hv[k]);
            stage_bf16(buf, lane, 0, v0);
            unstage_bf16(buf_g, lane, 4, hv);
#pragma unroll
            for (int k = 0; k < 32; k++) v1[k] *= gelu_bwd(hv[k]);
            stage_bf16(buf, lane, 4, v1);
          } else {
            // the head's 64 columns: products of the stored (bf16) values with aux, in column order
            float d = 0.f;
            unstage_bf16(buf_g, lane, 0, hv);
            round_stage_bf16(buf, lane, 0, v0);
#pragma unroll
            for (int k = 0; k < 32; k++) d = fmaf(v0[k], hv[k], d);
            unstage_bf16(buf_g, lane, 4, hv);
            round_stage_bf16(buf, lane, 4, v1);
#pragma unroll
            for (int k = 0; k < 32; k++) d = fmaf(v1[k], hv[k], d);
            const int row = rbase + lane;
            if (row < p.M) {
              const int bb = row / p.dT, t = row - bb * p.dT;
              p.dvec[((size_t)bb * p.dH + col0 / 64) * p.dT + t] = d;
            }
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&td, col0, rbase, z, buf);
            bulk_commit();
          }
          ci++;
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) release_acc(tempty0 + 8 * a);
      if (!ok) break;
      if (p.rowstats && rows_in && rbase + lane < p.M)
        *reinterpret_cast<float2*>(p.rowstats + ((size_t)(rbase + lane) * num_n + n0 / BN) * 2) =
            make_float2(st_m, st_s);
    }
    // an aux load cut short by an abort must land before the CTA exits
    if (pending >= 0) mbar_settle(auxbar + 8 * pending, pending_par);
    // the staging buffers must stay valid until every store has read them
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }
  fence_before();
  __syncthreads();
  // neither CTA of a pair may leave while the other can still write into it
  if (CL > 1) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    if (CL == 1) tmem_dealloc(tmem, 2 * BN);
    else tmem_dealloc_pair(tmem, 2 * BN);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.flags, FLAG_TIMEOUT);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// K splits for an fp32-accumulate launch: the count (1..16, at least 8
// k-blocks each) whose units fill the `slots` concurrent CTAs (or CTA pairs)
// best, the smallest among near ties
int choose_splits(int tiles, int nk, int slots) {
  int best = 1;
  double best_eff = 0;
  for (int s = 1; s <= 16 && nk / s >= 8; s++) {
    const long long units = (long long)tiles * s;
    const double eff = (double)units / (double)(((units + slots - 1) / slots) * slots);
    if (eff > best_eff + 0.02) best = s, best_eff = eff;
  }
  return best;
}

// 3-D tiled map with 128-byte swizzle: [depth][outer][inner] with row stride
// ld and item stride bstride (elements); box = box_inner x box_outer x 1
bool make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t ld, uint64_t depth, uint64_t bstride, uint32_t box_inner,
                 uint32_t box_outer);

template <int BN, int STAGES, int CL, int EPI_WARPS>
constexpr size_t smem_bytes() {
  return (size_t)STAGES * (BM * BK * 2 + (BN / CL) * BK * 2) + 2 * EPI_WARPS * STG + 1024 + 512;
}

template <int BN, int STAGES, int CL, int EPI_WARPS>
cudaError_t launch(const GemmArgs& g, int splits, int* flags, cudaStream_t st, const GemmArgs* g2 = nullptr) {
  constexpr size_t smem = smem_bytes<BN, STAGES, CL, EPI_WARPS>();
  static_assert(smem <= 232448, "shared memory per CTA");
  static_assert((2 * STAGES + 4 + 2 * EPI_WARPS) * 8 + 8 <= 512,
                "barriers, TMEM address and abort flag after the staging buffers");
  static_assert((BN * 4 / EPI_WARPS) % 64 == 0, "each epilogue warp takes whole 64-column chunks");
  {
    cudaError_t e = kernel_smem_attr(gemm_tc_kernel<BN, STAGES, CL, EPI_WARPS>, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // every operand map is 3-D: depth = batch items, g.sX elements apart
  CUtensorMap ta, tb, td, tx;
  const uint64_t nb = (uint64_t)(g.batch > 1 ? g.batch : 1);
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  bool ok = g.a_kmajor ? make_map_3d(&ta, bf, 2, g.A, g.K, g.M, g.lda, nb, g.sA, 64, BM)
                       : make_map_3d(&ta, bf, 2, g.A, g.M, g.K, g.lda, nb, g.sA, 64, 64);
  ok = ok && (g.b_kmajor ? make_map_3d(&tb, bf, 2, g.B, g.K, g.N, g.ldb, nb, g.sB, 64, BN / CL)
                         : make_map_3d(&tb, bf, 2, g.B, g.N, g.K, g.ldb, nb, g.sB, 64, 64));
  if (g.epi == EPI_ACC_F32)
    ok = ok && make_map_3d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.D, g.N, g.M, g.ldd, nb, g.sD, 32, 32);
  else ok = ok && make_map_3d(&td, bf, 2, g.D, g.N, g.M, g.ldd, nb, g.sD, 64, 32);
  if (g.epi == EPI_GELU || g.epi == EPI_GELU_BWD || g.epi == EPI_ROWDOT)
    ok = ok && make_map_3d(&tx, bf, 2, g.aux, g.N, g.M, g.ldaux, nb, g.sAux, 64, 32);
  else if (g.epi == EPI_ACC_F32 && splits > 1) ok = ok && tc_make_map_f32_3d(&tx, g.ws, g.N, g.M, splits - 1, 32, 32);
  else tx = td;
  // the second product of a grouped launch (EPI_ACC_F32, same N, K and operand majors)
  CUtensorMap ta2 = ta, tb2 = tb, td2 = td;
  long long nb2 = 0;
  if (g2) {
    nb2 = g2->batch > 1 ? g2->batch : 1;
    ok = ok && (g2->a_kmajor ? make_map_3d(&ta2, bf, 2, g2->A, g2->K, g2->M, g2->lda, nb2, g2->sA, 64, BM)
                             : make_map_3d(&ta2, bf, 2, g2->A, g2->M, g2->K, g2->lda, nb2, g2->sA, 64, 64));
    ok = ok && (g2->b_kmajor ? make_map_3d(&tb2, bf, 2, g2->B, g2->K, g2->N, g2->ldb, nb2, g2->sB, 64, BN / CL)
                             : make_map_3d(&tb2, bf, 2, g2->B, g2->N, g2->K, g2->ldb, nb2, g2->sB, 64, 64));
    ok = ok && make_map_3d(&td2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g2->D, g2->N, g2->M, g2->ldd, nb2, g2->sD, 32, 32);
  }
  if (!ok) return cudaErrorInvalidValue;
  const int sms = tc_num_sms();
  const long long tiles = ((g.M + CL * BM - 1) / (CL * BM)) * (long long)((g.N + BN - 1) / BN);
  TcParams p{g.M, g.N, g.K, g.a_kmajor ? 0 : 1, g.b_kmajor ? 0 : 1, g.epi, (const bf16*)g.bias, flags, splits,
             (int)nb, g.dvec, g.dT, g.dH, g.acc_store, g.rowstats, g.stats_cols, g2 ? g2->M : 0, (int)nb2,
             g.ln_mean, g.ln_rstd, g.ln_s, g.ln_c};
  const long long tiles2 = g2 ? ((g2->M + CL * BM - 1) / (CL * BM)) * (long long)((g.N + BN - 1) / BN) : 0;
  const long long units = tiles * splits * (long long)nb + tiles2 * nb2;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(64 + 32 * EPI_WARPS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  long long slots = sms / CL;  // clusters that can run at once
  if (CL > 1) {
    static int max_clusters = 0;
    if (!max_clusters) {
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = CL;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      cfg.gridDim = dim3((unsigned)(slots * CL));
      if (cudaOccupancyMaxActiveClusters(&max_clusters, gemm_tc_kernel<BN, STAGES, CL, EPI_WARPS>, &cfg) != cudaSuccess ||
          max_clusters <= 0)
        max_clusters = (int)slots;
    }
    if (max_clusters < slots) slots = max_clusters;
  }
  const unsigned grid = (unsigned)((units < slots ? units : slots) * CL);
  cfg.gridDim = dim3(grid);
  // programmatic dependent launch (the kernel waits for its predecessor
  // after its prologue), and the CTA-pair cluster
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (CL > 1) {
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = CL;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, STAGES, CL, EPI_WARPS>, ta, tb, td, tx, ta2, tb2, td2, p);
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

static bool make_map_dt(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool tc_make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                 uint32_t box_outer) {
  return make_map_dt(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, ld, box_inner, box_outer);
}

bool tc_make_map_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                     uint32_t box_inner, uint32_t box_outer) {
  return make_map_dt(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, inner, outer, ld, box_inner, box_outer);
}

namespace {
bool make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t ld, uint64_t depth, uint64_t bstride, uint32_t box_inner,
                 uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  if (depth <= 1) bstride = ld * outer;  // unused, any valid stride
  cuuint64_t dims[3] = {inner, outer, depth};
  cuuint64_t strides[2] = {ld * esize, bstride * esize};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}
}  // namespace

// dense fp32 [depth][outer][inner] (contiguous), box = box_inner x box_outer x 1
bool tc_make_map_f32_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t depth,
                        uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, outer, depth};
  cuuint64_t strides[2] = {inner * 4, inner * outer * 4};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_num_sms() {
  static int sms = 0;
  if (sms <= 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      sms = n;
  }
  return sms > 0 ? sms : 148;
}

extern void gpt2_count_launches(int n);

bool gemm_tc_supported(const GemmArgs& g) {
  auto al16 = [](const void* q) { return ((uintptr_t)q & 15) == 0; };
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return false;
  if (g.N % 8 || g.lda % 8 || g.ldb % 8 || !al16(g.A) || !al16(g.B) || !al16(g.D)) return false;
  if (g.epi == EPI_ACC_F32 ? (g.ldd % 4) : (g.ldd % 8)) return false;
  if (g.ldd < g.N) return false;
  if ((g.epi == EPI_GELU || g.epi == EPI_GELU_BWD || g.epi == EPI_ROWDOT) &&
      (!g.aux || g.ldaux % 8 || g.ldaux < g.N || !al16(g.aux)))
    return false;
  // rows are (b, t) with t < dT; 64-column heads; one product only
  if (g.epi == EPI_ROWDOT &&
      (!g.dvec || g.dT <= 0 || g.dH <= 0 || g.N != 64 * g.dH || g.M % g.dT || g.batch > 1 || g.bias))
    return false;
  if (g.bias && (!al16(g.bias) || (g.epi != EPI_STORE && g.epi != EPI_GELU))) return false;
  if (g.rowstats && (g.epi != EPI_STORE || g.batch > 1 || g.stats_cols <= 0)) return false;
  if (g.ln_mean || g.ln_rstd || g.ln_s || g.ln_c) {
    if (!g.ln_mean || !g.ln_rstd || !g.ln_s || !g.ln_c || !al16(g.ln_s) || !al16(g.ln_c)) return false;
    if ((g.epi != EPI_STORE && g.epi != EPI_GELU) || g.bias || g.rowstats || g.batch > 1 || !g.a_kmajor) return false;
  }
  if (g.a_kmajor ? g.lda < g.K : g.lda < g.M) return false;
  if (g.b_kmajor ? g.ldb < g.K : g.ldb < g.N) return false;
  if (g.batch > 1) {
    const bool f32 = g.epi == EPI_ACC_F32;
    if (g.bias || g.sA <= 0 || g.sB <= 0 || g.sD <= 0 || g.sA % 8 || g.sB % 8 || g.sD % (f32 ? 4 : 8)) return false;
    if (g.aux && (g.sAux <= 0 || g.sAux % 8)) return false;
  }
  return tc_available();
}

// K splits a weight-gradient (fp32 accumulate) product would use, and the
// workspace floats they need (splits * M * N, 0 when no split pays off)
// Split count of a weight-gradient (fp32 accumulate) product on CTA pairs and
// the workspace floats it needs: (splits - 1) * M * N, 0 when there is no split
static int splits_for(int M, int N, int K, size_t ws_floats, int sms) {
  const int BN = N >= 512 ? 256 : 128;
  const long long tiles = ((M + 2 * BM - 1) / (2 * BM)) * (long long)((N + BN - 1) / BN);
  int s = choose_splits((int)tiles, (K + BK - 1) / BK, sms / 2);
  while (s > 1 && (size_t)(s - 1) * M * N > ws_floats) s--;
  return s;
}
int gemm_tc_splits(int M, int N, int K, size_t ws_floats) { return splits_for(M, N, K, ws_floats, tc_num_sms()); }
// sized for a given SM count (the planner uses the B300's 148 so that the
// buffer size does not depend on the machine that asks); a run on a GPU with
// more SMs caps its splits to what fits
size_t gemm_tc_workspace_floats(int M, int N, int K, int sms) {
  const int s = splits_for(M, N, K, (size_t)-1, sms);
  return s > 1 ? (size_t)(s - 1) * M * N : 0;
}

__global__ void __launch_bounds__(256) splitk_reduce_kernel(float* __restrict__ D, long long ldd,
                                                            const float* __restrict__ ws, int M, int N, int splits) {
  pdl_enter();
  // D[m][n] += ws[0][m][n] + ws[1][m][n] + ... (the partials of splits 1, 2,
  // ... in order); four columns per thread, every load issued before the additions
  const long long nv = (long long)M * (N / 4);
  const size_t plane = (size_t)M * N;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(i / (N / 4)), n = (int)(i % (N / 4)) * 4;
    const float* src = ws + (size_t)m * N + n;
    float4 u[16];
#pragma unroll
    for (int sp = 0; sp < 16; sp++)
      if (sp < splits) u[sp] = __ldcs(reinterpret_cast<const float4*>(src + sp * plane));
    float4 t = u[0];
#pragma unroll
    for (int sp = 1; sp < 16; sp++)
      if (sp < splits) {
        t.x += u[sp].x; t.y += u[sp].y; t.z += u[sp].z; t.w += u[sp].w;
      }
    float4* d = reinterpret_cast<float4*>(D + (size_t)m * ldd + n);
    float4 o = *d;
    o.x += t.x; o.y += t.y; o.z += t.z; o.w += t.w;
    *d = o;
  }
}

int gemm_tc_stats_tiles(int N) { return N >= 512 ? (N + 255) / 256 : (N + 127) / 128; }

// two fp32-accumulate products with the same N, K and operand majors in one
// launch (the second's units after the first's), so the two share their last
// partial wave; falls back to two launches when the pair of them would not
// fill the CTA pairs or the shapes differ
cudaError_t gemm_tc_grouped(const GemmArgs& a, const GemmArgs& b, int* flags, cudaStream_t st) {
  if (!gemm_tc_supported(a) || !gemm_tc_supported(b)) return cudaErrorNotSupported;
  const int sms = tc_num_sms();
  auto row_tiles = [](const GemmArgs& g) { return (long long)(g.M + BM - 1) / BM; };
  auto items = [](const GemmArgs& g) { return (long long)(g.batch > 1 ? g.batch : 1); };
  const long long nt = (a.N + 255) / 256;
  const bool same = a.epi == EPI_ACC_F32 && b.epi == EPI_ACC_F32 && a.N == b.N && a.K == b.K &&
                    a.a_kmajor == b.a_kmajor && a.b_kmajor == b.b_kmajor && a.acc_store == b.acc_store && !a.bias &&
                    !b.bias && a.N >= 512;
  if (!same || row_tiles(a) < 2 || row_tiles(b) < 2 ||
      (row_tiles(a) * items(a) + row_tiles(b) * items(b)) * nt < sms) {
    cudaError_t e = gemm_tc(a, flags, st);
    return e != cudaSuccess ? e : gemm_tc(b, flags, st);
  }
  gpt2_count_launches(1);
  return launch<256, 6, 2, 4>(a, 1, flags, st, &b);
}

cudaError_t gemm_tc(const GemmArgs& g, int* flags, cudaStream_t st) {
  if (!gemm_tc_supported(g)) return cudaErrorNotSupported;
  gpt2_count_launches(1);
  const bool wide = g.N >= 512;  // 256-wide tiles (a ragged last column tile is clipped by TMA); as gemm_tc_stats_tiles
  const int sms = tc_num_sms();
  const long long mt = (g.M + BM - 1) / BM, nt = (g.N + (wide ? 256 : 128) - 1) / (wide ? 256 : 128);
  const long long nb = g.batch > 1 ? g.batch : 1;
  int splits = 1;
  if (g.epi == EPI_ACC_F32 && g.ws && g.N % 4 == 0 && mt >= 2 && nb == 1)
    splits = gemm_tc_splits(g.M, g.N, g.K, g.ws_floats);
  // CTA pairs (cta_group::2) when there are enough row tiles to pair up, or for a split K
  const bool pair = mt >= 2 && (splits > 1 || mt * nt * nb >= sms);
  cudaError_t e;
  // the GELU epilogues are bound by their arithmetic: eight epilogue warps (two
  // per SM sub-partition, the ring one stage shorter to make room for their
  // staging buffers); the others keep four warps and the deeper ring
  // (measured on the 124M shapes: fc forward with GELU 100 -> 88 us, fc
  // projection dgrad with GELU' 104 -> 90 us; plain epilogues 4-10% slower
  // with eight warps)
  const bool gelu = g.epi == EPI_GELU || g.epi == EPI_GELU_BWD;
  if (wide && pair) e = gelu ? launch<256, 5, 2, 8>(g, splits, flags, st) : launch<256, 6, 2, 4>(g, splits, flags, st);
  else if (wide) e = launch<256, 4, 1, 4>(g, 1, flags, st);
  else e = pair ? launch<128, 8, 2, 4>(g, splits, flags, st) : launch<128, 6, 1, 4>(g, 1, flags, st);
  if (e != cudaSuccess || splits == 1) return e;
  gpt2_count_launches(1);
  const long long nv = (long long)g.M * (g.N / 4);
  const unsigned grid = (unsigned)std::min<long long>((nv + 255) / 256, (long long)sms * 8);
  launch_k(splitk_reduce_kernel, dim3(grid), dim3(256), 0, st, (float*)g.D, g.ldd, g.ws, g.M, g.N, splits - 1);
  return cudaGetLastError();
}
