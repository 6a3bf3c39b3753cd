// Causal multi-head attention on the sm_103a tensor cores (bf16, head size
// 64, T a multiple of 128): a flash-style forward that keeps the score
// matrix on chip and saves only the per-row log-sum-exp, and a backward that
// recomputes the probabilities from that LSE.  The mathematics is the
// attention layer of "llm.c: GPT-2 training in plain C, with every gradient
// written by hand", §2 How the code works: scores q.k/sqrt(hd) over keys
// t2 <= t, softmax, weighted sum of values; backward
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(dO * O)),
//   dQ = dS K / sqrt(hd),  dK = dS^T Q / sqrt(hd).
// The tiling replaces the page's T x T score buffers ("preatt", "att"):
// nothing of size T x T ever reaches HBM.
//
// Layout: qkv [B*T][3C] (columns Q | K | V, head h at h*64..h*64+63 of
// each), out / dout [B*T][C], lse and D [B][H][T] fp32.  Every 128 x 64
// tile is one TMA box with 128-byte swizzle; P, dS (bf16) are written by
// the softmax warps into shared memory in the same swizzled layout and fed
// to tcgen05.mma as the A operand.  Accumulators live in TMEM.
//
// Forward (one CTA per pair of 128-row query tiles of one (b, h), 320
// threads): warp 0 issues TMA (both Q tiles once, then K/V tiles through a
// ring), one thread of warp 1 issues S = Q K^T and O_j = P V (M=128, K=16
// per instruction), warps 2-5 run the online softmax of query tile 0 and
// warps 6-9 that of tile 1, one query row per thread.  The two tiles share
// every K/V tile, and their softmax phases interleave on the tensor core.
// Each softmax warp reads its 128 scores with four TMEM loads and one wait,
// then releases the S accumulator at once, so the next Q K^T runs while it
// computes the exponentials; P is double-buffered, and O accumulates in TMEM
// (rescaled in place only when a row's maximum jumps by more than 2^8).
//
// Backward: two kernels, so that no gradient is accumulated with atomics
// (the result is deterministic).  The dQ kernel walks the key tiles of one
// query tile (S, dP, then dQ += dS K in TMEM) and also writes
// D = rowsum(dO * O); the dK/dV kernel then walks the query tiles of one key
// tile (S^T, dP^T, then dV += P^T dO and dK += dS^T Q in TMEM).  Eight
// elementwise warps split each 128-wide row of S into two halves.
//
// Every mbarrier wait is bounded; on expiry the CTA raises FLAG_TIMEOUT,
// stops, frees its TMEM and returns.
#include "kernels.cuh"
#include "tc_common.cuh"

extern void gpt2_count_launches(int n);

namespace {

using namespace tc;

constexpr int HD = 64;                       // head size handled here
constexpr uint32_t TILE = 128 * HD * 2;      // one 128 x 64 bf16 tile: 16 KB
constexpr uint32_t PTILE = 2 * TILE;         // one 128 x 128 bf16 tile (two 64-wide halves)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// K-major operand: 128-byte rows, 8-row groups 1024 B apart; a 16-wide k
// step advances 32 B inside the swizzled row
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk) { return sdesc(base + kk * 32, 16, 1024); }
// K-major 128 x 128 operand stored as two 64-wide halves 16 KB apart
__device__ __forceinline__ uint64_t desc_k128(uint32_t base, int kk) {
  return sdesc(base + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024);
}
// MN-major operand (the 64-wide MN extent in one 128-byte row, k along
// rows): a 16-wide k step is 16 rows = 2048 B
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int kk) { return sdesc(base + kk * 2048, 8192, 1024); }

// write 32 consecutive columns [c0, c0+32) (c0 % 32 == 0) of row r of a
// 128-wide bf16 operand tile
__device__ __forceinline__ void store_row32(uint32_t tile, uint32_t r, int c0, const float (&v)[32]) {
  const uint32_t half = tile + (uint32_t)(c0 >> 6) * TILE;
  const uint32_t ch0 = (uint32_t)(c0 & 63) >> 3;  // first 16-byte chunk
#pragma unroll
  for (int u = 0; u < 4; u++)
    st_shared_v4(half + swz(r, ch0 + u), pack_bf16(v[8 * u], v[8 * u + 1]), pack_bf16(v[8 * u + 2], v[8 * u + 3]),
                 pack_bf16(v[8 * u + 4], v[8 * u + 5]), pack_bf16(v[8 * u + 6], v[8 * u + 7]));
}

// 32 fp32 values -> 64 bytes of bf16 at a global address
__device__ __forceinline__ void store_global32(bf16* dst, const float (&v)[32], float mul) {
#pragma unroll
  for (int u = 0; u < 4; u++) {
    uint4 w;
    w.x = pack_bf16(v[8 * u] * mul, v[8 * u + 1] * mul);
    w.y = pack_bf16(v[8 * u + 2] * mul, v[8 * u + 3] * mul);
    w.z = pack_bf16(v[8 * u + 4] * mul, v[8 * u + 5] * mul);
    w.w = pack_bf16(v[8 * u + 6] * mul, v[8 * u + 7] * mul);
    reinterpret_cast<uint4*>(dst)[u] = w;
  }
}

struct AttnParams {
  bf16* out;          // forward: [B*T][C];  backward: dqkv [B*T][3C]
  float* lse;         // [B][H][T]
  float* D;           // backward: [B][H][T]
  const bf16* o;      // backward: forward output [B*T][C]
  const bf16* dout;   // backward: [B*T][C]
  int B, T, C, H;
  float sl2;          // softmax scale * log2(e)
  float scale;        // softmax scale
  int* flags;
};

// ============================================================================
// forward
// ============================================================================
// 32 lanes x 32 consecutive fp32 columns into TMEM (the inverse of tmem_ld32)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
      "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
      "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
// 32 lanes x 128 consecutive fp32 columns, four loads in flight, one wait
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
#pragma unroll
  for (int c = 0; c < 4; c++) tmem_ld32_async(taddr + 32 * c, *reinterpret_cast<float(*)[32]>(v + 32 * c));
  tmem_wait_ld();
}

// Online softmax with a lazily rescaled accumulator: the probabilities of a
// row are taken against a reference max m_ref; O (in TMEM) and the row sum l
// are only rescaled when a new block's max exceeds m_ref by more than
// RESCALE_LOG2 (then P stays <= 2^RESCALE_LOG2, harmless in fp32 and bf16).
// The result is the same softmax: every term and l share one reference.
constexpr float RESCALE_LOG2 = 8.f;
constexpr int FWD_STAGES = 2;
constexpr uint32_t FWD_KV = 2 * TILE;  // K tile then V tile
constexpr size_t FWD_SMEM = 1024 + 2 * TILE + FWD_STAGES * FWD_KV + 4 * PTILE + 256;

__global__ void __launch_bounds__(320, 1) attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tqkv, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sQ = smem_u32(smem);                  // 2 query tiles
  const uint32_t sKV = sQ + 2 * TILE;                  // ring of K/V tiles
  const uint32_t sP = sKV + FWD_STAGES * FWD_KV;       // P tiles [query tile][buffer] (128 x 128)
  uint64_t* bars = (uint64_t*)(smem + 2 * TILE + FWD_STAGES * FWD_KV + 4 * PTILE);
  const uint32_t b_q = smem_u32(bars);
  const uint32_t b_kvfull = b_q + 8, b_kvempty = b_kvfull + 8 * FWD_STAGES;
  const uint32_t b_sfull = b_kvempty + 8 * FWD_STAGES;  // [2] S of tile t computed
  const uint32_t b_sfree = b_sfull + 16;                // [2] S of tile t read by its softmax warps
  const uint32_t b_pfull = b_sfree + 16;                // [2 tiles][2 buffers] P written
  const uint32_t b_pempty = b_pfull + 32;               // [2 tiles][2 buffers] P V done with it
  uint32_t* tmem_holder = (uint32_t*)(bars + 1 + 2 * FWD_STAGES + 12);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, npair = (nq + 1) / 2;
  const int BH = p.B * p.H;
  // heaviest pairs (most key tiles) first
  const int pr = npair - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH), b = bh / p.H, h = bh % p.H;
  const int qt0 = 2 * pr;
  const bool two = qt0 + 1 < nq;         // does query tile 1 exist
  const int nkv = two ? qt0 + 2 : qt0 + 1;
  const int row0 = b * p.T;              // first row of this sequence in qkv

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < FWD_STAGES; s++) {
      mbar_init(b_kvfull + 8 * s, 1);
      mbar_init(b_kvempty + 8 * s, 1);
    }
    for (int t = 0; t < 2; t++) {
      mbar_init(b_sfull + 8 * t, 1);
      mbar_init(b_sfree + 8 * t, 4);
      for (int u = 0; u < 2; u++) {
        mbar_init(b_pfull + 16 * t + 8 * u, 4);
        mbar_init(b_pempty + 16 * t + 8 * u, 1);
      }
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
  if (warp == 0 && lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tqkv) : "memory");
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  // TMEM columns: S of tile t at 128 t, O of tile t at 256 + 64 t

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      mbar_expect_tx(b_q, (two ? 2 : 1) * TILE);
      tma_load_2d(sQ, &tqkv, h * HD, row0 + qt0 * 128, b_q);
      if (two) tma_load_2d(sQ + TILE, &tqkv, h * HD, row0 + qt0 * 128 + 128, b_q);
      for (int j = 0; j < nkv; j++) {
        const uint32_t s = j % FWD_STAGES, ph = (j / FWD_STAGES) & 1;
        if (!mbar_wait(b_kvempty + 8 * s, ph ^ 1, abort_flag)) break;
        const uint32_t dst = sKV + s * FWD_KV, fb = b_kvfull + 8 * s;
        mbar_expect_tx(fb, FWD_KV);
        tma_load_2d(dst, &tqkv, p.C + h * HD, row0 + j * 128, fb);
        tma_load_2d(dst + TILE, &tqkv, 2 * p.C + h * HD, row0 + j * 128, fb);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);  // S = Q K^T
      constexpr uint32_t ID_O = idesc_bf16(128, HD, 0, 1);   // O += P V (V is MN-major)
      auto active = [&](int t, int j) { return t == 0 ? j <= qt0 : (two && j <= qt0 + 1); };
      int kv_ready = -1;
      auto wait_kv = [&](int j) {
        if (kv_ready >= j) return true;
        if (!mbar_wait(b_kvfull + 8 * (j % FWD_STAGES), (j / FWD_STAGES) & 1, abort_flag)) return false;
        kv_ready = j;
        fence_after();
        return true;
      };
      auto issue_s = [&](int t, int j) {
        const uint32_t k = sKV + (j % FWD_STAGES) * FWD_KV, q = sQ + t * TILE;
#pragma unroll
        for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem + 128 * t, desc_k(q, kk), desc_k(k, kk), ID_S, kk > 0);
        mma_commit(b_sfull + 8 * t);
      };
      bool ok = mbar_wait(b_q, 0, abort_flag) && wait_kv(0);
      if (ok) {
        fence_after();
        issue_s(0, 0);
        if (active(1, 0)) issue_s(1, 0);
      }
      for (int j = 0; ok && j < nkv; j++) {
        // next scores first: S of tile t is free as soon as its softmax warps have read it
        for (int t = 0; t < 2 && ok; t++) {
          if (j + 1 >= nkv || !active(t, j + 1)) continue;
          if (!mbar_wait(b_sfree + 8 * t, j & 1, abort_flag) || !wait_kv(j + 1)) { ok = false; break; }
          fence_after();
          issue_s(t, j + 1);
        }
        const uint32_t v = sKV + (j % FWD_STAGES) * FWD_KV + TILE;
        for (int t = 0; t < 2 && ok; t++) {
          if (!active(t, j)) continue;
          const uint32_t pb = b_pfull + 16 * t + 8 * (j & 1);
          if (!mbar_wait(pb, (j >> 1) & 1, abort_flag)) { ok = false; break; }
          fence_after();
          const uint32_t pt = sP + (2 * t + (j & 1)) * PTILE;
#pragma unroll
          for (int kk = 0; kk < 128 / 16; kk++)
            mma_bf16(tmem + 256 + HD * t, desc_k128(pt, kk), desc_mn(v, kk), ID_O, (j | kk) > 0);
          mma_commit(b_pempty + 16 * t + 8 * (j & 1));
        }
        if (ok) mma_commit(b_kvempty + 8 * (j % FWD_STAGES));
      }
    }
  } else {  // ---- softmax warps: tile t, TMEM lane quarter q, one query row per thread
    const int t = (warp - 2) >> 2, q = warp & 3;
    const int qt = qt0 + t;
    if (qt < nq) {
      const uint32_t r = q * 32 + lane;             // row inside the tile
      const uint32_t lrow = (uint32_t)(q * 32) << 16;
      const uint32_t tS = tmem + lrow + 128 * t, tO = tmem + lrow + 256 + HD * t;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j <= qt; j++) {
        if (!mbar_wait_warp(b_sfull + 8 * t, j & 1, abort_flag)) { ok = false; break; }
        fence_after();
        float sv[128];
        tmem_ld128(tS, sv);
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sfree + 8 * t);  // the MMA may overwrite S now
        const bool diag = j == qt;
        float mx = -INFINITY;
        if (diag) {
#pragma unroll
          for (int i = 0; i < 128; i++)
            if (i <= (int)r) mx = fmaxf(mx, sv[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 128; i++) mx = fmaxf(mx, sv[i]);
        }
        mx *= p.sl2;
        // move the reference when this block's max runs too far above it; O and
        // l are rescaled below, once the probabilities no longer need registers
        const bool need = j > 0 && mx > m_ref + RESCALE_LOG2;
        const float m_old = j == 0 ? mx : m_ref;
        if (j == 0 || need) m_ref = mx;
        // P buffer (j & 1) is free once the P V of block j-2 is done
        const uint32_t pt = sP + (2 * t + (j & 1)) * PTILE;
        if (j >= 2 && !mbar_wait_warp(b_pempty + 16 * t + 8 * (j & 1), ((j - 2) >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 4; c++) {
          float(&pv)[32] = *reinterpret_cast<float(*)[32]>(sv + 32 * c);  // probabilities overwrite the scores
#pragma unroll
          for (int i = 0; i < 32; i++) {
            float e = ex2(fmaf(pv[i], p.sl2, -m_ref));
            if (diag && 32 * c + i > (int)r) e = 0.f;
            pv[i] = e;
            rs += e;
          }
          store_row32(pt, r, 32 * c, pv);
        }
        if (__any_sync(0xffffffffu, need)) {
          // the previous block's P V must have landed in O before O is rescaled
          if (!mbar_wait_warp(b_pempty + 16 * t + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          fence_after();
          const float alpha = need ? ex2(m_old - m_ref) : 1.f;
#pragma unroll
          for (int c = 0; c < 2; c++) {
            float ov[32];
            tmem_ld32(tO + 32 * c, ov);
#pragma unroll
            for (int i = 0; i < 32; i++) ov[i] *= alpha;
            tmem_st32(tO + 32 * c, ov);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          l *= alpha;
        }
        l += rs;
        fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull + 16 * t + 8 * (j & 1));
      }
      // the last block's P V completes the accumulator
      if (ok && mbar_wait_warp(b_pempty + 16 * t + 8 * (qt & 1), (qt >> 1) & 1, abort_flag)) {
        fence_after();
        const float inv = 1.f / l;
        bf16* dst = p.out + (size_t)(row0 + qt * 128 + r) * p.C + h * HD;
#pragma unroll
        for (int c = 0; c < 2; c++) {
          float v[32];
          tmem_ld32(tO + 32 * c, v);
          store_global32(dst + 32 * c, v, inv);
        }
        p.lse[((size_t)b * p.H + h) * p.T + qt * 128 + r] = (m_ref + log2f(l)) * LN2;
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.flags, FLAG_TIMEOUT);
}

// ============================================================================
// backward, dQ (+ D = rowsum(dO * O)): one CTA per (b, h, query tile)
// ============================================================================
constexpr int BWD_STAGES = 2;
constexpr uint32_t BWD_KV = 2 * TILE;
constexpr size_t DQ_SMEM = 1024 + 2 * TILE + BWD_STAGES * BWD_KV + PTILE + 256;

__global__ void __launch_bounds__(320, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                          AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sQ = smem_u32(smem), sDO = sQ + TILE;
  const uint32_t sKV = sQ + 2 * TILE;
  const uint32_t sDS = sKV + BWD_STAGES * BWD_KV;
  uint64_t* bars = (uint64_t*)(smem + 2 * TILE + BWD_STAGES * BWD_KV + PTILE);
  const uint32_t b_q = smem_u32(bars);
  const uint32_t b_kvfull = b_q + 8, b_kvempty = b_kvfull + 8 * BWD_STAGES;
  const uint32_t b_sfull = b_kvempty + 8 * BWD_STAGES;  // S and dP in TMEM
  const uint32_t b_sfree = b_sfull + 8;                 // ... read by all 8 warps
  const uint32_t b_dsfull = b_sfree + 8;                // dS tile written
  const uint32_t b_dsfree = b_dsfull + 8;               // dQ MMA done reading dS
  const uint32_t b_dqfull = b_dsfree + 8;
  uint32_t* tmem_holder = (uint32_t*)(bars + 1 + 2 * BWD_STAGES + 5);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, BH = p.B * p.H;
  const int qt = nq - 1 - (int)(blockIdx.x / BH);  // heaviest tiles first
  const int bh = (int)(blockIdx.x % BH), b = bh / p.H, h = bh % p.H;
  const int row0 = b * p.T;
  const int nkv = qt + 1;

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < BWD_STAGES; s++) {
      mbar_init(b_kvfull + 8 * s, 1);
      mbar_init(b_kvempty + 8 * s, 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, 8);
    mbar_init(b_dsfull, 8);
    mbar_init(b_dsfree, 1);
    mbar_init(b_dqfull, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tqkv) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tdo) : "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  // TMEM columns: S at 0, dP at 128, dQ at 256

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(b_q, 2 * TILE);
      tma_load_2d(sQ, &tqkv, h * HD, row0 + qt * 128, b_q);
      tma_load_2d(sDO, &tdo, h * HD, row0 + qt * 128, b_q);
      for (int j = 0; j < nkv; j++) {
        const uint32_t s = j % BWD_STAGES, ph = (j / BWD_STAGES) & 1;
        if (!mbar_wait(b_kvempty + 8 * s, ph ^ 1, abort_flag)) break;
        const uint32_t dst = sKV + s * BWD_KV, fb = b_kvfull + 8 * s;
        mbar_expect_tx(fb, BWD_KV);
        tma_load_2d(dst, &tqkv, p.C + h * HD, row0 + j * 128, fb);
        tma_load_2d(dst + TILE, &tqkv, 2 * p.C + h * HD, row0 + j * 128, fb);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);   // S = Q K^T, dP = dO V^T
      constexpr uint32_t ID_DQ = idesc_bf16(128, HD, 0, 1);   // dQ += dS K (K is MN-major here)
      auto issue_dq = [&](int j) {
        if (!mbar_wait(b_dsfull, j & 1, abort_flag)) return false;
        fence_after();
        const uint32_t k = sKV + (j % BWD_STAGES) * BWD_KV;
#pragma unroll
        for (int kk = 0; kk < 128 / 16; kk++) mma_bf16(tmem + 256, desc_k128(sDS, kk), desc_mn(k, kk), ID_DQ, (j | kk) > 0);
        mma_commit(b_dsfree);
        mma_commit(b_kvempty + 8 * (j % BWD_STAGES));
        return true;
      };
      bool ok = mbar_wait(b_q, 0, abort_flag);
      for (int j = 0; ok && j < nkv; j++) {
        const uint32_t s = j % BWD_STAGES;
        if (!mbar_wait(b_kvfull + 8 * s, (j / BWD_STAGES) & 1, abort_flag)) { ok = false; break; }
        if (j > 0 && !mbar_wait(b_sfree, (j - 1) & 1, abort_flag)) { ok = false; break; }
        fence_after();
        const uint32_t k = sKV + s * BWD_KV, v = k + TILE;
#pragma unroll
        for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem, desc_k(sQ, kk), desc_k(k, kk), ID_S, kk > 0);
#pragma unroll
        for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem + 128, desc_k(sDO, kk), desc_k(v, kk), ID_S, kk > 0);
        mma_commit(b_sfull);
        if (j > 0 && !issue_dq(j - 1)) { ok = false; break; }
      }
      if (ok && issue_dq(nkv - 1)) mma_commit(b_dqfull);
    }
  } else {  // ---- elementwise warps: lane quarter q, column half hf
    const int q = warp & 3, hf = (warp - 2) >> 2;
    const uint32_t r = q * 32 + lane;
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    const int tq = qt * 128 + r;                     // query position in the sequence
    const size_t grow = (size_t)(row0 + tq);
    const size_t sidx = ((size_t)b * p.H + h) * p.T + tq;
    // D = rowsum(dO * O) for this row (both halves compute it, half 0 stores it)
    float Dr = 0.f;
    {
      const bf16* dor = p.dout + grow * p.C + h * HD;
      const bf16* orow = p.o + grow * p.C + h * HD;
#pragma unroll
      for (int u = 0; u < HD / 8; u++) {
        float a[8], c[8];
        ld16(dor + 8 * u, a);
        ld16(orow + 8 * u, c);
#pragma unroll
        for (int i = 0; i < 8; i++) Dr = fmaf(a[i], c[i], Dr);
      }
      if (hf == 0) p.D[sidx] = Dr;
    }
    const float lse2 = p.lse[sidx] * LOG2E;
    bool ok = true;
    for (int j = 0; j < nkv; j++) {
      if (!mbar_wait_warp(b_sfull, j & 1, abort_flag)) { ok = false; break; }
      fence_after();
      float s[2][32], dp[2][32];
#pragma unroll
      for (int c = 0; c < 2; c++) {
        tmem_ld32_async(tmem + lrow + hf * 64 + 32 * c, s[c]);
        tmem_ld32_async(tmem + lrow + 128 + hf * 64 + 32 * c, dp[c]);
      }
      tmem_wait_ld();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sfree);
      const bool diag = j == qt;
#pragma unroll
      for (int c = 0; c < 2; c++) {
#pragma unroll
        for (int i = 0; i < 32; i++) {
          const int col = hf * 64 + 32 * c + i;
          float pv = ex2(fmaf(s[c][i], p.sl2, -lse2));
          if (diag && col > (int)r) pv = 0.f;
          s[c][i] = pv * (dp[c][i] - Dr);
        }
      }
      // the dS tile is free once the previous dQ MMA has read it
      if (j > 0 && !mbar_wait_warp(b_dsfree, (j - 1) & 1, abort_flag)) { ok = false; break; }
#pragma unroll
      for (int c = 0; c < 2; c++) store_row32(sDS, r, hf * 64 + 32 * c, s[c]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_dsfull);
    }
    if (ok && mbar_wait_warp(b_dqfull, 0, abort_flag)) {
      fence_after();
      float v[32];
      tmem_ld32(tmem + lrow + 256 + 32 * hf, v);
      store_global32(p.out + grow * 3 * p.C + h * HD + 32 * hf, v, p.scale);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.flags, FLAG_TIMEOUT);
}

// ============================================================================
// backward, dK and dV: one CTA per (b, h, key tile); needs D from the dQ kernel
// ============================================================================
constexpr uint32_t BWD_QD = 2 * TILE + 1024;  // Q tile, dO tile, lse[128], D[128]
constexpr size_t DKV_SMEM = 1024 + 2 * TILE + BWD_STAGES * BWD_QD + 2 * PTILE + 256;

__global__ void __launch_bounds__(320, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                           AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sK = smem_u32(smem), sV = sK + TILE;
  const uint32_t sQD = sK + 2 * TILE;                 // ring: Q, dO, lse, D
  const uint32_t sPT = sQD + BWD_STAGES * BWD_QD;     // P^T tile
  const uint32_t sDST = sPT + PTILE;                  // dS^T tile
  const uint8_t* ring_gen = smem + 2 * TILE;          // generic view of the ring
  uint64_t* bars = (uint64_t*)(smem + 2 * TILE + BWD_STAGES * BWD_QD + 2 * PTILE);
  const uint32_t b_kv = smem_u32(bars);
  const uint32_t b_qfull = b_kv + 8, b_qempty = b_qfull + 8 * BWD_STAGES;
  const uint32_t b_sfull = b_qempty + 8 * BWD_STAGES;
  const uint32_t b_sfree = b_sfull + 8;
  const uint32_t b_pfull = b_sfree + 8;   // P^T and dS^T written
  const uint32_t b_pfree = b_pfull + 8;   // dV/dK MMAs done reading them
  const uint32_t b_accfull = b_pfree + 8;
  uint32_t* tmem_holder = (uint32_t*)(bars + 1 + 2 * BWD_STAGES + 5);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, BH = p.B * p.H;
  const int kt = (int)(blockIdx.x / BH);  // key tile; small kt = more query tiles = heavier, first
  const int bh = (int)(blockIdx.x % BH), b = bh / p.H, h = bh % p.H;
  const int row0 = b * p.T;
  const int nit = nq - kt;                // query tiles kt .. nq-1
  const size_t sbase = ((size_t)b * p.H + h) * p.T;

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int s = 0; s < BWD_STAGES; s++) {
      mbar_init(b_qfull + 8 * s, 1);
      mbar_init(b_qempty + 8 * s, 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, 8);
    mbar_init(b_pfull, 8);
    mbar_init(b_pfree, 1);
    mbar_init(b_accfull, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tqkv) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tdo) : "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  // TMEM columns: S^T at 0, dP^T at 128, dV at 256, dK at 320

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(b_kv, 2 * TILE);
      tma_load_2d(sK, &tqkv, p.C + h * HD, row0 + kt * 128, b_kv);
      tma_load_2d(sV, &tqkv, 2 * p.C + h * HD, row0 + kt * 128, b_kv);
      for (int it = 0; it < nit; it++) {
        const int qt = kt + it;
        const uint32_t s = it % BWD_STAGES, ph = (it / BWD_STAGES) & 1;
        if (!mbar_wait(b_qempty + 8 * s, ph ^ 1, abort_flag)) break;
        const uint32_t dst = sQD + s * BWD_QD, fb = b_qfull + 8 * s;
        mbar_expect_tx(fb, BWD_QD);
        tma_load_2d(dst, &tqkv, h * HD, row0 + qt * 128, fb);
        tma_load_2d(dst + TILE, &tdo, h * HD, row0 + qt * 128, fb);
        bulk_load(dst + 2 * TILE, p.lse + sbase + qt * 128, 512, fb);
        bulk_load(dst + 2 * TILE + 512, p.D + sbase + qt * 128, 512, fb);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);  // S^T = K Q^T, dP^T = V dO^T
      constexpr uint32_t ID_G = idesc_bf16(128, HD, 0, 1);   // dV += P^T dO, dK += dS^T Q
      auto issue_grad = [&](int it) {
        if (!mbar_wait(b_pfull, it & 1, abort_flag)) return false;
        fence_after();
        const uint32_t qd = sQD + (it % BWD_STAGES) * BWD_QD;
#pragma unroll
        for (int kk = 0; kk < 128 / 16; kk++) {
          mma_bf16(tmem + 256, desc_k128(sPT, kk), desc_mn(qd + TILE, kk), ID_G, (it | kk) > 0);
          mma_bf16(tmem + 320, desc_k128(sDST, kk), desc_mn(qd, kk), ID_G, (it | kk) > 0);
        }
        mma_commit(b_pfree);
        mma_commit(b_qempty + 8 * (it % BWD_STAGES));
        return true;
      };
      bool ok = mbar_wait(b_kv, 0, abort_flag);
      for (int it = 0; ok && it < nit; it++) {
        const uint32_t s = it % BWD_STAGES;
        if (!mbar_wait(b_qfull + 8 * s, (it / BWD_STAGES) & 1, abort_flag)) { ok = false; break; }
        if (it > 0 && !mbar_wait(b_sfree, (it - 1) & 1, abort_flag)) { ok = false; break; }
        fence_after();
        const uint32_t qd = sQD + s * BWD_QD;
#pragma unroll
        for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem, desc_k(sK, kk), desc_k(qd, kk), ID_S, kk > 0);
#pragma unroll
        for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem + 128, desc_k(sV, kk), desc_k(qd + TILE, kk), ID_S, kk > 0);
        mma_commit(b_sfull);
        if (it > 0 && !issue_grad(it - 1)) { ok = false; break; }
      }
      if (ok && issue_grad(nit - 1)) mma_commit(b_accfull);
    }
  } else {  // ---- elementwise warps: key row r (lane quarter q), query-column half hf
    const int q = warp & 3, hf = (warp - 2) >> 2;
    const uint32_t r = q * 32 + lane;
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    bool ok = true;
    for (int it = 0; it < nit; it++) {
      if (!mbar_wait_warp(b_sfull, it & 1, abort_flag)) { ok = false; break; }
      fence_after();
      float s[2][32], dp[2][32];
#pragma unroll
      for (int c = 0; c < 2; c++) {
        tmem_ld32_async(tmem + lrow + hf * 64 + 32 * c, s[c]);
        tmem_ld32_async(tmem + lrow + 128 + hf * 64 + 32 * c, dp[c]);
      }
      tmem_wait_ld();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sfree);
      // lse and D of this stage's 128 queries (loaded with the Q tile)
      const float* lq = (const float*)(ring_gen + (it % BWD_STAGES) * BWD_QD + 2 * TILE);
      const float* dq = lq + 128;
      const bool diag = it == 0;  // query tile == key tile
#pragma unroll
      for (int c = 0; c < 2; c++) {
#pragma unroll
        for (int i = 0; i < 32; i++) {
          const int col = hf * 64 + 32 * c + i;  // query row inside the tile
          float pv = ex2(fmaf(s[c][i], p.sl2, -lq[col] * LOG2E));
          if (diag && (int)r > col) pv = 0.f;
          s[c][i] = pv;
          dp[c][i] = pv * (dp[c][i] - dq[col]);
        }
      }
      if (it > 0 && !mbar_wait_warp(b_pfree, (it - 1) & 1, abort_flag)) { ok = false; break; }
#pragma unroll
      for (int c = 0; c < 2; c++) {
        store_row32(sPT, r, hf * 64 + 32 * c, s[c]);
        store_row32(sDST, r, hf * 64 + 32 * c, dp[c]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull);
    }
    if (ok && mbar_wait_warp(b_accfull, 0, abort_flag)) {
      fence_after();
      float v[32];
      const size_t grow = (size_t)(row0 + kt * 128 + r);
      tmem_ld32(tmem + lrow + 256 + 32 * hf, v);
      store_global32(p.out + grow * 3 * p.C + 2 * p.C + h * HD + 32 * hf, v, 1.f);
      tmem_ld32(tmem + lrow + 320 + 32 * hf, v);
      store_global32(p.out + grow * 3 * p.C + p.C + h * HD + 32 * hf, v, p.scale);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.flags, FLAG_TIMEOUT);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

bool attention_tc_supported(int B, int T, int C, int H) {
  if (B <= 0 || T <= 0 || H <= 0 || C % H || C / H != HD || T % 128) return false;
  if ((long long)B * H * (T / 128) > 0x7fffffffLL) return false;
  return tc_available();
}

cudaError_t attention_forward_tc(bf16* out, float* lse, const bf16* qkv, int B, int T, int C, int H, int* flags,
                                 cudaStream_t st) {
  if (!attention_tc_supported(B, T, C, H) || !flags) return cudaErrorNotSupported;
  if (((uintptr_t)qkv & 15) || ((uintptr_t)out & 15)) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(attn_fwd_tc_kernel, FWD_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap tq;
  if (!tc_make_map(&tq, qkv, 3 * (uint64_t)C, (uint64_t)B * T, 3 * (uint64_t)C, HD, 128)) return cudaErrorInvalidValue;
  AttnParams p{out, lse, nullptr, nullptr, nullptr, B, T, C, H, LOG2E / sqrtf((float)HD), 1.f / sqrtf((float)HD), flags};
  const int npair = (T / 128 + 1) / 2;
  gpt2_count_launches(1);
  attn_fwd_tc_kernel<<<(unsigned)(B * H * npair), 320, FWD_SMEM, st>>>(tq, p);
  return cudaGetLastError();
}

cudaError_t attention_backward_tc(bf16* dqkv, float* Dbuf, const bf16* dout, const bf16* qkv, const bf16* out,
                                  const float* lse, int B, int T, int C, int H, int* flags, cudaStream_t st) {
  if (!attention_tc_supported(B, T, C, H) || !flags) return cudaErrorNotSupported;
  if (((uintptr_t)qkv & 15) || ((uintptr_t)out & 15) || ((uintptr_t)dout & 15) || ((uintptr_t)dqkv & 15) ||
      ((uintptr_t)lse & 15) || ((uintptr_t)Dbuf & 15))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(attn_bwd_dq_tc_kernel, DQ_SMEM);
    if (e == cudaSuccess) e = set_smem(attn_bwd_dkv_tc_kernel, DKV_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap tq, td;
  if (!tc_make_map(&tq, qkv, 3 * (uint64_t)C, (uint64_t)B * T, 3 * (uint64_t)C, HD, 128) ||
      !tc_make_map(&td, dout, (uint64_t)C, (uint64_t)B * T, (uint64_t)C, HD, 128))
    return cudaErrorInvalidValue;
  AttnParams p{dqkv, const_cast<float*>(lse), Dbuf, out, dout, B, T, C, H, LOG2E / sqrtf((float)HD),
               1.f / sqrtf((float)HD), flags};
  const unsigned grid = (unsigned)(B * H * (T / 128));
  gpt2_count_launches(2);
  attn_bwd_dq_tc_kernel<<<grid, 320, DQ_SMEM, st>>>(tq, td, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_dkv_tc_kernel<<<grid, 320, DKV_SMEM, st>>>(tq, td, p);
  return cudaGetLastError();
}
