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
// Forward (persistent: one CTA per SM walks the work items, an item being a
// pair of 128-row query tiles of one (b, h); 576 threads): warp 0 issues TMA
// (both Q tiles once, then K/V tiles through a ring), one thread of warp 1
// issues S = Q K^T and O += P V (M=128, K=16 per instruction), warps 2-9 run
// the online softmax of query tile 0 and warps 10-17 that of tile 1: two
// warps share each row, one per 64-column half, and combine row maxima and
// sums through shared memory.  The two tiles share
// every K/V tile, and their softmax phases interleave on the tensor core.
// Each softmax warp reads its 128 scores with four TMEM loads and one wait,
// then releases the S accumulator at once, so the next Q K^T runs while it
// computes the exponentials; O accumulates in TMEM
// (rescaled in place only when a row's maximum jumps by more than 2^8).
//
// Backward: two persistent kernels, so that no gradient is accumulated with
// atomics (the result is deterministic).  The dQ kernel walks the key tiles of one
// query tile (S, dP, then dQ += dS K in TMEM) and also writes
// D = rowsum(dO * O); the dK/dV kernel then walks the query tiles of one key
// tile (S^T, dP^T, then dV += P^T dO and dK += dS^T Q in TMEM).  The
// elementwise warps (EW_WARPS, a multiple of four: one per TMEM lane quarter
// and column group) split each 128-wide row of S into column groups.
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

// 2^x on the FMA pipe, for x >= -126 (clamped below), relative error < 1.1e-4:
// n = round(x) from the 1.5*2^23 shift, 2^(x-n) by a cubic in f = x - n on
// [-0.5, 0.5] (coefficients from a relative-error-weighted least-squares fit
// of 2^f with p(0) = 1), and 2^n added into the exponent field.  Used for a
// quarter of the exponentials so that the MUFU unit, which does the rest,
// is not the only pipe busy; P is rounded to bf16 (2^-8) afterwards anyway.
__device__ __forceinline__ float exp2_poly(float x) {
  x = fmaxf(x, -126.f);
  const float t = x + 12582912.f;
  const float f = x - (t - 12582912.f);
  const float q = fmaf(fmaf(fmaf(0.0550089069f, f, 0.242210984f), f, 0.693282962f), f, 1.f);
  return __int_as_float(__float_as_int(q) + (__float_as_int(t) << 23));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
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
constexpr int FWD_STAGES = 3;
constexpr uint32_t FWD_KV = 2 * TILE;  // K tile then V tile
constexpr size_t FWD_SMEM = 1024 + 2 * TILE + FWD_STAGES * FWD_KV + 2 * PTILE + 256 + (2 * 2 * 2 + 2 * 2) * 128 * 4;
constexpr int FWD_THREADS = 64 + 32 * 16;  // producer, MMA, 16 softmax warps

// Persistent: each CTA takes work items blockIdx.x, blockIdx.x + gridDim.x, ...
// (item = one pair of query tiles of one (b, h), heaviest first).  Every
// barrier phase is tracked by a running counter across items, so the next
// item's Q load, first Q K^T and K/V loads overlap the tail of the current one.
__global__ void __launch_bounds__(FWD_THREADS, 1) attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tqkv, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sQ = smem_u32(smem);                  // 2 query tiles
  const uint32_t sKV = sQ + 2 * TILE;                  // ring of K/V tiles
  const uint32_t sP = sKV + FWD_STAGES * FWD_KV;       // P tile of each query tile (128 x 128)
  uint64_t* bars = (uint64_t*)(smem + 2 * TILE + FWD_STAGES * FWD_KV + 2 * PTILE);
  const uint32_t b_qfull = smem_u32(bars), b_qempty = b_qfull + 8;
  const uint32_t b_kvfull = b_qempty + 8, b_kvempty = b_kvfull + 8 * FWD_STAGES;
  const uint32_t b_sfull = b_kvempty + 8 * FWD_STAGES;  // [2] S of tile t computed
  const uint32_t b_sfree = b_sfull + 16;                // [2] S of tile t read by its softmax warps
  const uint32_t b_pfull = b_sfree + 16;                // [2] P of tile t written
  const uint32_t b_pempty = b_pfull + 16;               // [2] P V of tile t done with it (O updated)
  const uint32_t b_ofree = b_pempty + 16;               // [2] finished O of tile t read out
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 + 2 * FWD_STAGES + 10);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);
  // row statistics exchanged between the two warps that share a row:
  // red[block parity][tile][half][row] (maxima), then lsum[tile][half][row]
  float* red = (float*)(smem + 2 * TILE + FWD_STAGES * FWD_KV + 2 * PTILE + 256);
  float* lsum = red + 2 * 2 * 2 * 128;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, npair = (nq + 1) / 2;
  const int BH = p.B * p.H;
  const int n_items = BH * npair;
  struct Item { int qt0, nkv, b, h, row0; bool two; };
  auto item = [&](int i) {
    Item it;
    const int pr = npair - 1 - i / BH;  // heaviest pairs (most key tiles) first
    const int bh = i % BH;
    it.b = bh / p.H;
    it.h = bh % p.H;
    it.qt0 = 2 * pr;
    it.two = it.qt0 + 1 < nq;           // does query tile 1 exist
    it.nkv = it.two ? it.qt0 + 2 : it.qt0 + 1;
    it.row0 = it.b * p.T;               // first row of this sequence in qkv
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    for (int s = 0; s < FWD_STAGES; s++) {
      mbar_init(b_kvfull + 8 * s, 1);
      mbar_init(b_kvempty + 8 * s, 1);
    }
    for (int t = 0; t < 2; t++) {
      mbar_init(b_sfull + 8 * t, 1);
      mbar_init(b_sfree + 8 * t, 8);
      mbar_init(b_ofree + 8 * t, 8);
      mbar_init(b_pfull + 8 * t, 8);
      mbar_init(b_pempty + 8 * t, 1);
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
      uint32_t g = 0, n = 0;  // K/V blocks and items loaded so far
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, n++) {
        const Item it = item(i);
        // the Q tiles are free once the previous item's last Q K^T has completed
        if (!mbar_wait(b_qempty, (n & 1) ^ 1, abort_flag)) break;
        mbar_expect_tx(b_qfull, (it.two ? 2 : 1) * TILE);
        tma_load_2d(sQ, &tqkv, it.h * HD, it.row0 + it.qt0 * 128, b_qfull);
        if (it.two) tma_load_2d(sQ + TILE, &tqkv, it.h * HD, it.row0 + it.qt0 * 128 + 128, b_qfull);
        for (int j = 0; j < it.nkv; j++, g++) {
          const uint32_t s = g % FWD_STAGES, ph = (g / FWD_STAGES) & 1;
          if (!mbar_wait(b_kvempty + 8 * s, ph ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t dst = sKV + s * FWD_KV, fb = b_kvfull + 8 * s;
          mbar_expect_tx(fb, FWD_KV);
          tma_load_2d(dst, &tqkv, p.C + it.h * HD, it.row0 + j * 128, fb);
          tma_load_2d(dst + TILE, &tqkv, 2 * p.C + it.h * HD, it.row0 + j * 128, fb);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);  // S = Q K^T
      constexpr uint32_t ID_O = idesc_bf16(128, HD, 0, 1);   // O += P V (V is MN-major)
      uint32_t g0 = 0, n = 0;                 // K/V blocks before this item, items so far
      uint32_t nS[2] = {0, 0}, nP[2] = {0, 0}, nO[2] = {0, 0};  // per tile: S issued, P V issued, items
      int kv_ready = -1;                      // highest K/V block known loaded (global index)
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, n++) {
        const Item it = item(i);
        auto active = [&](int t, int j) { return t == 0 ? j <= it.qt0 : (it.two && j <= it.qt0 + 1); };
        auto wait_kv = [&](int j) {
          const int gj = (int)g0 + j;
          if (kv_ready >= gj) return true;
          if (!mbar_wait(b_kvfull + 8 * (gj % FWD_STAGES), (gj / FWD_STAGES) & 1, abort_flag)) return false;
          kv_ready = gj;
          fence_after();
          return true;
        };
        // S of tile t for block j; S of the tile must have been read out first
        auto issue_s = [&](int t, int j) {
          if (nS[t] > 0 && !mbar_wait(b_sfree + 8 * t, (nS[t] - 1) & 1, abort_flag)) return false;
          if (!wait_kv(j)) return false;
          fence_after();
          const uint32_t k = sKV + ((g0 + j) % FWD_STAGES) * FWD_KV, q = sQ + t * TILE;
#pragma unroll
          for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem + 128 * t, desc_k(q, kk), desc_k(k, kk), ID_S, kk > 0);
          mma_commit(b_sfull + 8 * t);
          nS[t]++;
          return true;
        };
        if (!mbar_wait(b_qfull, n & 1, abort_flag)) break;
        fence_after();
        ok = issue_s(0, 0) && (!active(1, 0) || issue_s(1, 0));
        if (ok && it.nkv == 1) mma_commit(b_qempty);
        for (int j = 0; ok && j < it.nkv; j++) {
          // next scores first: S of tile t is free as soon as its softmax warps have read it
          for (int t = 0; t < 2 && ok; t++)
            if (j + 1 < it.nkv && active(t, j + 1)) ok = issue_s(t, j + 1);
          if (ok && j + 2 == it.nkv) mma_commit(b_qempty);  // the item's last Q K^T is issued
          const uint32_t v = sKV + ((g0 + j) % FWD_STAGES) * FWD_KV + TILE;
          for (int t = 0; t < 2 && ok; t++) {
            if (!active(t, j)) continue;
            if (!mbar_wait(b_pfull + 8 * t, nP[t] & 1, abort_flag)) { ok = false; break; }
            // the first P V of an item overwrites O: the previous item's O must be read out
            if (j == 0 && nO[t] > 0 && !mbar_wait(b_ofree + 8 * t, (nO[t] - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            fence_after();
            const uint32_t pt = sP + t * PTILE;
#pragma unroll
            for (int kk = 0; kk < 128 / 16; kk++)
              mma_bf16(tmem + 256 + HD * t, desc_k128(pt, kk), desc_mn(v, kk), ID_O, (j | kk) > 0);
            mma_commit(b_pempty + 8 * t);
            nP[t]++;
          }
          if (ok) mma_commit(b_kvempty + 8 * ((g0 + j) % FWD_STAGES));
        }
        for (int t = 0; t < 2; t++)
          if (t == 0 || it.two) nO[t]++;
        g0 += it.nkv;
      }
    }
  } else {  // ---- softmax warps: tile t, TMEM lane quarter q, column half hf; one row per thread pair
    const int wt = warp - 2;
    const int t = wt >> 3, hf = (wt >> 2) & 1, q = warp & 3;
    const uint32_t r = q * 32 + lane;             // row inside the tile
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    const uint32_t tS = tmem + lrow + 128 * t + 64 * hf, tO = tmem + lrow + 256 + HD * t + 32 * hf;
    const int bar_id = 1 + 4 * t + q;             // named barrier of the two warps sharing these rows
    float* my_red = red + (t * 2 + hf) * 128 + r;
    const float* peer_red = red + (t * 2 + (hf ^ 1)) * 128 + r;
    uint32_t nS = 0, nP = 0;                      // S blocks consumed, P blocks produced
    bool ok = true;
    for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
      const Item it = item(i);
      const int qt = it.qt0 + t;
      if (qt >= nq) continue;                     // this item has no tile t
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j <= qt; j++) {
        if (!mbar_wait_warp(b_sfull + 8 * t, nS & 1, abort_flag)) { ok = false; break; }
        fence_after();
        float sv[64];
        tmem_ld32_async(tS, *reinterpret_cast<float(*)[32]>(sv));
        tmem_ld32_async(tS + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
        tmem_wait_ld();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sfree + 8 * t);  // the MMA may overwrite S now
        const int c0 = 64 * hf;                      // first column of this half
        const bool diag = j == qt;
        // row maximum: four independent chains, then the partner half through shared memory
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (!diag) {
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            m4[0] = max3(m4[0], sv[c], sv[c + 1]);
            m4[1] = max3(m4[1], sv[c + 2], sv[c + 3]);
            m4[2] = max3(m4[2], sv[c + 4], sv[c + 5]);
            m4[3] = max3(m4[3], sv[c + 6], sv[c + 7]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; c++)
            if (c0 + c <= (int)r) m4[c & 3] = fmaxf(m4[c & 3], sv[c]);
        }
        float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        float* slot = my_red + (nS & 1) * 512;
        *slot = mx;
        asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");
        mx = fmaxf(mx, peer_red[(nS & 1) * 512]) * p.sl2;
        nS++;
        // move the reference when this block's max runs too far above it; O and
        // l are rescaled below, once the probabilities no longer need registers
        const bool need = j > 0 && mx > m_ref + RESCALE_LOG2;
        const float m_old = j == 0 ? mx : m_ref;
        if (j == 0 || need) m_ref = mx;
        // the P tile is free, and O holds every earlier block, once the previous P V is done
        const uint32_t pt = sP + t * PTILE;
        if (nP >= 1 && !mbar_wait_warp(b_pempty + 8 * t, (nP - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        fence_after();
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 2; c++) {
          float(&pv)[32] = *reinterpret_cast<float(*)[32]>(sv + 32 * c);  // probabilities overwrite the scores
#pragma unroll
          for (int e = 0; e < 32; e++) {
            const float x = fmaf(pv[e], p.sl2, -m_ref);
            pv[e] = (e & 3) == 3 ? exp2_poly(x) : ex2(x);
          }
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; e++)
              if (c0 + 32 * c + e > (int)r) pv[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 32; e++) rs4[e & 3] += pv[e];
          store_row32(pt, r, c0 + 32 * c, pv);
        }
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m_old - m_ref) : 1.f;
          float ov[32];
          tmem_ld32(tO, ov);
#pragma unroll
          for (int e = 0; e < 32; e++) ov[e] *= alpha;
          tmem_st32(tO, ov);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          l *= alpha;
        }
        l += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull + 8 * t);
        nP++;
      }
      if (!ok) break;
      // the row sum is split over the two halves
      lsum[(t * 2 + hf) * 128 + r] = l;
      // the item's last P V completes the accumulator
      if (!mbar_wait_warp(b_pempty + 8 * t, (nP - 1) & 1, abort_flag)) break;
      fence_after();
      float o[32];
      tmem_ld32(tO, o);
      fence_before();
      asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");  // both halves stored l and read O
      if (lane == 0) mbar_arrive(b_ofree + 8 * t);  // the next item may overwrite O
      const float lt = l + lsum[(t * 2 + (hf ^ 1)) * 128 + r];
      bf16* dst = p.out + (size_t)(it.row0 + qt * 128 + r) * p.C + it.h * HD + 32 * hf;
      store_global32(dst, o, 1.f / lt);
      if (hf == 0) p.lse[((size_t)it.b * p.H + it.h) * p.T + qt * 128 + r] = (m_ref + log2f(lt)) * LN2;
      // lsum is rewritten by the next item only after both halves pass the next block's barrier
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
// backward, dQ (+ D = rowsum(dO * O)).  Persistent: items are (b, h, query
// tile), heaviest first; per item the key tiles 0..qt stream through a ring.
// ============================================================================
constexpr int DQ_STAGES = 5;             // K/V ring of the dQ kernel
constexpr int DKV_STAGES = 3;            // Q/dO/lse/D ring of the dK/dV kernel
constexpr int EW_WARPS = 8;              // elementwise warps of the backward kernels
constexpr int EW_COLS = 128 / (EW_WARPS / 4);  // columns of S each elementwise warp handles
constexpr int BWD_THREADS = 64 + 32 * EW_WARPS;
constexpr uint32_t BWD_KV = 2 * TILE;
constexpr size_t DQ_SMEM = 1024 + 2 * TILE + DQ_STAGES * BWD_KV + PTILE + 256;

__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                          AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sQ = smem_u32(smem), sDO = sQ + TILE;
  const uint32_t sKV = sQ + 2 * TILE;
  const uint32_t sDS = sKV + DQ_STAGES * BWD_KV;
  uint64_t* bars = (uint64_t*)(smem + 2 * TILE + DQ_STAGES * BWD_KV + PTILE);
  const uint32_t b_qfull = smem_u32(bars), b_qempty = b_qfull + 8;  // Q and dO tiles of an item
  const uint32_t b_kvfull = b_qempty + 8, b_kvempty = b_kvfull + 8 * DQ_STAGES;
  const uint32_t b_sfull = b_kvempty + 8 * DQ_STAGES;  // S and dP in TMEM
  const uint32_t b_sfree = b_sfull + 8;                 // ... read by all 8 warps
  const uint32_t b_dsfull = b_sfree + 8;                // dS tile written
  const uint32_t b_dsfree = b_dsfull + 8;               // dQ MMA done reading dS
  const uint32_t b_dqfull = b_dsfree + 8;               // an item's dQ complete in TMEM
  const uint32_t b_dqfree = b_dqfull + 8;               // ... and read out
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 + 2 * DQ_STAGES + 6);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, BH = p.B * p.H;
  const int n_items = BH * nq;
  struct Item { int qt, b, h, row0; };
  auto item = [&](int i) {
    Item it;
    it.qt = nq - 1 - i / BH;  // heaviest tiles first
    const int bh = i % BH;
    it.b = bh / p.H;
    it.h = bh % p.H;
    it.row0 = it.b * p.T;
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    for (int s = 0; s < DQ_STAGES; s++) {
      mbar_init(b_kvfull + 8 * s, 1);
      mbar_init(b_kvempty + 8 * s, 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, EW_WARPS);
    mbar_init(b_dsfull, EW_WARPS);
    mbar_init(b_dsfree, 1);
    mbar_init(b_dqfull, 1);
    mbar_init(b_dqfree, EW_WARPS);
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
      uint32_t g = 0, n = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, n++) {
        const Item it = item(i);
        if (!mbar_wait(b_qempty, (n & 1) ^ 1, abort_flag)) break;
        mbar_expect_tx(b_qfull, 2 * TILE);
        tma_load_2d(sQ, &tqkv, it.h * HD, it.row0 + it.qt * 128, b_qfull);
        tma_load_2d(sDO, &tdo, it.h * HD, it.row0 + it.qt * 128, b_qfull);
        for (int j = 0; j <= it.qt; j++, g++) {
          const uint32_t s = g % DQ_STAGES, ph = (g / DQ_STAGES) & 1;
          if (!mbar_wait(b_kvempty + 8 * s, ph ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t dst = sKV + s * BWD_KV, fb = b_kvfull + 8 * s;
          mbar_expect_tx(fb, BWD_KV);
          tma_load_2d(dst, &tqkv, p.C + it.h * HD, it.row0 + j * 128, fb);
          tma_load_2d(dst + TILE, &tqkv, 2 * p.C + it.h * HD, it.row0 + j * 128, fb);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);   // S = Q K^T, dP = dO V^T
      constexpr uint32_t ID_DQ = idesc_bf16(128, HD, 0, 1);   // dQ += dS K (K is MN-major here)
      uint32_t g0 = 0, n = 0, nS = 0, nD = 0;
      bool ok = true;
      // dQ += dS_j K_j for the item's block j (global K/V block g0 + j)
      auto issue_dq = [&](int j) {
        if (!mbar_wait(b_dsfull, nD & 1, abort_flag)) return false;
        // the first dQ MMA of an item overwrites dQ: the previous item's must be read out
        if (j == 0 && n > 0 && !mbar_wait(b_dqfree, (n - 1) & 1, abort_flag)) return false;
        fence_after();
        const uint32_t k = sKV + ((g0 + j) % DQ_STAGES) * BWD_KV;
#pragma unroll
        for (int kk = 0; kk < 128 / 16; kk++)
          mma_bf16(tmem + 256, desc_k128(sDS, kk), desc_mn(k, kk), ID_DQ, (j | kk) > 0);
        mma_commit(b_dsfree);
        mma_commit(b_kvempty + 8 * ((g0 + j) % DQ_STAGES));
        nD++;
        return true;
      };
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, n++) {
        const Item it = item(i);
        const int nkv = it.qt + 1;
        if (!mbar_wait(b_qfull, n & 1, abort_flag)) break;
        for (int j = 0; ok && j < nkv; j++) {
          const uint32_t gj = g0 + j, s = gj % DQ_STAGES;
          if (!mbar_wait(b_kvfull + 8 * s, (gj / DQ_STAGES) & 1, abort_flag)) { ok = false; break; }
          if (nS > 0 && !mbar_wait(b_sfree, (nS - 1) & 1, abort_flag)) { ok = false; break; }
          fence_after();
          const uint32_t k = sKV + s * BWD_KV, v = k + TILE;
#pragma unroll
          for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem, desc_k(sQ, kk), desc_k(k, kk), ID_S, kk > 0);
#pragma unroll
          for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem + 128, desc_k(sDO, kk), desc_k(v, kk), ID_S, kk > 0);
          mma_commit(b_sfull);
          nS++;
          if (j == nkv - 1) mma_commit(b_qempty);  // the item's last use of Q and dO is issued
          if (j > 0 && !issue_dq(j - 1)) { ok = false; break; }
        }
        if (ok && issue_dq(nkv - 1)) mma_commit(b_dqfull);
        else ok = false;
        g0 += nkv;
      }
    }
  } else {  // ---- elementwise warps: lane quarter q, column group cq (EW_COLS columns)
    const int q = warp & 3, cq = (warp - 2) >> 2;
    const int c0 = cq * EW_COLS;
    const uint32_t r = q * 32 + lane;
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    uint32_t n = 0, nS = 0, nD = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, n++) {
      const Item it = item(i);
      const int tq = it.qt * 128 + r;                  // query position in the sequence
      const size_t grow = (size_t)(it.row0 + tq);
      const size_t sidx = ((size_t)it.b * p.H + it.h) * p.T + tq;
      // D = rowsum(dO * O) for this row (every column group computes it, group 0 stores it)
      float Dr = 0.f;
      {
        const bf16* dor = p.dout + grow * p.C + it.h * HD;
        const bf16* orow = p.o + grow * p.C + it.h * HD;
#pragma unroll
        for (int u = 0; u < HD / 8; u++) {
          float a[8], c[8];
          ld16(dor + 8 * u, a);
          ld16(orow + 8 * u, c);
#pragma unroll
          for (int e = 0; e < 8; e++) Dr = fmaf(a[e], c[e], Dr);
        }
        if (cq == 0) p.D[sidx] = Dr;
      }
      const float lse2 = p.lse[sidx] * LOG2E;
      for (int j = 0; j <= it.qt; j++) {
        if (!mbar_wait_warp(b_sfull, nS & 1, abort_flag)) { ok = false; break; }
        fence_after();
        float sv[EW_COLS], dp[EW_COLS];
#pragma unroll
        for (int c = 0; c < EW_COLS / 32; c++) {
          tmem_ld32_async(tmem + lrow + c0 + 32 * c, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
          tmem_ld32_async(tmem + lrow + 128 + c0 + 32 * c, *reinterpret_cast<float(*)[32]>(dp + 32 * c));
        }
        tmem_wait_ld();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sfree);
        nS++;
        const bool diag = j == it.qt;
#pragma unroll
        for (int e = 0; e < EW_COLS; e++) {
          const float x = fmaf(sv[e], p.sl2, -lse2);
          sv[e] = (e & 3) == 3 ? exp2_poly(x) : ex2(x);
        }
        if (diag) {
#pragma unroll
          for (int e = 0; e < EW_COLS; e++)
            if (c0 + e > (int)r) sv[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < EW_COLS; e++) sv[e] *= dp[e] - Dr;
        // the dS tile is free once the previous dQ MMA has read it
        if (nD > 0 && !mbar_wait_warp(b_dsfree, (nD - 1) & 1, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < EW_COLS / 32; c++)
          store_row32(sDS, r, c0 + 32 * c, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_dsfull);
        nD++;
      }
      if (!ok || !mbar_wait_warp(b_dqfull, n & 1, abort_flag)) break;
      fence_after();
      // dQ has 64 columns: the first two column groups take 32 each
      constexpr int DQ_GROUPS = EW_WARPS / 4 < 2 ? EW_WARPS / 4 : 2;
      float v[32];
      if (cq < DQ_GROUPS) tmem_ld32(tmem + lrow + 256 + 32 * cq, v);
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_dqfree);
      if (cq < DQ_GROUPS) store_global32(p.out + grow * 3 * p.C + it.h * HD + 32 * cq, v, p.scale);
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
// backward, dK and dV.  Persistent: items are (b, h, key tile), heaviest
// first; per item the query tiles kt..nq-1 stream through a ring (Q, dO and
// their lse and D).  Needs D from the dQ kernel.
// ============================================================================
constexpr uint32_t BWD_QD = 2 * TILE + 1024;  // Q tile, dO tile, lse[128], D[128]
constexpr size_t DKV_SMEM = 1024 + 2 * TILE + DKV_STAGES * BWD_QD + 2 * PTILE + 256;

__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                           AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sK = smem_u32(smem), sV = sK + TILE;
  const uint32_t sQD = sK + 2 * TILE;                 // ring: Q, dO, lse, D
  const uint32_t sPT = sQD + DKV_STAGES * BWD_QD;     // P^T tile
  const uint32_t sDST = sPT + PTILE;                  // dS^T tile
  const uint8_t* ring_gen = smem + 2 * TILE;          // generic view of the ring
  uint64_t* bars = (uint64_t*)(smem + 2 * TILE + DKV_STAGES * BWD_QD + 2 * PTILE);
  const uint32_t b_kvfull = smem_u32(bars), b_kvempty = b_kvfull + 8;  // K and V tiles of an item
  const uint32_t b_qfull = b_kvempty + 8, b_qempty = b_qfull + 8 * DKV_STAGES;
  const uint32_t b_sfull = b_qempty + 8 * DKV_STAGES;
  const uint32_t b_sfree = b_sfull + 8;
  const uint32_t b_pfull = b_sfree + 8;   // P^T and dS^T written
  const uint32_t b_pfree = b_pfull + 8;   // dV/dK MMAs done reading them
  const uint32_t b_accfull = b_pfree + 8;
  const uint32_t b_accfree = b_accfull + 8;
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 + 2 * DKV_STAGES + 6);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, BH = p.B * p.H;
  const int n_items = BH * nq;
  struct Item { int kt, nit, b, h, row0; size_t sbase; };
  auto item = [&](int i) {
    Item it;
    it.kt = i / BH;  // key tile; small kt = more query tiles = heavier, first
    const int bh = i % BH;
    it.b = bh / p.H;
    it.h = bh % p.H;
    it.row0 = it.b * p.T;
    it.nit = nq - it.kt;  // query tiles kt .. nq-1
    it.sbase = ((size_t)it.b * p.H + it.h) * p.T;
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(b_kvfull, 1);
    mbar_init(b_kvempty, 1);
    for (int s = 0; s < DKV_STAGES; s++) {
      mbar_init(b_qfull + 8 * s, 1);
      mbar_init(b_qempty + 8 * s, 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, EW_WARPS);
    mbar_init(b_pfull, EW_WARPS);
    mbar_init(b_pfree, 1);
    mbar_init(b_accfull, 1);
    mbar_init(b_accfree, EW_WARPS);
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
      uint32_t g = 0, n = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, n++) {
        const Item it = item(i);
        if (!mbar_wait(b_kvempty, (n & 1) ^ 1, abort_flag)) break;
        mbar_expect_tx(b_kvfull, 2 * TILE);
        tma_load_2d(sK, &tqkv, p.C + it.h * HD, it.row0 + it.kt * 128, b_kvfull);
        tma_load_2d(sV, &tqkv, 2 * p.C + it.h * HD, it.row0 + it.kt * 128, b_kvfull);
        for (int k = 0; k < it.nit; k++, g++) {
          const int qt = it.kt + k;
          const uint32_t s = g % DKV_STAGES, ph = (g / DKV_STAGES) & 1;
          if (!mbar_wait(b_qempty + 8 * s, ph ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t dst = sQD + s * BWD_QD, fb = b_qfull + 8 * s;
          mbar_expect_tx(fb, BWD_QD);
          tma_load_2d(dst, &tqkv, it.h * HD, it.row0 + qt * 128, fb);
          tma_load_2d(dst + TILE, &tdo, it.h * HD, it.row0 + qt * 128, fb);
          bulk_load(dst + 2 * TILE, p.lse + it.sbase + qt * 128, 512, fb);
          bulk_load(dst + 2 * TILE + 512, p.D + it.sbase + qt * 128, 512, fb);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);  // S^T = K Q^T, dP^T = V dO^T
      constexpr uint32_t ID_G = idesc_bf16(128, HD, 0, 1);   // dV += P^T dO, dK += dS^T Q
      uint32_t g0 = 0, n = 0, nS = 0, nG = 0;
      bool ok = true;
      auto issue_grad = [&](int k) {
        if (!mbar_wait(b_pfull, nG & 1, abort_flag)) return false;
        // the first gradient MMAs of an item overwrite dV, dK: the previous item's must be read out
        if (k == 0 && n > 0 && !mbar_wait(b_accfree, (n - 1) & 1, abort_flag)) return false;
        fence_after();
        const uint32_t qd = sQD + ((g0 + k) % DKV_STAGES) * BWD_QD;
#pragma unroll
        for (int kk = 0; kk < 128 / 16; kk++) {
          mma_bf16(tmem + 256, desc_k128(sPT, kk), desc_mn(qd + TILE, kk), ID_G, (k | kk) > 0);
          mma_bf16(tmem + 320, desc_k128(sDST, kk), desc_mn(qd, kk), ID_G, (k | kk) > 0);
        }
        mma_commit(b_pfree);
        mma_commit(b_qempty + 8 * ((g0 + k) % DKV_STAGES));
        nG++;
        return true;
      };
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, n++) {
        const Item it = item(i);
        if (!mbar_wait(b_kvfull, n & 1, abort_flag)) break;
        for (int k = 0; ok && k < it.nit; k++) {
          const uint32_t gk = g0 + k, s = gk % DKV_STAGES;
          if (!mbar_wait(b_qfull + 8 * s, (gk / DKV_STAGES) & 1, abort_flag)) { ok = false; break; }
          if (nS > 0 && !mbar_wait(b_sfree, (nS - 1) & 1, abort_flag)) { ok = false; break; }
          fence_after();
          const uint32_t qd = sQD + s * BWD_QD;
#pragma unroll
          for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem, desc_k(sK, kk), desc_k(qd, kk), ID_S, kk > 0);
#pragma unroll
          for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem + 128, desc_k(sV, kk), desc_k(qd + TILE, kk), ID_S, kk > 0);
          mma_commit(b_sfull);
          nS++;
          if (k == it.nit - 1) mma_commit(b_kvempty);  // the item's last use of K and V is issued
          if (k > 0 && !issue_grad(k - 1)) { ok = false; break; }
        }
        if (ok && issue_grad(it.nit - 1)) mma_commit(b_accfull);
        else ok = false;
        g0 += it.nit;
      }
    }
  } else {  // ---- elementwise warps: key row r (lane quarter q), query-column group cq
    const int q = warp & 3, cq = (warp - 2) >> 2;
    const int c0 = cq * EW_COLS;
    const uint32_t r = q * 32 + lane;
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    uint32_t g0 = 0, n = 0, nS = 0, nG = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, n++) {
      const Item it = item(i);
      for (int k = 0; k < it.nit; k++) {
        if (!mbar_wait_warp(b_sfull, nS & 1, abort_flag)) { ok = false; break; }
        fence_after();
        float sv[EW_COLS], dp[EW_COLS];
#pragma unroll
        for (int c = 0; c < EW_COLS / 32; c++) {
          tmem_ld32_async(tmem + lrow + c0 + 32 * c, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
          tmem_ld32_async(tmem + lrow + 128 + c0 + 32 * c, *reinterpret_cast<float(*)[32]>(dp + 32 * c));
        }
        tmem_wait_ld();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sfree);
        nS++;
        // lse and D of this stage's 128 queries (bulk-loaded with the Q tile)
        const uint32_t gk = g0 + k;
        if (!mbar_wait_warp(b_qfull + 8 * (gk % DKV_STAGES), (gk / DKV_STAGES) & 1, abort_flag)) { ok = false; break; }
        const float* lq = (const float*)(ring_gen + (gk % DKV_STAGES) * BWD_QD + 2 * TILE) + c0;
        const float* dq = lq + 128;
        const bool diag = k == 0;  // query tile == key tile
#pragma unroll
        for (int e = 0; e < EW_COLS; e++) {
          const float x = fmaf(sv[e], p.sl2, -lq[e] * LOG2E);
          sv[e] = (e & 3) == 3 ? exp2_poly(x) : ex2(x);
        }
        if (diag) {
#pragma unroll
          for (int e = 0; e < EW_COLS; e++)
            if ((int)r > c0 + e) sv[e] = 0.f;  // key after query
        }
#pragma unroll
        for (int e = 0; e < EW_COLS; e++) dp[e] = sv[e] * (dp[e] - dq[e]);
        if (nG > 0 && !mbar_wait_warp(b_pfree, (nG - 1) & 1, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < EW_COLS / 32; c++) {
          store_row32(sPT, r, c0 + 32 * c, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
          store_row32(sDST, r, c0 + 32 * c, *reinterpret_cast<float(*)[32]>(dp + 32 * c));
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull);
        nG++;
      }
      if (!ok || !mbar_wait_warp(b_accfull, n & 1, abort_flag)) break;
      fence_after();
      // dV (TMEM 256..319) and dK (320..383): 128 columns over the column groups
      constexpr int EPI_COLS = 128 / (EW_WARPS / 4);
      float v[EPI_COLS];
#pragma unroll
      for (int c = 0; c < EPI_COLS / 32; c++)
        tmem_ld32_async(tmem + lrow + 256 + cq * EPI_COLS + 32 * c, *reinterpret_cast<float(*)[32]>(v + 32 * c));
      tmem_wait_ld();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_accfree);
      const size_t grow = (size_t)(it.row0 + it.kt * 128 + r);
#pragma unroll
      for (int c = 0; c < EPI_COLS / 32; c++) {
        const int col = cq * EPI_COLS + 32 * c;  // 0..63 dV, 64..127 dK
        if (col < 64)
          store_global32(p.out + grow * 3 * p.C + 2 * p.C + it.h * HD + col, *reinterpret_cast<float(*)[32]>(v + 32 * c), 1.f);
        else
          store_global32(p.out + grow * 3 * p.C + p.C + it.h * HD + col - 64, *reinterpret_cast<float(*)[32]>(v + 32 * c),
                         p.scale);
      }
      g0 += it.nit;
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
  const long long items = (long long)B * H * npair;
  const int sms = tc_num_sms();
  gpt2_count_launches(1);
  attn_fwd_tc_kernel<<<(unsigned)(items < sms ? items : sms), FWD_THREADS, FWD_SMEM, st>>>(tq, p);
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
  const long long items = (long long)B * H * (T / 128);
  const int sms = tc_num_sms();
  const unsigned grid = (unsigned)(items < sms ? items : sms);
  gpt2_count_launches(2);
  attn_bwd_dq_tc_kernel<<<grid, BWD_THREADS, DQ_SMEM, st>>>(tq, td, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_dkv_tc_kernel<<<grid, BWD_THREADS, DKV_SMEM, st>>>(tq, td, p);
  return cudaGetLastError();
}
