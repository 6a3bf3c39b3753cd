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
// pair of 128-row query tiles of one (b, h); 320 threads): warp 0 issues TMA,
// one thread of warp 1 issues S = Q K^T and O += P [V | 1], and two softmax
// warpgroups (one per query tile) hold one score row per thread.  P goes
// back into TMEM over its own scores and is the A operand of the P V product,
// whose B operand is V extended by a block of ones, so the row sums come out
// of the tensor core beside O.  See attn_fwd_tc_kernel.
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
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

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
// (a0, a1) * b + (c, c) on the packed fp32 pipe: two FMAs in one instruction
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\tmov.b64 z, {%5, %5};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// packed fp32 pairs: (a0, a1) op (b0, b1), one instruction for two lanes' worth
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%6, %7};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "sub.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
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
  uint8_t* ds;        // backward: dS blocks (see ds_block)
};

// Which work items each persistent CTA takes.  The items of a kernel differ in
// length (a causal query tile of index qt spans qt + 1 key tiles), so taking
// items i = blockIdx.x, blockIdx.x + gridDim.x, ... left the busiest CTA 10-15%
// above the mean at T = 1024.  The host assigns the items, heaviest first, each
// to the CTA with the least work so far (longest-processing-time first, lowest
// index on ties): every CTA then ends within one item of the mean.  The table
// is a pure function of the shape and travels as a kernel parameter, so a
// captured launch replays it unchanged.  n = 0: more items or CTAs than the
// table holds; the kernels then stride over the items.
constexpr int SCHED_MAX_ITEMS = 4096;
constexpr int SCHED_MAX_CTAS = 256;
struct AttnSched {
  int n;                                 // items in the table (0: stride over them)
  uint16_t first[SCHED_MAX_CTAS + 1];    // CTA c takes item[first[c] .. first[c + 1] - 1], in order
  uint16_t item[SCHED_MAX_ITEMS];
};

__device__ __forceinline__ int sched_count(const AttnSched& s, int n_items) {
  if (s.n) return s.first[blockIdx.x + 1] - s.first[blockIdx.x];
  return n_items > (int)blockIdx.x ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
}
__device__ __forceinline__ int sched_item(const AttnSched& s, int k) {
  return s.n ? (int)s.item[s.first[blockIdx.x] + k] : (int)blockIdx.x + k * (int)gridDim.x;
}

// ============================================================================
// forward
// ============================================================================
// TMEM accesses of one warp: 32 lanes x N consecutive 32-bit columns
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
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
__device__ __forceinline__ void tmem_ld1(uint32_t taddr, float& v) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
  v = __uint_as_float(r);
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(__float_as_uint(v)) : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 32 lanes x 128 consecutive fp32 columns, four loads in flight, one wait
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
#pragma unroll
  for (int c = 0; c < 4; c++) tmem_ld32_async(taddr + 32 * c, *reinterpret_cast<float(*)[32]>(v + 32 * c));
  tmem_wait_ld();
}
// O (+)= P V with P read from TMEM (A operand, M=128 x K=16 per instruction:
// 8 columns of packed bf16 pairs) and V from shared memory
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

constexpr int FWD_POLY = 16;  // one exponential in this many columns from the FMA-pipe polynomial
constexpr float RESCALE_LOG2 = 8.f;
// P of one block in TMEM, as the A operand of O += P [V | 1]: 64 columns of
// packed bf16 pairs, keys 0..63 in the 32 columns at tP0 (beside O, which
// leaves them free) and keys 64..127 over the first 32 columns of S (whose
// scores of keys 0..63 have been read by then).

// 32 probabilities p = 2^(x) of columns col0 .. col0 + 31 from x = s sl2 -
// m_ref, packed into 16 bf16 pairs; m2 tracks the maximum of x.  One
// exponential in FWD_POLY from the FMA-pipe polynomial (none on the diagonal
// block, whose keys after the query get x = -inf, p = 0).
template <bool DIAG>
__device__ __forceinline__ void fwd_chunk(const float* sv, int col0, uint32_t r, float sl2, float m_ref, float (&m2)[2],
                                          uint32_t* pk) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const int col = col0 + e;
    float x0, x1;
    ffma2(x0, x1, sv[e], sv[e + 1], sl2, -m_ref);
    if (DIAG) {
      if (col > (int)r) x0 = -INFINITY;
      if (col + 1 > (int)r) x1 = -INFINITY;
    }
    m2[(e >> 1) & 1] = max3(m2[(e >> 1) & 1], x0, x1);
    if (!DIAG && (col % FWD_POLY) == FWD_POLY - 2) x0 = exp2_poly(x0);
    else x0 = ex2(x0);
    x1 = ex2(x1);
    pk[e >> 1] = pack_bf16(x0, x1);
  }
}

// The probabilities of one 128-wide score row (TMEM lane r of the warp's
// quarter, scores at tS) against the reference m_ref, read 64 columns at a
// time and written to the P layout above.
template <bool DIAG>
__device__ __forceinline__ void fwd_probs(uint32_t tS, uint32_t tP0, uint32_t r, float sl2, float m_ref) {
  float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int h = 0; h < 2; h++) {
    float sv[64];
    tmem_ld32_async(tS + 64 * h, *reinterpret_cast<float(*)[32]>(sv));
    tmem_ld32_async(tS + 64 * h + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < 2; c++) {
      uint32_t pk[16];
      fwd_chunk<DIAG>(sv + 32 * c, 64 * h + 32 * c, r, sl2, m_ref, m2, pk);
      tmem_st16((h ? tS : tP0) + 16 * c, pk);
    }
  }
}

// The same probabilities in one read of the scores, for a block after the
// first below the diagonal: the row's maximum is tracked while p is taken against the current
// reference.  Keys 0..63 are written at once (to tP0, which leaves the scores
// intact); keys 64..127 stay in registers and are written only when no row of
// the warp has run more than RESCALE_LOG2 above its reference.  Otherwise
// false is returned with the scores untouched (fwd_probs then redoes the
// block); mrel = max over the valid columns of s sl2 - m_ref for this row.
__device__ __forceinline__ bool fwd_probs_once(uint32_t tS, uint32_t tP0, uint32_t r, float sl2, float m_ref,
                                               float& mrel) {
  float m2[2] = {-INFINITY, -INFINITY};
  {
    float sv[64];
    tmem_ld32_async(tS, *reinterpret_cast<float(*)[32]>(sv));
    tmem_ld32_async(tS + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < 2; c++) {
      uint32_t pk[16];
      fwd_chunk<false>(sv + 32 * c, 32 * c, r, sl2, m_ref, m2, pk);
      tmem_st16(tP0 + 16 * c, pk);
    }
  }
  uint32_t pk[32];
  {
    float a[32], b[32];
    tmem_ld32_async(tS + 64, a);
    tmem_wait_ld();
    tmem_ld32_async(tS + 96, b);  // in flight while keys 64..95 are worked
    fwd_chunk<false>(a, 64, r, sl2, m_ref, m2, pk);
    tmem_wait_ld();
    fwd_chunk<false>(b, 96, r, sl2, m_ref, m2, pk + 16);
  }
  mrel = fmaxf(m2[0], m2[1]);
  if (!__all_sync(0xffffffffu, !(mrel > RESCALE_LOG2))) return false;
  tmem_st16(tS, *reinterpret_cast<const uint32_t(*)[16]>(pk));
  tmem_st16(tS + 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16));
  return true;
}

// Online softmax with a lazily rescaled accumulator: the probabilities of a
// row are taken against a reference max m_ref; O (in TMEM) is only rescaled
// when a new block's max exceeds m_ref by more than RESCALE_LOG2 (then P
// stays <= 2^RESCALE_LOG2, harmless in fp32 and bf16).  The result is the
// same softmax: every term and the row sum share one reference.
//
// Forward kernel layout (persistent, one CTA per SM, 320 threads): an item is
// a pair of 128-row query tiles of one (b, h); warp 0 issues TMA (both Q tiles,
// then K/V tiles through a ring), one thread of warp 1 issues the MMAs, warps
// 2-5 run the softmax of query tile 0 and warps 6-9 that of tile 1, one
// thread per query row with the whole 128-wide score row in registers.  Per
// key block j and tile t:
//   S_t = Q_t K_j^T                  (TMEM columns 128 t .. 128 t + 127)
//   P_t = exp2(S_t sl2 - m_ref)      written as bf16 pairs into TMEM (keys
//                                     0..63 beside O_t, keys 64..127 over the
//                                     first 32 columns of S_t; no shared-memory
//                                     trip)
//   O_t += P_t [V_j | 1]             A = P_t from TMEM, B = V_j and a block of
//                                     ones from shared memory: N = 80, so
//                                     column 64 of O_t accumulates the row
//                                     sum of the same bf16 P (free)
// and S_t of block j+1 is issued right behind that P V (the tensor core takes
// them in order, so it reads P_t before overwriting it).  The two tiles'
// softmax phases interleave: one tile's exponentials overlap the other's MMAs.
// O *= alpha for this thread's row: the 64 value columns and the row sum
// (column 64); the columns after it hold P (see FWD_P0) and stay as they are
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
  float ov[32], l;
#pragma unroll
  for (int c = 0; c < 2; c++) {
    tmem_ld32(tO + 32 * c, ov);
#pragma unroll
    for (int e = 0; e < 32; e++) ov[e] *= alpha;
    tmem_st32(tO + 32 * c, ov);
  }
  tmem_ld1(tO + 64, l);
  tmem_wait_ld();
  tmem_st1(tO + 64, l * alpha);
}

constexpr int FWD_STAGES = 3;
constexpr uint32_t FWD_KV = 2 * TILE;  // K tile then V tile
constexpr int FWD_ON = 80;             // P V width: 64 value columns + the row-sum column (+ 15 unused)
constexpr uint32_t FWD_P0 = 256 + FWD_ON;  // P of keys 0..63, relative to the tile's S columns (beside O)
constexpr size_t FWD_SMEM = 1024 + 2 * TILE + FWD_STAGES * FWD_KV + TILE + 256;
constexpr int FWD_THREADS = 64 + 32 * 8;  // producer, MMA, two softmax warpgroups

// Persistent: each CTA takes the work items its schedule table lists (item =
// one pair of query tiles of one (b, h); item indices run heaviest first).  Every
// barrier phase is tracked by a running counter across items, so the next
// item's Q load, first Q K^T and K/V loads overlap the tail of the current one.
__global__ void __launch_bounds__(FWD_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tqkv, AttnParams p, const __grid_constant__ AttnSched sch) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sQ = smem_u32(smem);                  // 2 query tiles
  const uint32_t sKV = sQ + 2 * TILE;                  // ring of K/V tiles
  const uint32_t sOnes = sKV + FWD_STAGES * FWD_KV;    // 128 x 64 bf16 ones: the row-sum columns of V
  uint64_t* bars = (uint64_t*)(smem + 2 * TILE + FWD_STAGES * FWD_KV + TILE);
  const uint32_t b_qfull = smem_u32(bars), b_qempty = b_qfull + 8;
  const uint32_t b_kvfull = b_qempty + 8, b_kvempty = b_kvfull + 8 * FWD_STAGES;
  const uint32_t b_sfull = b_kvempty + 8 * FWD_STAGES;  // [2] S of tile t computed
  const uint32_t b_pfull = b_sfull + 16;                // [2] P of tile t written (4 warps)
  const uint32_t b_pvdone = b_pfull + 16;               // [2] a P V of tile t completed
  const uint32_t b_ofree = b_pvdone + 16;               // [2] finished O of tile t read out (4 warps)
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 + 2 * FWD_STAGES + 8);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, npair = (nq + 1) / 2;
  const int BH = p.B * p.H;
  const int n_items = BH * npair;
  const int n_mine = sched_count(sch, n_items);
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
      mbar_init(b_pfull + 8 * t, 4);
      mbar_init(b_pvdone + 8 * t, 1);
      mbar_init(b_ofree + 8 * t, 4);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the ones block (bf16 1.0 everywhere, so its swizzle does not matter)
  for (uint32_t o = threadIdx.x * 16; o < TILE; o += FWD_THREADS * 16) st_shared_v4(sOnes + o, 0x3f803f80u, 0x3f803f80u,
                                                                                        0x3f803f80u, 0x3f803f80u);
  fence_async_smem();
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
  if (warp == 0 && lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tqkv) : "memory");
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_enter();  // global memory only from here on
  // TMEM columns: S of tile t at 128 t, O of tile t at 256 + 128 t (80 wide), P of tile t:
  // keys 0..63 at 336 + 128 t (32 columns), keys 64..127 at 128 t (32 columns)

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      uint32_t g = 0, n = 0;  // K/V blocks and items loaded so far
      bool ok = true;
      for (int ki = 0; ok && ki < n_mine; ki++, n++) {
        const int i = sched_item(sch, ki);
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
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);     // S = Q K^T
      constexpr uint32_t ID_O = idesc_bf16(128, FWD_ON, 0, 1);  // O += P [V | 1] (V is MN-major)
      uint32_t g0 = 0, n = 0;                                   // K/V blocks before this item, items so far
      uint32_t nP[2] = {0, 0}, nO[2] = {0, 0};                  // per tile: P blocks consumed, items finished
      int kv_ready = -1;                                        // highest K/V block known loaded (global index)
      bool ok = true;
      for (int ki = 0; ok && ki < n_mine; ki++, n++) {
        const int i = sched_item(sch, ki);
        const Item it = item(i);
        const int last_t = it.two ? 1 : 0;
        auto active = [&](int t, int j) { return t == 0 ? j <= it.qt0 : (it.two && j <= it.qt0 + 1); };
        auto wait_kv = [&](int j) {
          const int gj = (int)g0 + j;
          if (kv_ready >= gj) return true;
          if (!mbar_wait(b_kvfull + 8 * (gj % FWD_STAGES), (gj / FWD_STAGES) & 1, abort_flag)) return false;
          kv_ready = gj;
          return true;
        };
        auto issue_s = [&](int t, int j) {
          if (!wait_kv(j)) return false;
          fence_after();
          const uint32_t k = sKV + ((g0 + j) % FWD_STAGES) * FWD_KV, q = sQ + t * TILE;
#pragma unroll
          for (int kk = 0; kk < HD / 16; kk++) mma_bf16(tmem + 128 * t, desc_k(q, kk), desc_k(k, kk), ID_S, kk > 0);
          mma_commit(b_sfull + 8 * t);
          // the item's last Q K^T: the Q tiles may be reloaded once it completes
          if (t == last_t && j == it.nkv - 1) mma_commit(b_qempty);
          return true;
        };
        if (!mbar_wait(b_qfull, n & 1, abort_flag)) break;
        fence_after();
        ok = issue_s(0, 0) && (!active(1, 0) || issue_s(1, 0));
        for (int j = 0; ok && j < it.nkv; j++) {
          const uint32_t v = sKV + ((g0 + j) % FWD_STAGES) * FWD_KV + TILE;
          // V and the ones block are one MN-major operand of N = 80 columns:
          // the ones sit at a fixed distance after this stage's V tile
          const uint32_t lbo = sOnes - v;
          for (int t = 0; t < 2 && ok; t++) {
            if (!active(t, j)) continue;
            if (!mbar_wait(b_pfull + 8 * t, nP[t] & 1, abort_flag)) { ok = false; break; }
            // the first P V of an item overwrites O: the previous item's O must be read out
            if (j == 0 && nO[t] > 0 && !mbar_wait(b_ofree + 8 * t, (nO[t] - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            fence_after();
#pragma unroll
            for (int kk = 0; kk < 128 / 16; kk++)
              mma_bf16_ts(tmem + 256 + 128 * t, tmem + 128 * t + (kk < 4 ? FWD_P0 + 8 * kk : 8 * (kk - 4)),
                          sdesc(v + kk * 2048, lbo, 1024), ID_O,
                          (j | kk) > 0);
            mma_commit(b_pvdone + 8 * t);
            nP[t]++;
            // the next scores of this tile, behind the P V that reads P from the same columns
            if (active(t, j + 1) && !issue_s(t, j + 1)) { ok = false; break; }
          }
          if (ok) mma_commit(b_kvempty + 8 * ((g0 + j) % FWD_STAGES));
        }
        for (int t = 0; t < 2; t++)
          if (t == 0 || it.two) nO[t]++;
        g0 += it.nkv;
      }
    }
  } else {  // ---- softmax warps: tile t, TMEM lane quarter q; one query row per thread
    const int t = (warp - 2) >> 2, q = warp & 3;
    const uint32_t r = q * 32 + lane;  // row inside the tile
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    const uint32_t tS = tmem + lrow + 128 * t, tO = tmem + lrow + 256 + 128 * t, tP0 = tS + FWD_P0;
    uint32_t nS = 0, nPV = 0;  // S blocks consumed; P V products of this tile before the current item
    bool ok = true;
    for (int ki = 0; ok && ki < n_mine; ki++) {
      const int i = sched_item(sch, ki);
      const Item it = item(i);
      const int qt = it.qt0 + t;
      if (qt >= nq) continue;  // this item has no tile t
      float m_ref = -INFINITY;
      for (int j = 0; j <= qt; j++) {
        if (!mbar_wait_warp(b_sfull + 8 * t, nS & 1, abort_flag)) { ok = false; break; }
        nS++;
        fence_after();
        const bool diag = j == qt;
        if (j > 0 && !diag) {
          // one read of the scores against the current reference; a row that
          // ran too far above it moves the reference, and the block is redone
          float mrel;
          if (!fwd_probs_once(tS, tP0, r, p.sl2, m_ref, mrel)) {
            const bool need = mrel > RESCALE_LOG2;
            const float m_old = m_ref;
            if (need) m_ref += mrel;
            tmem_wait_st();  // the first half's stores land before they are redone
            fwd_probs<false>(tS, tP0, r, p.sl2, m_ref);
            // O holds blocks 0 .. j-1 once the previous P V has completed
            if (!mbar_wait_warp(b_pvdone + 8 * t, (nPV + j - 1) & 1, abort_flag)) { ok = false; break; }
            fence_after();
            rescale_o(tO, need ? ex2(m_old - m_ref) : 1.f);
          }
          tmem_wait_st();
          fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_pfull + 8 * t);
          continue;
        }
        // the first and the diagonal block: two reads of the scores
        float mx;
        {  // pass 1: the row maximum over the valid columns (c <= r on the diagonal block)
          float sv[128];
          tmem_ld128(tS, sv);
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (!diag) {
#pragma unroll
            for (int c = 0; c < 128; c += 8) {
              m4[0] = max3(m4[0], sv[c], sv[c + 1]);
              m4[1] = max3(m4[1], sv[c + 2], sv[c + 3]);
              m4[2] = max3(m4[2], sv[c + 4], sv[c + 5]);
              m4[3] = max3(m4[3], sv[c + 6], sv[c + 7]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 128; c++)
              if (c <= (int)r) m4[c & 3] = fmaxf(m4[c & 3], sv[c]);
          }
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.sl2;
        }
        // move the reference when this block's max runs too far above it
        const bool need = j > 0 && mx > m_ref + RESCALE_LOG2;
        const float m_old = m_ref;
        if (j == 0 || need) m_ref = mx;
        // pass 2: the scores again, 64 columns at a time, into P
        if (!diag) fwd_probs<false>(tS, tP0, r, p.sl2, m_ref);
        else fwd_probs<true>(tS, tP0, r, p.sl2, m_ref);
        if (__any_sync(0xffffffffu, need)) {
          // O holds blocks 0 .. j-1 once the previous P V has completed
          if (!mbar_wait_warp(b_pvdone + 8 * t, (nPV + j - 1) & 1, abort_flag)) { ok = false; break; }
          fence_after();
          rescale_o(tO, need ? ex2(m_old - m_ref) : 1.f);
        }
        tmem_wait_st();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull + 8 * t);
      }
      if (!ok) break;
      // the item's last P V completes the accumulator and the row sum
      if (!mbar_wait_warp(b_pvdone + 8 * t, (nPV + qt) & 1, abort_flag)) break;
      nPV += qt + 1;
      fence_after();
      float o[64], lt;
      tmem_ld32_async(tO, *reinterpret_cast<float(*)[32]>(o));
      tmem_ld32_async(tO + 32, *reinterpret_cast<float(*)[32]>(o + 32));
      tmem_ld1(tO + 64, lt);
      tmem_wait_ld();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ofree + 8 * t);  // the next item may overwrite O
      bf16* dst = p.out + (size_t)(it.row0 + qt * 128 + r) * p.C + it.h * HD;
      const float inv = 1.f / lt;
      store_global32(dst, *reinterpret_cast<float(*)[32]>(o), inv);
      store_global32(dst + 32, *reinterpret_cast<float(*)[32]>(o + 32), inv);
      p.lse[((size_t)it.b * p.H + it.h) * p.T + qt * 128 + r] = (m_ref + log2f(lt)) * LN2;
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
// backward.  D = rowsum(dO * O) first (attn_rowdot_kernel); then the dK/dV
// kernel, which also writes every dS block it forms to global memory; then
// the dQ kernel, a plain blocked product dQ = dS K over those blocks.
// ============================================================================
constexpr int DKV_STAGES = 3;            // Q/dO/lse/D ring of the dK/dV kernel
constexpr int EW_WARPS = 16;             // elementwise warps of the dK/dV kernel
constexpr int EW_COLS = 128 / (EW_WARPS / 4);  // columns of S each elementwise warp handles
constexpr int BWD_THREADS = 64 + 32 * EW_WARPS + 32;  // producer, MMA, elementwise warps, dS store warp

// D[b][h][t] = sum over the head's 64 channels of dO * O: one thread per 8
// channels, the 8 threads of a head added by a fixed shuffle tree.
__global__ void __launch_bounds__(256) attn_rowdot_kernel(float* D, const bf16* dout, const bf16* o, long long n8,
                                                          int T, int C, int H) {
  pdl_enter();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  float acc = 0.f;
  if (i < n8) {
    float a[8], c[8];
    ld16(dout + i * 8, a);
    ld16(o + i * 8, c);
#pragma unroll
    for (int e = 0; e < 8; e++) acc = fmaf(a[e], c[e], acc);
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (i < n8 && (i & 7) == 0) {
    const long long row = i / (C / 8);
    const int h = (int)(i % (C / 8)) / 8;
    const long long b = row / T, t = row % T;
    D[(b * H + h) * T + t] = acc;
  }
}

// dS blocks in global memory: for each (b, h), the causal blocks (key tile
// kt, query tile qt >= kt) in order of kt then qt, each the 32 KB shared-memory
// image of the dS^T tile (two 64-query halves of 128 key rows, 128-byte
// swizzled), so that a 1024-aligned bulk copy brings it back operand-ready.
__host__ __device__ __forceinline__ long long ds_block(int bh, int nq, int kt, int qt) {
  const long long per_bh = (long long)nq * (nq + 1) / 2;
  return bh * per_bh + (long long)kt * nq - (long long)kt * (kt - 1) / 2 + (qt - kt);
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"((uint64_t)dst), "r"(src),
               "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- dQ = dS K: persistent, items (b, h, query tile) heaviest first; per
// item the blocks kt = 0..qt stream through a ring (dS^T block + K tile) and
// accumulate into one of two TMEM accumulators, so that one item's read-out
// overlaps the next item's products.  Bandwidth-bound: 48 KB in per block
// for 2*128*128*64 flops.
constexpr int DQ_STAGES = 4;
constexpr uint32_t DQ_STAGE = PTILE + TILE;  // dS^T block, K tile
constexpr int DQ_THREADS = 64 + 32 * 4;      // producer, MMA, 4 read-out warps
constexpr size_t DQ_SMEM = 1024 + DQ_STAGES * DQ_STAGE + 256;

__global__ void __launch_bounds__(DQ_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tqkv, const uint8_t* __restrict__ ds, AttnParams p,
                          const __grid_constant__ AttnSched sch) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t ring = smem_u32(smem);
  uint64_t* bars = (uint64_t*)(smem + DQ_STAGES * DQ_STAGE);
  const uint32_t b_full = smem_u32(bars), b_empty = b_full + 8 * DQ_STAGES;
  const uint32_t b_accfull = b_empty + 8 * DQ_STAGES;  // [2] an item's dQ complete in TMEM
  const uint32_t b_accfree = b_accfull + 16;           // [2] ... and read out
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 * DQ_STAGES + 4);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, BH = p.B * p.H;
  const int n_items = BH * nq;
  const int n_mine = sched_count(sch, n_items);
  auto item_qt = [&](int i) { return nq - 1 - i / BH; };  // heaviest tiles first

  if (threadIdx.x == 0) {
    for (int s = 0; s < DQ_STAGES; s++) {
      mbar_init(b_full + 8 * s, 1);
      mbar_init(b_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; a++) {
      mbar_init(b_accfull + 8 * a, 1);
      mbar_init(b_accfree + 8 * a, 4);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 128);
  if (warp == 0 && lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tqkv) : "memory");
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_enter();  // global memory only from here on
  // TMEM columns: dQ accumulator a at 64 a

  if (warp == 0) {
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      for (int ki = 0; ok && ki < n_mine; ki++) {
        const int i = sched_item(sch, ki);
        const int qt = item_qt(i), bh = i % BH, h = bh % p.H, row0 = (bh / p.H) * p.T;
        for (int kt = 0; kt <= qt; kt++, g++) {
          const uint32_t s = g % DQ_STAGES, ph = (g / DQ_STAGES) & 1;
          if (!mbar_wait(b_empty + 8 * s, ph ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t dst = ring + s * DQ_STAGE, fb = b_full + 8 * s;
          mbar_expect_tx(fb, DQ_STAGE);
          bulk_load(dst, ds + ds_block(bh, nq, kt, qt) * PTILE, PTILE, fb);
          tma_load_2d(dst + PTILE, &tqkv, p.C + h * HD, row0 + kt * 128, fb);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // A = dS (M = 128 queries, MN-major: the dS^T tile's 64-query halves
      // 16 KB apart, 16 key rows per step); B = K tile (N = 64, MN-major)
      constexpr uint32_t ID_DQ = idesc_bf16(128, HD, 1, 1);
      uint32_t g = 0, n = 0;
      bool ok = true;
      for (int ki = 0; ok && ki < n_mine; ki++, n++) {
        const int i = sched_item(sch, ki);
        const int qt = item_qt(i);
        const uint32_t a = n & 1, acc = tmem + 64 * a;
        if (!mbar_wait(b_accfree + 8 * a, ((n >> 1) & 1) ^ 1, abort_flag)) break;
        fence_after();
        for (int kt = 0; kt <= qt; kt++, g++) {
          const uint32_t s = g % DQ_STAGES;
          if (!mbar_wait(b_full + 8 * s, (g / DQ_STAGES) & 1, abort_flag)) { ok = false; break; }
          fence_after();
          const uint32_t st = ring + s * DQ_STAGE;
#pragma unroll
          for (int kk = 0; kk < 128 / 16; kk++)
            mma_bf16(acc, sdesc(st + kk * 2048, TILE, 1024), desc_mn(st + PTILE, kk), ID_DQ, (kt | kk) > 0);
          mma_commit(b_empty + 8 * s);
        }
        if (ok) mma_commit(b_accfull + 8 * a);
      }
    }
  } else {  // ---- read-out warps: lane quarter q, rows q*32 .. q*32+31 of the item's query tile
    const int q = warp & 3;
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    uint32_t n = 0;
    for (int ki = 0; ki < n_mine; ki++, n++) {
      const int i = sched_item(sch, ki);
      const int qt = item_qt(i), bh = i % BH, h = bh % p.H, row0 = (bh / p.H) * p.T;
      const uint32_t a = n & 1;
      if (!mbar_wait_warp(b_accfull + 8 * a, (n >> 1) & 1, abort_flag)) break;
      fence_after();
      float v0[32], v1[32];
      tmem_ld32_async(tmem + lrow + 64 * a, v0);
      tmem_ld32_async(tmem + lrow + 64 * a + 32, v1);
      tmem_wait_ld();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_accfree + 8 * a);
      bf16* dst = p.out + (size_t)(row0 + qt * 128 + q * 32 + lane) * 3 * p.C + h * HD;
      store_global32(dst, v0, p.scale);
      store_global32(dst + 32, v1, p.scale);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    tmem_dealloc(tmem, 128);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.flags, FLAG_TIMEOUT);
}

// ============================================================================
// backward, dK and dV.  Persistent: items are (b, h, key tile), heaviest
// first; per item the query tiles kt..nq-1 stream through a ring (Q, dO and
// their lse and D).  Needs D (from attn_rowdot_kernel or the producer of dO);
// writes each dS^T tile it forms to the dS block buffer for the dQ kernel:
// the last warp bulk-copies the whole 32 KB tile once the elementwise warps
// have written it, and releases it when the copy has read it.
// ============================================================================
constexpr uint32_t BWD_QD = 2 * TILE + 1024;  // Q tile, dO tile, lse[128], D[128]
constexpr size_t DKV_SMEM = 1024 + 2 * TILE + DKV_STAGES * BWD_QD + 2 * PTILE + 256;

__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tqkv, const __grid_constant__ CUtensorMap tdo,
                           AttnParams p, const __grid_constant__ AttnSched sch) {
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
  const uint32_t b_dsfree = b_accfree + 8;  // dS^T tile copied out
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 + 2 * DKV_STAGES + 7);
  volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = p.T / 128, BH = p.B * p.H;
  const int n_items = BH * nq;
  const int n_mine = sched_count(sch, n_items);
  struct Item { int kt, nit, bh, b, h, row0; size_t sbase; };
  auto item = [&](int i) {
    Item it;
    it.kt = i / BH;  // key tile; small kt = more query tiles = heavier, first
    const int bh = i % BH;
    it.bh = bh;
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
    mbar_init(b_dsfree, 1);
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
  pdl_enter();  // global memory only from here on
  // TMEM columns: S^T at 0, dP^T at 128, dV at 256, dK at 320

  if (warp == 0) {
    if (lane == 0) {
      uint32_t g = 0, n = 0;
      bool ok = true;
      for (int ki = 0; ok && ki < n_mine; ki++, n++) {
        const int i = sched_item(sch, ki);
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
      for (int ki = 0; ok && ki < n_mine; ki++, n++) {
        const int i = sched_item(sch, ki);
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
  } else if (warp < 2 + EW_WARPS) {  // ---- elementwise warps: key row r (lane quarter q), query-column group cq
    const int q = warp & 3, cq = (warp - 2) >> 2;
    const int c0 = cq * EW_COLS;
    const uint32_t r = q * 32 + lane;
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    uint32_t g0 = 0, n = 0, nS = 0, nG = 0;
    bool ok = true;
    for (int ki = 0; ok && ki < n_mine; ki++, n++) {
      const int i = sched_item(sch, ki);
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
        // this group's 32 queries' lse and D (four floats per shared-memory load)
        const float4* lq4 = reinterpret_cast<const float4*>(ring_gen + (gk % DKV_STAGES) * BWD_QD + 2 * TILE) + c0 / 4;
        const float4* dq4 = lq4 + 32;
        // P^T = 2^(S^T sl2 - lse log2 e) and dS^T = P^T (dP^T - D), on packed fp32 pairs
#pragma unroll
        for (int g = 0; g < EW_COLS / 4; g++) {
          const float4 lv = lq4[g], dv = dq4[g];
          float n0, n1, n2, n3;
          mul2(n0, n1, lv.x, lv.y, -LOG2E, -LOG2E);
          mul2(n2, n3, lv.z, lv.w, -LOG2E, -LOG2E);
          float x0, x1, x2, x3;
          fma2(x0, x1, sv[4 * g], sv[4 * g + 1], p.sl2, p.sl2, n0, n1);
          fma2(x2, x3, sv[4 * g + 2], sv[4 * g + 3], p.sl2, p.sl2, n2, n3);
          sv[4 * g] = (g & 3) == 3 ? exp2_poly(x0) : ex2(x0);  // one exponential in 16 on the FMA pipe
          sv[4 * g + 1] = ex2(x1);
          sv[4 * g + 2] = ex2(x2);
          sv[4 * g + 3] = ex2(x3);
          sub2(dp[4 * g], dp[4 * g + 1], dp[4 * g], dp[4 * g + 1], dv.x, dv.y);
          sub2(dp[4 * g + 2], dp[4 * g + 3], dp[4 * g + 2], dp[4 * g + 3], dv.z, dv.w);
        }
        if (k == 0) {  // the diagonal tile: a key after its query gets P = 0
#pragma unroll
          for (int e = 0; e < EW_COLS; e++)
            if ((int)r > c0 + e) sv[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < EW_COLS; e += 2) mul2(dp[e], dp[e + 1], sv[e], sv[e + 1], dp[e], dp[e + 1]);
        // the P^T / dS^T tiles are free once the dV/dK MMAs have read them
        // and the copy of the previous dS^T has read it
        if (nG > 0 && (!mbar_wait_warp(b_pfree, (nG - 1) & 1, abort_flag) ||
                       !mbar_wait_warp(b_dsfree, (nG - 1) & 1, abort_flag))) { ok = false; break; }
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
  } else {  // ---- the dS store warp: each finished dS^T tile to its block of the dS buffer
    uint32_t nG = 0;
    bool ok = true;
    for (int ki = 0; ok && ki < n_mine; ki++) {
      const int i = sched_item(sch, ki);
      const Item it = item(i);
      for (int k = 0; k < it.nit; k++, nG++) {
        if (!mbar_wait_warp(b_pfull, nG & 1, abort_flag)) { ok = false; break; }
        if (lane == 0) {
          bulk_store(p.ds + ds_block(it.bh, nq, it.kt, it.kt + k) * PTILE, sDST, PTILE);
          bulk_wait_read();
          mbar_arrive(b_dsfree);
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait_all();
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
  return kernel_smem_attr(kernel, (int)bytes);
}

// The schedule table of one kernel at one shape (see AttnSched).  kind 0: the
// forward (item i = pair of query tiles qt0, qt0 + 1 with qt0 = 2 (npair - 1 -
// i / BH): qt0 + 1 + qt0 + 2 key tiles); kind 1: dK/dV (key tile kt = i / BH:
// nq - kt query tiles); kind 2: dQ (query tile qt = nq - 1 - i / BH: qt + 1 key
// tiles).  Built once per (kind, BH, nq, grid) and kept.
const AttnSched& attn_schedule(int kind, int BH, int nq, int grid) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, std::unique_ptr<AttnSched>> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto& slot = cache[std::make_tuple(kind, BH, nq, grid)];
  if (slot) return *slot;
  slot.reset(new AttnSched());
  AttnSched& s = *slot;
  const int npair = (nq + 1) / 2;
  const long long n_items = (long long)BH * (kind == 0 ? npair : nq);
  s.n = 0;
  if (n_items <= 0 || n_items > SCHED_MAX_ITEMS || grid <= 0 || grid > SCHED_MAX_CTAS) return s;
  auto weight = [&](int i) -> long long {
    const int cls = i / BH;
    if (kind == 0) {
      const int qt0 = 2 * (npair - 1 - cls);
      return qt0 + 1 + (qt0 + 1 < nq ? qt0 + 2 : 0);
    }
    if (kind == 1) return nq - cls;
    return nq - cls;  // dQ: qt + 1 with qt = nq - 1 - cls
  };
  using Slot = std::pair<long long, int>;  // (work so far, CTA)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> pq;
  for (int c = 0; c < grid; c++) pq.push({0, c});
  std::vector<int> owner((size_t)n_items), count((size_t)grid, 0);
  for (int i = 0; i < (int)n_items; i++) {
    const Slot top = pq.top();
    pq.pop();
    owner[i] = top.second;
    count[top.second]++;
    pq.push({top.first + weight(i), top.second});
  }
  s.first[0] = 0;
  for (int c = 0; c < grid; c++) s.first[c + 1] = (uint16_t)(s.first[c] + count[c]);
  std::vector<int> pos(s.first, s.first + grid);
  for (int i = 0; i < (int)n_items; i++) s.item[pos[owner[i]]++] = (uint16_t)i;
  s.n = (int)n_items;
  return s;
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
  {
    cudaError_t e = set_smem(attn_fwd_tc_kernel, FWD_SMEM);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tq;
  if (!tc_make_map(&tq, qkv, 3 * (uint64_t)C, (uint64_t)B * T, 3 * (uint64_t)C, HD, 128)) return cudaErrorInvalidValue;
  AttnParams p{out, lse, nullptr, nullptr, nullptr, B, T, C, H, LOG2E / sqrtf((float)HD), 1.f / sqrtf((float)HD), flags};
  const int npair = (T / 128 + 1) / 2;
  const long long items = (long long)B * H * npair;
  const int sms = tc_num_sms();
  gpt2_count_launches(1);
  const int grid = (int)(items < sms ? items : sms);
  const AttnSched& sch = attn_schedule(0, B * H, T / 128, grid);
  launch_k(attn_fwd_tc_kernel, dim3((unsigned)grid), dim3(FWD_THREADS), FWD_SMEM, st, tq, p, sch);
  return cudaGetLastError();
}

size_t attention_tc_ds_bytes(int B, int T, int H) {
  if (B <= 0 || T <= 0 || H <= 0 || T % 128) return 0;
  const long long nq = T / 128;
  return (size_t)((long long)B * H * nq * (nq + 1) / 2) * PTILE;
}

cudaError_t attention_backward_tc(bf16* dqkv, float* Dbuf, void* dS, const bf16* dout, const bf16* qkv,
                                  const bf16* out, const float* lse, int B, int T, int C, int H, int* flags,
                                  cudaStream_t st, bool d_ready) {
  if (!attention_tc_supported(B, T, C, H) || !flags) return cudaErrorNotSupported;
  if (((uintptr_t)qkv & 15) || ((uintptr_t)out & 15) || ((uintptr_t)dout & 15) || ((uintptr_t)dqkv & 15) ||
      ((uintptr_t)lse & 15) || ((uintptr_t)Dbuf & 15) || !dS || ((uintptr_t)dS & 15))
    return cudaErrorInvalidValue;
  {
    cudaError_t e = set_smem(attn_bwd_dq_tc_kernel, DQ_SMEM);
    if (e == cudaSuccess) e = set_smem(attn_bwd_dkv_tc_kernel, DKV_SMEM);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tq, td;
  if (!tc_make_map(&tq, qkv, 3 * (uint64_t)C, (uint64_t)B * T, 3 * (uint64_t)C, HD, 128) ||
      !tc_make_map(&td, dout, (uint64_t)C, (uint64_t)B * T, (uint64_t)C, HD, 128))
    return cudaErrorInvalidValue;
  AttnParams p{dqkv, const_cast<float*>(lse), Dbuf, out, dout, B, T, C, H, LOG2E / sqrtf((float)HD),
               1.f / sqrtf((float)HD), flags, (uint8_t*)dS};
  const long long items = (long long)B * H * (T / 128);
  const int sms = tc_num_sms();
  const unsigned grid = (unsigned)(items < sms ? items : sms);
  const long long n8 = (long long)B * T * C / 8;
  gpt2_count_launches(d_ready ? 2 : 3);
  cudaError_t e;
  if (!d_ready) {
    launch_k(attn_rowdot_kernel, dim3((unsigned)((n8 + 255) / 256)), dim3(256), 0, st, Dbuf, dout, out, n8, T, C, H);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  launch_k(attn_bwd_dkv_tc_kernel, dim3(grid), dim3(BWD_THREADS), DKV_SMEM, st, tq, td, p,
           attn_schedule(1, B * H, T / 128, (int)grid));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_k(attn_bwd_dq_tc_kernel, dim3(grid), dim3(DQ_THREADS), DQ_SMEM, st, tq, (const uint8_t*)dS, p,
           attn_schedule(2, B * H, T / 128, (int)grid));
  return cudaGetLastError();
}
