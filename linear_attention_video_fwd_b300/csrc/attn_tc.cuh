// Block-sparse flash-attention forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 inputs, head_dim D in {64, 128}, 128-token
// blocks. A D = 128 tile is two 64-dim halves (one 128B swizzle atom wide
// each); a D = 64 tile is one.
//
// Work unit: one CTA per (batch*head, query-block pair {2P, 2P+1}). The two
// query tiles share one stream of K/V tiles: the union of the two CSR rows,
// precomputed at mask build time as entries (J << 2 | live bits), so every
// key block that either tile needs is fetched once. CTAs run head-major and,
// within a head, longest pair first (LPT), so the K/V working set in flight
// stays in L2 and the grid tail holds the shortest pairs.
//
// 384 threads (12 warps):
//   warp 0       TMA producer: Q tiles once, then K_u and V_u of every union
//                entry u into rings of NK and NV stages (128B-swizzled);
//   warp 1       MMA issuer (one thread): for tile t live at u,
//                S_t = Q_t K_u^T into TMEM, and O_t += P_t V_u once the
//                softmax of tile t has written P_t;
//   warps 2, 3   idle (they only take part in set-up and tear-down);
//   warps 4..7   softmax / correction / epilogue of tile 0,
//   warps 8..11  the same for tile 1; thread r of a group owns query row r
//                (TMEM lane r), so row max and row sum need no shuffles.
// Tensor-pipe order per union entry: PV_0(prev), QK_0(u), PV_1(prev), QK_1(u):
// the softmax of tile 0 overlaps the MMAs of tile 1 and the other way round.
//
// TMEM (512 columns): tile t uses columns [256t, 256t + 128) for S_t (fp32;
// P_t is written back over its first 64 columns as packed bf16 pairs) and
// [256t + 128, 256t + 128 + D) for the O_t accumulator.
//
// Online softmax in the log2 domain: the running max used for exponentiation
// is only raised when a block's max exceeds it by more than TAU = 16 (so
// P <= 2^16, far inside bf16 and fp32 range, and O and l stay exact to
// rounding); raising it rescales O_t in TMEM after waiting for the previous
// PV_t to complete. A block is first exponentiated against the running max
// with no max pass; only when its weights sum above 2^(TAU - 1) (or m_used
// is still -inf) does the warp take the max, maybe rescale, and exponentiate
// again, so the weights are those of the max-first order either way.
//
// Every mbarrier wait is bounded (clock64 limit): on a timeout the CTA records
// VA_ERR_TIMEOUT in the device error word, drains its own copies and MMAs
// with bounded waits, frees its TMEM and exits.
#pragma once

#include "common.cuh"

namespace va {

constexpr int TC_BLK = 128;
constexpr int TC_D = 128;
constexpr int TC_NK = 2;                    // K ring stages
constexpr int TC_NV = 2;                    // V ring stages
constexpr int TC_THREADS = 384;
constexpr int TC_TILE_BYTES = TC_BLK * TC_D * 2;  // 32 KB: one 128 x 128 bf16 tile
constexpr int TC_HALF_BYTES = TC_TILE_BYTES / 2;  // 16 KB: 128 rows x 64 dims
constexpr int TC_SMEM_BYTES = 1024 + TC_TILE_BYTES * (2 + TC_NK + TC_NV);
// Rescale threshold of the online softmax (log2 units), and the block sum
// below which a block needs no max pass (every weight is then below
// 2^(TAU - 1)); the compensated attention uses both as well.
constexpr float TC_TAU = 16.0f;
constexpr float TC_FAST_SUM = 32768.0f;
// Register split (setmaxnreg): the kernel is compiled to TC_LAUNCH_REGS per
// thread; warpgroup 0 (producer, MMA, idle warps) gives registers back and the
// two softmax warpgroups take them. 128 * DEC + 256 * INC must not exceed
// 384 * TC_LAUNCH_REGS, or the increase would wait forever; the host checks
// the compiled register count before every first launch.
constexpr int TC_LAUNCH_REGS = 168;
constexpr int TC_REGS_DEC = 72;
constexpr int TC_REGS_INC = 216;
static_assert(128 * TC_REGS_DEC + 256 * TC_REGS_INC <= TC_THREADS * TC_LAUNCH_REGS,
              "register split exceeds the launch allocation");
static_assert(TC_NV >= 2 && TC_NV <= 4, "V stage bookkeeping assumes 2..4 stages");

// Sizes that depend on the head dimension D of the forward kernel.
template <int D>
struct TcDim {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kTileBytes = TC_BLK * D * 2;   // one 128 x D bf16 tile
  static constexpr int kHalves = D / 64;              // 64-dim TMA boxes per tile
  static constexpr int kSmemBytes = 1024 + kTileBytes * (2 + TC_NK + TC_NV);
};

struct TcArgs {
  const int* row_ptr;  // [nqb + 1] CSR rows
  const int* col;      // [nnz] live key blocks per row (ascending)
  const int* pcol;     // pair unions: pair P's entries start at row_ptr[2P]
  const int* plen;     // [npairs] union length per pair
  const int* porder;   // [npairs] pairs, longest first
  __nv_bfloat16* out;
  float* lse;
  int N, nqb, npairs;
  float scale_log2;
  long long wait_limit;
};

// barrier slots
enum : int {
  B_Q_FULL = 0,                  // 2 (per tile)
  B_K_FULL = B_Q_FULL + 2,
  B_K_EMPTY = B_K_FULL + TC_NK,
  B_V_FULL = B_K_EMPTY + TC_NK,
  B_V_EMPTY = B_V_FULL + TC_NV,
  B_S_FULL = B_V_EMPTY + TC_NV,  // 2 (per tile)
  B_P_FULL = B_S_FULL + 2,       // 2 (per tile), 128 arrivals
  B_O_DONE = B_P_FULL + 2,       // 2 (per tile)
  B_DRAIN = B_O_DONE + 2,
  B_COUNT = B_DRAIN + 1
};

// S = Q K^T over the 128 dims (8 steps of K = 16) into TMEM at s_tmem; Q and
// K are 128B-swizzled K-major tiles (two 64-dim halves). Used by the kernels
// whose issue loops are not grouped.
__device__ __forceinline__ void tc_issue_qk(uint32_t s_tmem, uint32_t sQ, uint32_t sK) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
  for (int k = 0; k < TC_D / 16; ++k) {
    const uint32_t off = (k >> 2) * TC_HALF_BYTES + (k & 3) * 32;
    umma_ss(s_tmem, sw128_desc(sQ + off, 16, 1024), sw128_desc(sK + off, 16, 1024), idesc, k > 0);
  }
}

// O (+)= P V with P from TMEM at p_tmem and V an MN-major tile at sV.
__device__ __forceinline__ void tc_issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t sV,
                                            bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int k = 0; k < TC_BLK / 16; ++k) {
    umma_ts(o_tmem, p_tmem + k * 8, sw128_desc(sV + k * 2048, TC_HALF_BYTES, 1024), idesc,
            (accumulate || k > 0) ? 1u : 0u);
  }
}

// The tensor pipe accepts an MMA about as fast as it runs one (64 cycles for
// 128 x 128 x 16), so every instruction the issuing thread spends between
// two MMAs of a product is idle pipe. A product's eight K = 16 steps are
// therefore issued from one asm block, with descriptors precomputed: a step
// changes only the start address field (low 14 bits) of a 128B-swizzled
// tile's descriptor, i.e. low word + (byte offset >> 4), with no carry since
// shared-memory addresses stay below 256 KB.

// S = Q K^T: A and B are K-major tiles, steps 16 elements (32 B) apart
// within a 64-wide half and TC_HALF_BYTES between the halves.
template <int D>
__device__ __forceinline__ void tc_qk_group(uint32_t d, uint32_t alo, uint32_t blo, uint32_t hi);

// D = 64: four steps within the one 64-dim atom.
template <>
__device__ __forceinline__ void tc_qk_group<64>(uint32_t d, uint32_t alo, uint32_t blo,
                                                uint32_t hi) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t"
      "setp.ne.b32 pf, %3, %3;\n\tsetp.eq.b32 pt, %3, %3;\n\t"
      "mov.b64 a, {%4, %2};\n\tmov.b64 b, {%5, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pf;\n\t"
      "mov.b64 a, {%6, %2};\n\tmov.b64 b, {%7, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t"
      "mov.b64 a, {%8, %2};\n\tmov.b64 b, {%9, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t"
      "mov.b64 a, {%10, %2};\n\tmov.b64 b, {%11, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t}"
      ::"r"(d), "r"(idesc), "r"(hi), "r"(0u), "r"(alo), "r"(blo), "r"(alo + 2u), "r"(blo + 2u),
      "r"(alo + 4u), "r"(blo + 4u), "r"(alo + 6u), "r"(blo + 6u)
      : "memory");
}

// D = 128: four steps per 64-dim half.
template <>
__device__ __forceinline__ void tc_qk_group<128>(uint32_t d, uint32_t alo, uint32_t blo,
                                                 uint32_t hi) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#define TC_QK_OFS(k) ((((k) >> 2) * TC_HALF_BYTES + ((k) & 3) * 32) >> 4)
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t"
      "setp.ne.b32 pf, %3, %3;\n\tsetp.eq.b32 pt, %3, %3;\n\t"
      "mov.b64 a, {%4, %2};\n\tmov.b64 b, {%5, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pf;\n\t"
      "mov.b64 a, {%6, %2};\n\tmov.b64 b, {%7, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t"
      "mov.b64 a, {%8, %2};\n\tmov.b64 b, {%9, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t"
      "mov.b64 a, {%10, %2};\n\tmov.b64 b, {%11, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t"
      "mov.b64 a, {%12, %2};\n\tmov.b64 b, {%13, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t"
      "mov.b64 a, {%14, %2};\n\tmov.b64 b, {%15, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t"
      "mov.b64 a, {%16, %2};\n\tmov.b64 b, {%17, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t"
      "mov.b64 a, {%18, %2};\n\tmov.b64 b, {%19, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %1, pt;\n\t}"
      ::"r"(d), "r"(idesc), "r"(hi), "r"(0u),
      "r"(alo + TC_QK_OFS(0)), "r"(blo + TC_QK_OFS(0)), "r"(alo + TC_QK_OFS(1)),
      "r"(blo + TC_QK_OFS(1)), "r"(alo + TC_QK_OFS(2)), "r"(blo + TC_QK_OFS(2)),
      "r"(alo + TC_QK_OFS(3)), "r"(blo + TC_QK_OFS(3)), "r"(alo + TC_QK_OFS(4)),
      "r"(blo + TC_QK_OFS(4)), "r"(alo + TC_QK_OFS(5)), "r"(blo + TC_QK_OFS(5)),
      "r"(alo + TC_QK_OFS(6)), "r"(blo + TC_QK_OFS(6)), "r"(alo + TC_QK_OFS(7)),
      "r"(blo + TC_QK_OFS(7))
      : "memory");
#undef TC_QK_OFS
}

// O (+)= P V: A (P, bf16 pairs) from TMEM columns p + 8k, B (V) an MN-major
// tile of D columns whose start advances 16 rows (2048 B) per step (the
// 64-dim halves of a D = 128 tile lie TC_HALF_BYTES apart). The first step
// accumulates only if `accumulate`.
template <int D>
__device__ __forceinline__ void tc_pv_group(uint32_t d, uint32_t p, uint32_t blo, uint32_t hi,
                                            bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 b;\n\t"
      "setp.ne.b32 pf, %3, 0;\n\tsetp.eq.b32 pt, %3, %3;\n\t"
      "mov.b64 b, {%5, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], b, %1, pf;\n\t"
      "mov.b64 b, {%7, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], b, %1, pt;\n\t"
      "mov.b64 b, {%9, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], b, %1, pt;\n\t"
      "mov.b64 b, {%11, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%10], b, %1, pt;\n\t"
      "mov.b64 b, {%13, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%12], b, %1, pt;\n\t"
      "mov.b64 b, {%15, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%14], b, %1, pt;\n\t"
      "mov.b64 b, {%17, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%16], b, %1, pt;\n\t"
      "mov.b64 b, {%19, %2};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%18], b, %1, pt;\n\t}"
      ::"r"(d), "r"(idesc), "r"(hi), "r"(accumulate ? 1u : 0u),
      "r"(p + 0), "r"(blo + 0 * 128), "r"(p + 8), "r"(blo + 1 * 128),
      "r"(p + 16), "r"(blo + 2 * 128), "r"(p + 24), "r"(blo + 3 * 128),
      "r"(p + 32), "r"(blo + 4 * 128), "r"(p + 40), "r"(blo + 5 * 128),
      "r"(p + 48), "r"(blo + 6 * 128), "r"(p + 56), "r"(blo + 7 * 128)
      : "memory");
}


__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (d0, d1) = (a0 * b + c, a1 * b + c) as one packed f32x2 FMA.
__device__ __forceinline__ void ffma2_bc(float& d0, float& d1, float a0, float a1, float b,
                                         float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// Softmax of one tile: its CSR row, its TMEM columns and its barriers. With
// SUB (64-token mask blocks) the tile is two query blocks and an entry two key
// blocks: the tile walks the CTA's union stream (entries pbeg .. pbeg + nu)
// for those with its tile bit, and a 64-key half that is not live for this
// row's query block takes part in neither the max nor the sum.
template <int D, bool SUB = false>
__device__ __forceinline__ void tc_softmax_tile(const TcArgs& a, int tile, int I, int bh,
                                                uint32_t tmem, uint64_t* bars,
                                                volatile int* abort_p, int pbeg = 0,
                                                int nu = 0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;               // TMEM lane quarter of this warp
  const int r = wq * 32 + lane;          // query row within the tile
  const int row = I * TC_BLK + r;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + tile * 256 + lane_off;
  const uint32_t tO = tS + 128;
  const uint32_t bS = smem_u32(&bars[B_S_FULL + tile]);
  const uint32_t bP = smem_u32(&bars[B_P_FULL + tile]);
  const uint32_t bO = smem_u32(&bars[B_O_DONE + tile]);
  const long long lim = a.wait_limit;
  const float sl2 = a.scale_log2;
  int n = nu, tail_valid = TC_BLK;
  if constexpr (!SUB) {
    const int beg = a.row_ptr[I];
    n = a.row_ptr[I + 1] - beg;
    // Only the last live block of a row can be the ragged tail block.
    if (n > 0 && a.col[beg + n - 1] == a.nqb - 1) tail_valid = a.N - (a.nqb - 1) * TC_BLK;
  }

  float m_used = -INFINITY, l = 0.f;
  bool ok = true;
  int nl = 0;  // entries of this tile so far (SUB: the union entries with its bit)
  for (int it = 0; it < n; ++it) {
    int valid = TC_BLK, lo_end = 64, hi_end = 128;  // live key columns [0, lo_end), [64, hi_end)
    if constexpr (SUB) {
      const int e = a.pcol[pbeg + it];
      if (!((e >> tile) & 1)) continue;
      const int jc = e >> 10;
      const int sb = (e >> (2 + 4 * tile + 2 * (r >> 6))) & 3;  // this row's block, both key halves
      valid = jc == a.nqb - 1 ? a.N - jc * TC_BLK : TC_BLK;
      lo_end = (sb & 1) ? min(valid, 64) : 0;
      hi_end = (sb & 2) ? valid : 64;
    } else {
      valid = it == n - 1 ? tail_valid : TC_BLK;
    }
    const int j = nl++;
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(bS, j & 1, lim, abort_p));
    if (!ok) break;
    tc_fence_after();
    float s[128];
    auto load_s = [&]() {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[i]);
      }
      tmem_wait_ld();
    };
    // P = 2^(s * sl2 - m_used), dead key columns zeroed
    auto exponentiate = [&]() {
      const float neg_m = -m_used;
#pragma unroll
      for (int i = 0; i < 128; i += 2) {
        ffma2_bc(s[i], s[i + 1], s[i], s[i + 1], sl2, neg_m);
        s[i] = ex2_approx(s[i]);
        s[i + 1] = ex2_approx(s[i + 1]);
      }
      if constexpr (SUB) {
        if (lo_end < 64) {
#pragma unroll
          for (int i = 0; i < 64; ++i) s[i] = i < lo_end ? s[i] : 0.f;
        }
        if (hi_end < 128) {
#pragma unroll
          for (int i = 64; i < 128; ++i) s[i] = i < hi_end ? s[i] : 0.f;
        }
      } else if (valid < TC_BLK) {
#pragma unroll
        for (int i = 1; i < 128; ++i) s[i] = (i < valid) ? s[i] : 0.f;
      }
    };
    float r0, r1, r2, r3;
    uint32_t pk[64];
    auto sum_pack = [&]() {
      r0 = r1 = r2 = r3 = 0.f;
#pragma unroll
      for (int i = 0; i < 128; i += 4) {
        fadd2_acc(r0, r1, s[i], s[i + 1]);
        fadd2_acc(r2, r3, s[i + 2], s[i + 3]);
        pk[i / 2] = pack_bf16x2(s[i], s[i + 1]);
        pk[i / 2 + 1] = pack_bf16x2(s[i + 2], s[i + 3]);
      }
    };
    load_s();
    // SUB: the entry may hold no live key of this row (a row of the other query
    // block of the tile is live): it then adds nothing (warp-uniform, as a
    // warp's 32 rows lie in one block)
    const bool row_live = !SUB || lo_end > 0 || hi_end > 64;
    // Pass 0 tries the block against the running max, with no max pass. A
    // block sum of at most 2^(TAU - 1) bounds every weight by it, so the block
    // max lies more than one below m_used + TAU and the rescale test of pass 1
    // would keep m_used: the weights are exactly those of pass 1. Any larger
    // sum, an infinite one (no max yet) or NaN sends the whole warp to pass 1,
    // which reloads S (P is not written over it yet), takes the max and maybe
    // rescales before exponentiating.
#pragma unroll 1
    for (int pass = 0;; ++pass) {
      if (pass == 1) {
        load_s();
        if constexpr (SUB) {
          if (row_live) {
            // dead columns take a live value of the block for the max, and a
            // zero weight in exponentiate()
            const float rep = lo_end > 0 ? s[0] : s[64];
            if (lo_end < 64) {
#pragma unroll
              for (int i = 0; i < 64; ++i) s[i] = i < lo_end ? s[i] : rep;
            }
            if (hi_end < 128) {
#pragma unroll
              for (int i = 64; i < 128; ++i) s[i] = i < hi_end ? s[i] : rep;
            }
          }
        } else if (valid < TC_BLK) {
          // Key columns >= valid hold zero-filled rows: give them a real value
          // of the block for the max, and a zero weight in exponentiate().
#pragma unroll
          for (int i = 1; i < 128; ++i) s[i] = (i < valid) ? s[i] : s[0];
        }
        // Largest scaled logit of the block (sl2 may be negative).
        float mx;
        if (sl2 >= 0.f) {
          float m0 = fmax3(s[0], s[1], s[2]), m1 = fmax3(s[3], s[4], s[5]);
          float m2 = fmax3(s[6], s[7], s[8]), m3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
          for (int i = 12; i < 124; i += 8) {
            m0 = fmax3(m0, s[i], s[i + 1]);
            m1 = fmax3(m1, s[i + 2], s[i + 3]);
            m2 = fmax3(m2, s[i + 4], s[i + 5]);
            m3 = fmax3(m3, s[i + 6], s[i + 7]);
          }
          mx = fmax3(fmax3(m0, m1, s[124]), fmax3(m2, m3, s[125]), fmaxf(s[126], s[127]));
        } else {
          float m0 = fmin3(s[0], s[1], s[2]), m1 = fmin3(s[3], s[4], s[5]);
          float m2 = fmin3(s[6], s[7], s[8]), m3 = fmin3(s[9], s[10], s[11]);
#pragma unroll
          for (int i = 12; i < 124; i += 8) {
            m0 = fmin3(m0, s[i], s[i + 1]);
            m1 = fmin3(m1, s[i + 2], s[i + 3]);
            m2 = fmin3(m2, s[i + 4], s[i + 5]);
            m3 = fmin3(m3, s[i + 6], s[i + 7]);
          }
          mx = fmin3(fmin3(m0, m1, s[124]), fmin3(m2, m3, s[125]), fminf(s[126], s[127]));
        }
        const float m_cand = mx * sl2;
        const bool need = row_live && m_cand > m_used + TC_TAU;
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m_used - m_cand);
          m_used = m_cand;
          l *= alpha;
        }
        if (__any_sync(0xffffffffu, need && j > 0)) {
          // O_t holds the sum up to PV_t(j-1): wait for it, then rescale in TMEM.
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(bO, (j - 1) & 1, lim, abort_p));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tO + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(tO + c * 32, v);
          }
        }
      }
      exponentiate();
      sum_pack();
      if (pass == 1 ||
          !__any_sync(0xffffffffu, !((r0 + r1) + (r2 + r3) <= TC_FAST_SUM)))
        break;
    }
    if (!ok) break;
    l += (r0 + r1) + (r2 + r3);
    {
      uint32_t (&lo)[32] = *reinterpret_cast<uint32_t (*)[32]>(&pk[0]);
      uint32_t (&hi)[32] = *reinterpret_cast<uint32_t (*)[32]>(&pk[32]);
      tmem_st32(tS, lo);
      tmem_st32(tS + 32, hi);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bP);
  }
  // epilogue (SUB: a row that no entry made live ends with l = 0 and is
  // written as a row without live blocks)
  const long long obase = (static_cast<long long>(bh) * a.N + row) * D;
  if (nl > 0 && ok)
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(bO, (nl - 1) & 1, lim, abort_p));
  const bool empty_row = SUB && l == 0.f;
  if (nl > 0 && ok && !empty_row) {
    tc_fence_after();
    const float inv = 1.f / l;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tO + c * 32, v);
      tmem_wait_ld();
      if (row < a.N) {
        uint4* dst = reinterpret_cast<uint4*>(a.out + obase + c * 32);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]) * inv, __uint_as_float(v[q4 * 8 + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]) * inv, __uint_as_float(v[q4 * 8 + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]) * inv, __uint_as_float(v[q4 * 8 + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]) * inv, __uint_as_float(v[q4 * 8 + 7]) * inv);
          dst[q4] = w;
        }
      }
    }
    if (row < a.N && a.lse != nullptr)
      a.lse[static_cast<long long>(bh) * a.N + row] = (m_used + log2f(l)) * 0.69314718055994530942f;
  } else if ((nl == 0 || (empty_row && ok)) && row < a.N) {
    uint4* dst = reinterpret_cast<uint4*>(a.out + obase);
#pragma unroll
    for (int q4 = 0; q4 < D / 8; ++q4) dst[q4] = make_uint4(0, 0, 0, 0);
    if (a.lse != nullptr) a.lse[static_cast<long long>(bh) * a.N + row] = -INFINITY;
  }
}

template <int D, bool SUB = false>
__global__ void __launch_bounds__(TC_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[B_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ0 = smem_u32(smem);
  constexpr int kTile = TcDim<D>::kTileBytes;
  const uint32_t sK0 = sQ0 + 2 * kTile;
  const uint32_t sV0 = sK0 + TC_NK * kTile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int bh = blockIdx.x / a.npairs;
  const int P = a.porder[blockIdx.x % a.npairs];
  const int I0 = 2 * P, I1 = 2 * P + 1;
  const bool has1 = I1 < a.nqb;
  // SUB: the CTA's union starts at the offset of its first 64-token query row
  const int pbeg = a.row_ptr[SUB ? 2 * I0 : I0];
  const int nu = a.plen[P];
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (tid == 0) {
    abort_flag = 0;
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(B_Q_FULL + t), 1);
      mbar_init(bar(B_S_FULL + t), 1);
      mbar_init(bar(B_P_FULL + t), 128);
      mbar_init(bar(B_O_DONE + t), 1);
    }
    for (int s = 0; s < TC_NK; ++s) {
      mbar_init(bar(B_K_FULL + s), 1);
      mbar_init(bar(B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < TC_NV; ++s) {
      mbar_init(bar(B_V_FULL + s), 1);
      mbar_init(bar(B_V_EMPTY + s), 1);
    }
    mbar_init(bar(B_DRAIN), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile int* abort_p = &abort_flag;
  const long long lim = a.wait_limit;

  if (warp >= 4) {
    // ------------------------------------------- softmax / correction / out --
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(TC_REGS_INC));
    const int tile = (warp - 4) >> 2;
    if (tile == 0 || has1)
      tc_softmax_tile<D, SUB>(a, tile, tile == 0 ? I0 : I1, bh, tmem, bars, abort_p, pbeg, nu);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(TC_REGS_DEC));
  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && nu > 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      // a tile is kHalves boxes of 64 dims x 128 rows, TC_HALF_BYTES apart
      auto load_tile = [&](uint32_t dst, const CUtensorMap* map, uint32_t b, int row0) {
        mbar_arrive_expect_tx(b, kTile);
#pragma unroll
        for (int h = 0; h < TcDim<D>::kHalves; ++h)
          tma_load_3d(dst + h * TC_HALF_BYTES, map, b, 64 * h, row0, bh);
      };
      load_tile(sQ0, &map_q, bar(B_Q_FULL + 0), I0 * TC_BLK);
      if (has1) load_tile(sQ0 + kTile, &map_q, bar(B_Q_FULL + 1), I1 * TC_BLK);
      int issued_k = 0, issued_v = 0;
      for (int u = 0; u < nu; ++u) {
        const int J = a.pcol[pbeg + u] >> (SUB ? 10 : 2);
        const int sk = u % TC_NK, sv = u % TC_NV;
        const uint32_t sK = sK0 + sk * kTile, sV = sV0 + sv * kTile;
        if (u >= TC_NK &&
            !mbar_wait_bounded(bar(B_K_EMPTY + sk), ((u / TC_NK) & 1) ^ 1, lim, abort_p))
          break;
        load_tile(sK, &map_k, bar(B_K_FULL + sk), J * TC_BLK);
        issued_k = u + 1;
        if (u >= TC_NV &&
            !mbar_wait_bounded(bar(B_V_EMPTY + sv), ((u / TC_NV) & 1) ^ 1, lim, abort_p))
          break;
        load_tile(sV, &map_v, bar(B_V_FULL + sv), J * TC_BLK);
        issued_v = u + 1;
      }
      if (*abort_p) {
        // Drain: every copy issued must land before this CTA's shared memory
        // is released. Only the last NK (NV) loads of a ring can still be in
        // flight: a stage is reloaded only after its previous copy was used.
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(B_Q_FULL + 0), 0, lim, &no_abort);
        if (has1) {
          no_abort = 0;
          mbar_wait_bounded(bar(B_Q_FULL + 1), 0, lim, &no_abort);
        }
        for (int u = issued_k > TC_NK ? issued_k - TC_NK : 0; u < issued_k; ++u) {
          no_abort = 0;
          mbar_wait_bounded(bar(B_K_FULL + u % TC_NK), (u / TC_NK) & 1, lim, &no_abort);
        }
        for (int u = issued_v > TC_NV ? issued_v - TC_NV : 0; u < issued_v; ++u) {
          no_abort = 0;
          mbar_wait_bounded(bar(B_V_FULL + u % TC_NV), (u / TC_NV) & 1, lim, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0 && nu > 0) {
      const uint32_t sQ1 = sQ0 + kTile;
      bool ok = mbar_wait_bounded(bar(B_Q_FULL + 0), 0, lim, abort_p);
      if (ok && has1) ok = mbar_wait_bounded(bar(B_Q_FULL + 1), 0, lim, abort_p);
      // Descriptor halves of the Q tiles and of stage 0 of the K and V rings;
      // a stage's descriptor is the low word + stage * (tile bytes >> 4).
      const uint64_t dq0 = sw128_desc(sQ0, 16, 1024), dq1 = sw128_desc(sQ1, 16, 1024);
      const uint64_t dk = sw128_desc(sK0, 16, 1024);
      const uint64_t dv = sw128_desc(sV0, TC_HALF_BYTES, 1024);
      const uint32_t q_lo[2] = {static_cast<uint32_t>(dq0), static_cast<uint32_t>(dq1)};
      const uint32_t k_lo = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
      const uint32_t v_lo = static_cast<uint32_t>(dv), v_hi = static_cast<uint32_t>(dv >> 32);
      int pend[2] = {-1, -1};   // union entry whose PV is still to issue, per tile
      int cnt[2] = {0, 0};      // QKs issued per tile
      uint32_t outst = 0;       // per V stage, 2 bits: tiles still to read it
      // Issue PV_t for the pending entry of tile t (after its softmax wrote P_t).
      auto issue_pv = [&](int t) -> bool {
        const int pu = pend[t];
        const int jj = cnt[t] - 1;
        if (!mbar_wait_bounded(bar(B_P_FULL + t), jj & 1, lim, abort_p)) return false;
        const int sv = pu % TC_NV;
        if (!mbar_wait_bounded(bar(B_V_FULL + sv), (pu / TC_NV) & 1, lim, abort_p)) return false;
        tc_fence_after();
        tc_pv_group<D>(tmem + t * 256 + 128, tmem + t * 256, v_lo + sv * (kTile >> 4), v_hi,
                       jj > 0);
        umma_commit(bar(B_O_DONE + t));
        outst &= ~(1u << (2 * sv + t));
        if (((outst >> (2 * sv)) & 3u) == 0) umma_commit(bar(B_V_EMPTY + sv));
        pend[t] = -1;
        return true;
      };
      for (int u = 0; ok && u < nu; ++u) {
        const uint32_t f = static_cast<uint32_t>(a.pcol[pbeg + u]) & 3u;
        const int sk = u % TC_NK;
        outst |= f << (2 * (u % TC_NV));
        if (!(ok = mbar_wait_bounded(bar(B_K_FULL + sk), (u / TC_NK) & 1, lim, abort_p))) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (pend[t] >= 0 && !(ok = issue_pv(t))) break;
          if ((f >> t) & 1u) {
            tc_qk_group<D>(tmem + t * 256, q_lo[t], k_lo + sk * (kTile >> 4), k_hi);
            umma_commit(bar(B_S_FULL + t));
            pend[t] = u;
            ++cnt[t];
          }
        }
        if (!ok) break;
        umma_commit(bar(B_K_EMPTY + sk));
      }
      if (ok && pend[0] >= 0) ok = issue_pv(0);
      if (ok && pend[1] >= 0) ok = issue_pv(1);
      if (!ok) {
        // Drain this thread's MMAs before TMEM is released.
        umma_commit(bar(B_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(B_DRAIN), 0, lim, &no_abort);
      }
    }
  }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace va
