// Linear attention and LinVideo's mixed attention (LinVideo, gist.science
// 2510.08318, technical summary sec. 1: O(n) linear attention; sec. 2 A: per
// layer a scalar r mixes quadratic (r = 1) and linear (r = 0) attention) on
// the 5th-generation tensor cores, bf16, head_dim D = 64 or 128. Feature map
// phi(x) = elu(x) + 1; non-causal:
//   lin_i = phi(q_i)^T S / phi(q_i)^T z,  S = sum_j phi(k_j) v_j^T,  z = sum_j phi(k_j)
//   mix_i = r att_i + (1 - r) lin_i
//
// Three kernels, each HBM-bound (one read of K and V, one of Q, one write of
// the output):
//   lin_state_kernel  CTA (split, batch*head) streams 128-token tiles of K
//                     and V through rings of LN_NS stages; a warpgroup applies phi to the K tile in place
//                     (tokens >= N get 0), then S += phi(K)^T V and
//                     z += phi(K)^T 1 on the tensor cores (TMEM), and the
//                     split's partial {S, z} goes to global memory;
//   lin_prep_kernel   sums the partials and writes [S | z]^T ((D + 16) x D,
//                     rows past D zero) as bf16 pieces hi + lo (16 significant
//                     bits, so the product keeps fp32-level accuracy);
//   lin_out_kernel    persistent CTAs keep the pieces resident and stream
//                     128-token tiles of Q; num | den = phi(Q) [S | z] on the
//                     tensor cores, the epilogue writes num / den (mixed with
//                     the attention output already in `out` when r < 1).
// Every mbarrier wait is bounded; on a timeout the CTA records
// VA_ERR_TIMEOUT, drains its copies and MMAs and frees its TMEM.
#pragma once

#include "common.cuh"

namespace va {

constexpr int LN_HALF = 128 * 64 * 2;    // 16 KB: 128 tokens x 64 dims bf16 (one TMA box)
constexpr int LN_KSTAGE = 2 * LN_HALF;   // a K stage: phi(K) is the M = 128 MMA operand
constexpr int LN_STATE_THREADS = 640;    // producer, MMA, 2 idle warps, 4 phi warpgroups
constexpr int LN_OUT_THREADS = 768;
constexpr int LN_NS = 3;                 // ring stages (K and V, or Q)

// Sizes that depend on the head dimension D.
template <int D>
struct LnDim {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kHalves = D / 64;           // 64-dim TMA boxes per tile
  static constexpr int kTile = 128 * D * 2;        // 128 tokens x D dims bf16
  static constexpr int kNext = D + 16;             // rows of [S | z]^T (D + z + padding)
  static constexpr int kPieceHalf = kNext * 128;   // kNext rows x 64 dims bf16
  static constexpr int kPiece = kNext * D * 2;     // one bf16 piece of [S | z]^T
  static constexpr int kRow = D + 1;               // partial rows per split: S[.][n], n < D, z
  // K and V rings and the ones tile. With D = 64 the upper half of each K stage
  // stays zero, so phi(K)^T keeps M = 128 and S's rows past D come out zero.
  static constexpr int kStateSmem = 1024 + LN_NS * (LN_KSTAGE + kTile) + 4096;
  static constexpr int kOutSmem = 1024 + 2 * kPiece + (LN_NS + 1) * kTile;  // pieces, Q ring, O
};

// phi(x) = elu(x) + 1 = max(x, 0) + exp(n), n = max(min(x, 0), -100), on a
// pair of bf16 values in bf16x2 arithmetic. max and min are exact; exp(n) =
// 2^(n log2 e) with the argument formed as fma(n, c_hi, n c_lo) (c_hi + c_lo
// equals log2 e to 2^-17, so the constant adds no bias), then the hardware 2^x
// in bf16; the final add rounds once. For x > 0 the result is bf16(x + 1)
// exactly. For x <= 0 the relative error (measured over every bf16 input) is
// at most 0.75% on [-1, 0) and 1.5% on [-4, -1) and grows with |x| (the
// argument keeps 8 bits), while the absolute error stays below 0.008; after the
// fp32 sums this is below the bf16 rounding of the output. The clamp at -100
// (where exp is below the smallest bf16 normal) keeps -inf from forming
// -inf + inf: -inf gives 0, +inf gives +inf, NaN stays NaN.
__device__ __forceinline__ uint32_t lin_phi_bf16x2(uint32_t x) {
  uint32_t m, n, t, y, ex, r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(x), "r"(0u));
  asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(n) : "r"(x), "r"(0u));
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(n) : "r"(n), "r"(0xc2c8c2c8u));              // -100
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(n), "r"(0xbb2cbb2cu));               // c_lo = -0.0026245
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(y) : "r"(n), "r"(0x3fb93fb9u), "r"(t));  // c_hi = 1.4453125
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(ex) : "r"(y));
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(ex));
  return r;
}

// phi in place on NC 16-byte chunks (c0 .. c0 + NC - 1) of token row `row` of
// a 128-row x 64-dim 128B-swizzled half tile; rows with token >= N become 0.
// The chunks are visited in an order rotated by the row, so the warp's
// 16-byte accesses fall on distinct banks (the swizzle only permutes chunks
// within a row, and phi is elementwise); all loads are issued before the
// stores.
template <int NC>
__device__ __forceinline__ void lin_phi_chunks(uint8_t* half, int row, int c0, bool valid) {
  uint4 w[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c)
    w[c] = *reinterpret_cast<const uint4*>(half + row * 128 + ((c0 + c + row) & 7) * 16);
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    uint32_t* e = reinterpret_cast<uint32_t*>(&w[c]);
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = valid ? lin_phi_bf16x2(e[i]) : 0u;
    *reinterpret_cast<uint4*>(half + row * 128 + ((c0 + c + row) & 7) * 16) = w[c];
  }
}

// phi on a 128-token tile of D dims by the two warpgroups (h = 0, 1) of a
// pair, thread r of each: with D = 128 warpgroup h takes 64-dim half h, one
// row per thread; with D = 64 the 256 threads take half a row each. Rows
// >= nvalid become 0.
template <int D>
__device__ __forceinline__ void lin_phi_tile(uint8_t* tile, int h, int r, int nvalid) {
  if constexpr (D == 128) {
    lin_phi_chunks<8>(tile + h * LN_HALF, r, 0, r < nvalid);
  } else {
    const int t = h * 128 + r, row = t >> 1;
    lin_phi_chunks<4>(tile, row, (t & 1) * 4, row < nvalid);
  }
}

enum : int {
  LS_KF = 0,                   // LN_NS: K tile loaded
  LS_VF = LS_KF + LN_NS,       // LN_NS: V tile loaded
  LS_PHI = LS_VF + LN_NS,      // LN_NS: phi(K) written (256 arrivals)
  LS_EMPTY = LS_PHI + LN_NS,   // LN_NS: K and V tiles consumed by the MMAs
  LS_DONE = LS_EMPTY + LN_NS,  // accumulators complete
  LS_DRAIN = LS_DONE + 1,
  LS_COUNT = LS_DRAIN + 1
};

// Token tiles [t_lo, t_hi) of split `split` of `nsplit` over ntiles.
__device__ __forceinline__ void lin_range(int ntiles, int nsplit, int split, int& t_lo, int& t_hi) {
  const int per = (ntiles + nsplit - 1) / nsplit;
  t_lo = min(ntiles, split * per);
  t_hi = min(ntiles, t_lo + per);
}

// Grid (nsplit, BH), 640 threads. part[bh][split][n][dim]: n < D S[dim][n],
// n = D z[dim] (dims contiguous, so both the stores here and the loads of
// lin_prep_kernel are coalesced).
template <int D>
__global__ void __launch_bounds__(LN_STATE_THREADS, 1)
    lin_state_kernel(const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v, int N, float* __restrict__ part,
                     long long lim) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[LS_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  using Dm = LnDim<D>;
  uint8_t* kt = smem;                    // stage s at kt + s KSTAGE
  uint8_t* vt = smem + LN_NS * LN_KSTAGE;  // stage s at vt + s Dm::kTile
  uint8_t* ones = vt + LN_NS * Dm::kTile;  // 16 rows x 128 tokens of 1.0 (K-major halves)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bh = blockIdx.y, nsplit = gridDim.x;
  const int ntiles = (N + 127) / 128;
  int t_lo, t_hi;
  lin_range(ntiles, nsplit, split, t_lo, t_hi);
  const int nt = t_hi - t_lo;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < LN_NS; ++s) {
      mbar_init(bar(LS_KF + s), 1);
      mbar_init(bar(LS_VF + s), 1);
      mbar_init(bar(LS_PHI + s), 256);
      mbar_init(bar(LS_EMPTY + s), 1);
    }
    mbar_init(bar(LS_DONE), 1);
    mbar_init(bar(LS_DRAIN), 1);
    fence_barrier_init();
  }
  for (int i = tid; i < 4096 / 4; i += LN_STATE_THREADS)
    reinterpret_cast<uint32_t*>(ones)[i] = 0x3f803f80u;  // bf16 1.0 pairs
  if constexpr (D == 64) {  // the upper 64 dims of phi(K), never loaded, stay zero
    for (int i = tid; i < LN_NS * LN_HALF / 16; i += LN_STATE_THREADS) {
      const int s = i / (LN_HALF / 16), o = i % (LN_HALF / 16);
      reinterpret_cast<uint4*>(kt + s * LN_KSTAGE + LN_HALF)[o] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;  // S at [0, 128), z at [128, 144)
  volatile int* abort_p = &abort_flag;
  grid_dep_launch();  // lin_prep_kernel may be scheduled now; it waits for this grid

  if (warp == 0) {
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int issued = 0;
      for (int u = 0; u < nt; ++u) {
        const int s = u % LN_NS, row = (t_lo + u) * 128;
        if (u >= LN_NS &&
            !mbar_wait_bounded(bar(LS_EMPTY + s), ((u / LN_NS) & 1) ^ 1, lim, abort_p))
          break;
        mbar_arrive_expect_tx(bar(LS_KF + s), Dm::kTile);
        for (int hh = 0; hh < Dm::kHalves; ++hh)
          tma_load_3d(smem_u32(kt + s * LN_KSTAGE + hh * LN_HALF), &map_k, bar(LS_KF + s), 64 * hh,
                      row, bh);
        mbar_arrive_expect_tx(bar(LS_VF + s), Dm::kTile);
        for (int hh = 0; hh < Dm::kHalves; ++hh)
          tma_load_3d(smem_u32(vt + s * Dm::kTile + hh * LN_HALF), &map_v, bar(LS_VF + s),
                      64 * hh, row, bh);
        issued = u + 1;
      }
      if (*abort_p) {
        volatile int no_abort = 0;
        for (int u = issued > LN_NS ? issued - LN_NS : 0; u < issued; ++u) {
          no_abort = 0;
          mbar_wait_bounded(bar(LS_KF + u % LN_NS), (u / LN_NS) & 1, lim, &no_abort);
          no_abort = 0;
          mbar_wait_bounded(bar(LS_VF + u % LN_NS), (u / LN_NS) & 1, lim, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nt > 0) {
      // S (+)= phi(K)^T V: A = phi(K) (M = 128 dims) and B = V (N = D), both
      // MN-major (dims contiguous), K = 16 tokens per MMA; z (+)= phi(K)^T 1
      // with a K-major ones tile, N = 16.
      constexpr uint32_t id_s = idesc_bf16_f32(128, D, 1, 1);
      constexpr uint32_t id_z = idesc_bf16_f32(128, 16, 1, 0);
      const uint32_t sOnes = smem_u32(ones);
      bool ok = true;
      for (int u = 0; u < nt; ++u) {
        const int s = u % LN_NS;
        const uint32_t ph = (u / LN_NS) & 1;
        if (!(ok = mbar_wait_bounded(bar(LS_PHI + s), ph, lim, abort_p))) break;
        if (!(ok = mbar_wait_bounded(bar(LS_VF + s), ph, lim, abort_p))) break;
        tc_fence_after();
        const uint32_t sK = smem_u32(kt + s * LN_KSTAGE), sV = smem_u32(vt + s * Dm::kTile);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a = sw128_desc(sK + k * 2048, LN_HALF, 1024);
          umma_ss(tmem, a, sw128_desc(sV + k * 2048, LN_HALF, 1024), id_s, (u | k) ? 1u : 0u);
          umma_ss(tmem + 128, a, sw128_desc(sOnes + (k >> 2) * 2048 + (k & 3) * 32, 16, 1024),
                  id_z, (u | k) ? 1u : 0u);
        }
        umma_commit(bar(LS_EMPTY + s));
      }
      if (ok) umma_commit(bar(LS_DONE));
      else {
        umma_commit(bar(LS_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(LS_DRAIN), 0, lim, &no_abort);
      }
    }
  } else if (warp >= 4) {
    // Two pairs of warpgroups take alternate tiles: pair g transforms tiles
    // u = g, g + 2, ... (lin_phi_tile splits a tile between the pair). Tile u - 3,
    // the previous user of stage s, belongs to the other pair, so the pair
    // first waits for that tile's phi: until then the K-full barrier of stage s
    // may sit two phases behind tile u and its parity would match too early.
    const int r = (warp & 3) * 32 + lane, h = ((warp - 4) >> 2) & 1, g = (warp - 4) >> 3;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    for (int u = g; u < nt; u += 2) {
      const int s = u % LN_NS;
      const uint32_t ph = (u / LN_NS) & 1;
      if (u >= LN_NS &&
          !(ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(LS_PHI + s), ph ^ 1, lim, abort_p))))
        break;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(LS_KF + s), ph, lim, abort_p))))
        break;
      lin_phi_tile<D>(kt + s * LN_KSTAGE, h, r, N - (t_lo + u) * 128);
      fence_proxy_async_smem();
      mbar_arrive(bar(LS_PHI + s));
    }
    // The epilogue is the warps of 4..7 whose TMEM lanes hold dims (r < D);
    // thread r stores column r.
    if (h == 0 && g == 0 && (warp & 3) * 32 < D) {
      float* out = part + (static_cast<long long>(bh) * nsplit + split) * Dm::kRow * D + r;
      if (nt == 0) {
        for (int n = 0; n < Dm::kRow; ++n) out[n * D] = 0.f;
      } else if (ok && __all_sync(0xffffffffu, mbar_wait_bounded(bar(LS_DONE), 0, lim, abort_p))) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) out[(c * 32 + i) * D] = __uint_as_float(v[i]);
        }
        uint32_t zv[16];
        tmem_ld16(tmem + lane_off + 128, zv);
        tmem_wait_ld();
        out[D * D] = __uint_as_float(zv[0]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// [S | z]^T of each batch*head from the split partials, as bf16 pieces:
// piece[bh][p][n][dim], p = 0 hi, 1 lo, n < D S[dim][n], n = D z[dim],
// n > D zero. Grid (D + 16, BH), D threads (one per dim). Launched as a
// programmatic dependent of lin_state_kernel: it waits for that grid before
// reading the partials.
template <int D>
__global__ void lin_prep_kernel(const float* __restrict__ part, int nsplit,
                                __nv_bfloat16* __restrict__ piece) {
  constexpr int kRow = LnDim<D>::kRow, kNext = LnDim<D>::kNext;
  grid_dep_launch();
  grid_dep_wait();
  const int n = blockIdx.x, bh = blockIdx.y, dim = threadIdx.x;
  float acc = 0.f;
  if (n <= D) {
    const float* pp = part + static_cast<long long>(bh) * nsplit * kRow * D + n * D + dim;
    for (int s = 0; s < nsplit; ++s) acc += pp[static_cast<long long>(s) * kRow * D];
  }
  const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
  const __nv_bfloat16 lo = __float2bfloat16_rn(acc - __bfloat162float(hi));
  const long long o = ((static_cast<long long>(bh) * 2) * kNext + n) * D + dim;
  piece[o] = hi;
  piece[o + static_cast<long long>(kNext) * D] = lo;
}

enum : int {
  LO_PF = 0,                 // pieces loaded
  LO_QF = 1,                 // LN_NS: Q tile loaded
  LO_QE = LO_QF + LN_NS,     // LN_NS: Q tile read into registers by its phi pair (256 arrivals)
  LO_PHI = LO_QE + LN_NS,    // 2: phi(Q) written to TMEM operand buffer a (256 arrivals)
  LO_ABE = LO_PHI + 2,       // 2: operand buffer a read by the MMAs
  LO_AF = LO_ABE + 2,        // 2: accumulator full
  LO_AE = LO_AF + 2,         // 2: accumulator read (128 arrivals)
  LO_DRAIN = LO_AE + 2,
  LO_COUNT = LO_DRAIN + 1
};

// TMEM columns of the output kernel: accumulator b at [256 b, 256 b + D + 16);
// phi(Q) operand buffer a (128 rows x D bf16, two per 32-bit column) at
// column 160 + 256 a, past the accumulator of its half.
__device__ __forceinline__ uint32_t ln_opd(int a) { return 160u + 256u * static_cast<uint32_t>(a); }

// Grid (nsplit, BH), 768 threads: warp 0 TMA producer, warp 1 MMA issuer,
// warps 8..11 epilogue (thread r owns token row r of the tile; the tile goes
// out through shared memory and a TMA store), and two pairs of warpgroups
// that take alternate tiles: warps 4..7 and 12..15 the even tiles (TMEM
// operand buffer 0), warps 16..19 and 20..23 the odd ones (buffer 1). A pair
// reads its Q tile into registers, releases the ring stage at once, and writes
// phi(Q) as the MMA's A operand into its TMEM buffer; the MMA is then
// TMEM x shared memory (the [S | z]^T pieces). out = num / den, or
// r_mix * out + (1 - r_mix) * num / den when mix != 0 (out then holds the
// attention output on entry).
template <int D>
__global__ void __launch_bounds__(LN_OUT_THREADS, 1)
    lin_out_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_p, const __grid_constant__ CUtensorMap map_o,
                   int N, __nv_bfloat16* __restrict__ out,
                   int mix, float r_mix, long long lim) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[LO_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  using Dm = LnDim<D>;
  uint8_t* pc = smem;                    // piece p at pc + p kPiece
  uint8_t* qt = smem + 2 * Dm::kPiece;   // Q stage s at qt + s kTile
  uint8_t* ot = qt + LN_NS * Dm::kTile;  // output tile staged for the TMA store
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int ntiles = (N + 127) / 128;
  int t_lo, t_hi;
  lin_range(ntiles, gridDim.x, split, t_lo, t_hi);
  const int nt = t_hi - t_lo;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar(LO_PF), 1);
    for (int s = 0; s < LN_NS; ++s) {
      mbar_init(bar(LO_QF + s), 1);
      mbar_init(bar(LO_QE + s), 256);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(LO_PHI + b), 256);
      mbar_init(bar(LO_ABE + b), 1);
      mbar_init(bar(LO_AF + b), 1);
      mbar_init(bar(LO_AE + b), 128);
    }
    mbar_init(bar(LO_DRAIN), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;  // accumulator b at [256 b, 256 b + 144)
  volatile int* abort_p = &abort_flag;

  if (warp == 0) {
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_p);
      tma_prefetch_desc(&map_o);
      int issued = 0;
      auto load_q = [&](int u) {
        const int s = u % LN_NS, row = (t_lo + u) * 128;
        mbar_arrive_expect_tx(bar(LO_QF + s), Dm::kTile);
        for (int hh = 0; hh < Dm::kHalves; ++hh)
          tma_load_3d(smem_u32(qt + s * Dm::kTile + hh * LN_HALF), &map_q, bar(LO_QF + s), 64 * hh,
                      row, bh);
        issued = u + 1;
      };
      // The first Q tiles need no wait. The pieces are the previous kernel's
      // output, so under a programmatic dependent launch they load after it.
      for (int u = 0; u < nt && u < LN_NS; ++u) load_q(u);
      grid_dep_wait();
      mbar_arrive_expect_tx(bar(LO_PF), 2 * Dm::kPiece);
      for (int p = 0; p < 2; ++p)
        for (int h = 0; h < Dm::kHalves; ++h)
          tma_load_3d(smem_u32(pc + p * Dm::kPiece + h * Dm::kPieceHalf), &map_p, bar(LO_PF),
                      64 * h, p * Dm::kNext, bh);
      for (int u = LN_NS; u < nt; ++u) {
        if (!mbar_wait_bounded(bar(LO_QE + u % LN_NS), ((u / LN_NS) & 1) ^ 1, lim, abort_p)) break;
        load_q(u);
      }
      if (*abort_p) {
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(LO_PF), 0, lim, &no_abort);
        for (int u = issued > LN_NS ? issued - LN_NS : 0; u < issued; ++u) {
          no_abort = 0;
          mbar_wait_bounded(bar(LO_QF + u % LN_NS), (u / LN_NS) & 1, lim, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nt > 0) {
      // num | den = phi(Q) [S | z]: A = phi(Q) from TMEM (K-major), B = [S | z]^T
      // K-major in shared memory (D + 16 rows), two pieces accumulated in fp32.
      constexpr uint32_t id = idesc_bf16_f32(128, Dm::kNext, 0, 0);
      const uint32_t sP = smem_u32(pc);
      bool ok = mbar_wait_bounded(bar(LO_PF), 0, lim, abort_p);
      for (int u = 0; ok && u < nt; ++u) {
        const int b = u & 1;  // operand buffer and accumulator of the tile
        if (!(ok = mbar_wait_bounded(bar(LO_PHI + b), (u >> 1) & 1, lim, abort_p))) break;
        if (u >= 2 &&
            !(ok = mbar_wait_bounded(bar(LO_AE + b), ((u >> 1) & 1) ^ 1, lim, abort_p)))
          break;
        tc_fence_after();
        const uint32_t tA = tmem + ln_opd(b);
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            umma_ts(tmem + b * 256, tA + k * 8,
                    sw128_desc(sP + p * Dm::kPiece + (k >> 2) * Dm::kPieceHalf + (k & 3) * 32, 16,
                               1024),
                    id, (p | k) ? 1u : 0u);
        umma_commit(bar(LO_ABE + b));
        umma_commit(bar(LO_AF + b));
      }
      if (!ok) {
        umma_commit(bar(LO_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(LO_DRAIN), 0, lim, &no_abort);
      }
    }
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    const int r = (warp & 3) * 32 + lane;
    const int h = (warp >= 12 && warp < 16) || warp >= 20 ? 1 : 0;
    const int g = warp >= 16 ? 1 : 0;
    // Thread r of warpgroup h: chunks [c0, c0 + NC) of token row r (TMEM lane
    // r, in this warp's lane quarter), i.e. dims 8 c0 .. 8 (c0 + NC) - 1.
    constexpr int NC = D / 16;                       // 16-byte chunks per thread
    uint8_t* const half0 = qt + (D == 128 ? h * LN_HALF : 0);
    const int c0 = D == 128 ? 0 : 4 * h;
    const uint32_t tOpd = tmem + ln_opd(g) + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                          static_cast<uint32_t>(h * NC * 4);
    for (int u = g; u < nt; u += 2) {
      // As in lin_state_kernel: first the other pair's release of tile u - 3,
      // the previous user of stage s, so the Q-full parity cannot match too
      // early; then this pair's operand buffer, read by the MMAs of tile u - 2.
      const int s = u % LN_NS;
      const uint32_t ph = (u / LN_NS) & 1;
      if (u >= LN_NS &&
          !__all_sync(0xffffffffu, mbar_wait_bounded(bar(LO_QE + s), ph ^ 1, lim, abort_p)))
        break;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(LO_QF + s), ph, lim, abort_p)))
        break;
      if (u >= 2 && !__all_sync(0xffffffffu, mbar_wait_bounded(bar(LO_ABE + g),
                                                               ((u >> 1) - 1) & 1, lim, abort_p)))
        break;
      // chunk j of row r sits at 16-byte position j ^ (r & 7) (128-byte
      // swizzle); in logical order the warp's loads still hit distinct banks
      const uint8_t* rowp = half0 + s * Dm::kTile + r * 128;
      uint4 w[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c)
        w[c] = *reinterpret_cast<const uint4*>(rowp + (((c0 + c) ^ (r & 7)) * 16));
      mbar_arrive(bar(LO_QE + s));  // the stage may be reloaded (release: loads done)
      uint32_t e[NC * 4];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        e[4 * c + 0] = lin_phi_bf16x2(w[c].x);
        e[4 * c + 1] = lin_phi_bf16x2(w[c].y);
        e[4 * c + 2] = lin_phi_bf16x2(w[c].z);
        e[4 * c + 3] = lin_phi_bf16x2(w[c].w);
      }
      if constexpr (NC * 4 == 32) tmem_st32(tOpd, e);
      else tmem_st16(tOpd, e);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(LO_PHI + g));
    }
  } else if (warp >= 8) {
    // Thread r converts token row r of the tile into the staging tile (the
    // 128B-swizzled layout of the Q tiles, so the 16-byte stores of a warp hit
    // distinct banks), then one thread writes the tile with two TMA stores
    // (rows past N are clipped by the tensor map). Before the staging tile is
    // rewritten, the previous stores must have read it; the four warps decide
    // together (bar.red) whether to go on, so none is left at the barrier.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool issuer = warp == 8 && lane == 0;
    for (int u = 0; u < nt; ++u) {
      const int b = u & 1;
      const bool full =
          __all_sync(0xffffffffu, mbar_wait_bounded(bar(LO_AF + b), (u >> 1) & 1, lim, abort_p));
      if (issuer) bulk_wait_read_all();
      if (!named_bar_and(1, 128, full)) break;
      tc_fence_after();
      const uint32_t tA = tmem + b * 256 + lane_off;
      uint32_t dv[16];
      tmem_ld16(tA + D, dv);
      tmem_wait_ld();
      const float inv = 1.f / __uint_as_float(dv[0]);
      const int tok = (t_lo + u) * 128 + r;
      const __nv_bfloat16* arow = out + (static_cast<long long>(bh) * N + tok) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tA + c * 32, v);
        tmem_wait_ld();
        if (c == D / 32 - 1) {
          tc_fence_before();
          mbar_arrive(bar(LO_AE + b));
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(v[q4 * 8 + e]) * inv;
          if (mix && tok < N) {
            const uint4 a = reinterpret_cast<const uint4*>(arow + c * 32)[q4];
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              o[2 * e] = fmaf(r_mix, __uint_as_float(aw[e] << 16) - o[2 * e], o[2 * e]);
              o[2 * e + 1] =
                  fmaf(r_mix, __uint_as_float(aw[e] & 0xffff0000u) - o[2 * e + 1], o[2 * e + 1]);
            }
          }
          uint4 w;
          w.x = pack_bf16x2(o[0], o[1]);
          w.y = pack_bf16x2(o[2], o[3]);
          w.z = pack_bf16x2(o[4], o[5]);
          w.w = pack_bf16x2(o[6], o[7]);
          const int j = (c & 1) * 4 + q4;  // 16-byte chunk within the 64-dim half c / 2
          *reinterpret_cast<uint4*>(ot + (c >> 1) * LN_HALF + r * 128 + ((j ^ (r & 7)) * 16)) = w;
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (issuer) {
        for (int hh = 0; hh < Dm::kHalves; ++hh)
          tma_store_3d(&map_o, smem_u32(ot + hh * LN_HALF), 64 * hh, (t_lo + u) * 128, bh);
        bulk_commit();
      }
    }
    if (issuer) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace va
