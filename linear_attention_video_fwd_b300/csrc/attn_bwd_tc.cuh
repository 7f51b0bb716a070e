// Block-sparse attention backward on the 5th-generation tensor cores (tcgen05
// + TMEM + TMA), bf16, head_dim D in {64, 128}, 128-token blocks (a D = 128
// tile is two 64-dim halves, a D = 64 tile one). The gradients are
// those of the float32 kernels' header (chain rule of the attention
// definition); p is recomputed from the forward's lse, in the log2 domain:
// p = exp2(scale_log2 s + nlse2), nlse2 = -lse log2(e) (-inf on padding rows).
//
// Two kernels, each one CTA per (batch*head, 128-token block), longest list
// first, no atomics (the results are deterministic):
//   bwd_dkdv_tc_kernel  key block J resident (K, V); walks the query blocks
//                       of the transposed CSR with Q and G (= dL/dO) tiles in
//                       a ring. Per query block, on the tensor cores:
//                         S^T  = K Q^T,  dP^T = V G^T            (SS, TMEM)
//                         dV  += P^T G,  dK  += dS^T Q           (TS: P^T, dS^T in TMEM)
//                       and in between, two warpgroups (64 query columns
//                       each) turn S^T into P^T and dP^T into
//                       dS^T = P^T (dP^T - delta), both written back to TMEM
//                       as bf16 over the columns they came from;
//   bwd_dq_tc_kernel    query block I resident (Q, G); walks its live key
//                       blocks with K and V tiles in a ring:
//                         S = Q K^T,  dP = G V^T,  dQ += dS K.
// 384 threads: warp 0 TMA producer, warp 1 MMA issuer (one thread), warps 2-3
// idle, warps 4-7 and 8-11 the two column halves; thread r of a warpgroup owns
// TMEM lane r (a key row in the first kernel, a query row in the second).
// MMA order per block u of the first kernel: dV(u), S(u+1), then after dS(u)
// is written dK(u), dP(u+1); the tensor pipe executes them in issue order, so
// an MMA that overwrites a TMEM region is issued after the one that reads it.
// Every mbarrier wait is bounded; on a timeout the CTA records
// VA_ERR_TIMEOUT, drains its copies and MMAs and frees its TMEM.
#pragma once

#include "attn_tc.cuh"

namespace va {

constexpr int BW_THREADS = 384;
constexpr int BW_NS = 2;  // ring stages
constexpr int BW_ROWVEC = 1024;  // per stage: nlse2 and ndelta of one 128-row block
template <int D>
struct BwDim {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kTileBytes = TC_BLK * D * 2;
  static constexpr int kSmemBytes = 1024 + kTileBytes * (2 + 2 * BW_NS) + BW_NS * BW_ROWVEC;
};

// A (rows x D) B^T over the D dims into TMEM: both operands 128-row K-major
// tiles of D dims (D / 16 steps), e.g. S = Q K^T.
template <int D>
__device__ __forceinline__ void bw_issue_ss(uint32_t d_tmem, uint32_t sA, uint32_t sB) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t off = (k >> 2) * TC_HALF_BYTES + (k & 3) * 32;
    umma_ss(d_tmem, sw128_desc(sA + off, 16, 1024), sw128_desc(sB + off, 16, 1024), idesc, k > 0);
  }
}

struct BwArgs {
  const int* ptr;    // CSR (query side) or transposed CSR (key side) offsets
  const int* idx;    // the blocks of each list
  const int* order;  // blocks by descending list length
  const int* len;    // 64-token blocks: coarse list lengths (entries c << 4 | 2 x 2 live bits)
  const float* ndelta;  // [BH, Np]: -(dO . O)
  const float* nlse2;   // [BH, Np]: -lse log2(e)
  __nv_bfloat16* d0;   // dq (query side) or dv (key side)
  __nv_bfloat16* d1;   // dk (key side)
  int N, Np, nb;
  float scale, scale_log2;
  long long wait_limit;
};

// TMEM column of K-step k (16 elements) of a 128 x 128 bf16 operand that two
// warpgroups packed: warpgroup h wrote its 64 elements as 32 columns at 64 h.
__device__ __forceinline__ uint32_t bw_pcol(int k) {
  return static_cast<uint32_t>((k >> 2) * 64 + (k & 3) * 8);
}

// D (+)= A x B, A = 128 x 128 bf16 packed in TMEM (bw_pcol), B a 128-token
// tile in shared memory whose D dims are the N side (MN-major).
template <int D>
__device__ __forceinline__ void bw_issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t sB,
                                            bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    umma_ts(d_tmem, a_tmem + bw_pcol(k), sw128_desc(sB + k * 2048, TC_HALF_BYTES, 1024), idesc,
            (accumulate || k > 0) ? 1u : 0u);
}

// 64 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void bw_ld64(uint32_t taddr, float (&x)[64]) {
  uint32_t a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    x[i] = __uint_as_float(a[i]);
    x[32 + i] = __uint_as_float(b[i]);
  }
}

// Store 64 values as 32 packed bf16 columns and publish them to the MMA.
__device__ __forceinline__ void bw_st_packed(uint32_t taddr, const float (&x)[64]) {
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
  tmem_st32(taddr, pk);
  tmem_wait_st();
}

// Write 64 fp32 TMEM columns (times mul) as bf16 to dst (64 elements).
__device__ __forceinline__ void bw_store64(uint32_t taddr, float mul, __nv_bfloat16* dst,
                                           bool valid) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + c * 32, v);
    tmem_wait_ld();
    if (valid) {
      uint4* d = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]) * mul, __uint_as_float(v[q4 * 8 + 1]) * mul);
        w.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]) * mul, __uint_as_float(v[q4 * 8 + 3]) * mul);
        w.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]) * mul, __uint_as_float(v[q4 * 8 + 5]) * mul);
        w.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]) * mul, __uint_as_float(v[q4 * 8 + 7]) * mul);
        d[q4] = w;
      }
    }
  }
}

// (d0, d1) = (a0 * b0, a1 * b1) as one packed f32x2 multiply.
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bw_bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

template <int D>
__device__ __forceinline__ void bw_load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int row, int bh) {
#pragma unroll
  for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * TC_HALF_BYTES, map, bar, 64 * h, row, bh);
}

enum : int {
  KA_RES = 0,                    // resident pair of tiles loaded
  KA_FULL = KA_RES + 1,          // BW_NS: streamed pair loaded
  KA_EMPTY = KA_FULL + BW_NS,    // BW_NS: streamed pair consumed
  KA_S = KA_EMPTY + BW_NS,       // S (or S^T) computed
  KA_DP = KA_S + 1,              // dP computed
  KA_P = KA_DP + 1,              // 256 arrivals: P^T written (key side) / S read (query side)
  KA_DS = KA_P + 1,              // 256 arrivals: dS written
  KA_DONE = KA_DS + 1,
  KA_DRAIN = KA_DONE + 1,
  KA_COUNT = KA_DRAIN + 1
};

// Shared set-up of both kernels: barriers and a 512-column TMEM allocation.
__device__ __forceinline__ void bw_setup(uint64_t* bars, uint32_t* tmem_base_s, int* abort_flag) {
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(smem_u32(&bars[KA_RES]), 1);
    for (int s = 0; s < BW_NS; ++s) {
      mbar_init(smem_u32(&bars[KA_FULL + s]), 1);
      mbar_init(smem_u32(&bars[KA_EMPTY + s]), 1);
    }
    mbar_init(smem_u32(&bars[KA_S]), 1);
    mbar_init(smem_u32(&bars[KA_DP]), 1);
    mbar_init(smem_u32(&bars[KA_P]), 256);
    mbar_init(smem_u32(&bars[KA_DS]), 256);
    mbar_init(smem_u32(&bars[KA_DONE]), 1);
    mbar_init(smem_u32(&bars[KA_DRAIN]), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_base_s), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Producer of both kernels: the resident pair of tiles at block `own`, then
// the streamed pair for every entry of the list (block list[u] >> shift).
// With rv0 != nullptr each entry also brings the 128 floats of rv0 and rv1 at
// its block (the nlse2 and ndelta rows of a query block) to sX + stage *
// BW_ROWVEC.
template <int D>
__device__ __forceinline__ void bw_produce(const CUtensorMap* r0, const CUtensorMap* r1,
                                           const CUtensorMap* s0, const CUtensorMap* s1,
                                           uint32_t sR, uint32_t sA, uint32_t sB, int own,
                                           const int* list, int n, int bh, uint64_t* bars,
                                           long long lim, volatile int* abort_p,
                                           const float* rv0 = nullptr,
                                           const float* rv1 = nullptr, uint32_t sX = 0,
                                           int shift = 0) {
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  tma_prefetch_desc(r0);
  tma_prefetch_desc(r1);
  tma_prefetch_desc(s0);
  tma_prefetch_desc(s1);
  constexpr int kTile = BwDim<D>::kTileBytes;
  mbar_arrive_expect_tx(bar(KA_RES), 2 * kTile);
  bw_load_tile<D>(sR, r0, bar(KA_RES), own * TC_BLK, bh);
  bw_load_tile<D>(sR + kTile, r1, bar(KA_RES), own * TC_BLK, bh);
  int issued = 0;
  for (int u = 0; u < n; ++u) {
    const int s = u % BW_NS, blk = list[u] >> shift;
    if (u >= BW_NS &&
        !mbar_wait_bounded(bar(KA_EMPTY + s), ((u / BW_NS) & 1) ^ 1, lim, abort_p))
      break;
    mbar_arrive_expect_tx(bar(KA_FULL + s), 2 * kTile + (rv0 ? BW_ROWVEC : 0));
    bw_load_tile<D>(sA + s * kTile, s0, bar(KA_FULL + s), blk * TC_BLK, bh);
    bw_load_tile<D>(sB + s * kTile, s1, bar(KA_FULL + s), blk * TC_BLK, bh);
    if (rv0 != nullptr) {
      bw_bulk_load(sX + s * BW_ROWVEC, rv0 + blk * TC_BLK, 512, bar(KA_FULL + s));
      bw_bulk_load(sX + s * BW_ROWVEC + 512, rv1 + blk * TC_BLK, 512, bar(KA_FULL + s));
    }
    issued = u + 1;
  }
  if (*abort_p) {
    // Every copy issued must land before the CTA's shared memory is released;
    // only the last BW_NS streamed loads can still be in flight.
    volatile int no_abort = 0;
    mbar_wait_bounded(bar(KA_RES), 0, lim, &no_abort);
    for (int u = issued > BW_NS ? issued - BW_NS : 0; u < issued; ++u) {
      no_abort = 0;
      mbar_wait_bounded(bar(KA_FULL + u % BW_NS), (u / BW_NS) & 1, lim, &no_abort);
    }
  }
}

__device__ __forceinline__ void bw_mma_drain(uint64_t* bars, bool ok, long long lim) {
  if (ok) {
    umma_commit(smem_u32(&bars[KA_DONE]));
  } else {
    umma_commit(smem_u32(&bars[KA_DRAIN]));
    volatile int no_abort = 0;
    mbar_wait_bounded(smem_u32(&bars[KA_DRAIN]), 0, lim, &no_abort);
  }
}

// dK and dV of key block J = order[blockIdx % nb] of head blockIdx / nb.
// TMEM: S^T [0, 128) (P^T packed over it), dP^T [128, 256) (dS^T packed over
// it), dV [256, 384), dK [384, 512). Shared memory: K, V, then the Q ring and
// the G ring. SUB (64-token mask blocks): J is a pair of key blocks and each
// entry a pair of query blocks; p is zero in the 64 x 64 quarters whose key
// block does not see the query block.
template <int D, bool SUB = false>
__global__ void __launch_bounds__(BW_THREADS, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                       const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v,
                       const __grid_constant__ CUtensorMap map_g, const BwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[KA_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kTile = BwDim<D>::kTileBytes;
  const uint32_t sK = smem_u32(smem), sV = sK + kTile;
  const uint32_t sQ0 = sV + kTile, sG0 = sQ0 + BW_NS * kTile;
  const uint32_t sX = sG0 + BW_NS * kTile;  // nlse2 | ndelta per stage
  const float* rowvec = reinterpret_cast<const float*>(smem + (sX - sK));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / a.nb;
  const int J = a.order[blockIdx.x % a.nb];
  const int beg = a.ptr[SUB ? 2 * J : J];
  const int n = SUB ? a.len[J] : a.ptr[J + 1] - beg;
  const int* list = a.idx + beg;
  bw_setup(bars, &tmem_base_s, &abort_flag);
  const uint32_t tmem = tmem_base_s;
  const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;
  volatile int* abort_p = &abort_flag;
  const long long lim = a.wait_limit;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (warp == 0) {
    if (lane == 0 && n > 0)
      bw_produce<D>(&map_k, &map_v, &map_q, &map_g, sK, sQ0, sG0, J, list, n, bh, bars, lim,
                    abort_p, a.nlse2 + static_cast<long long>(bh) * a.Np,
                    a.ndelta + static_cast<long long>(bh) * a.Np, sX, SUB ? 4 : 0);
  } else if (warp == 1) {
    if (lane == 0 && n > 0) {
      bool ok = mbar_wait_bounded(bar(KA_RES), 0, lim, abort_p) &&
                mbar_wait_bounded(bar(KA_FULL), 0, lim, abort_p);
      if (ok) {
        tc_fence_after();
        bw_issue_ss<D>(tS, sK, sQ0);
        umma_commit(bar(KA_S));
        bw_issue_ss<D>(tDP, sV, sG0);
        umma_commit(bar(KA_DP));
      }
      for (int u = 0; ok && u < n; ++u) {
        const int s = u % BW_NS, s1 = (u + 1) % BW_NS;
        if (!(ok = mbar_wait_bounded(bar(KA_P), u & 1, lim, abort_p))) break;
        tc_fence_after();
        bw_issue_ts<D>(tDV, tS, sG0 + s * kTile, u > 0);
        if (u + 1 < n) {
          if (!(ok = mbar_wait_bounded(bar(KA_FULL + s1), ((u + 1) / BW_NS) & 1, lim, abort_p)))
            break;
          tc_fence_after();
          bw_issue_ss<D>(tS, sK, sQ0 + s1 * kTile);
          umma_commit(bar(KA_S));
        }
        if (!(ok = mbar_wait_bounded(bar(KA_DS), u & 1, lim, abort_p))) break;
        tc_fence_after();
        bw_issue_ts<D>(tDK, tDP, sQ0 + s * kTile, u > 0);
        umma_commit(bar(KA_EMPTY + s));
        if (u + 1 < n) {
          bw_issue_ss<D>(tDP, sV, sG0 + s1 * kTile);
          umma_commit(bar(KA_DP));
        }
      }
      bw_mma_drain(bars, ok, lim);
    }
  } else if (warp >= 4) {
    const int h = (warp - 4) >> 2;  // query-column half
    const int wq = warp & 3, r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t col = lane_off + h * 64;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int u = 0; u < n; ++u) {
      // nlse2 and ndelta of this query block's 64 columns, staged with its tiles
      // (the stage cannot be refilled before this iteration's dS is written)
      const int s = u % BW_NS;
      const float* l2b = rowvec + s * (BW_ROWVEC / 4) + h * 64;
      const float* dlb = l2b + 128;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(KA_FULL + s), (u / BW_NS) & 1,
                                                          lim, abort_p))))
        break;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(KA_S), u & 1, lim, abort_p))))
        break;
      tc_fence_after();
      float p[64];
      bw_ld64(tS + col, p);
      // SUB: does this key row's block see this half's query block (warp-uniform)
      const bool live = !SUB || ((list[u] >> (2 * (r >> 6) + h)) & 1);
      if (live) {
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 l = *reinterpret_cast<const float4*>(l2b + c);
          ffma2_v(p[c], p[c + 1], p[c], p[c + 1], sl2, l.x, l.y);
          ffma2_v(p[c + 2], p[c + 3], p[c + 2], p[c + 3], sl2, l.z, l.w);
#pragma unroll
          for (int i = 0; i < 4; ++i) p[c + i] = ex2_approx(p[c + i]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = 0.f;
      }
      bw_st_packed(tS + col, p);
      tc_fence_before();
      mbar_arrive(bar(KA_P));
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(KA_DP), u & 1, lim, abort_p))))
        break;
      tc_fence_after();
      float ds[64];
      bw_ld64(tDP + col, ds);
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 dl = *reinterpret_cast<const float4*>(dlb + c);
        fadd2_acc(ds[c], ds[c + 1], dl.x, dl.y);
        fadd2_acc(ds[c + 2], ds[c + 3], dl.z, dl.w);
        fmul2(ds[c], ds[c + 1], ds[c], ds[c + 1], p[c], p[c + 1]);
        fmul2(ds[c + 2], ds[c + 3], ds[c + 2], ds[c + 3], p[c + 2], p[c + 3]);
      }
      bw_st_packed(tDP + col, ds);
      tc_fence_before();
      mbar_arrive(bar(KA_DS));
    }
    // epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK
    const int key = J * TC_BLK + r;
    __nv_bfloat16* dst = (h == 0 ? a.d0 : a.d1) + (static_cast<long long>(bh) * a.N + key) * D;
    if (n > 0 && ok)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(KA_DONE), 0, lim, abort_p));
    if (n > 0 && ok) {
      tc_fence_after();
      const uint32_t src = (h == 0 ? tDV : tDK) + lane_off;
      const float mul = h == 0 ? 1.f : a.scale;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) bw_store64(src + 64 * c, mul, dst + 64 * c, key < a.N);
    } else if (n == 0 && key < a.N) {
      uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int q4 = 0; q4 < D / 8; ++q4) d[q4] = make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// dQ of query block I = order[blockIdx % nb] of head blockIdx / nb.
// TMEM: S [0, 128), dP [128, 256) (dS packed over it), dQ [256, 384).
// Shared memory: Q, G, then the K ring and the V ring. SUB (64-token mask
// blocks): I is a pair of query blocks and each entry a pair of key blocks;
// p is zero in the 64 x 64 quarters that are not live.
template <int D, bool SUB = false>
__global__ void __launch_bounds__(BW_THREADS, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v,
                     const __grid_constant__ CUtensorMap map_g, const BwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[KA_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kTile = BwDim<D>::kTileBytes;
  const uint32_t sQ = smem_u32(smem), sG = sQ + kTile;
  const uint32_t sK0 = sG + kTile, sV0 = sK0 + BW_NS * kTile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / a.nb;
  const int I = a.order[blockIdx.x % a.nb];
  const int beg = a.ptr[SUB ? 2 * I : I];
  const int n = SUB ? a.len[I] : a.ptr[I + 1] - beg;
  const int* list = a.idx + beg;
  bw_setup(bars, &tmem_base_s, &abort_flag);
  const uint32_t tmem = tmem_base_s;
  const uint32_t tS = tmem, tDP = tmem + 128, tDQ = tmem + 256;
  volatile int* abort_p = &abort_flag;
  const long long lim = a.wait_limit;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (warp == 0) {
    if (lane == 0 && n > 0)
      bw_produce<D>(&map_q, &map_g, &map_k, &map_v, sQ, sK0, sV0, I, list, n, bh, bars, lim,
                    abort_p, nullptr, nullptr, 0, SUB ? 4 : 0);
  } else if (warp == 1) {
    if (lane == 0 && n > 0) {
      bool ok = mbar_wait_bounded(bar(KA_RES), 0, lim, abort_p) &&
                mbar_wait_bounded(bar(KA_FULL), 0, lim, abort_p);
      if (ok) {
        tc_fence_after();
        bw_issue_ss<D>(tS, sQ, sK0);
        umma_commit(bar(KA_S));
        bw_issue_ss<D>(tDP, sG, sV0);
        umma_commit(bar(KA_DP));
      }
      for (int u = 0; ok && u < n; ++u) {
        const int s = u % BW_NS, s1 = (u + 1) % BW_NS;
        if (u + 1 < n) {
          // S(u) has been read into registers: compute S(u + 1) meanwhile.
          if (!(ok = mbar_wait_bounded(bar(KA_P), u & 1, lim, abort_p))) break;
          if (!(ok = mbar_wait_bounded(bar(KA_FULL + s1), ((u + 1) / BW_NS) & 1, lim, abort_p)))
            break;
          tc_fence_after();
          bw_issue_ss<D>(tS, sQ, sK0 + s1 * kTile);
          umma_commit(bar(KA_S));
        }
        if (!(ok = mbar_wait_bounded(bar(KA_DS), u & 1, lim, abort_p))) break;
        tc_fence_after();
        bw_issue_ts<D>(tDQ, tDP, sK0 + s * kTile, u > 0);
        umma_commit(bar(KA_EMPTY + s));
        if (u + 1 < n) {
          bw_issue_ss<D>(tDP, sG, sV0 + s1 * kTile);
          umma_commit(bar(KA_DP));
        }
      }
      bw_mma_drain(bars, ok, lim);
    }
  } else if (warp >= 4) {
    const int h = (warp - 4) >> 2;  // key-column half
    const int wq = warp & 3, r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t col = lane_off + h * 64;
    const int row = I * TC_BLK + r;
    const float nl2 = a.nlse2[static_cast<long long>(bh) * a.Np + row];  // -inf on padding rows
    const float ndl = a.ndelta[static_cast<long long>(bh) * a.Np + row];
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int u = 0; u < n; ++u) {
      // key columns of this half that are real tokens (the last block is ragged);
      // SUB: none if this row's query block does not see this half's key block
      const int e = list[u];
      const int kvalid = (!SUB || ((e >> (2 * (r >> 6) + h)) & 1))
                             ? a.N - (e >> (SUB ? 4 : 0)) * TC_BLK - h * 64
                             : 0;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(KA_S), u & 1, lim, abort_p))))
        break;
      tc_fence_after();
      float p[64];
      bw_ld64(tS + col, p);
      tc_fence_before();
      mbar_arrive(bar(KA_P));
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        ffma2_bc(p[c], p[c + 1], p[c], p[c + 1], sl2, nl2);
        p[c] = ex2_approx(p[c]);
        p[c + 1] = ex2_approx(p[c + 1]);
      }
      if (kvalid < 64) {  // warp-uniform: the ragged last key block (SUB: or a dead quarter)
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = c < kvalid ? p[c] : 0.f;
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(KA_DP), u & 1, lim, abort_p))))
        break;
      tc_fence_after();
      float ds[64];
      bw_ld64(tDP + col, ds);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        ffma2_bc(ds[c], ds[c + 1], ds[c], ds[c + 1], 1.f, ndl);
        fmul2(ds[c], ds[c + 1], ds[c], ds[c + 1], p[c], p[c + 1]);
      }
      bw_st_packed(tDP + col, ds);
      tc_fence_before();
      mbar_arrive(bar(KA_DS));
    }
    // dQ has D columns: warpgroup h writes columns [64 h, 64 h + 64) of them
    __nv_bfloat16* dst = a.d0 + (static_cast<long long>(bh) * a.N + row) * D + h * 64;
    if (n > 0 && ok)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(KA_DONE), 0, lim, abort_p));
    if (h * 64 >= D) {
      // D = 64: the second key-column half has no dQ columns to write
    } else if (n > 0 && ok) {
      tc_fence_after();
      bw_store64(tDQ + col, a.scale, dst, row < a.N);
    } else if (n == 0 && row < a.N) {
      uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) d[q4] = make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace va
