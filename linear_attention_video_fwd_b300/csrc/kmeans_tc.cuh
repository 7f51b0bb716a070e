// k-means assignment on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA) for bf16 points with d = 128: the distance cross term x . c of the
// Lloyd assign step (SVG-EAR, gist.science 2603.08982, technical summary
// sec. 2, idea 1: semantic clustering of queries and keys).
//
// The float32 centroid is split as c = c_hi + c_lo with both parts bf16
// (|c - c_hi - c_lo| <= 2^-17 |c|), so x . c = x . c_hi + x . c_lo is two
// exact-product bf16 MMAs accumulated in one fp32 TMEM accumulator (K = 256).
// dist(i, c) = |c|^2 - 2 x_i . c; the argmin takes the lowest c on ties.
//
// One CTA per (batch*head, pair of 128-point tiles); 256 threads:
//   warp 0      TMA producer: the two point tiles once, then the hi and lo
//               halves of every 128-cluster tile into a ring of KA_NS stages
//               (each cluster tile is fetched once for both point tiles);
//   warp 1      MMA issuer: cluster tile t against point tile q into TMEM
//               columns [256 (t & 1) + 128 q, +128);
//   warps 2, 3  idle;
//   warps 4..7  argmin epilogue, thread r owns point r of both tiles (TMEM
//               lane r); a buffer is released right after its tcgen05.ld, so
//               the next cluster tile's MMAs overlap these comparisons.
// Every mbarrier wait is bounded; see attn_tc.cuh for the timeout protocol.
#pragma once

#include "common.cuh"

namespace va {

constexpr int KA_THREADS = 256;
constexpr int KA_NS = 2;
constexpr int KA_TILE = 128 * 128 * 2;   // 32 KB: 128 rows x 128 bf16
constexpr int KA_HALF = KA_TILE / 2;
constexpr int KA_PTS = 2;  // 128-point tiles per CTA
constexpr int KA_SMEM_BYTES = 1024 + KA_TILE * (KA_PTS + 2 * KA_NS);

enum : int {
  KB_X_FULL = 0,
  KB_C_FULL = 1,
  KB_C_EMPTY = KB_C_FULL + KA_NS,
  KB_ACC_FULL = KB_C_EMPTY + KA_NS,   // 2
  KB_ACC_EMPTY = KB_ACC_FULL + 2,     // 2, 128 arrivals
  KB_DRAIN = KB_ACC_EMPTY + 2,
  KB_COUNT = KB_DRAIN + 1
};

// D (+)= A[128 x 128] . B[128 x 128]^T, both K-major 128B-swizzled halves.
__device__ __forceinline__ void ka_issue(uint32_t d_tmem, uint32_t sA, uint32_t sB,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t off = (k >> 2) * KA_HALF + (k & 3) * 32;
    umma_ss(d_tmem, sw128_desc(sA + off, 16, 1024), sw128_desc(sB + off, 16, 1024), idesc,
            (accumulate || k > 0) ? 1u : 0u);
  }
}

__global__ void __launch_bounds__(KA_THREADS, 1)
    km_assign_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                        const __grid_constant__ CUtensorMap map_hi,
                        const __grid_constant__ CUtensorMap map_lo,
                        const float* __restrict__ cnorm, int N, int C, int* __restrict__ assign,
                        int* __restrict__ count, long long lim) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[KB_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sX = smem_u32(smem);  // point tile q at sX + q TILE
  const uint32_t sC0 = sX + KA_PTS * KA_TILE;  // stage s: hi at sC0 + 2 s TILE, lo right after
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, i0 = blockIdx.x * 128 * KA_PTS;
  const int ntiles = (C + 127) / 128;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar(KB_X_FULL), 1);
    for (int s = 0; s < KA_NS; ++s) {
      mbar_init(bar(KB_C_FULL + s), 1);
      mbar_init(bar(KB_C_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(KB_ACC_FULL + b), 1);
      mbar_init(bar(KB_ACC_EMPTY + b), 128);
    }
    mbar_init(bar(KB_DRAIN), 1);
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

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&map_x);
      tma_prefetch_desc(&map_hi);
      tma_prefetch_desc(&map_lo);
      mbar_arrive_expect_tx(bar(KB_X_FULL), KA_PTS * KA_TILE);
      for (int q = 0; q < KA_PTS; ++q) {
        tma_load_3d(sX + q * KA_TILE, &map_x, bar(KB_X_FULL), 0, i0 + 128 * q, bh);
        tma_load_3d(sX + q * KA_TILE + KA_HALF, &map_x, bar(KB_X_FULL), 64, i0 + 128 * q, bh);
      }
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % KA_NS;
        if (t >= KA_NS &&
            !mbar_wait_bounded(bar(KB_C_EMPTY + s), ((t / KA_NS) & 1) ^ 1, lim, abort_p))
          break;
        const uint32_t hi = sC0 + 2 * s * KA_TILE, lo = hi + KA_TILE;
        mbar_arrive_expect_tx(bar(KB_C_FULL + s), 2 * KA_TILE);
        tma_load_3d(hi, &map_hi, bar(KB_C_FULL + s), 0, t * 128, bh);
        tma_load_3d(hi + KA_HALF, &map_hi, bar(KB_C_FULL + s), 64, t * 128, bh);
        tma_load_3d(lo, &map_lo, bar(KB_C_FULL + s), 0, t * 128, bh);
        tma_load_3d(lo + KA_HALF, &map_lo, bar(KB_C_FULL + s), 64, t * 128, bh);
        issued = t + 1;
      }
      if (*abort_p) {
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(KB_X_FULL), 0, lim, &no_abort);
        for (int t = issued > KA_NS ? issued - KA_NS : 0; t < issued; ++t) {
          no_abort = 0;
          mbar_wait_bounded(bar(KB_C_FULL + t % KA_NS), (t / KA_NS) & 1, lim, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait_bounded(bar(KB_X_FULL), 0, lim, abort_p);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int s = t % KA_NS, b = t & 1;
        if (!(ok = mbar_wait_bounded(bar(KB_C_FULL + s), (t / KA_NS) & 1, lim, abort_p))) break;
        if (t >= 2 &&
            !(ok = mbar_wait_bounded(bar(KB_ACC_EMPTY + b), ((t >> 1) & 1) ^ 1, lim, abort_p)))
          break;
        tc_fence_after();
        const uint32_t hi = sC0 + 2 * s * KA_TILE, lo = hi + KA_TILE;
#pragma unroll
        for (int q = 0; q < KA_PTS; ++q) {
          ka_issue(tmem + b * 256 + q * 128, sX + q * KA_TILE, hi, false);
          ka_issue(tmem + b * 256 + q * 128, sX + q * KA_TILE, lo, true);
        }
        umma_commit(bar(KB_C_EMPTY + s));
        umma_commit(bar(KB_ACC_FULL + b));
      }
      if (!ok) {
        umma_commit(bar(KB_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(KB_DRAIN), 0, lim, &no_abort);
      }
    }
  } else if (warp >= 4) {
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float* cn = cnorm + static_cast<long long>(bh) * C;
    float best[KA_PTS];
    int besti[KA_PTS];
#pragma unroll
    for (int q = 0; q < KA_PTS; ++q) {
      best[q] = INFINITY;
      besti[q] = 0x7fffffff;
    }
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int b = t & 1;
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(bar(KB_ACC_FULL + b), (t >> 1) & 1, lim, abort_p));
      if (!ok) break;
      tc_fence_after();
      const int c0 = t * 128;
      const int nc = min(128, C - c0);
#pragma unroll 1
      for (int q = 0; q < KA_PTS; ++q) {
        float acc[128];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(tmem + b * 256 + q * 128 + lane_off + c4 * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[c4 * 32 + i] = __uint_as_float(v[i]);
        }
        tmem_wait_ld();
        if (q == KA_PTS - 1) {
          tc_fence_before();
          mbar_arrive(bar(KB_ACC_EMPTY + b));
        }
        float bq = best[q];
        int iq = besti[q];
        if (nc == 128) {
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            const float dist = fmaf(-2.f, acc[i], __ldg(cn + c0 + i));
            if (dist < bq) {
              bq = dist;
              iq = c0 + i;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            if (i < nc) {
              const float dist = fmaf(-2.f, acc[i], __ldg(cn + c0 + i));
              if (dist < bq) {
                bq = dist;
                iq = c0 + i;
              }
            }
          }
        }
        best[q] = bq;
        besti[q] = iq;
      }
    }
#pragma unroll
    for (int q = 0; q < KA_PTS; ++q) {
      const int i = i0 + 128 * q + r;
      if (ok && i < N) {
        assign[static_cast<long long>(bh) * N + i] = besti[q];
        atomicAdd(&count[static_cast<long long>(bh) * C + besti[q]], 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// c = hi + lo with hi = bf16(c) and lo = bf16(c - hi), for [rows, 128] fp32.
__global__ void km_split_kernel(const float* __restrict__ cent, long long n,
                                __nv_bfloat16* __restrict__ hi, __nv_bfloat16* __restrict__ lo) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float c = cent[i];
  const __nv_bfloat16 h = __float2bfloat16_rn(c);
  hi[i] = h;
  lo[i] = __float2bfloat16_rn(c - __bfloat162float(h));
}

}  // namespace va
