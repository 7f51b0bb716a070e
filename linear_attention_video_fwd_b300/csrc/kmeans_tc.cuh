// k-means assignment on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA) for bf16 points with d = D (64 or 128): the distance cross term x . c of the
// Lloyd assign step (SVG-EAR, gist.science 2603.08982, technical summary
// sec. 2, idea 1: semantic clustering of queries and keys).
//
// The float32 centroid is split as c = c_hi + c_lo with both parts bf16
// (|c - c_hi - c_lo| <= 2^-17 |c|), so x . c = x . c_hi + x . c_lo is two
// exact-product bf16 MMAs accumulated in one fp32 TMEM accumulator (K = 2 D).
// dist(i, c) = |c|^2 - 2 x_i . c; the argmin takes the lowest c on ties.
//
// Persistent CTAs with resident centroids: CTA (split, chunk, batch*head)
// holds the hi and lo parts of one chunk of 256 clusters in shared memory
// (128 KB at D = 128) and streams its share of the 128-point tiles through a two-stage
// TMA ring; the accumulators of consecutive point tiles alternate between two
// TMEM halves, so the argmin of one tile overlaps the MMAs of the next. With
// several chunks the per-chunk (distance, index) results are merged by
// ka_merge_kernel in chunk order (strict <, so the lowest index still wins
// ties). 256 threads:
//   warp 0      TMA producer: the centroid chunk once, then the point tiles;
//   warp 1      MMA issuer: point tile i against cluster tiles 0, 1 into TMEM
//               columns [256 (i & 1) + 128 t, +128);
//   warps 2, 3  idle;
//   warps 4..7  argmin epilogue, thread r owns point r of the tile (TMEM lane
//               r); the accumulators are released right after tcgen05.ld.
// Every mbarrier wait is bounded; see attn_tc.cuh for the timeout protocol.
#pragma once

#include "common.cuh"

namespace va {

constexpr int KA_THREADS = 256;
constexpr int KA_CHUNK = 256;            // clusters resident per CTA
constexpr int KA_HALF = 128 * 64 * 2;    // 16 KB: 128 rows x 64 bf16 (one TMA box)
constexpr int KA_NX = 2;                 // point-tile ring stages

// Sizes that depend on the head dimension D.
template <int D>
struct KaDim {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kHalves = D / 64;
  static constexpr int kTile = 128 * D * 2;   // 128 rows x D bf16
  static constexpr int kSmemBytes = 1024 + kTile * (4 + KA_NX);
};

enum : int {
  KB_C_FULL = 0,
  KB_X_FULL = 1,
  KB_X_EMPTY = KB_X_FULL + KA_NX,
  KB_ACC_FULL = KB_X_EMPTY + KA_NX,   // 2
  KB_ACC_EMPTY = KB_ACC_FULL + 2,     // 2, 128 arrivals
  KB_DRAIN = KB_ACC_EMPTY + 2,
  KB_COUNT = KB_DRAIN + 1
};

__device__ __forceinline__ float ka_min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Acc (+)= A[128 x D] . B[128 x D]^T, both K-major 128B-swizzled halves.
template <int D>
__device__ __forceinline__ void ka_issue(uint32_t d_tmem, uint32_t sA, uint32_t sB,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t off = (k >> 2) * KA_HALF + (k & 3) * 32;
    umma_ss(d_tmem, sw128_desc(sA + off, 16, 1024), sw128_desc(sB + off, 16, 1024), idesc,
            (accumulate || k > 0) ? 1u : 0u);
  }
}

// Point tiles [t_lo, t_hi) of split blockIdx.x over the ntiles of a head.
__device__ __forceinline__ void ka_range(int ntiles, int nsplit, int split, int& t_lo, int& t_hi) {
  const int per = (ntiles + nsplit - 1) / nsplit;
  t_lo = min(ntiles, split * per);
  t_hi = min(ntiles, t_lo + per);
}

// Grid (nsplit, nchunks, BH). With one chunk the result is the assignment
// (assign, count += 1); with several, (pdist, pidx)[bh][chunk][i] for the merge.
template <int D>
__global__ void __launch_bounds__(KA_THREADS, 1)
    km_assign_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                        const __grid_constant__ CUtensorMap map_hi,
                        const __grid_constant__ CUtensorMap map_lo,
                        const float* __restrict__ cnorm, int N, int C,
                        int* __restrict__ assign, int* __restrict__ count,
                        float* __restrict__ pdist, int* __restrict__ pidx, long long lim) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[KB_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ __align__(8) float cn_s[KA_CHUNK];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kTile = KaDim<D>::kTile, kHalves = KaDim<D>::kHalves;
  const uint32_t sHi = smem_u32(smem);          // cluster tile t: hi at sHi + t kTile
  const uint32_t sLo = sHi + 2 * kTile;         // lo at sLo + t kTile
  const uint32_t sX0 = sLo + 2 * kTile;         // point-tile stage s at sX0 + s kTile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, chunk = blockIdx.y, bh = blockIdx.z;
  const int nchunks = gridDim.y;
  const int c0 = chunk * KA_CHUNK;
  const int ntiles = (N + 127) / 128;
  int t_lo, t_hi;
  ka_range(ntiles, gridDim.x, split, t_lo, t_hi);
  const int nt = t_hi - t_lo;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar(KB_C_FULL), 1);
    for (int s = 0; s < KA_NX; ++s) {
      mbar_init(bar(KB_X_FULL + s), 1);
      mbar_init(bar(KB_X_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(KB_ACC_FULL + b), 1);
      mbar_init(bar(KB_ACC_EMPTY + b), 128);
    }
    mbar_init(bar(KB_DRAIN), 1);
    fence_barrier_init();
  }
  // |c|^2 of the chunk; +inf past C, so those columns never win
  for (int c = tid; c < KA_CHUNK; c += KA_THREADS)
    cn_s[c] = c0 + c < C ? cnorm[static_cast<long long>(bh) * C + c0 + c] : INFINITY;
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
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&map_x);
      tma_prefetch_desc(&map_hi);
      tma_prefetch_desc(&map_lo);
      mbar_arrive_expect_tx(bar(KB_C_FULL), 4 * kTile);
      for (int t = 0; t < 2; ++t)
        for (int h = 0; h < kHalves; ++h) {
          tma_load_3d(sHi + t * kTile + h * KA_HALF, &map_hi, bar(KB_C_FULL), 64 * h,
                      c0 + 128 * t, bh);
          tma_load_3d(sLo + t * kTile + h * KA_HALF, &map_lo, bar(KB_C_FULL), 64 * h,
                      c0 + 128 * t, bh);
        }
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int s = i % KA_NX;
        if (i >= KA_NX &&
            !mbar_wait_bounded(bar(KB_X_EMPTY + s), ((i / KA_NX) & 1) ^ 1, lim, abort_p))
          break;
        const int row = (t_lo + i) * 128;
        mbar_arrive_expect_tx(bar(KB_X_FULL + s), kTile);
        for (int h = 0; h < kHalves; ++h)
          tma_load_3d(sX0 + s * kTile + h * KA_HALF, &map_x, bar(KB_X_FULL + s), 64 * h, row, bh);
        issued = i + 1;
      }
      if (*abort_p) {
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(KB_C_FULL), 0, lim, &no_abort);
        for (int i = issued > KA_NX ? issued - KA_NX : 0; i < issued; ++i) {
          no_abort = 0;
          mbar_wait_bounded(bar(KB_X_FULL + i % KA_NX), (i / KA_NX) & 1, lim, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nt > 0) {
      bool ok = mbar_wait_bounded(bar(KB_C_FULL), 0, lim, abort_p);
      for (int i = 0; ok && i < nt; ++i) {
        const int s = i % KA_NX, b = i & 1;
        if (!(ok = mbar_wait_bounded(bar(KB_X_FULL + s), (i / KA_NX) & 1, lim, abort_p))) break;
        if (i >= 2 &&
            !(ok = mbar_wait_bounded(bar(KB_ACC_EMPTY + b), ((i >> 1) & 1) ^ 1, lim, abort_p)))
          break;
        tc_fence_after();
        const uint32_t sX = sX0 + s * kTile;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          ka_issue<D>(tmem + b * 256 + t * 128, sX, sHi + t * kTile, false);
          ka_issue<D>(tmem + b * 256 + t * 128, sX, sLo + t * kTile, true);
        }
        umma_commit(bar(KB_X_EMPTY + s));
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
    for (int i = 0; i < nt; ++i) {
      const int b = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(KB_ACC_FULL + b), (i >> 1) & 1, lim,
                                                      abort_p)))
        break;
      tc_fence_after();
      float best = INFINITY;
      int besti = 0x7fffffff;
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        float acc[128];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(tmem + b * 256 + t * 128 + lane_off + c4 * 32, v);
#pragma unroll
          for (int k = 0; k < 32; ++k) acc[c4 * 32 + k] = __uint_as_float(v[k]);
        }
        tmem_wait_ld();
        if (t == 1) {
          tc_fence_before();
          mbar_arrive(bar(KB_ACC_EMPTY + b));
        }
        // distances, two per packed FMA (columns past C have |c|^2 = +inf)
#pragma unroll
        for (int k = 0; k < 128; k += 2) {
          const float2 n2 = *reinterpret_cast<const float2*>(&cn_s[t * 128 + k]);
          ffma2_v(acc[k], acc[k + 1], acc[k], acc[k + 1], -2.f, n2.x, n2.y);
        }
        // the tile's minimum, then the lowest column that attains it (the
        // same choice as a strict-< scan in column order)
        float m0 = ka_min3(acc[0], acc[1], acc[2]), m1 = ka_min3(acc[3], acc[4], acc[5]);
#pragma unroll
        for (int k = 6; k < 126; k += 4) {
          m0 = ka_min3(m0, acc[k], acc[k + 1]);
          m1 = ka_min3(m1, acc[k + 2], acc[k + 3]);
        }
        const float mn = ka_min3(m0, m1, fminf(acc[126], acc[127]));
        int kmin = 0;
#pragma unroll
        for (int k = 127; k >= 0; --k) kmin = acc[k] == mn ? k : kmin;
        if (mn < best) {  // earlier tiles win ties
          best = mn;
          besti = c0 + t * 128 + kmin;
        }
      }
      const int p = (t_lo + i) * 128 + r;
      if (p < N) {
        if (nchunks == 1) {
          assign[static_cast<long long>(bh) * N + p] = besti;
          atomicAdd(&count[static_cast<long long>(bh) * C + besti], 1);
        } else {
          const long long o = (static_cast<long long>(bh) * nchunks + chunk) * N + p;
          pdist[o] = best;
          pidx[o] = besti;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// Argmin over the chunks' results in chunk order (strict <: the lowest index
// wins ties, as in one pass over all clusters); assign and count += 1.
// Grid (ceil(N / 256), BH).
__global__ void ka_merge_kernel(const float* __restrict__ pdist, const int* __restrict__ pidx,
                                int N, int C, int nchunks, int* __restrict__ assign,
                                int* __restrict__ count) {
  const int bh = blockIdx.y;
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= N) return;
  float best = INFINITY;
  int besti = 0x7fffffff;
  for (int ch = 0; ch < nchunks; ++ch) {
    const long long o = (static_cast<long long>(bh) * nchunks + ch) * N + p;
    const float d = pdist[o];
    if (d < best) {
      best = d;
      besti = pidx[o];
    }
  }
  if (besti >= 0 && besti < C) {
    assign[static_cast<long long>(bh) * N + p] = besti;
    atomicAdd(&count[static_cast<long long>(bh) * C + besti], 1);
  } else {
    raise_error(VA_ERR_DEVICE);
  }
}

// c = hi + lo with hi = bf16(c) and lo = bf16(c - hi), elementwise over n fp32.
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
