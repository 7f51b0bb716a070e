// Block-sparse flash-attention forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 inputs, head_dim 128, 128-token blocks.
//
// One CTA per (batch*head, query block I); CTAs are ordered head-major and,
// within a head, by descending CSR row length (longest first), so the K/V
// working set of the CTAs in flight stays within L2 and the grid tail holds
// the shortest rows. 192 threads:
//   warp 0      TMA producer: Q tile once, then K_j and V_j of every live key
//               block j of row I into a ring of NS stages (128B-swizzled);
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               score buffers, O += P_j V_j with P_j read from TMEM;
//   warps 2..5  softmax / correction / epilogue; thread r owns query row r
//               (TMEM lane r), so row max and row sum need no shuffles.
// Tensor-pipe order: QK(0), QK(1), PV(0), QK(2), PV(1), ... so the softmax of
// block j overlaps PV(j-1) and QK(j+1).
//
// TMEM (512 columns): S buffers at columns [0,128) and [128,256) (fp32; P_j
// is written back over the first 64 columns of its S buffer as packed bf16
// pairs), O accumulator at [256,384).
//
// Online softmax in the log2 domain: the running max used for exponentiation
// is only raised when a block's max exceeds it by more than TAU (so P <= 2^TAU
// and fp32 O/l stay exact to rounding); raising it rescales O in TMEM after
// waiting for the previous PV to complete.
//
// Every mbarrier wait is bounded (clock64 limit): on a timeout the CTA records
// VA_ERR_TIMEOUT in the device error word, drains its own copies and MMAs
// with bounded waits, frees its TMEM and exits.
#pragma once

#include "common.cuh"

namespace va {

constexpr int TC_BLK = 128;
constexpr int TC_D = 128;
constexpr int TC_NS = 2;                    // K/V ring stages
constexpr int TC_THREADS = 192;
constexpr int TC_TILE_BYTES = TC_BLK * TC_D * 2;  // 32 KB: one 128 x 128 bf16 tile
constexpr int TC_HALF_BYTES = TC_TILE_BYTES / 2;  // 16 KB: 128 rows x 64 dims
constexpr int TC_SMEM_BYTES = 1024 + TC_TILE_BYTES * (1 + 2 * TC_NS);
constexpr float TC_TAU = 8.0f;

struct TcArgs {
  const int* row_ptr;
  const int* col;
  const int* order;
  __nv_bfloat16* out;
  float* lse;
  int N, nqb;
  float scale_log2;
  long long wait_limit;
};

// barrier slots
enum : int {
  B_Q_FULL = 0,
  B_K_FULL = 1,
  B_K_EMPTY = B_K_FULL + TC_NS,
  B_V_FULL = B_K_EMPTY + TC_NS,
  B_V_EMPTY = B_V_FULL + TC_NS,
  B_S_FULL = B_V_EMPTY + TC_NS,  // 2
  B_P_FULL = B_S_FULL + 2,       // 2
  B_O_DONE = B_P_FULL + 2,
  B_DRAIN = B_O_DONE + 1,
  B_COUNT = B_DRAIN + 1
};

__device__ __forceinline__ void tc_issue_qk(uint32_t s_tmem, uint32_t sQ, uint32_t sK) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
  for (int k = 0; k < TC_D / 16; ++k) {
    const uint32_t off = (k >> 2) * TC_HALF_BYTES + (k & 3) * 32;
    umma_ss(s_tmem, sw128_desc(sQ + off, 16, 1024), sw128_desc(sK + off, 16, 1024), idesc, k > 0);
  }
}

__device__ __forceinline__ void tc_issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t sV,
                                            bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int k = 0; k < TC_BLK / 16; ++k) {
    umma_ts(o_tmem, p_tmem + k * 8, sw128_desc(sV + k * 2048, TC_HALF_BYTES, 1024), idesc,
            (accumulate || k > 0) ? 1u : 0u);
  }
}

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
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + TC_TILE_BYTES;
  const uint32_t sV0 = sK0 + TC_NS * TC_TILE_BYTES;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int bh = blockIdx.x / a.nqb;
  const int I = a.order[blockIdx.x % a.nqb];
  const int beg = a.row_ptr[I];
  const int n = a.row_ptr[I + 1] - beg;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar(B_Q_FULL), 1);
    for (int s = 0; s < TC_NS; ++s) {
      mbar_init(bar(B_K_FULL + s), 1);
      mbar_init(bar(B_K_EMPTY + s), 1);
      mbar_init(bar(B_V_FULL + s), 1);
      mbar_init(bar(B_V_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_S_FULL + b), 1);
      mbar_init(bar(B_P_FULL + b), 128);
    }
    mbar_init(bar(B_O_DONE), 1);
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
  const uint32_t tS0 = tmem, tO = tmem + 256;
  volatile int* abort_p = &abort_flag;
  const long long lim = a.wait_limit;

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(bar(B_Q_FULL), TC_TILE_BYTES);
      tma_load_3d(sQ, &map_q, bar(B_Q_FULL), 0, I * TC_BLK, bh);
      tma_load_3d(sQ + TC_HALF_BYTES, &map_q, bar(B_Q_FULL), 64, I * TC_BLK, bh);
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j % TC_NS;
        const uint32_t ph = (j / TC_NS) & 1;
        const int J = a.col[beg + j];
        const uint32_t sK = sK0 + st * TC_TILE_BYTES, sV = sV0 + st * TC_TILE_BYTES;
        if (j >= TC_NS && !mbar_wait_bounded(bar(B_K_EMPTY + st), ph ^ 1, lim, abort_p)) break;
        mbar_arrive_expect_tx(bar(B_K_FULL + st), TC_TILE_BYTES);
        tma_load_3d(sK, &map_k, bar(B_K_FULL + st), 0, J * TC_BLK, bh);
        tma_load_3d(sK + TC_HALF_BYTES, &map_k, bar(B_K_FULL + st), 64, J * TC_BLK, bh);
        issued_k = j + 1;
        if (j >= TC_NS && !mbar_wait_bounded(bar(B_V_EMPTY + st), ph ^ 1, lim, abort_p)) break;
        mbar_arrive_expect_tx(bar(B_V_FULL + st), TC_TILE_BYTES);
        tma_load_3d(sV, &map_v, bar(B_V_FULL + st), 0, J * TC_BLK, bh);
        tma_load_3d(sV + TC_HALF_BYTES, &map_v, bar(B_V_FULL + st), 64, J * TC_BLK, bh);
        issued_v = j + 1;
      }
      if (*abort_p) {
        // Drain: every copy issued must land before this CTA's shared memory
        // is released. Only the last TC_NS blocks can still be in flight (a
        // stage is reloaded only after its previous copy was consumed).
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(B_Q_FULL), 0, lim, &no_abort);
        for (int j = issued_k > TC_NS ? issued_k - TC_NS : 0; j < issued_k; ++j) {
          const int st = j % TC_NS;
          const uint32_t ph = (j / TC_NS) & 1;
          no_abort = 0;
          mbar_wait_bounded(bar(B_K_FULL + st), ph, lim, &no_abort);
          if (j < issued_v) {
            no_abort = 0;
            mbar_wait_bounded(bar(B_V_FULL + st), ph, lim, &no_abort);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0 && n > 0) {
      bool ok = mbar_wait_bounded(bar(B_Q_FULL), 0, lim, abort_p);
      if (ok) ok = mbar_wait_bounded(bar(B_K_FULL + 0), 0, lim, abort_p);
      if (ok) {
        tc_fence_after();
        tc_issue_qk(tS0, sQ, sK0);
        umma_commit(bar(B_K_EMPTY + 0));
        umma_commit(bar(B_S_FULL + 0));
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          const int st1 = (j + 1) % TC_NS;
          if (!(ok = mbar_wait_bounded(bar(B_K_FULL + st1), ((j + 1) / TC_NS) & 1, lim, abort_p)))
            break;
          tc_fence_after();
          tc_issue_qk(tS0 + ((j + 1) & 1) * 128, sQ, sK0 + st1 * TC_TILE_BYTES);
          umma_commit(bar(B_K_EMPTY + st1));
          umma_commit(bar(B_S_FULL + ((j + 1) & 1)));
        }
        const int st = j % TC_NS;
        if (!(ok = mbar_wait_bounded(bar(B_P_FULL + (j & 1)), (j >> 1) & 1, lim, abort_p))) break;
        if (!(ok = mbar_wait_bounded(bar(B_V_FULL + st), (j / TC_NS) & 1, lim, abort_p))) break;
        tc_fence_after();
        tc_issue_pv(tO, tS0 + (j & 1) * 128, sV0 + st * TC_TILE_BYTES, j > 0);
        umma_commit(bar(B_V_EMPTY + st));
        umma_commit(bar(B_O_DONE));
      }
      if (!ok) {
        // Drain this thread's MMAs before TMEM is released.
        umma_commit(bar(B_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(B_DRAIN), 0, lim, &no_abort);
      }
    }
  } else {
    // ------------------------------------------- softmax / correction / out --
    const int wq = warp & 3;               // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;          // query row within the tile
    const int row = I * TC_BLK + r;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_S_FULL + b), (j >> 1) & 1, lim, abort_p));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tS0 + b * 128 + lane_off;
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[i]);
      }
      tmem_wait_ld();
      const int J = a.col[beg + j];
      const int valid = min(TC_BLK, a.N - J * TC_BLK);
      // largest scaled logit of the valid columns (valid >= 1 for a live block)
      float mx = -INFINITY, mn = INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        if (i < valid) {
          mx = fmaxf(mx, s[i]);
          mn = fminf(mn, s[i]);
        }
      }
      const float m_cand = (sl2 >= 0.f ? mx : mn) * sl2;
      const bool need = m_cand > m_used + TC_TAU;
      float alpha = 1.f;
      if (need) {
        alpha = exp2f(m_used - m_cand);
        m_used = m_cand;
        l *= alpha;
      }
      if (__any_sync(0xffffffffu, need && j > 0)) {
        // O holds the sum up to PV(j-1): wait for it, then rescale in TMEM.
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_O_DONE), (j - 1) & 1, lim, abort_p));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + lane_off + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(tO + lane_off + c * 32, v);
        }
      }
      const float neg_m = -m_used;
      uint32_t pk[64];
      float rs = 0.f;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float p0 = (2 * i < valid) ? exp2f(fmaf(s[2 * i], sl2, neg_m)) : 0.f;
        const float p1 = (2 * i + 1 < valid) ? exp2f(fmaf(s[2 * i + 1], sl2, neg_m)) : 0.f;
        rs += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l += rs;
      {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t (*)[32]>(&pk[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t (*)[32]>(&pk[32]);
        const uint32_t tP = tS0 + b * 128 + lane_off;
        tmem_st32(tP, lo);
        tmem_st32(tP + 32, hi);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL + b));
    }
    // epilogue
    const long long obase = (static_cast<long long>(bh) * a.N + row) * TC_D;
    if (n > 0 && ok)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_O_DONE), (n - 1) & 1, lim, abort_p));
    if (n > 0 && ok) {
      tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + lane_off + c * 32, v);
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
    } else if (n == 0 && row < a.N) {
      uint4* dst = reinterpret_cast<uint4*>(a.out + obase);
#pragma unroll
      for (int q4 = 0; q4 < 16; ++q4) dst[q4] = make_uint4(0, 0, 0, 0);
      if (a.lse != nullptr) a.lse[static_cast<long long>(bh) * a.N + row] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace va
