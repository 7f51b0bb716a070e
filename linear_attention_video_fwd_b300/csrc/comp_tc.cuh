// SVG-EAR compensated attention on the 5th-generation tensor cores (bf16,
// d = D, 64 or 128): one softmax per query over (1) virtual centroid keys kc_c with
// logit bias ln n_c and values vc_c for every non-empty key cluster that is
// not selected for the query's cluster, and (2) the exact keys of the
// selected key clusters (SVG-EAR, gist.science 2603.08982, technical summary
// sec. 2, ideas 1 and 2).
//
// Layout: Q, K and V are first gathered into cluster order, so a query
// cluster is a contiguous row range of Qs and a key cluster one of Ks / Vs.
// A work unit is one 128-row chunk of one query cluster; a CTA takes two
// chunks (tiles t = 0, 1) whose key streams are interleaved entry by entry,
// reusing the two-tile pipeline of attn_tc.cuh (one MMA thread, one softmax
// warpgroup per tile, S_t and O_t in TMEM), with two TMA producer warps: one
// for Q, K and the column biases, one for V.
//
// Key stream of a query cluster p: nv virtual tiles (centroids 128j ..
// 128j + 127, one TMA box each for K and V), then exact tiles of 16 slots.
// A slot is 8 consecutive rows of one selected key cluster (an 8-row TMA box,
// which lands on a whole 128B-swizzle atom, so slots assemble into the same
// shared-memory layout as one 128-row box); a cluster of n_c keys takes
// ceil(n_c / 8) slots and the rows past n_c are masked. The K producer passes
// each entry's 128 column biases (log2 n_c of a virtual key, -inf for a
// selected or empty cluster; 0 / -inf for a valid / padding slot row) to the
// softmax through a small shared-memory ring with its own full / empty
// barriers; the softmax adds them with the logit scaling in one packed FMA.
#pragma once

#include <type_traits>

#include "attn_tc.cuh"

namespace va {

constexpr int CT_NM = 4;  // validity-mask ring entries
// K and V ring depths (two stages each, as in the attention kernel).
constexpr int CT_NK = 2;
constexpr int CT_NV = 2;
// Two Q tiles plus the K and V rings, tiles of 128 rows x D dims.
template <int D>
constexpr int ct_smem_bytes() { return 1024 + TcDim<D>::kTileBytes * (2 + CT_NK + CT_NV); }
// Register split of this kernel (launched at TC_LAUNCH_REGS per thread): the
// producer's slot search needs more than the attention kernel's producer.
constexpr int CT_REGS_DEC = 72;
constexpr int CT_REGS_INC = 216;
static_assert(128 * CT_REGS_DEC + 256 * CT_REGS_INC <= TC_THREADS * TC_LAUNCH_REGS,
              "register split exceeds the launch allocation");

struct CompArgs {
  const int* choff;    // [BH][Cq + 1] offsets of 128-row query chunks per cluster
  const int* qoff;     // [BH][Cq + 1] query cluster offsets in cluster order
  const int* qperm;    // [BH][N] token of each cluster-ordered query row
  const int* koff;     // [BH][Ck + 1] key cluster offsets in cluster order
  const int* nk;       // [BH][Ck]
  const int* seln;     // [BH][Cq] number of selected key clusters
  const int* selc;     // [BH][Cq][Ck] selected key clusters (ascending)
  const int* selbox;   // [BH][Cq][Ck + 1] exclusive prefix of ceil(n_c / 8) over selc
  const float* vbias;  // [BH][Cq][nv * 128] virtual-key bias, log2 units (-inf: none)
  const int* slots;    // slot table: (first key row << 4) | valid rows, 16 per exact tile
  const long long* slotbase;  // [BH] start of each (batch, head) in the slot table
  const int* slotoff;  // [BH][Cq + 1] start of each query cluster's slots
  __nv_bfloat16* out;  // [BH][N][128], token order
  int N, Cq, Ck, nv;
  float scale_log2;
  long long wait_limit;
};

enum : int {
  CB_Q_FULL = 0,                    // 2
  CB_K_FULL = CB_Q_FULL + 2,
  CB_K_EMPTY = CB_K_FULL + CT_NK,
  CB_V_FULL = CB_K_EMPTY + CT_NK,
  CB_V_EMPTY = CB_V_FULL + CT_NV,
  CB_M_FULL = CB_V_EMPTY + CT_NV,   // CT_NM
  CB_M_EMPTY = CB_M_FULL + CT_NM,   // CT_NM, 128 arrivals
  CB_S_FULL = CB_M_EMPTY + CT_NM,   // 2
  CB_P_FULL = CB_S_FULL + 2,        // 2, 128 arrivals
  CB_O_DONE = CB_P_FULL + 2,        // 2
  CB_DRAIN = CB_O_DONE + 2,
  CB_COUNT = CB_DRAIN + 1
};

// Row maps of the cluster-ordered K and V with box heights 8 << i (i < 5):
// a run of 2^i consecutive slots with contiguous source rows is one copy.
constexpr int CT_NBOX = 5;
struct CompSlotMaps {
  CUtensorMap k[CT_NBOX];
  CUtensorMap v[CT_NBOX];
};

struct CompTile {
  int p, r0, nrows, ns, nslots, n;  // cluster, first row, rows, selected, slots, blocks
};

// Entry u of the interleaved stream of two tiles with n0, n1 blocks.
__device__ __forceinline__ void ct_entry(int u, int n0, int n1, int& t, int& j) {
  const int nmin = min(n0, n1);
  if (u < 2 * nmin) {
    t = u & 1;
    j = u >> 1;
  } else {
    t = n0 > n1 ? 0 : 1;
    j = nmin + (u - 2 * nmin);
  }
}

__device__ __forceinline__ int ct_index(int t, int j, int n0, int n1) {
  const int nmin = min(n0, n1);
  return j < nmin ? 2 * j + t : 2 * nmin + (j - nmin);
}

// Softmax of one tile (thread r owns row r of the tile); O has D columns.
template <int D>
__device__ __forceinline__ void ct_softmax(const CompArgs& a, int tile, const CompTile& T,
                                           int n0, int n1, int bh, uint32_t tmem,
                                           uint64_t* bars, const float4* bias_ring,
                                           volatile int* abort_p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + tile * 256 + lane_off;
  const uint32_t tO = tS + 128;
  const uint32_t bS = smem_u32(&bars[CB_S_FULL + tile]);
  const uint32_t bP = smem_u32(&bars[CB_P_FULL + tile]);
  const uint32_t bO = smem_u32(&bars[CB_O_DONE + tile]);
  const long long lim = a.wait_limit;
  const float sl2 = a.scale_log2;

  float m_used = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < T.n; ++j) {
    const int u = ct_index(tile, j, n0, n1);
    const int ms = u % CT_NM;
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(bS, j & 1, lim, abort_p));
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars[CB_M_FULL + ms]),
                                                           (u / CT_NM) & 1, lim, abort_p));
    if (!ok) break;
    tc_fence_after();
    float s[128];
    // scaled logit plus the entry's column bias (log2 units): log2 n_c of a
    // virtual key (-inf for a selected or empty cluster), 0 / -inf for a
    // valid / padding row of an exact tile
    const float4* brow = bias_ring + ms * 32;
    auto load_biased = [&]() {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[i]);
      }
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        // volatile: each pass loads its own biases (held across the passes
        // they would take 128 registers)
        float4 bb;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(bb.x), "=f"(bb.y), "=f"(bb.z), "=f"(bb.w)
                     : "r"(smem_u32(brow + i)));
        ffma2_v(s[4 * i], s[4 * i + 1], s[4 * i], s[4 * i + 1], sl2, bb.x, bb.y);
        ffma2_v(s[4 * i + 2], s[4 * i + 3], s[4 * i + 2], s[4 * i + 3], sl2, bb.z, bb.w);
      }
    };
    float r0, r1, r2, r3;
    // P = 2^(logit - m_used) in s, row sums in r0..r3
    auto exp_sum = [&]() {
      const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
#pragma unroll
      for (int i = 0; i < 128; i += 2) {
        ffma2_bc(s[i], s[i + 1], s[i], s[i + 1], 1.f, neg_m);
        s[i] = ex2_approx(s[i]);
        s[i + 1] = ex2_approx(s[i + 1]);
      }
      r0 = r1 = r2 = r3 = 0.f;
#pragma unroll
      for (int i = 0; i < 128; i += 4) {
        fadd2_acc(r0, r1, s[i], s[i + 1]);
        fadd2_acc(r2, r3, s[i + 2], s[i + 3]);
      }
    };
    load_biased();
    // Pass 0 tries the entry against the running max with no max pass: a sum
    // of at most 2^(TAU - 1) bounds every weight by it, so pass 1 would
    // keep m_used and give exactly these weights. A larger sum, NaN, or a row
    // with no running max yet sends the warp to pass 1 (S reloaded, the bias
    // slot still held), which takes the max and maybe rescales.
#pragma unroll 1
    for (int pass = 0;; ++pass) {
      if (pass == 1) {
        load_biased();
        float m0 = fmax3(s[0], s[1], s[2]), m1 = fmax3(s[3], s[4], s[5]);
        float m2 = fmax3(s[6], s[7], s[8]), m3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
        for (int i = 12; i < 124; i += 8) {
          m0 = fmax3(m0, s[i], s[i + 1]);
          m1 = fmax3(m1, s[i + 2], s[i + 3]);
          m2 = fmax3(m2, s[i + 4], s[i + 5]);
          m3 = fmax3(m3, s[i + 6], s[i + 7]);
        }
        const float m_cand =
            fmax3(fmax3(m0, m1, s[124]), fmax3(m2, m3, s[125]), fmaxf(s[126], s[127]));
        const bool need = m_cand > m_used + TC_TAU;  // false while the block is all -inf
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m_used - m_cand);
          m_used = m_cand;
          l *= alpha;
        }
        if (__any_sync(0xffffffffu, need && j > 0)) {
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
      exp_sum();
      if (pass == 1 ||
          !__any_sync(0xffffffffu, m_used == -INFINITY ||
                                       !((r0 + r1) + (r2 + r3) <= TC_FAST_SUM)))
        break;
    }
    mbar_arrive(smem_u32(&bars[CB_M_EMPTY + ms]));
    if (!ok) break;
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // pack and store P in two halves of 64 keys
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const int c = h * 64 + i;
        pk[i / 2] = pack_bf16x2(s[c], s[c + 1]);
        pk[i / 2 + 1] = pack_bf16x2(s[c + 2], s[c + 3]);
      }
      tmem_st32(tS + h * 32, pk);
    }
    l += (r0 + r1) + (r2 + r3);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bP);
  }
  if (T.n > 0 && ok)
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(bO, (T.n - 1) & 1, lim, abort_p));
  if (T.n > 0 && ok) {
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const bool live = r < T.nrows;
    const int tok = live ? a.qperm[static_cast<long long>(bh) * a.N + T.r0 + r] : 0;
    __nv_bfloat16* orow = a.out + (static_cast<long long>(bh) * a.N + tok) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tO + c * 32, v);
      tmem_wait_ld();
      if (live) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
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
  }
}

__device__ __forceinline__ void ct_locate(const CompArgs& a, int bh, int chunk, CompTile& T) {
  const int* co = a.choff + static_cast<long long>(bh) * (a.Cq + 1);
  int lo = 0, hi = a.Cq - 1;  // last p with co[p] <= chunk (skips empty clusters)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (co[mid] <= chunk) lo = mid;
    else hi = mid - 1;
  }
  const int* qo = a.qoff + static_cast<long long>(bh) * (a.Cq + 1);
  const long long pc = static_cast<long long>(bh) * a.Cq + lo;
  T.p = lo;
  T.r0 = qo[lo] + (chunk - co[lo]) * 128;
  T.nrows = min(128, qo[lo + 1] - T.r0);
  T.ns = a.seln[pc];
  T.nslots = a.selbox[pc * (a.Ck + 1) + T.ns];
  T.n = a.nv + (T.nslots + 15) / 16;
}

template <int D>
__global__ void __launch_bounds__(TC_THREADS, 1)
    comp_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_kc,
                   const __grid_constant__ CUtensorMap map_vc,
                   const __grid_constant__ CompSlotMaps maps, const CompArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[CB_COUNT];
  __shared__ float4 bias_ring[CT_NM * 32];  // per entry: 128 column biases
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ CompTile tiles[2];

  const int bh = blockIdx.y;
  const int total = a.choff[static_cast<long long>(bh) * (a.Cq + 1) + a.Cq];
  const int c0 = 2 * blockIdx.x;
  if (c0 >= total) return;  // whole CTA, before any barrier or TMEM use
  const bool has1 = c0 + 1 < total;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kTile = TcDim<D>::kTileBytes, kHalves = TcDim<D>::kHalves;
  const uint32_t sQ0 = smem_u32(smem);
  const uint32_t sK0 = sQ0 + 2 * kTile;
  const uint32_t sV0 = sK0 + CT_NK * kTile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (tid == 0) {
    abort_flag = 0;
    ct_locate(a, bh, c0, tiles[0]);
    if (has1) ct_locate(a, bh, c0 + 1, tiles[1]);
    else tiles[1] = CompTile{0, 0, 0, 0, 0, 0};
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(CB_Q_FULL + t), 1);
      mbar_init(bar(CB_S_FULL + t), 1);
      mbar_init(bar(CB_P_FULL + t), 128);
      mbar_init(bar(CB_O_DONE + t), 1);
    }
    for (int s = 0; s < CT_NK; ++s) {
      mbar_init(bar(CB_K_FULL + s), 1);
      mbar_init(bar(CB_K_EMPTY + s), 1);
    }
    for (int s = 0; s < CT_NV; ++s) {
      mbar_init(bar(CB_V_FULL + s), 1);
      mbar_init(bar(CB_V_EMPTY + s), 1);
    }
    for (int s = 0; s < CT_NM; ++s) {
      mbar_init(bar(CB_M_FULL + s), 1);
      mbar_init(bar(CB_M_EMPTY + s), 128);
    }
    mbar_init(bar(CB_DRAIN), 1);
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
  const CompTile T0 = tiles[0], T1 = tiles[1];
  const int n0 = T0.n, n1 = T1.n, nent = n0 + n1;

  if (warp >= 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(CT_REGS_INC));
    const int tile = (warp - 4) >> 2;
    if (tile == 0 || has1)
      ct_softmax<D>(a, tile, tile == 0 ? T0 : T1, n0, n1, bh, tmem, bars, bias_ring, abort_p);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CT_REGS_DEC));
    if (warp == 0 || warp == 2) {
      // --------------------------------------------------------- producers --
      // Warp 0: the Q tiles, then the K copies and the column biases of every
      // entry; warp 2: the V copies. Each walks the whole stream on its own,
      // so K never waits behind a V stage (which frees only when an earlier
      // PV completed). Lane 0 waits and arms the barriers, lanes 0..15 issue
      // one slot's copies each.
      const bool kw = warp == 0;
      int issued = 0;
      if (lane == 0) {
        if (kw) {
          tma_prefetch_desc(&map_q);
          tma_prefetch_desc(&map_kc);
          for (int i = 0; i < CT_NBOX; ++i) tma_prefetch_desc(&maps.k[i]);
          mbar_arrive_expect_tx(bar(CB_Q_FULL + 0), kTile);
          for (int h = 0; h < kHalves; ++h)
            tma_load_3d(sQ0 + h * TC_HALF_BYTES, &map_q, bar(CB_Q_FULL + 0), 64 * h, T0.r0, bh);
          if (has1) {
            const uint32_t sQ1 = sQ0 + kTile;
            mbar_arrive_expect_tx(bar(CB_Q_FULL + 1), kTile);
            for (int h = 0; h < kHalves; ++h)
              tma_load_3d(sQ1 + h * TC_HALF_BYTES, &map_q, bar(CB_Q_FULL + 1), 64 * h, T1.r0, bh);
          }
        } else {
          tma_prefetch_desc(&map_vc);
          for (int i = 0; i < CT_NBOX; ++i) tma_prefetch_desc(&maps.v[i]);
        }
      }
      // Slot lists of the two tiles; the slot of the next entry is read one
      // entry ahead, so its global-memory latency overlaps this entry's waits.
      const int* slots_bh = a.slots + a.slotbase[bh];
      const int* so = a.slotoff + static_cast<long long>(bh) * (a.Cq + 1);
      const int* slot_list0 = slots_bh + so[T0.p];
      const int* slot_list1 = slots_bh + so[T1.p];
      const float* vb0 = a.vbias + (static_cast<long long>(bh) * a.Cq + T0.p) * (a.nv * 128);
      const float* vb1 = a.vbias + (static_cast<long long>(bh) * a.Cq + T1.p) * (a.nv * 128);
      auto slot_of = [&](int u) -> int {
        int t, j;
        ct_entry(u, n0, n1, t, j);
        const int* sl = t == 0 ? slot_list0 : slot_list1;
        return (j >= a.nv && lane < 16) ? sl[(j - a.nv) * 16 + lane] : 0;
      };
      const CUtensorMap* map_c = kw ? &map_kc : &map_vc;  // centroid rows (virtual tiles)
      const CUtensorMap* map_slots = kw ? maps.k : maps.v;  // slot runs (exact tiles)
      const int nst = kw ? CT_NK : CT_NV;
      const int b_full = kw ? CB_K_FULL : CB_V_FULL, b_empty = kw ? CB_K_EMPTY : CB_V_EMPTY;
      const uint32_t s0 = kw ? sK0 : sV0;
      int sd_next = nent > 0 ? slot_of(0) : 0;
      for (int u = 0; u < nent; ++u) {
        int t, j;
        ct_entry(u, n0, n1, t, j);
        const int st = u % nst;
        const uint32_t dst = s0 + st * kTile;
        // slot of this lane (exact tiles): source row and valid row count,
        // from the slot table (16 slots per exact tile, padding slots valid 0)
        const int sd = sd_next;
        if (u + 1 < nent) sd_next = slot_of(u + 1);
        const int src = sd >> 4, valid = sd & 15;
        bool ok = true;
        if (lane == 0) {
          if (u >= nst)
            ok = mbar_wait_bounded(bar(b_empty + st), ((u / nst) & 1) ^ 1, lim, abort_p);
          if (ok) mbar_arrive_expect_tx(bar(b_full + st), kTile);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        if (j < a.nv) {
          if (lane == 0) {
            for (int h = 0; h < kHalves; ++h)
              tma_load_3d(dst + h * TC_HALF_BYTES, map_c, bar(b_full + st), 64 * h, j * 128, bh);
          }
        } else {
          // Runs of slots with contiguous source rows (slot l continues slot
          // l - 1 when its first row is 8 further) are copied as greedy
          // power-of-two pieces, each one box of 8 * 2^i rows issued by the
          // lane of its first slot; together they cover the 16 slots once.
          const int prev = __shfl_up_sync(0xffffffffu, src, 1);
          const bool starts_run = lane < 16 && (lane == 0 || src != prev + 8);
          const uint32_t starts = __ballot_sync(0xffffffffu, starts_run);
          if (lane < 16) {
            const uint32_t upto = starts & ((2u << lane) - 1u);
            const int r0 = 31 - __clz(upto);
            const uint32_t above = starts & ~((2u << lane) - 1u);
            const int r1 = above ? __ffs(above) - 1 : 16;
            const int n = r1 - r0, pos = lane - r0;
            int lg = -1;
            for (int at = 0; at < n;) {
              const int l2 = 31 - __clz(n - at);
              if (at == pos) lg = l2;
              at += 1 << l2;
            }
            if (lg >= 0) {
              for (int h = 0; h < kHalves; ++h)
                tma_load_3d(dst + h * TC_HALF_BYTES + lane * 1024, map_slots + lg,
                            bar(b_full + st), 64 * h, src, bh);
            }
          }
        }
        if (lane == 0) issued = u + 1;
        if (!kw) continue;
        // column biases of the entry (lane l: columns 4l..4l+3, rows 4 (l & 1)..
        // of slot l / 2): the virtual bias row, or 0 / -inf for valid / padding
        // slot rows
        const int ms = u % CT_NM;
        const int vslot = __shfl_sync(0xffffffffu, valid, lane >> 1);
        float4 brow;
        if (j < a.nv) {
          brow = __ldg(reinterpret_cast<const float4*>((t == 0 ? vb0 : vb1) + j * 128) + lane);
        } else {
          const int r0 = (lane & 1) * 4;
          brow.x = r0 + 0 < vslot ? 0.f : -INFINITY;
          brow.y = r0 + 1 < vslot ? 0.f : -INFINITY;
          brow.z = r0 + 2 < vslot ? 0.f : -INFINITY;
          brow.w = r0 + 3 < vslot ? 0.f : -INFINITY;
        }
        if (lane == 0 && u >= CT_NM)
          ok = mbar_wait_bounded(bar(CB_M_EMPTY + ms), ((u / CT_NM) & 1) ^ 1, lim, abort_p);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        bias_ring[ms * 32 + lane] = brow;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(CB_M_FULL + ms));
      }
      if (lane == 0 && *abort_p) {
        // Drain: only the last nst copies of a ring can still be in flight.
        volatile int no_abort = 0;
        if (kw) {
          mbar_wait_bounded(bar(CB_Q_FULL + 0), 0, lim, &no_abort);
          if (has1) {
            no_abort = 0;
            mbar_wait_bounded(bar(CB_Q_FULL + 1), 0, lim, &no_abort);
          }
        }
        for (int u = issued > nst ? issued - nst : 0; u < issued; ++u) {
          no_abort = 0;
          mbar_wait_bounded(bar(b_full + u % nst), (u / nst) & 1, lim, &no_abort);
        }
      }
    } else if (warp == 1) {
      // --------------------------------------------------------------- MMA --
      if (lane == 0) {
        const uint32_t sQ1 = sQ0 + kTile;
        bool ok = mbar_wait_bounded(bar(CB_Q_FULL + 0), 0, lim, abort_p);
        if (ok && has1) ok = mbar_wait_bounded(bar(CB_Q_FULL + 1), 0, lim, abort_p);
        // Per-tile state in scalars selected at compile time: an array indexed
        // by the runtime tile number would live in local memory.
        int pend0 = -1, pend1 = -1;  // entry whose PV is still to issue
        int cnt0 = 0, cnt1 = 0;      // QKs issued
        // descriptor low words of the Q tiles and of stage 0 of the K and V
        // rings (a stage adds stage * (tile bytes >> 4); one asm block issues
        // a product's eight steps)
        const uint64_t dq0 = sw128_desc(sQ0, 16, 1024), dq1 = sw128_desc(sQ1, 16, 1024);
        const uint64_t dk = sw128_desc(sK0, 16, 1024);
        const uint64_t dv = sw128_desc(sV0, TC_HALF_BYTES, 1024);
        const uint32_t k_lo = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
        const uint32_t v_lo = static_cast<uint32_t>(dv), v_hi = static_cast<uint32_t>(dv >> 32);
        using Tile0 = std::integral_constant<int, 0>;
        using Tile1 = std::integral_constant<int, 1>;
        auto issue_pv = [&](auto tile) -> bool {
          constexpr int t = decltype(tile)::value;
          int& pend = t == 0 ? pend0 : pend1;
          const int pu = pend;
          const int jj = (t == 0 ? cnt0 : cnt1) - 1;
          if (!mbar_wait_bounded(bar(CB_P_FULL + t), jj & 1, lim, abort_p)) return false;
          const int sv = pu % CT_NV;
          if (!mbar_wait_bounded(bar(CB_V_FULL + sv), (pu / CT_NV) & 1, lim, abort_p)) return false;
          tc_fence_after();
          tc_pv_group<D>(tmem + t * 256 + 128, tmem + t * 256, v_lo + sv * (kTile >> 4), v_hi,
                         jj > 0);
          umma_commit(bar(CB_O_DONE + t));
          umma_commit(bar(CB_V_EMPTY + sv));  // every entry is read by one tile only
          pend = -1;
          return true;
        };
        auto issue_entry = [&](auto tile, int u) -> bool {
          constexpr int t = decltype(tile)::value;
          const int sk = u % CT_NK;
          if (!mbar_wait_bounded(bar(CB_K_FULL + sk), (u / CT_NK) & 1, lim, abort_p)) return false;
          if ((t == 0 ? pend0 : pend1) >= 0 && !issue_pv(tile)) return false;
          tc_fence_after();
          tc_qk_group<D>(tmem + t * 256, static_cast<uint32_t>(t == 0 ? dq0 : dq1),
                         k_lo + sk * (kTile >> 4), k_hi);
          umma_commit(bar(CB_S_FULL + t));
          umma_commit(bar(CB_K_EMPTY + sk));
          (t == 0 ? pend0 : pend1) = u;
          ++(t == 0 ? cnt0 : cnt1);
          return true;
        };
        for (int u = 0; ok && u < nent; ++u) {
          int t, j;
          ct_entry(u, n0, n1, t, j);
          // A V stage is reloaded NV entries later: release stale pending PVs.
          if (pend0 >= 0 && pend0 <= u - CT_NV && !(ok = issue_pv(Tile0{}))) break;
          if (pend1 >= 0 && pend1 <= u - CT_NV && !(ok = issue_pv(Tile1{}))) break;
          ok = t == 0 ? issue_entry(Tile0{}, u) : issue_entry(Tile1{}, u);
        }
        if (ok && pend0 >= 0) ok = issue_pv(Tile0{});
        if (ok && pend1 >= 0) ok = issue_pv(Tile1{});
        if (!ok) {
          umma_commit(bar(CB_DRAIN));
          volatile int no_abort = 0;
          mbar_wait_bounded(bar(CB_DRAIN), 0, lim, &no_abort);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ preparation --

// dst[bh][t] = src[bh][perm[bh][t]] for bf16 rows of D (D / 8 lanes per row,
// 16 bytes each). Grid (ceil(N / GR_ROWS<D>), BH), 128 threads.
template <int D>
constexpr int GR_ROWS = 128 / (D / 8);
template <int D>
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                   const int* __restrict__ perm, int N,
                                   __nv_bfloat16* __restrict__ dst) {
  constexpr int kLanes = D / 8, kRows = GR_ROWS<D>;
  const int bh = blockIdx.y;
  const int t = blockIdx.x * kRows + threadIdx.x / kLanes;
  const int c = threadIdx.x % kLanes;
  if (t >= N) return;
  const long long base = static_cast<long long>(bh) * N;
  const int row = perm[base + t];
  const uint4* s = reinterpret_cast<const uint4*>(src + (base + row) * D);
  uint4* d = reinterpret_cast<uint4*>(dst + (base + t) * D);
  d[c] = s[c];
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ x, long long n,
                                   __nv_bfloat16* __restrict__ y) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) y[i] = __float2bfloat16_rn(x[i]);
}

// ceil(n_p / rows) chunks per query cluster.
__global__ void chunk_count_kernel(const int* __restrict__ nq, int Cq, int rows,
                                   int* __restrict__ nch) {
  const int bh = blockIdx.y;
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= Cq) return;
  const int n = nq[static_cast<long long>(bh) * Cq + p];
  nch[static_cast<long long>(bh) * Cq + p] = (n + rows - 1) / rows;
}

// One warp per (bh, p): the slot prefix over the selected list and the
// virtual-key bias row (log2 n_c for non-empty unselected c, else -inf).
__global__ void comp_prep_kernel(const int* __restrict__ nk, const int* __restrict__ seln,
                                 const int* __restrict__ selc, const uint8_t* __restrict__ sel,
                                 int Cq, int Ck, int nv, int* __restrict__ selbox,
                                 float* __restrict__ vbias) {
  const int bh = blockIdx.y;
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= Cq) return;
  const long long pc = static_cast<long long>(bh) * Cq + p;
  const int* nkb = nk + static_cast<long long>(bh) * Ck;
  const int ns = seln[pc];
  const int* sl = selc + pc * Ck;
  int* sb = selbox + pc * (Ck + 1);
  int base = 0;
  for (int s0 = 0; s0 < ns; s0 += 32) {
    const int s = s0 + lane;
    const int boxes = s < ns ? (nkb[sl[s]] + 7) / 8 : 0;
    int incl = boxes;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (s < ns) sb[s] = base + incl - boxes;
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) sb[ns] = base;
  const uint8_t* sr = sel + pc * Ck;
  float* vb = vbias + pc * (nv * 128);
  for (int c = lane; c < nv * 128; c += 32) {
    const int n = c < Ck ? nkb[c] : 0;
    vb[c] = (n > 0 && !sr[c]) ? log2f(static_cast<float>(n)) : -INFINITY;
  }
}

// Padded slot count per query cluster: 16 * ceil(slots / 16).
__global__ void slot_count_kernel(const int* __restrict__ seln, const int* __restrict__ selbox,
                                  int Cq, int Ck, int* __restrict__ cnt) {
  const int bh = blockIdx.y;
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= Cq) return;
  const long long pc = static_cast<long long>(bh) * Cq + p;
  const int ns = selbox[pc * (Ck + 1) + seln[pc]];
  cnt[pc] = (ns + 15) / 16 * 16;
}

// base[b] = sum of off[b'][Cq] for b' < b; base[BH] = total (one thread).
__global__ void slot_base_kernel(const int* __restrict__ off, int Cq, int BH,
                                 long long* __restrict__ base) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  long long acc = 0;
  for (int b = 0; b < BH; ++b) {
    base[b] = acc;
    acc += off[static_cast<long long>(b) * (Cq + 1) + Cq];
  }
  base[BH] = acc;
}

// One thread per slot of one query cluster: (first key row << 4) | valid rows
// for slot i < slots (a slot is 8 rows of one selected key cluster, in cluster
// order), 0 for the padding up to a multiple of 16. Grid (Cq, BH).
__global__ void slot_fill_kernel(const int* __restrict__ koff, const int* __restrict__ seln,
                                 const int* __restrict__ selc, const int* __restrict__ selbox,
                                 int Cq, int Ck, const long long* __restrict__ base,
                                 const int* __restrict__ off, int* __restrict__ slots) {
  const int bh = blockIdx.y, p = blockIdx.x;
  const long long pc = static_cast<long long>(bh) * Cq + p;
  const int ns = seln[pc];
  const int* sb = selbox + pc * (Ck + 1);
  const int* sl = selc + pc * Ck;
  const int* ko = koff + static_cast<long long>(bh) * (Ck + 1);
  const int nslots = sb[ns];
  const int npad = (nslots + 15) / 16 * 16;
  int* out = slots + base[bh] + off[static_cast<long long>(bh) * (Cq + 1) + p];
  for (int i = threadIdx.x; i < npad; i += blockDim.x) {
    int v = 0;
    if (i < nslots) {
      int lo = 0, hi = ns - 1;  // last selected s with sb[s] <= i
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sb[mid] <= i) lo = mid;
        else hi = mid - 1;
      }
      const int c = sl[lo];
      const int src = ko[c] + 8 * (i - sb[lo]);
      v = (src << 4) | min(8, ko[c + 1] - src);
    }
    out[i] = v;
  }
}

}  // namespace va
