// Error probe of SVG-EAR (gist.science 2603.08982, technical summary sec. 2,
// idea 2: query-cluster centroids as proxies, streamed over the keys without
// storing logits) on the 5th-generation tensor cores, bf16 K/V, head_dim D
// (64 or 128).
//
// Per (batch*head, proxy tile of 128 query clusters, key split):
//   pass 1  sweep A: l = qc . k for every key of the split, row max m2 (log2
//           units); sweep B: e = 2^(l s log2e - m2), Z = sum e, O = sum e v;
//           the partials {m2, Z, O} of the splits are merged afterwards;
//   pass 2  with the merged m2, Z, O of each proxy: per key cluster c,
//           E_c = sum_{j in c} e_j v_j, Zc = sum_{j in c} e_j, then
//           r = E_c - Zc O - w_c (vc_c - O), w_c = n_c 2^(lbar s log2e - m2),
//           err(p, c) = |r| / Z, where lbar = mean_{j in c} l_j equals
//           qc . kc_c (kc_c is the member mean, and the dot product is
//           linear): taken from the same logits as the e_j, a singleton
//           cluster gets w_c = e_j exactly and r = 0 to rounding.
//
// Precision: the fp32 operands (proxies qc, weights e) are split into three
// bf16 pieces hi + mid + lo (24 significant bits, the fp32 mantissa), keys and
// values are exact in bf16, products are exact and the tensor cores accumulate
// in fp32; the logits of the hi piece and of the mid + lo pieces go to separate
// accumulators (added in fp32 by the softmax), so the large partial sums of
// the hi piece do not absorb the small ones.
//
// Key layout: keys and values are copied in key-cluster order with every
// cluster padded to a multiple of 16 rows (zero rows), so each K = 16 step of
// an MMA lies inside one cluster; a 16-row group carries (valid rows, first,
// last) metadata. A split is a range of whole clusters with about equal
// numbers of groups; a tile is 4 groups (64 rows).
//
// 384 threads: warp 0 TMA producer (proxy pieces once, K/V tiles through rings
// of 3); warp 1 MMA issuer (one thread): S_u = sum_i Qpiece_i K_u^T (M 128, N
// 64) into one of two TMEM stages, then, once the softmax wrote the three P
// pieces over that stage, O (pass 1) or E of the group's cluster (pass 2) +=
// sum_i Ppiece_i V_group (TMEM A operand); warps 4..7 softmax (thread r owns
// proxy row r); warps 8..11 (pass 2) per-cluster residual norm from the E
// accumulator (two TMEM buffers) and O held in registers.
// TMEM columns: stage b at [128b, 128b + 128) (S of the hi piece in the first
// 64, S of mid + lo in the next 64, then the P pieces over them in 3 x 32);
// pass 1 O at [256, 384); pass 2 E buffers at 256 and 384.
//
// Every mbarrier wait is bounded; on a timeout the CTA records
// VA_ERR_TIMEOUT, drains its copies and MMAs and frees its TMEM.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace va {

constexpr int PT_KT = 64;    // keys per tile (4 groups of 16)
constexpr int PT_NK = 3;     // K ring stages
constexpr int PT_NV = 3;     // V ring stages
constexpr int PT_THREADS = 384;
constexpr int PT_QP_HALF = 128 * 64 * 2;    // 128 proxy rows x 64 dims (one TMA box)
constexpr int PT_KV_HALF = PT_KT * 64 * 2;   // 64 key rows x 64 dims

// Sizes that depend on the head dimension D.
template <int D>
struct PtDim {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kHalves = D / 64;
  static constexpr int kQP = 128 * D * 2;     // one bf16 piece of a 128-proxy tile
  static constexpr int kKV = PT_KT * D * 2;   // one 64-key tile of K or V
  static constexpr int kSmem = 1024 + 3 * kQP + (PT_NK + PT_NV) * kKV;
  static constexpr int kRow = 2 + D;          // {m2, Z, O[D]} per proxy
};
constexpr int PT_G_FIRST = 1 << 5;
constexpr int PT_G_LAST = 1 << 6;
constexpr uint32_t PT_STAGE_COLS = 128;  // S of the hi piece, S of mid + lo, then P
constexpr uint32_t PT_T_ACC = 2 * PT_STAGE_COLS;
// Register split as in the attention kernel: warpgroup 0 gives registers to
// the softmax and residual warpgroups (the latter keeps O_p in 128 registers).
constexpr int PT_LAUNCH_REGS = 168;
constexpr int PT_REGS_DEC = 72;
constexpr int PT_REGS_INC = 216;
static_assert(128 * PT_REGS_DEC + 256 * PT_REGS_INC <= PT_THREADS * PT_LAUNCH_REGS,
              "register split exceeds the launch allocation");

struct ProbeArgs {
  const int* gmeta;   // [BH][G] per 16-row group: valid rows | PT_G_FIRST | PT_G_LAST |
                      // cluster << 8
  const int* kpoff;   // [BH][Ck + 1] first padded row of each key cluster
  const int* nq;      // [BH][Cq] query-cluster sizes
  const float* mzo;   // pass 2: [BH][Cq][D + 2] merged {m2, Z, O / Z}
  const float* vc;    // pass 2: [BH][Ck][D] value means
  float* part;        // pass 1: [BH][Cq][NS][D + 2] split partials {m2, Z, O}
  float* err;         // pass 2: [BH][Cq][Ck]
  int Cq, Ck, Cqp, G, NS;
  float sl2;          // scale * log2(e)
  long long wait_limit;
};

enum : int {
  PB_Q = 0,
  PB_KF = 1,
  PB_KE = PB_KF + PT_NK,
  PB_VF = PB_KE + PT_NK,
  PB_VE = PB_VF + PT_NV,
  PB_SF = PB_VE + PT_NV,  // 2 (per TMEM stage)
  PB_PF = PB_SF + 2,      // 2, 128 arrivals
  PB_EF = PB_PF + 2,      // 2 (per E buffer)
  PB_ZF = PB_EF + 2,      // 2, 128 arrivals
  PB_EE = PB_ZF + 2,      // 2, 128 arrivals
  PB_OD = PB_EE + 2,
  PB_DRAIN = PB_OD + 1,
  PB_COUNT = PB_DRAIN + 1
};

// First cluster of split s of NS: the smallest c with kp[c] / 16 >= s * G / NS
// (G = groups of the head); split NS starts at Ck.
__device__ __forceinline__ int pt_split_cluster(const int* kp, int Ck, int s, int NS) {
  if (s >= NS) return Ck;
  const long long t = static_cast<long long>(kp[Ck] >> 4) * s / NS;
  int lo = 0, hi = Ck;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((kp[mid] >> 4) >= t) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// x = hi + mid + lo, each bf16 (round to nearest), packed in pairs.
__device__ __forceinline__ void pt_split3(float x0, float x1, uint32_t& hi, uint32_t& mid,
                                          uint32_t& lo) {
  hi = pack_bf16x2(x0, x1);
  const float r0 = x0 - __uint_as_float(hi << 16);
  const float r1 = x1 - __uint_as_float(hi & 0xffff0000u);
  mid = pack_bf16x2(r0, r1);
  lo = pack_bf16x2(r0 - __uint_as_float(mid << 16), r1 - __uint_as_float(mid & 0xffff0000u));
}

// Softmax warpgroup: thread r owns proxy row r of the tile.
template <int PASS, int D>
__device__ __forceinline__ void pt_softmax(const ProbeArgs& a, int bh, int pt, int split,
                                           int g_lo, int g_hi, int nt, uint32_t tmem,
                                           uint64_t* bars, float (*zc_s)[128],
                                           float (*w_s)[128], float (*vc_s)[128], int* cid_s,
                                           volatile int* abort_p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;
  const int p = pt * 128 + r;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const long long lim = a.wait_limit;
  const float sl2 = a.sl2;
  const int nval0 = PASS == 1 ? nt : 0;
  const int ne = nval0 + nt;
  const int* gm = a.gmeta + static_cast<long long>(bh) * a.G;
  float m2 = -INFINITY, Z = 0.f, zc = 0.f, ls = 0.f, vc_pre = 0.f;
  int nv = 0, cur_c = 0;
  if constexpr (PASS == 2)
    m2 = a.mzo[(static_cast<long long>(bh) * a.Cq + min(p, a.Cq - 1)) * PtDim<D>::kRow];
  int ci = -1;
  bool ok = true;
  int mn[4] = {0, 0, 0, 0};  // group metadata, read one tile ahead
  auto tile_meta = [&](int u, int (&m4)[4]) {
    const int t = u >= nval0 ? u - nval0 : u;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int gg = g_lo + 4 * t + g;
      m4[g] = gg < g_hi ? gm[gg] : 0;
    }
  };
  if (ne > 0) tile_meta(0, mn);
  for (int u = 0; u < ne; ++u) {
    const int b = u & 1;
    const int m4[4] = {mn[0], mn[1], mn[2], mn[3]};
    if (u + 1 < ne) tile_meta(u + 1, mn);
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars[PB_SF + b]), (u >> 1) & 1,
                                                    lim, abort_p));
    if (!ok) break;
    tc_fence_after();
    const uint32_t tS = tmem + b * PT_STAGE_COLS + lane_off;
    float s[64];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v0[32], v1[32];
      tmem_ld32(tS + 32 * h, v0);
      tmem_ld32(tS + 64 + 32 * h, v1);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) s[32 * h + i] = __uint_as_float(v0[i]) + __uint_as_float(v1[i]);
    }
    if (PASS == 1 && u < nval0) {
      // sweep A: row max of the scaled logits over the valid keys
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if ((j & 15) < (m4[j >> 4] & 31)) mx = fmaxf(mx, s[j] * sl2);
      m2 = fmaxf(m2, mx);
      tc_fence_before();
      mbar_arrive(smem_u32(&bars[PB_PF + b]));
      continue;
    }
    float lsum[4] = {0.f, 0.f, 0.f, 0.f};  // per group: sum of the valid raw logits
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const bool valid = (j & 15) < (m4[j >> 4] & 31);
      if (PASS == 2 && valid) lsum[j >> 4] += s[j];
      s[j] = valid ? ex2_approx(fmaf(s[j], sl2, -m2)) : 0.f;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t hi[16], mi[16], lo[16];
#pragma unroll
      for (int w = 0; w < 16; ++w) pt_split3(s[32 * h + 2 * w], s[32 * h + 2 * w + 1], hi[w], mi[w], lo[w]);
      tmem_st16(tS + h * 16, hi);
      tmem_st16(tS + 32 + h * 16, mi);
      tmem_st16(tS + 64 + h * 16, lo);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(smem_u32(&bars[PB_PF + b]));
    if constexpr (PASS == 1) {
      float z0 = 0.f, z1 = 0.f;
#pragma unroll
      for (int j = 0; j < 64; j += 2) {
        z0 += s[j];
        z1 += s[j + 1];
      }
      Z += z0 + z1;
    } else {
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int mg = m4[g];
        if ((mg & 31) == 0) continue;
        if (mg & PT_G_FIRST) {
          ++ci;
          zc = 0.f;
          ls = 0.f;
          nv = 0;
          cur_c = mg >> 8;
          // value mean of the cluster (thread r holds dim r < D), read now and
          // published at its end
          vc_pre = r < D ? a.vc[(static_cast<long long>(bh) * a.Ck + cur_c) * D + r] : 0.f;
        }
        float gs = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) gs += s[16 * g + i];
        zc += gs;
        ls += lsum[g];
        nv += mg & 31;
        if (mg & PT_G_LAST) {
          const int slot = ci & 1;
          if (ci >= 2) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait_bounded(smem_u32(&bars[PB_EE + slot]), ((ci - 2) >> 1) & 1,
                                              lim, abort_p));
            if (!ok) break;
          }
          // compensated weight n_c 2^(lbar sl2 - m2) of the centroid
          const float nf = static_cast<float>(nv);
          zc_s[slot][r] = zc;
          w_s[slot][r] = nf * ex2_approx(fmaf(ls / nf, sl2, -m2));
          vc_s[slot][r] = vc_pre;
          if (r == 0) cid_s[slot] = cur_c;
          mbar_arrive(smem_u32(&bars[PB_ZF + slot]));
        }
      }
      if (!ok) break;
    }
  }
  if constexpr (PASS == 2) {
    // sentinel after the last cluster: the residual warpgroup stops there
    if (ok) {
      const int cn = ci + 1, slot = cn & 1;
      if (cn >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars[PB_EE + slot]),
                                                        ((cn - 2) >> 1) & 1, lim, abort_p));
      if (ok) {
        if (r == 0) cid_s[slot] = -1;
        mbar_arrive(smem_u32(&bars[PB_ZF + slot]));
      }
    }
  }
  if constexpr (PASS == 1) {
    // split partial {m2, Z, O} of this row (O unnormalised); a split without
    // keys reports m2 = -inf, Z = 0
    float* out = a.part + ((static_cast<long long>(bh) * a.Cq + min(p, a.Cq - 1)) * a.NS + split) *
                              PtDim<D>::kRow;
    const bool mine = p < a.Cq;
    if (nt > 0 && ok)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars[PB_OD]), 0, lim, abort_p));
    if (nt > 0 && ok) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + PT_T_ACC + c * 32 + lane_off, v);
        tmem_wait_ld();
        if (mine) {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            *reinterpret_cast<float2*>(out + 2 + c * 32 + i) =
                make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
        }
      }
      if (mine) {
        out[0] = m2;
        out[1] = Z;
      }
    } else if (nt == 0 && mine) {
      out[0] = -INFINITY;
      out[1] = 0.f;
      for (int i = 0; i < D; i += 2) *reinterpret_cast<float2*>(out + 2 + i) = make_float2(0.f, 0.f);
    }
  }
}

// Residual warpgroup (pass 2): thread r owns proxy row r. The softmax
// publishes each finished cluster through a slot of shared memory (its id,
// Zc and w_c per row, and its value mean), then a sentinel id -1 after the
// last one.
template <int D>
__device__ __forceinline__ void pt_residual(const ProbeArgs& a, int bh, int pt, uint32_t tmem,
                                            uint64_t* bars, const float (*zc_s)[128],
                                            const float (*w_s)[128], const float (*vc_s)[128],
                                            const int* cid_s, volatile int* abort_p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;
  const int p = pt * 128 + r;
  const int pr = min(p, a.Cq - 1);
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const long long lim = a.wait_limit;
  const float* mz = a.mzo + (static_cast<long long>(bh) * a.Cq + pr) * PtDim<D>::kRow;
  const float invZ = 1.f / mz[1];
  float O[D];
#pragma unroll
  for (int i = 0; i < D; i += 2) {
    const float2 t = *reinterpret_cast<const float2*>(mz + 2 + i);
    O[i] = t.x;
    O[i + 1] = t.y;
  }
  const bool write = p < a.Cq && a.nq[static_cast<long long>(bh) * a.Cq + pr] > 0;
  float* errr = a.err + (static_cast<long long>(bh) * a.Cq + pr) * a.Ck;
  for (int ci = 0;; ++ci) {
    const int slot = ci & 1;
    const uint32_t ph = (ci >> 1) & 1;
    if (!__all_sync(0xffffffffu,
                    mbar_wait_bounded(smem_u32(&bars[PB_ZF + slot]), ph, lim, abort_p)))
      break;
    const int c = cid_s[slot];
    if (c < 0) break;  // sentinel: no more clusters
    if (!__all_sync(0xffffffffu,
                    mbar_wait_bounded(smem_u32(&bars[PB_EF + slot]), ph, lim, abort_p)))
      break;
    tc_fence_after();
    const float zc = zc_s[slot][r];
    const float w = w_s[slot][r];
    const float4* vc4 = reinterpret_cast<const float4*>(vc_s[slot]);
    const uint32_t tE = tmem + PT_T_ACC + slot * 128 + lane_off;
    // r = E_c - Zc O - w (vc - O) = (E_c + (w - Zc) O) - w vc, two packed
    // FMAs per pair of dims, and |r|^2 accumulated by a third.
    const float al = w - zc, nw = -w;
    float n2a = 0.f, n2b = 0.f;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
      uint32_t v[32];
      tmem_ld32(tE + q * 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 vv = vc4[(q * 32 + i) / 4];
        const int o = q * 32 + i;
        float t0, t1, t2, t3;
        ffma2_v(t0, t1, O[o], O[o + 1], al, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
        ffma2_v(t2, t3, O[o + 2], O[o + 3], al, __uint_as_float(v[i + 2]),
                __uint_as_float(v[i + 3]));
        ffma2_v(t0, t1, vv.x, vv.y, nw, t0, t1);
        ffma2_v(t2, t3, vv.z, vv.w, nw, t2, t3);
        fsq2_acc(n2a, n2b, t0, t1);
        fsq2_acc(n2a, n2b, t2, t3);
      }
    }
    tc_fence_before();
    mbar_arrive(smem_u32(&bars[PB_EE + slot]));
    if (write) errr[c] = sqrtf(n2a + n2b) * invZ;
  }
}

template <int PASS, int D>
__global__ void __launch_bounds__(PT_THREADS, 1)
    probe_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const ProbeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[PB_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ float zc_s[2][128];  // per E buffer: Zc and w_c of each proxy row,
  __shared__ float w_s[2][128];   // the cluster's value mean and its id
  __shared__ __align__(16) float vc_s[2][128];
  __shared__ int cid_s[2];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  using Pd = PtDim<D>;
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + 3 * Pd::kQP;
  const uint32_t sV0 = sK0 + PT_NK * Pd::kKV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, pt = blockIdx.y, bh = blockIdx.z;
  const int* kp = a.kpoff + static_cast<long long>(bh) * (a.Ck + 1);
  const int c_lo = pt_split_cluster(kp, a.Ck, split, a.NS);
  const int c_hi = pt_split_cluster(kp, a.Ck, split + 1, a.NS);
  const int g_lo = kp[c_lo] >> 4, g_hi = kp[c_hi] >> 4;
  const int nt = (g_hi - g_lo + 3) >> 2;
  const int nval0 = PASS == 1 ? nt : 0;
  const int ne = nval0 + nt;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar(PB_Q), 1);
    for (int s = 0; s < PT_NK; ++s) {
      mbar_init(bar(PB_KF + s), 1);
      mbar_init(bar(PB_KE + s), 1);
    }
    for (int s = 0; s < PT_NV; ++s) {
      mbar_init(bar(PB_VF + s), 1);
      mbar_init(bar(PB_VE + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(PB_SF + b), 1);
      mbar_init(bar(PB_PF + b), 128);
      mbar_init(bar(PB_EF + b), 1);
      mbar_init(bar(PB_ZF + b), 128);
      mbar_init(bar(PB_EE + b), 128);
    }
    mbar_init(bar(PB_OD), 1);
    mbar_init(bar(PB_DRAIN), 1);
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PT_REGS_INC));
    if (warp < 8) {
      pt_softmax<PASS, D>(a, bh, pt, split, g_lo, g_hi, nt, tmem, bars, zc_s, w_s, vc_s, cid_s,
                          abort_p);
    } else if constexpr (PASS == 2) {
      pt_residual<D>(a, bh, pt, tmem, bars, zc_s, w_s, vc_s, cid_s, abort_p);
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PT_REGS_DEC));
  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && ne > 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(bar(PB_Q), 3 * Pd::kQP);
      for (int i = 0; i < 3; ++i)
        for (int h = 0; h < Pd::kHalves; ++h)
          tma_load_3d(sQ + i * Pd::kQP + h * PT_QP_HALF, &map_q, bar(PB_Q), 64 * h,
                      i * a.Cqp + pt * 128, bh);
      const int row0 = 16 * g_lo;
      int issued_k = 0, issued_v = 0;
      for (int u = 0; u < ne; ++u) {
        const int t = u >= nval0 ? u - nval0 : u;
        const int sk = u % PT_NK;
        if (u >= PT_NK &&
            !mbar_wait_bounded(bar(PB_KE + sk), ((u / PT_NK) & 1) ^ 1, lim, abort_p))
          break;
        mbar_arrive_expect_tx(bar(PB_KF + sk), Pd::kKV);
        for (int h = 0; h < Pd::kHalves; ++h)
          tma_load_3d(sK0 + sk * Pd::kKV + h * PT_KV_HALF, &map_k, bar(PB_KF + sk), 64 * h,
                      row0 + PT_KT * t, bh);
        issued_k = u + 1;
        if (u >= nval0) {
          const int vu = u - nval0, sv = vu % PT_NV;
          if (vu >= PT_NV &&
              !mbar_wait_bounded(bar(PB_VE + sv), ((vu / PT_NV) & 1) ^ 1, lim, abort_p))
            break;
          mbar_arrive_expect_tx(bar(PB_VF + sv), Pd::kKV);
          for (int h = 0; h < Pd::kHalves; ++h)
            tma_load_3d(sV0 + sv * Pd::kKV + h * PT_KV_HALF, &map_v, bar(PB_VF + sv), 64 * h,
                        row0 + PT_KT * t, bh);
          issued_v = vu + 1;
        }
      }
      if (*abort_p) {
        // Drain: only the last NK (NV) loads of a ring can still be in flight.
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(PB_Q), 0, lim, &no_abort);
        for (int u = issued_k > PT_NK ? issued_k - PT_NK : 0; u < issued_k; ++u) {
          no_abort = 0;
          mbar_wait_bounded(bar(PB_KF + u % PT_NK), (u / PT_NK) & 1, lim, &no_abort);
        }
        for (int u = issued_v > PT_NV ? issued_v - PT_NV : 0; u < issued_v; ++u) {
          no_abort = 0;
          mbar_wait_bounded(bar(PB_VF + u % PT_NV), (u / PT_NV) & 1, lim, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0 && ne > 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(128, PT_KT, 0, 0);
      constexpr uint32_t id_pv = idesc_bf16_f32(128, D, 0, 1);
      const int* gm = a.gmeta + static_cast<long long>(bh) * a.G;
      bool ok = mbar_wait_bounded(bar(PB_Q), 0, lim, abort_p);
      int ci = -1;
      // P_u V_u once the softmax of entry u released its TMEM stage.
      auto issue_pv = [&](int u, const int (&m4)[4]) -> bool {
        const int b = u & 1;
        if (!mbar_wait_bounded(bar(PB_PF + b), (u >> 1) & 1, lim, abort_p)) return false;
        if (u < nval0) return true;
        const int vu = u - nval0, sv = vu % PT_NV;
        if (!mbar_wait_bounded(bar(PB_VF + sv), (vu / PT_NV) & 1, lim, abort_p)) return false;
        tc_fence_after();
        const uint32_t tP = tmem + b * PT_STAGE_COLS;
        const uint32_t sV = sV0 + sv * Pd::kKV;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int mg = m4[g];
          if ((mg & 31) == 0) continue;
          const uint64_t bd = sw128_desc(sV + g * 2048, PT_KV_HALF, 1024);
          uint32_t dst = tmem + PT_T_ACC;
          bool first;
          if constexpr (PASS == 1) {
            first = vu == 0 && g == 0;
          } else {
            first = (mg & PT_G_FIRST) != 0;
            if (first) {
              ++ci;
              if (ci >= 2) {
                if (!mbar_wait_bounded(bar(PB_EE + (ci & 1)), ((ci - 2) >> 1) & 1, lim, abort_p))
                  return false;
                tc_fence_after();
              }
            }
            dst += (ci & 1) * 128;
          }
#pragma unroll
          for (int i = 0; i < 3; ++i)
            umma_ts(dst, tP + i * 32 + g * 8, bd, id_pv, (first && i == 0) ? 0u : 1u);
          if constexpr (PASS == 2) {
            if (mg & PT_G_LAST) umma_commit(bar(PB_EF + (ci & 1)));
          }
        }
        umma_commit(bar(PB_VE + sv));
        return true;
      };
      int mcur[4] = {0, 0, 0, 0}, mnext[4];
      for (int u = 0; ok && u < ne; ++u) {
        const int t = u >= nval0 ? u - nval0 : u;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int gg = g_lo + 4 * t + g;
          mnext[g] = gg < g_hi ? gm[gg] : 0;
        }
        const int sk = u % PT_NK, b = u & 1;
        if (!(ok = mbar_wait_bounded(bar(PB_KF + sk), (u / PT_NK) & 1, lim, abort_p))) break;
        tc_fence_after();
        const uint32_t sK = sK0 + sk * Pd::kKV;
#pragma unroll
        for (int i = 0; i < 3; ++i)
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            umma_ss(tmem + b * PT_STAGE_COLS + (i > 0 ? 64 : 0),
                    sw128_desc(sQ + i * Pd::kQP + (k >> 2) * PT_QP_HALF + (k & 3) * 32, 16, 1024),
                    sw128_desc(sK + (k >> 2) * PT_KV_HALF + (k & 3) * 32, 16, 1024), id_qk,
                    (i == 2 || k > 0) ? 1u : 0u);
        umma_commit(bar(PB_SF + b));
        umma_commit(bar(PB_KE + sk));
        if (u >= 1 && !(ok = issue_pv(u - 1, mcur))) break;
#pragma unroll
        for (int g = 0; g < 4; ++g) mcur[g] = mnext[g];
      }
      if (ok) ok = issue_pv(ne - 1, mcur);
      if (ok && PASS == 1) umma_commit(bar(PB_OD));
      if (!ok) {
        umma_commit(bar(PB_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_bounded(bar(PB_DRAIN), 0, lim, &no_abort);
      }
    }
  }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// mzo[bh][p] = {m2, Z, O / Z} from the NS split partials. Grid (Cq, BH), D
// threads (one per dim).
template <int D>
__global__ void probe_tc_combine_kernel(const float* __restrict__ part, int Cq, int NS,
                                        float* __restrict__ mzo) {
  constexpr int kRow = PtDim<D>::kRow;
  const int bh = blockIdx.y, p = blockIdx.x, d = threadIdx.x;
  const float* pp = part + (static_cast<long long>(bh) * Cq + p) * NS * kRow;
  float m = -INFINITY;
  for (int s = 0; s < NS; ++s) m = fmaxf(m, pp[s * kRow]);
  float Z = 0.f, O = 0.f;
  for (int s = 0; s < NS; ++s) {
    const float ms = pp[s * kRow];
    if (ms == -INFINITY) continue;
    const float wgt = exp2f(ms - m);
    Z = fmaf(pp[s * kRow + 1], wgt, Z);
    O = fmaf(pp[s * kRow + 2 + d], wgt, O);
  }
  float* out = mzo + (static_cast<long long>(bh) * Cq + p) * kRow;
  if (d == 0) {
    out[0] = m;
    out[1] = Z;
  }
  out[2 + d] = O / Z;
}

// ------------------------------------------------------------------ prep --

// cnt16[bh][c] = n_c rounded up to a multiple of 16.
__global__ void pad16_count_kernel(const int* __restrict__ nk, int n, int* __restrict__ cnt16) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) cnt16[i] = (nk[i] + 15) & ~15;
}

// Padded cluster-ordered copies of K and V ([BH][Npad][D]) and the group
// metadata; block (c, bh) copies cluster c (its members, then zero rows up to
// a multiple of 16); block (Ck, bh) zeroes the 64 rows after the last cluster,
// which a tile may read past its split. 128 threads, one warp per row (D / 32
// values per lane).
template <int D>
__global__ void pad_gather_kernel(const __nv_bfloat16* __restrict__ k,
                                  const __nv_bfloat16* __restrict__ v, int N, int Ck,
                                  const int* __restrict__ nk, const int* __restrict__ koff,
                                  const int* __restrict__ kperm, const int* __restrict__ kpoff,
                                  long long Npad, int G, __nv_bfloat16* __restrict__ kpad,
                                  __nv_bfloat16* __restrict__ vpad, int* __restrict__ gmeta) {
  const int c = blockIdx.x, bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* kp = kpoff + static_cast<long long>(bh) * (Ck + 1);
  const long long base = static_cast<long long>(bh) * Npad + kp[c];
  int n = 0, rows = 64;
  if (c < Ck) {
    n = nk[static_cast<long long>(bh) * Ck + c];
    rows = (n + 15) & ~15;
  }
  const int src0 = c < Ck ? koff[static_cast<long long>(bh) * (Ck + 1) + c] : 0;
  for (int row = warp; row < rows; row += 4) {
    const int j = row < n ? kperm[static_cast<long long>(bh) * N + src0 + row] : -1;
    using W = typename std::conditional<D == 128, uint2, uint32_t>::type;  // D / 32 bf16
    W kv{}, vv{};
    if (j >= 0) {
      const long long src = (static_cast<long long>(bh) * N + j) * D + lane * (D / 32);
      kv = *reinterpret_cast<const W*>(k + src);
      vv = *reinterpret_cast<const W*>(v + src);
    }
    const long long dst = (base + row) * D + lane * (D / 32);
    *reinterpret_cast<W*>(kpad + dst) = kv;
    *reinterpret_cast<W*>(vpad + dst) = vv;
  }
  if (c < Ck) {
    const int ng = rows >> 4;
    for (int g = threadIdx.x; g < ng; g += blockDim.x) {
      const int valid = min(16, n - 16 * g);
      gmeta[static_cast<long long>(bh) * G + (kp[c] >> 4) + g] =
          valid | (g == 0 ? PT_G_FIRST : 0) | (g == ng - 1 ? PT_G_LAST : 0) | (c << 8);
    }
  }
}

// Three bf16 pieces of the proxies: qp[bh][i][p][d], p < Cqp (rows >= Cq
// zero). Grid (Cqp, BH), D threads.
template <int D>
__global__ void proxy_pieces_kernel(const float* __restrict__ qc, int Cq, int Cqp,
                                    __nv_bfloat16* __restrict__ qp) {
  const int p = blockIdx.x, bh = blockIdx.y, d = threadIdx.x;
  const float x = p < Cq ? qc[(static_cast<long long>(bh) * Cq + p) * D + d] : 0.f;
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  const long long o = (static_cast<long long>(bh) * 3 * Cqp + p) * D + d;
  const long long piece = static_cast<long long>(Cqp) * D;
  qp[o] = hi;
  qp[o + piece] = mid;
  qp[o + 2 * piece] = lo;
}

}  // namespace va
