// SVG-EAR compensated sparse attention with error-aware routing (SVG-EAR,
// gist.science 2603.08982, technical summary sec. 2):
//   idea 1  parameter-free linear compensation: a skipped (query cluster p,
//           key cluster c) block contributes through the cluster centroids,
//           a virtual key kc_c with logit bias ln n_c and value vc_c;
//   idea 2  error-aware routing: a light probe with the query-cluster
//           centroid as proxy (O(C_q N_k d) instead of O(N_q N_k d)),
//           streamed without storing logits, estimates each block's
//           compensation error; under a density budget the blocks with the
//           highest error-to-cost ratio are computed exactly.
// The page gives no formulas; the readings implemented here are
//   probe    l_j = s qc_p . k_j, m_p = max_j l_j, e_j = exp(l_j - m_p),
//            Z_p = sum_j e_j, O_p = sum_j e_j v_j / Z_p,
//            r(p, c) = sum_{j in c} e_j (v_j - O_p) - w_c (vc_c - O_p),
//            w_c = n_c exp(s qc_p . kc_c - m_p), err(p, c) = |r(p, c)| / Z_p
//            (= |dE - O_p dZ| / Z_p, the first-order change of the proxy's
//            normalised output when the block is compensated);
//   routing  ratio = err / n_c (fp32), ordered by ratio descending, then p,
//            then c; the longest prefix whose summed cost n_p n_c is at most
//            floor(density N^2) is computed exactly; empty clusters never;
//   output   one softmax per query over the exact keys of its cluster's
//            selected key clusters and the virtual keys of every other
//            non-empty key cluster.
#pragma once

#include "kmeans.cuh"

namespace va {

// ------------------------------------------------------------------ probe --
//
// Pass 1 splits the keys of every proxy over PR_SPLIT CTAs (partial max, sum
// and unnormalised value sum, merged by probe_combine_kernel); pass 2 splits
// the key clusters over PR_CSPLIT CTAs (a cluster's residual only needs the
// merged m_p, Z_p, O_p and its own keys). A CTA holds PR_PG = 32 proxies; warp
// w owns proxies 4w..4w+3: each lane computes their logits for keys 2 lane,
// 2 lane + 1 of a 64-key tile, and their value sums for the DV = d / 32 dims
// DV lane.. (register tiles of 4 x 2 and 4 x DV, shared-memory operands read
// as vectors).

constexpr int PR_PG = 32;  // query clusters (proxies) per CTA
constexpr int PR_KT = 64;  // keys per tile
constexpr int PR_THREADS = 256;
constexpr int PR_SPLIT = 8;    // key splits of pass 1
constexpr int PR_CSPLIT = 8;   // key-cluster splits of pass 2
// Row stride (floats) of the per-key weight tile es[key][proxy]: 36 keeps the
// float4 rows of consecutive keys on different bank groups.
constexpr int PR_ES_LD = PR_PG + 4;
constexpr int PR_NO_KEY = 0x7fffffff;  // tile slot past the range's last key

template <int D>
constexpr int probe_smem_bytes(int Ck) {
  return (D * PR_PG + D * PR_KT + PR_KT * D + PR_KT * PR_ES_LD) * 4 + 2 * PR_KT * 4 + (Ck + 1) * 4;
}

// acc[a][b] = qc_{4w+a} . k_{2 lane + b}
template <int D>
__device__ __forceinline__ void probe_logits(const float* qcT, const float* kT, int w, int lane,
                                             float (&acc)[4][2]) {
#pragma unroll
  for (int a = 0; a < 4; ++a) acc[a][0] = acc[a][1] = 0.f;
#pragma unroll 8
  for (int dd = 0; dd < D; ++dd) {
    const float4 qv = *reinterpret_cast<const float4*>(&qcT[dd * PR_PG + 4 * w]);
    const float2 kv = *reinterpret_cast<const float2*>(&kT[dd * PR_KT + 2 * lane]);
    const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      acc[a][0] = fmaf(qa[a], kv.x, acc[a][0]);
      acc[a][1] = fmaf(qa[a], kv.y, acc[a][1]);
    }
  }
}

// out[e] = src[e], e < DV, as one vector load (src aligned to DV floats).
template <int DV>
__device__ __forceinline__ void load_vec(const float* src, float (&out)[DV]) {
  if constexpr (DV == 4) {
    const float4 t = *reinterpret_cast<const float4*>(src);
    out[0] = t.x;
    out[1] = t.y;
    out[2] = t.z;
    out[3] = t.w;
  } else if constexpr (DV == 2) {
    const float2 t = *reinterpret_cast<const float2*>(src);
    out[0] = t.x;
    out[1] = t.y;
  } else {
#pragma unroll
    for (int e = 0; e < DV; ++e) out[e] = src[e];
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// part[bh][p][split] = {m, Z, O[0..D)} over keys of this split (O unnormalised).
// Grid (ceil(Cq / PR_PG), PR_SPLIT, BH).
template <typename T, int D>
__global__ void __launch_bounds__(PR_THREADS)
    probe_pass1_kernel(const T* __restrict__ k, const T* __restrict__ v, int N, int Cq,
                       const float* __restrict__ qc, float scale, float* __restrict__ part) {
  static_assert(D == 64 || D == 128, "the probe tiles assume d = 64 or 128");
  constexpr int DV = D / 32;
  extern __shared__ float pr_smem[];
  float* qcT = pr_smem;                       // [D][PR_PG]
  float* kT = qcT + D * PR_PG;                // [D][PR_KT]
  float* vs = kT + D * PR_KT;                 // [PR_KT][D]
  float* es = vs + PR_KT * D;                 // [PR_KT][PR_ES_LD]
  const int bh = blockIdx.z, split = blockIdx.y;
  const int p0 = blockIdx.x * PR_PG;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const long long kvb = static_cast<long long>(bh) * N * D;
  const int per = ((N + PR_SPLIT - 1) / PR_SPLIT + PR_KT - 1) / PR_KT * PR_KT;
  const int jb = split * per, je = min(N, jb + per);
  stage_transposed<float, D, PR_PG, PR_THREADS>(qcT, [&](int pp) -> const float* {
    return p0 + pp < Cq ? qc + (static_cast<long long>(bh) * Cq + p0 + pp) * D : nullptr;
  });
  float m[4], Z[4], O[4][DV];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -INFINITY;
    Z[a] = 0.f;
#pragma unroll
    for (int e = 0; e < DV; ++e) O[a][e] = 0.f;
  }
  for (int j0 = jb; j0 < je; j0 += PR_KT) {
    __syncthreads();
    stage_transposed<T, D, PR_KT, PR_THREADS>(kT, [&](int kk) -> const T* {
      return j0 + kk < je ? k + kvb + static_cast<long long>(j0 + kk) * D : nullptr;
    });
    stage_rows<T, D, PR_KT, PR_THREADS>(vs, [&](int kk) -> const T* {
      return j0 + kk < je ? v + kvb + static_cast<long long>(j0 + kk) * D : nullptr;
    });
    __syncthreads();
    float acc[4][2];
    probe_logits<D>(qcT, kT, w, lane, acc);
    const bool v0 = j0 + 2 * lane < je, v1 = j0 + 2 * lane + 1 < je;
    float e0[4], e1[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float l0 = v0 ? acc[a][0] * scale : -INFINITY;
      const float l1 = v1 ? acc[a][1] * scale : -INFINITY;
      const float mn = fmaxf(m[a], warp_max(fmaxf(l0, l1)));
      const float alpha = expf(m[a] - mn);  // m = -inf on the first tile: alpha = 0
      m[a] = mn;
      e0[a] = expf(l0 - mn);
      e1[a] = expf(l1 - mn);
      Z[a] = Z[a] * alpha + warp_sum(e0[a] + e1[a]);
#pragma unroll
      for (int e = 0; e < DV; ++e) O[a][e] *= alpha;
    }
    *reinterpret_cast<float4*>(&es[(2 * lane) * PR_ES_LD + 4 * w]) =
        make_float4(e0[0], e0[1], e0[2], e0[3]);
    *reinterpret_cast<float4*>(&es[(2 * lane + 1) * PR_ES_LD + 4 * w]) =
        make_float4(e1[0], e1[1], e1[2], e1[3]);
    __syncwarp();
#pragma unroll 4
    for (int kk = 0; kk < PR_KT; ++kk) {
      const float4 ev = *reinterpret_cast<const float4*>(&es[kk * PR_ES_LD + 4 * w]);
      const float ea[4] = {ev.x, ev.y, ev.z, ev.w};
      float va4[DV];
      load_vec<DV>(&vs[kk * D + DV * lane], va4);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < DV; ++e) O[a][e] = fmaf(ea[a], va4[e], O[a][e]);
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int p = p0 + 4 * w + a;
    if (p < Cq) {
      float* out = part + ((static_cast<long long>(bh) * Cq + p) * PR_SPLIT + split) * (D + 2);
      if (lane == 0) {
        out[0] = m[a];
        out[1] = Z[a];
      }
      float* o4 = out + 2 + DV * lane;
#pragma unroll
      for (int e = 0; e < DV; ++e) o4[e] = O[a][e];
    }
  }
}

// mzo[bh][p] = {m_p, Z_p, O_p[0..D)} (O_p normalised) from the split partials.
// Grid (Cq, BH), D threads.
template <int D>
__global__ void probe_combine_kernel(const float* __restrict__ part, int Cq,
                                     float* __restrict__ mzo) {
  const int bh = blockIdx.y, p = blockIdx.x, d = threadIdx.x;
  const float* pp = part + (static_cast<long long>(bh) * Cq + p) * PR_SPLIT * (D + 2);
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < PR_SPLIT; ++s) m = fmaxf(m, pp[s * (D + 2)]);
  float Z = 0.f, O = 0.f;
#pragma unroll
  for (int s = 0; s < PR_SPLIT; ++s) {
    const float ms = pp[s * (D + 2)];
    if (ms == -INFINITY) continue;
    const float wgt = expf(ms - m);
    Z = fmaf(pp[s * (D + 2) + 1], wgt, Z);
    O = fmaf(pp[s * (D + 2) + 2 + d], wgt, O);
  }
  float* out = mzo + (static_cast<long long>(bh) * Cq + p) * (D + 2);
  if (d == 0) {
    out[0] = m;
    out[1] = Z;
  }
  out[2 + d] = O / Z;
}

// err[bh][p][c] for non-empty p and the clusters c of this CTA's cluster range
// (keys in cluster order). Grid (ceil(Cq / PR_PG), PR_CSPLIT, BH).
template <typename T, int D>
__global__ void __launch_bounds__(PR_THREADS)
    probe_pass2_kernel(const T* __restrict__ k, const T* __restrict__ v, int N, int Cq, int Ck,
                       const float* __restrict__ qc, const int* __restrict__ nq,
                       const float* __restrict__ kc, const float* __restrict__ vc,
                       const int* __restrict__ nk, const int* __restrict__ koff,
                       const int* __restrict__ kperm, const int* __restrict__ kassign,
                       const float* __restrict__ mzo, float scale, float* __restrict__ err) {
  static_assert(D == 64 || D == 128, "the probe tiles assume d = 64 or 128");
  constexpr int DV = D / 32;
  extern __shared__ float pr_smem[];
  float* qcT = pr_smem;                       // [D][PR_PG]
  float* kT = qcT + D * PR_PG;                // [D][PR_KT]
  float* vs = kT + D * PR_KT;                 // [PR_KT][D]
  float* es = vs + PR_KT * D;                 // [PR_KT][PR_ES_LD]
  int* cid = reinterpret_cast<int*>(es + PR_KT * PR_ES_LD);  // [PR_KT]: cluster, or
                                              // -1 - cluster for its last key
  int* kidx = cid + PR_KT;                    // [PR_KT]
  int* offs = kidx + PR_KT;                   // [Ck + 1] (this range's part)

  const int bh = blockIdx.z, split = blockIdx.y;
  const int p0 = blockIdx.x * PR_PG;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const long long kvb = static_cast<long long>(bh) * N * D;
  const int* ko = koff + static_cast<long long>(bh) * (Ck + 1);
  const int* kp = kperm + static_cast<long long>(bh) * N;
  const int* ka = kassign + static_cast<long long>(bh) * N;
  const int cper = (Ck + PR_CSPLIT - 1) / PR_CSPLIT;
  const int c_lo = min(Ck, split * cper), c_hi = min(Ck, c_lo + cper);
  const int tb = ko[c_lo], te = ko[c_hi];

  stage_transposed<float, D, PR_PG, PR_THREADS>(qcT, [&](int pp) -> const float* {
    return p0 + pp < Cq ? qc + (static_cast<long long>(bh) * Cq + p0 + pp) * D : nullptr;
  });
  for (int e = tid; e <= c_hi - c_lo; e += PR_THREADS) offs[e] = ko[c_lo + e];
  // Per cluster: E = sum e_j v_j and Zc = sum e_j over its keys; at its last
  // key r = E - Zc O - w (vc - O) (the same residual, one subtraction per
  // cluster instead of per key).
  float m[4], invZ[4], O[4][DV], r[4][DV], zc[4];
  bool write[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int p = p0 + 4 * w + a;
    const int pr = min(p, Cq - 1);
    const float* mz = mzo + (static_cast<long long>(bh) * Cq + pr) * (D + 2);
    m[a] = mz[0];
    invZ[a] = 1.f / mz[1];
#pragma unroll
    for (int e = 0; e < DV; ++e) {
      O[a][e] = mz[2 + DV * lane + e];
      r[a][e] = 0.f;
    }
    zc[a] = 0.f;
    write[a] = p < Cq && nq[static_cast<long long>(bh) * Cq + pr] > 0;
  }
  for (int t0 = tb; t0 < te; t0 += PR_KT) {
    __syncthreads();
    for (int kk = tid; kk < PR_KT; kk += PR_THREADS) {
      const int j = (t0 + kk < te) ? kp[t0 + kk] : -1;
      kidx[kk] = j;
      int c = PR_NO_KEY;
      if (j >= 0) {
        c = ka[j];
        if (t0 + kk == offs[c - c_lo + 1] - 1) c = -1 - c;  // last key of cluster c
      }
      cid[kk] = c;
    }
    __syncthreads();
    stage_transposed<T, D, PR_KT, PR_THREADS>(kT, [&](int kk) -> const T* {
      return kidx[kk] >= 0 ? k + kvb + static_cast<long long>(kidx[kk]) * D : nullptr;
    });
    stage_rows<T, D, PR_KT, PR_THREADS>(vs, [&](int kk) -> const T* {
      return kidx[kk] >= 0 ? v + kvb + static_cast<long long>(kidx[kk]) * D : nullptr;
    });
    __syncthreads();
    float acc[4][2];
    probe_logits<D>(qcT, kT, w, lane, acc);
    const bool v0 = t0 + 2 * lane < te, v1 = t0 + 2 * lane + 1 < te;
    float e0[4], e1[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      e0[a] = v0 ? expf(fmaf(acc[a][0], scale, -m[a])) : 0.f;
      e1[a] = v1 ? expf(fmaf(acc[a][1], scale, -m[a])) : 0.f;
    }
    *reinterpret_cast<float4*>(&es[(2 * lane) * PR_ES_LD + 4 * w]) =
        make_float4(e0[0], e0[1], e0[2], e0[3]);
    *reinterpret_cast<float4*>(&es[(2 * lane + 1) * PR_ES_LD + 4 * w]) =
        make_float4(e1[0], e1[1], e1[2], e1[3]);
    __syncwarp();
    for (int kk = 0; kk < PR_KT; ++kk) {
      const int cc = cid[kk];
      if (cc == PR_NO_KEY) break;
      const float4 ev = *reinterpret_cast<const float4*>(&es[kk * PR_ES_LD + 4 * w]);
      const float ea[4] = {ev.x, ev.y, ev.z, ev.w};
      float va4[DV];
      load_vec<DV>(&vs[kk * D + DV * lane], va4);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        zc[a] += ea[a];
#pragma unroll
        for (int e = 0; e < DV; ++e) r[a][e] = fmaf(ea[a], va4[e], r[a][e]);
      }
      if (cc < 0) {
        const int c = -1 - cc;
        // last key of cluster c: subtract Zc O and the compensated term, then |r| / Z
        const float* kcc = kc + (static_cast<long long>(bh) * Ck + c) * D + DV * lane;
        const float* vcc = vc + (static_cast<long long>(bh) * Ck + c) * D + DV * lane;
        float kca[DV], vca[DV];
#pragma unroll
        for (int e = 0; e < DV; ++e) {
          kca[e] = kcc[e];
          vca[e] = vcc[e];
        }
        const float ncf = static_cast<float>(nk[static_cast<long long>(bh) * Ck + c]);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < DV; ++e) dot = fmaf(qcT[(DV * lane + e) * PR_PG + 4 * w + a], kca[e], dot);
          dot = warp_sum(dot);
          const float wc = ncf * expf(fmaf(dot, scale, -m[a]));
          float n2 = 0.f;
#pragma unroll
          for (int e = 0; e < DV; ++e) {
            const float re = fmaf(-wc, vca[e] - O[a][e], fmaf(-zc[a], O[a][e], r[a][e]));
            n2 = fmaf(re, re, n2);
            r[a][e] = 0.f;
          }
          zc[a] = 0.f;
          n2 = warp_sum(n2);
          if (write[a] && lane == 0)
            err[(static_cast<long long>(bh) * Cq + p0 + 4 * w + a) * Ck + c] = sqrtf(n2) * invZ[a];
        }
      }
    }
  }
}

// ---------------------------------------------------------------- routing --

__device__ __forceinline__ unsigned long long route_key(float ratio, int p, int c, int Ck) {
  // ascending key order = ratio descending (non-negative floats order like
  // their bit patterns), then p ascending, then c ascending
  const uint32_t hi = 0xFFFFFFFFu - __float_as_uint(ratio);
  return (static_cast<unsigned long long>(hi) << 32) |
         static_cast<unsigned long long>(p * Ck + c);
}

// Sort keys and costs of every (p, c) block: key = route_key(err / n_c, p, c)
// and cost n_p n_c, or (~0, 0) for a block with an empty cluster.
// Grid (ceil(Cq * Ck / 256), BH).
__global__ void route_keys_kernel(const float* __restrict__ err, const int* __restrict__ nq,
                                  const int* __restrict__ nk, int Cq, int Ck,
                                  unsigned long long* __restrict__ keys,
                                  unsigned long long* __restrict__ costs) {
  const int bh = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= Cq * Ck) return;
  const int p = e / Ck, c = e - p * Ck;
  const int np = nq[static_cast<long long>(bh) * Cq + p];
  const int nc = nk[static_cast<long long>(bh) * Ck + c];
  const long long i = static_cast<long long>(bh) * Cq * Ck + e;
  if (np <= 0 || nc <= 0) {
    keys[i] = ~0ull;
    costs[i] = 0;
    return;
  }
  const float ratio = __fdiv_rn(err[i], static_cast<float>(nc));
  keys[i] = route_key(ratio, p, c, Ck);
  costs[i] = static_cast<unsigned long long>(np) * static_cast<unsigned long long>(nc);
}


// Weighted MSB-first radix select, 8 bits per pass, spread over many CTAs:
// per bh, the smallest key K whose prefix (all keys <= K) costs more than the
// budget; blocks with key < K are computed exactly, cut[bh] = ~0 when every
// valid block fits. State per bh: {prefix, mask, remaining budget, done}.
// Each pass: every CTA adds the costs of its slice's keys that match the
// prefix into a per-bh global histogram of the next 8 bits (64-bit integer
// sums, so the result does not depend on the order); the last CTA to finish
// scans the histogram, extends the prefix and clears the histogram.
constexpr int RS_THREADS = 256;
constexpr int RS_PER_CTA = 4096;  // keys per CTA and pass

// state[bh] = {0, 0, budget, 0}; hist and the CTA counters zeroed.
__global__ void route_init_kernel(long long budget, int BH, unsigned long long* __restrict__ state,
                                  unsigned long long* __restrict__ hist,
                                  unsigned int* __restrict__ counter) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < BH * 256) hist[i] = 0;
  if (i < BH) {
    state[4 * i + 0] = 0;
    state[4 * i + 1] = 0;
    state[4 * i + 2] = static_cast<unsigned long long>(budget);
    state[4 * i + 3] = 0;
    counter[i] = 0;
  }
}

// One pass at bit offset `shift`. Grid (ceil(total / RS_PER_CTA), BH), RS_THREADS.
__global__ void __launch_bounds__(RS_THREADS)
    route_pass_kernel(const unsigned long long* __restrict__ keys,
                      const unsigned long long* __restrict__ costs, int total, int shift,
                      unsigned long long* __restrict__ state, unsigned long long* __restrict__ hist,
                      unsigned int* __restrict__ counter) {
  __shared__ unsigned long long h[256];
  __shared__ int s_last;
  const int bh = blockIdx.y, tid = threadIdx.x;
  unsigned long long* st = state + 4 * bh;
  if (st[3]) return;  // uniform: every key already fits
  const unsigned long long prefix = st[0], mask = st[1];
  h[tid] = 0;
  __syncthreads();
  const unsigned long long* kb = keys + static_cast<long long>(bh) * total;
  const unsigned long long* cb = costs + static_cast<long long>(bh) * total;
  const int e0 = blockIdx.x * RS_PER_CTA, e1 = min(total, e0 + RS_PER_CTA);
  for (int e = e0 + tid; e < e1; e += RS_THREADS) {
    const unsigned long long key = kb[e];
    const unsigned long long cost = cb[e];
    if (cost == 0 || (key & mask) != prefix) continue;
    atomicAdd(&h[(key >> shift) & 255u], cost);
  }
  __syncthreads();
  unsigned long long* gh = hist + 256 * static_cast<long long>(bh);
  if (h[tid] != 0) atomicAdd(&gh[tid], h[tid]);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&counter[bh], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last CTA of this bh: read the complete histogram, extend the prefix
  h[tid] = atomicExch(&gh[tid], 0ull);
  __syncthreads();
  if (tid == 0) {
    long long remaining = static_cast<long long>(st[2]);
    long long cum = 0;
    int b = 0;
    for (; b < 256; ++b) {
      const long long hb = static_cast<long long>(h[b]);
      if (cum + hb > remaining) break;
      cum += hb;
    }
    if (b == 256) {
      // everything under this prefix fits (only possible on the first pass:
      // the whole set fits the budget)
      st[0] = ~0ull;
      st[3] = 1;
    } else {
      st[2] = static_cast<unsigned long long>(remaining - cum);
      st[0] = prefix | (static_cast<unsigned long long>(b) << shift);
      st[1] = mask | (255ull << shift);
    }
    counter[bh] = 0;
  }
}

// cut[bh] = state prefix after the last pass.
__global__ void route_cut_kernel(const unsigned long long* __restrict__ state, int BH,
                                 unsigned long long* __restrict__ cut) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < BH) cut[i] = state[4 * i];
}

// sel[bh][p][c] = 1 for exactly computed blocks (if sel != nullptr) and the
// ascending list of selected c per p: selc[bh][p][0..seln[bh][p]).
// Grid (Cq, BH), 256 threads.
__global__ void route_mark_kernel(const float* __restrict__ err, const int* __restrict__ nq,
                                  const int* __restrict__ nk, int Cq, int Ck,
                                  const unsigned long long* __restrict__ cut,
                                  uint8_t* __restrict__ sel, int* __restrict__ seln,
                                  int* __restrict__ selc) {
  __shared__ int warp_tot[8];
  __shared__ int base_s;
  const int bh = blockIdx.y, p = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned long long K = cut[bh];
  const int np = nq[static_cast<long long>(bh) * Cq + p];
  const float* eb = err + (static_cast<long long>(bh) * Cq + p) * Ck;
  const int* nkb = nk + static_cast<long long>(bh) * Ck;
  int* list = selc + (static_cast<long long>(bh) * Cq + p) * Ck;
  if (tid == 0) base_s = 0;
  __syncthreads();
  for (int c0 = 0; c0 < Ck; c0 += 256) {
    const int c = c0 + tid;
    bool s = false;
    if (c < Ck) {
      const int nc = nkb[c];
      if (np > 0 && nc > 0) {
        const float ratio = __fdiv_rn(eb[c], static_cast<float>(nc));
        s = route_key(ratio, p, c, Ck) < K;
      }
      if (sel != nullptr) sel[(static_cast<long long>(bh) * Cq + p) * Ck + c] = s ? 1 : 0;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, s);
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int before = base_s;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    if (s) list[before + __popc(bal & ((1u << lane) - 1u))] = c;
    __syncthreads();
    if (tid == 0) {
      int t = 0;
      for (int w = 0; w < 8; ++w) t += warp_tot[w];
      base_s += t;
    }
    __syncthreads();
  }
  if (tid == 0) seln[static_cast<long long>(bh) * Cq + p] = base_s;
}

// ----------------------------------------------------- compensated output --

constexpr int CA_QT = 64;  // queries per CTA (one query cluster)
constexpr int CA_KT = 64;  // keys per tile
constexpr int CA_THREADS = 256;

template <int D>
constexpr int comp_smem_bytes(int Ck) {
  return (D * CA_QT + D * CA_KT + CA_KT * D + CA_QT * CA_KT + CA_KT) * 4 + CA_QT * 4 +
         CA_KT * 4 + (Ck + 1) * 4 + Ck * 4 + ((Ck + 31) / 32) * 4;
}

// ceil(n_p / CA_QT) chunks per query cluster (input to the offsets scan).
__global__ void comp_chunks_kernel(const int* __restrict__ nq, int Cq, int* __restrict__ nch) {
  const int bh = blockIdx.y;
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= Cq) return;
  const int n = nq[static_cast<long long>(bh) * Cq + p];
  nch[static_cast<long long>(bh) * Cq + p] = (n + CA_QT - 1) / CA_QT;
}

// One CTA per (bh, chunk of up to 64 queries of one query cluster p): online
// softmax over (1) the virtual keys of the non-empty, non-selected key
// clusters and (2) the keys of the selected clusters (cluster order), then
// out[token] for each query token. Grid (max chunks, BH).
template <typename T, int D>
__global__ void __launch_bounds__(CA_THREADS)
    comp_attn_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     int N, int Cq, int Ck, const int* __restrict__ choff,
                     const int* __restrict__ qoff, const int* __restrict__ qperm,
                     const int* __restrict__ koff, const int* __restrict__ kperm,
                     const float* __restrict__ kc, const float* __restrict__ vc,
                     const int* __restrict__ nk, const int* __restrict__ seln,
                     const int* __restrict__ selc, float scale_log2, T* __restrict__ out) {
  constexpr int DV = D / 16;
  extern __shared__ float ca_smem[];
  float* qT = ca_smem;                  // [D][CA_QT]
  float* kT = qT + D * CA_QT;           // [D][CA_KT]
  float* vs = kT + D * CA_KT;           // [CA_KT][D]
  float* ps = vs + CA_KT * D;           // [CA_QT][CA_KT]
  float* bias = ps + CA_QT * CA_KT;     // [CA_KT] (log2 units)
  int* qrow = reinterpret_cast<int*>(bias + CA_KT);  // [CA_QT]
  int* kidx = qrow + CA_QT;             // [CA_KT]: key token of each tile column
  int* spos = kidx + CA_KT;             // [Ck + 1]: stream start of selected cluster s
  int* sc = spos + Ck + 1;              // [Ck]: selected clusters
  uint32_t* smask = reinterpret_cast<uint32_t*>(sc + Ck);  // [ceil(Ck/32)]
  __shared__ int s_p, s_first, s_nq;

  const int bh = blockIdx.y, tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int* co = choff + static_cast<long long>(bh) * (Cq + 1);
  const int chunk = blockIdx.x;
  if (chunk >= co[Cq]) return;
  if (tid == 0) {
    int lo = 0, hi = Cq - 1;  // last p with co[p] <= chunk
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (co[mid] <= chunk) lo = mid;
      else hi = mid - 1;
    }
    const int* qo = qoff + static_cast<long long>(bh) * (Cq + 1);
    s_p = lo;
    s_first = qo[lo] + (chunk - co[lo]) * CA_QT;
    s_nq = min(CA_QT, qo[lo + 1] - s_first);
  }
  __syncthreads();
  const int p = s_p, nqc = s_nq;
  const long long base = static_cast<long long>(bh) * N * D;
  const int* ko = koff + static_cast<long long>(bh) * (Ck + 1);
  const int* kp = kperm + static_cast<long long>(bh) * N;
  const int ns = seln[static_cast<long long>(bh) * Cq + p];
  const int* sl = selc + (static_cast<long long>(bh) * Cq + p) * Ck;
  const int nwords = (Ck + 31) / 32;

  for (int r = tid; r < CA_QT; r += CA_THREADS)
    qrow[r] = r < nqc ? qperm[static_cast<long long>(bh) * N + s_first + r] : -1;
  for (int w = tid; w < nwords; w += CA_THREADS) smask[w] = 0;
  __syncthreads();
  stage_transposed<T, D, CA_QT, CA_THREADS>(qT, [&](int r) -> const T* {
    return qrow[r] >= 0 ? q + base + static_cast<long long>(qrow[r]) * D : nullptr;
  });
  for (int s = tid; s < ns; s += CA_THREADS) {
    const int c = sl[s];
    sc[s] = c;
    atomicOr(&smask[c >> 5], 1u << (c & 31));
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int s = 0; s < ns; ++s) {
      spos[s] = acc;
      acc += ko[sc[s] + 1] - ko[sc[s]];
    }
    spos[ns] = acc;
  }
  __syncthreads();
  const int n_exact = spos[ns];
  const int n_virt_tiles = (Ck + CA_KT - 1) / CA_KT;
  const int n_exact_tiles = (n_exact + CA_KT - 1) / CA_KT;

  float m[4], l[4], O[4][DV];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
#pragma unroll
    for (int e = 0; e < DV; ++e) O[a][e] = 0.f;
  }
  for (int t = 0; t < n_virt_tiles + n_exact_tiles; ++t) {
    const bool virt = t < n_virt_tiles;
    __syncthreads();
    if (virt) {
      const int c0 = t * CA_KT;
      const float* kcb = kc + static_cast<long long>(bh) * Ck * D;
      const float* vcb = vc + static_cast<long long>(bh) * Ck * D;
      stage_transposed<float, D, CA_KT, CA_THREADS>(kT, [&](int kk) -> const float* {
        return c0 + kk < Ck ? kcb + static_cast<long long>(c0 + kk) * D : nullptr;
      });
      stage_rows<float, D, CA_KT, CA_THREADS>(vs, [&](int kk) -> const float* {
        return c0 + kk < Ck ? vcb + static_cast<long long>(c0 + kk) * D : nullptr;
      });
      for (int kk = tid; kk < CA_KT; kk += CA_THREADS) {
        const int c = c0 + kk;
        const int n = c < Ck ? nk[static_cast<long long>(bh) * Ck + c] : 0;
        const bool live = n > 0 && !((smask[c >> 5] >> (c & 31)) & 1u);
        bias[kk] = live ? log2f(static_cast<float>(n)) : -INFINITY;
      }
    } else {
      const int s0 = (t - n_virt_tiles) * CA_KT;
      for (int kk = tid; kk < CA_KT; kk += CA_THREADS) {
        const int pos = s0 + kk;
        int j = -1;
        if (pos < n_exact) {
          int lo = 0, hi = ns - 1;  // selected cluster holding stream position pos
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (spos[mid] <= pos) lo = mid;
            else hi = mid - 1;
          }
          j = kp[ko[sc[lo]] + (pos - spos[lo])];
        }
        kidx[kk] = j;
        bias[kk] = j >= 0 ? 0.f : -INFINITY;
      }
      __syncthreads();
      stage_transposed<T, D, CA_KT, CA_THREADS>(kT, [&](int kk) -> const T* {
        return kidx[kk] >= 0 ? k + base + static_cast<long long>(kidx[kk]) * D : nullptr;
      });
      stage_rows<T, D, CA_KT, CA_THREADS>(vs, [&](int kk) -> const T* {
        return kidx[kk] >= 0 ? v + base + static_cast<long long>(kidx[kk]) * D : nullptr;
      });
    }
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
    for (int dd = 0; dd < D; ++dd) {
      const float4 qv = *reinterpret_cast<const float4*>(&qT[dd * CA_QT + ty * 4]);
      const float4 kv = *reinterpret_cast<const float4*>(&kT[dd * CA_KT + tx * 4]);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
      const float kb[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qa[a], kb[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float tmax = -INFINITY;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        acc[a][b] = fmaf(acc[a][b], scale_log2, bias[tx * 4 + b]);
        tmax = fmaxf(tmax, acc[a][b]);
      }
#pragma unroll
      for (int o = 8; o; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float mn = fmaxf(m[a], tmax);
      const float alpha = (mn == -INFINITY) ? 1.f : exp2f(m[a] - mn);
      float ts = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float e = (mn == -INFINITY) ? 0.f : exp2f(acc[a][b] - mn);
        ps[(ty * 4 + a) * CA_KT + tx * 4 + b] = e;
        ts += e;
      }
#pragma unroll
      for (int o = 8; o; o >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, o);
      m[a] = mn;
      l[a] = l[a] * alpha + ts;
#pragma unroll
      for (int e = 0; e < DV; ++e) O[a][e] *= alpha;
    }
    __syncwarp();
    for (int kk = 0; kk < CA_KT; ++kk) {
      float vv[DV];
#pragma unroll
      for (int e = 0; e < DV; ++e) vv[e] = vs[kk * D + tx * DV + e];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float w = ps[(ty * 4 + a) * CA_KT + kk];
#pragma unroll
        for (int e = 0; e < DV; ++e) O[a][e] = fmaf(w, vv[e], O[a][e]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int r = ty * 4 + a;
    const int tok = qrow[r];
    if (tok < 0) continue;
    const float inv = l[a] > 0.f ? 1.f / l[a] : 0.f;
    T* dst = out + base + static_cast<long long>(tok) * D + tx * DV;
#pragma unroll
    for (int e = 0; e < DV; ++e) {
      if constexpr (sizeof(T) == 4) dst[e] = O[a][e] * inv;
      else dst[e] = __float2bfloat16_rn(O[a][e] * inv);
    }
  }
}

}  // namespace va
