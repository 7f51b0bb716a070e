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

constexpr int PR_PG = 16;  // query clusters per CTA
constexpr int PR_KT = 64;  // keys per tile
constexpr int PR_THREADS = 256;

template <int D>
constexpr int probe_smem_bytes(int Ck) {
  return (D * PR_PG + D * PR_KT + PR_KT * D + PR_PG * PR_KT) * 4 + 2 * PR_KT * 4 + (Ck + 1) * 4;
}

// err[bh][p][c] for every non-empty p and c (other entries are left as the
// caller initialised them). Grid: (ceil(Cq / PR_PG), BH), 256 threads;
// thread (ty, tx): query cluster p0 + ty, keys tx*4..tx*4+3 of a tile and
// dims tx*(D/16).. of the value accumulators.
template <typename T, int D>
__global__ void __launch_bounds__(PR_THREADS)
    probe_kernel(const T* __restrict__ k, const T* __restrict__ v, int N, int Cq, int Ck,
                 const float* __restrict__ qc, const int* __restrict__ nq,
                 const float* __restrict__ kc, const float* __restrict__ vc,
                 const int* __restrict__ nk, const int* __restrict__ koff,
                 const int* __restrict__ kperm, const int* __restrict__ kassign, float scale,
                 float* __restrict__ err) {
  constexpr int DV = D / 16;  // value dims per thread
  extern __shared__ float pr_smem[];
  float* qcT = pr_smem;                       // [D][PR_PG]
  float* kT = qcT + D * PR_PG;                // [D][PR_KT]
  float* vs = kT + D * PR_KT;                 // [PR_KT][D]
  float* es = vs + PR_KT * D;                 // [PR_PG][PR_KT]
  int* cid = reinterpret_cast<int*>(es + PR_PG * PR_KT);  // [PR_KT]
  int* kidx = cid + PR_KT;                    // [PR_KT]
  int* offs = kidx + PR_KT;                   // [Ck + 1]

  const int bh = blockIdx.y;
  const int p0 = blockIdx.x * PR_PG;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int p = p0 + ty;
  const long long kvb = static_cast<long long>(bh) * N * D;
  const int* ko = koff + static_cast<long long>(bh) * (Ck + 1);
  const int* kp = kperm + static_cast<long long>(bh) * N;
  const int* ka = kassign + static_cast<long long>(bh) * N;

  stage_transposed<float, D, PR_PG, PR_THREADS>(qcT, [&](int pp) -> const float* {
    return p0 + pp < Cq ? qc + (static_cast<long long>(bh) * Cq + p0 + pp) * D : nullptr;
  });
  for (int e = tid; e <= Ck; e += PR_THREADS) offs[e] = ko[e];

  // ---- pass 1: m_p, Z_p, O_p over all keys (token order) -------------------
  float m = -INFINITY, Z = 0.f;
  float O[DV];
#pragma unroll
  for (int e = 0; e < DV; ++e) O[e] = 0.f;
  for (int j0 = 0; j0 < N; j0 += PR_KT) {
    __syncthreads();
    stage_transposed<T, D, PR_KT, PR_THREADS>(kT, [&](int kk) -> const T* {
      return j0 + kk < N ? k + kvb + static_cast<long long>(j0 + kk) * D : nullptr;
    });
    stage_rows<T, D, PR_KT, PR_THREADS>(vs, [&](int kk) -> const T* {
      return j0 + kk < N ? v + kvb + static_cast<long long>(j0 + kk) * D : nullptr;
    });
    __syncthreads();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int dd = 0; dd < D; ++dd) {
      const float qv = qcT[dd * PR_PG + ty];
      const float4 kv = *reinterpret_cast<const float4*>(&kT[dd * PR_KT + tx * 4]);
      acc[0] = fmaf(qv, kv.x, acc[0]);
      acc[1] = fmaf(qv, kv.y, acc[1]);
      acc[2] = fmaf(qv, kv.z, acc[2]);
      acc[3] = fmaf(qv, kv.w, acc[3]);
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      acc[b] = (j0 + tx * 4 + b < N) ? acc[b] * scale : -INFINITY;
      tmax = fmaxf(tmax, acc[b]);
    }
#pragma unroll
    for (int o = 8; o; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    const float mn = fmaxf(m, tmax);
    const float alpha = expf(m - mn);  // m = -inf on the first tile: alpha = 0
    m = mn;
    float ts = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float e = expf(acc[b] - mn);
      es[ty * PR_KT + tx * 4 + b] = e;
      ts += e;
    }
#pragma unroll
    for (int o = 8; o; o >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, o);
    Z = Z * alpha + ts;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < DV; ++e) O[e] *= alpha;
    for (int kk = 0; kk < PR_KT; ++kk) {
      const float w = es[ty * PR_KT + kk];
#pragma unroll
      for (int e = 0; e < DV; ++e) O[e] = fmaf(w, vs[kk * D + tx * DV + e], O[e]);
    }
  }
  const float invZ = 1.f / Z;
#pragma unroll
  for (int e = 0; e < DV; ++e) O[e] *= invZ;

  // ---- pass 2: per key cluster residual, keys in cluster order -------------
  const bool write = p < Cq && nq[static_cast<long long>(bh) * Cq + min(p, Cq - 1)] > 0;
  float r[DV];
#pragma unroll
  for (int e = 0; e < DV; ++e) r[e] = 0.f;
  for (int t0 = 0; t0 < N; t0 += PR_KT) {
    __syncthreads();
    for (int kk = tid; kk < PR_KT; kk += PR_THREADS) {
      const int j = (t0 + kk < N) ? kp[t0 + kk] : -1;
      kidx[kk] = j;
      cid[kk] = j >= 0 ? ka[j] : -1;
    }
    __syncthreads();
    stage_transposed<T, D, PR_KT, PR_THREADS>(kT, [&](int kk) -> const T* {
      return kidx[kk] >= 0 ? k + kvb + static_cast<long long>(kidx[kk]) * D : nullptr;
    });
    stage_rows<T, D, PR_KT, PR_THREADS>(vs, [&](int kk) -> const T* {
      return kidx[kk] >= 0 ? v + kvb + static_cast<long long>(kidx[kk]) * D : nullptr;
    });
    __syncthreads();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int dd = 0; dd < D; ++dd) {
      const float qv = qcT[dd * PR_PG + ty];
      const float4 kv = *reinterpret_cast<const float4*>(&kT[dd * PR_KT + tx * 4]);
      acc[0] = fmaf(qv, kv.x, acc[0]);
      acc[1] = fmaf(qv, kv.y, acc[1]);
      acc[2] = fmaf(qv, kv.z, acc[2]);
      acc[3] = fmaf(qv, kv.w, acc[3]);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b)
      es[ty * PR_KT + tx * 4 + b] =
          (t0 + tx * 4 + b < N) ? expf(fmaf(acc[b], scale, -m)) : 0.f;
    __syncwarp();
    for (int kk = 0; kk < PR_KT; ++kk) {
      const int c = cid[kk];
      if (c < 0) break;
      const float w = es[ty * PR_KT + kk];
#pragma unroll
      for (int e = 0; e < DV; ++e) r[e] = fmaf(w, vs[kk * D + tx * DV + e] - O[e], r[e]);
      if (t0 + kk == offs[c + 1] - 1) {
        // last key of cluster c: subtract the compensated term, then |r| / Z
        const float* kcc = kc + (static_cast<long long>(bh) * Ck + c) * D;
        const float* vcc = vc + (static_cast<long long>(bh) * Ck + c) * D;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < DV; ++e) dot = fmaf(qcT[(tx * DV + e) * PR_PG + ty], kcc[tx * DV + e], dot);
#pragma unroll
        for (int o = 8; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const float wc = static_cast<float>(nk[static_cast<long long>(bh) * Ck + c]) *
                         expf(fmaf(dot, scale, -m));
        float n2 = 0.f;
#pragma unroll
        for (int e = 0; e < DV; ++e) {
          const float re = fmaf(-wc, vcc[tx * DV + e] - O[e], r[e]);
          n2 = fmaf(re, re, n2);
          r[e] = 0.f;
        }
#pragma unroll
        for (int o = 8; o; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
        if (write && tx == 0)
          err[(static_cast<long long>(bh) * Cq + p) * Ck + c] = sqrtf(n2) * invZ;
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

// Per bh (one CTA of 1024 threads): the smallest key K whose prefix (all keys
// <= K) costs more than the budget; blocks with key < K are computed exactly.
// cut[bh] = ~0 when every valid block fits. Weighted MSB-first radix select,
// 8 bits per pass.
__global__ void __launch_bounds__(1024)
    route_select_kernel(const float* __restrict__ err, const int* __restrict__ nq,
                        const int* __restrict__ nk, int Cq, int Ck, long long budget,
                        unsigned long long* __restrict__ cut) {
  __shared__ unsigned long long hist[256];
  __shared__ unsigned long long s_prefix, s_mask;
  __shared__ long long s_remaining;
  __shared__ int s_done;
  const int bh = blockIdx.x, tid = threadIdx.x;
  const float* eb = err + static_cast<long long>(bh) * Cq * Ck;
  const int* nqb = nq + static_cast<long long>(bh) * Cq;
  const int* nkb = nk + static_cast<long long>(bh) * Ck;
  if (tid == 0) {
    s_prefix = 0;
    s_mask = 0;
    s_remaining = budget;
    s_done = 0;
  }
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += 1024) hist[b] = 0;
    __syncthreads();
    if (s_done) break;
    const unsigned long long prefix = s_prefix, mask = s_mask;
    const int total = Cq * Ck;
    for (int e = tid; e < total; e += 1024) {
      const int p = e / Ck, c = e - p * Ck;
      const int np = nqb[p], nc = nkb[c];
      if (np <= 0 || nc <= 0) continue;
      const float ratio = __fdiv_rn(eb[e], static_cast<float>(nc));
      const unsigned long long key = route_key(ratio, p, c, Ck);
      if ((key & mask) != prefix) continue;
      atomicAdd(&hist[(key >> shift) & 255u],
                static_cast<unsigned long long>(np) * static_cast<unsigned long long>(nc));
    }
    __syncthreads();
    if (tid == 0) {
      long long cum = 0;
      int b = 0;
      for (; b < 256; ++b) {
        const long long h = static_cast<long long>(hist[b]);
        if (cum + h > s_remaining) break;
        cum += h;
      }
      if (b == 256) {
        // everything under this prefix fits
        s_done = 1;
        if (shift == 56) s_prefix = ~0ull;  // the whole set fits the budget
        else s_prefix = prefix | ((1ull << (shift + 8)) - 1ull) ;
      } else {
        s_remaining -= cum;
        s_prefix = prefix | (static_cast<unsigned long long>(b) << shift);
        s_mask = mask | (255ull << shift);
      }
    }
    __syncthreads();
  }
  if (tid == 0) cut[bh] = s_prefix;
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
