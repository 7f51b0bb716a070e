// Static spatiotemporal block masks as CSR lists (integer arithmetic only).
//
// Token rules (readings of the pages; identical for every batch and head):
//   radial (Radial Attention news page, hyper.ai: the window shrinks
//     exponentially with temporal distance):
//       live(i, j) <=> |s_i - s_j| <= W0 >> octave(|t_i - t_j|),
//       octave(0) = 0, octave(dt) = bit length of dt;
//   LVSA (LVSA review, secrett2633 blog, sec. 3 and Fig. 2: local frame window
//     plus periodic global anchor frames that rotate per denoising step):
//       live(i, j) <=> |t_i - t_j| <= L  or  (t_j - a0 - rho*step) mod P == 0
//       (P == 0: t_j == a0);
//   dense: always live.
// A block pair is live iff some real token pair in it is live. Blocks are
// split into runs of one frame each; for two runs the smallest in-frame
// distance is max(0, lo_j - hi_i, lo_i - hi_j), which decides the radial rule.
#pragma once

#include "common.cuh"

namespace va {

struct MaskDesc {
  int kind, T, F, N, block, nb;
  int w0, local, period, anchor0, rot_stride, step;
  // 1: count and fill the transposed lists (for key block I, the query blocks
  // J that see it), which the backward's key-side kernels walk.
  int transpose = 0;
};

__device__ __forceinline__ bool run_pair_live(const MaskDesc& m, int ti, int lo_i, int hi_i,
                                              int tj, int lo_j, int hi_j) {
  if (m.kind == VA_MASK_DENSE) return true;
  const int dt = ti > tj ? ti - tj : tj - ti;
  if (m.kind == VA_MASK_RADIAL) {
    const int oct = 32 - __clz(dt);  // bit length; __clz(0) == 32
    const int w = oct >= 31 ? 0 : (m.w0 >> oct);
    const int gap = max(0, max(lo_j - hi_i, lo_i - hi_j));
    return gap <= w;
  }
  if (dt <= m.local) return true;
  if (m.period > 0) {
    long long r = (static_cast<long long>(tj) - m.anchor0 -
                   static_cast<long long>(m.rot_stride) * m.step) % m.period;
    if (r < 0) r += m.period;
    return r == 0;
  }
  return tj == m.anchor0;
}

__device__ bool block_pair_live(const MaskDesc& m, int I, int J) {
  const int qs = I * m.block, qe = min(m.N, qs + m.block);
  const int ks = J * m.block, ke = min(m.N, ks + m.block);
  for (int n = qs; n < qe;) {
    const int ti = n / m.F;
    const int qstop = min(qe, (ti + 1) * m.F);
    const int lo_i = n - ti * m.F, hi_i = qstop - 1 - ti * m.F;
    for (int j = ks; j < ke;) {
      const int tj = j / m.F;
      const int kstop = min(ke, (tj + 1) * m.F);
      if (run_pair_live(m, ti, lo_i, hi_i, tj, j - tj * m.F, kstop - 1 - tj * m.F)) return true;
      j = kstop;
    }
    n = qstop;
  }
  return false;
}

// One warp per query block: number of live key blocks and the number of key
// tokens they hold.
__global__ void mask_count_kernel(MaskDesc m, int* __restrict__ cnt,
                                  long long* __restrict__ key_tokens) {
  const int I = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (I >= m.nb) return;
  int c = 0;
  long long kt = 0;
  for (int J0 = 0; J0 < m.nb; J0 += 32) {
    const int J = J0 + lane;
    const bool live = J < m.nb && (m.transpose ? block_pair_live(m, J, I) : block_pair_live(m, I, J));
    c += __popc(__ballot_sync(0xffffffffu, live));
    if (live) kt += min(m.N, (J + 1) * m.block) - J * m.block;
  }
  for (int o = 16; o; o >>= 1) kt += __shfl_xor_sync(0xffffffffu, kt, o);
  if (lane == 0) {
    cnt[I] = c;
    key_tokens[I] = kt;
  }
}

// Single CTA: exclusive scan of the counts into row_ptr, nnz and live token
// pairs into summary[0..1], and the rows ordered by descending length
// (stable), the longest-first order the attention kernel schedules in.
// hist must hold nb + 1 ints.
__global__ void mask_scan_kernel(MaskDesc m, const int* __restrict__ cnt,
                                 const long long* __restrict__ key_tokens,
                                 int* __restrict__ row_ptr, long long* __restrict__ summary,
                                 int* __restrict__ order, int* __restrict__ hist) {
  __shared__ long long part[1024];
  __shared__ long long part_pairs[1024];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (m.nb + nt - 1) / nt;
  const int lo = min(m.nb, tid * per), hi = min(m.nb, lo + per);
  long long s = 0, pairs = 0;
  for (int i = lo; i < hi; ++i) {
    s += cnt[i];
    const long long rows = min(m.N, (i + 1) * m.block) - i * m.block;
    pairs += rows * key_tokens[i];
  }
  part[tid] = s;
  part_pairs[tid] = pairs;
  __syncthreads();
  if (tid == 0) {
    long long acc = 0, accp = 0;
    for (int t = 0; t < nt; ++t) {
      const long long v = part[t];
      part[t] = acc;
      acc += v;
      accp += part_pairs[t];
    }
    summary[0] = acc;
    summary[1] = accp;
    row_ptr[m.nb] = static_cast<int>(acc);
  }
  __syncthreads();
  long long base = part[tid];
  for (int i = lo; i < hi; ++i) {
    row_ptr[i] = static_cast<int>(base);
    base += cnt[i];
  }
  // stable counting sort of rows by descending count (counts are 0..nb)
  for (int i = tid; i <= m.nb; i += nt) hist[i] = 0;
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < m.nb; ++i) hist[m.nb - cnt[i]]++;
    int acc = 0;
    for (int b = 0; b <= m.nb; ++b) {
      const int v = hist[b];
      hist[b] = acc;
      acc += v;
    }
    for (int i = 0; i < m.nb; ++i) order[hist[m.nb - cnt[i]]++] = i;
  }
}

// One warp per query block: write the live key blocks in ascending order.
__global__ void mask_fill_kernel(MaskDesc m, const int* __restrict__ row_ptr,
                                 int* __restrict__ col) {
  const int I = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (I >= m.nb) return;
  int base = row_ptr[I];
  const int end = row_ptr[I + 1];
  if (base < 0 || end < base) {
    // offsets that wrapped or run backwards: write nothing
    if (lane == 0) raise_error(VA_ERR_DEVICE);
    return;
  }
  for (int J0 = 0; J0 < m.nb; J0 += 32) {
    const int J = J0 + lane;
    const bool live = J < m.nb && (m.transpose ? block_pair_live(m, J, I) : block_pair_live(m, I, J));
    const unsigned bal = __ballot_sync(0xffffffffu, live);
    const int pos = base + __popc(bal & ((1u << lane) - 1u));
    if (live) {
      if (pos < end) {
        col[pos] = J;
      } else {
        raise_error(VA_ERR_DEVICE);
      }
    }
    base += __popc(bal);
  }
}

}  // namespace va

namespace va {

// Query-block pairs {2P, 2P+1} for the two-tile attention kernel: the merged
// (union) key-block list of the two rows, entry = J << 2 | live bits (bit 0:
// row 2P, bit 1: row 2P+1). Pair P's entries start at row_ptr[2P] (the union
// is never longer than both rows together). One thread per pair.
__global__ void pair_merge_kernel(int nb, const int* __restrict__ row_ptr,
                                  const int* __restrict__ col, int* __restrict__ pcol,
                                  int* __restrict__ plen) {
  const int P = blockIdx.x * blockDim.x + threadIdx.x;
  const int npairs = (nb + 1) / 2;
  if (P >= npairs) return;
  int a = row_ptr[2 * P];
  const int ae = row_ptr[2 * P + 1];
  int b = ae;
  const int be = (2 * P + 1 < nb) ? row_ptr[2 * P + 2] : ae;
  const int out = row_ptr[2 * P];
  int k = 0;
  while (a < ae || b < be) {
    const int ja = a < ae ? col[a] : 0x7fffffff;
    const int jb = b < be ? col[b] : 0x7fffffff;
    int e;
    if (ja < jb) {
      e = (ja << 2) | 1;
      ++a;
    } else if (jb < ja) {
      e = (jb << 2) | 2;
      ++b;
    } else {
      e = (ja << 2) | 3;
      ++a;
      ++b;
    }
    pcol[out + k] = e;
    ++k;
  }
  plen[P] = k;
}

// Quads for the two-tile kernel on 64-token blocks: tile t of quad Q covers
// the 128 query rows of blocks 4Q + 2t and 4Q + 2t + 1, and an entry covers
// the 128 keys of blocks 2J' and 2J' + 1. The union over the four rows is
// keyed by J'; entry = J' << 10 | sub << 2 | tile bits, where sub bit
// 4t + 2a + b says that block 4Q + 2t + a sees block 2J' + b, and tile bit t
// that any of tile t's four sub bits is set. Quad Q's entries start at
// row_ptr[4Q] (the union is never longer than the four rows together). One
// thread per quad.
__global__ void quad_merge_kernel(int nb, const int* __restrict__ row_ptr,
                                  const int* __restrict__ col, int* __restrict__ qcol,
                                  int* __restrict__ qlen) {
  const int Q = blockIdx.x * blockDim.x + threadIdx.x;
  const int nquads = (nb + 3) / 4;
  if (Q >= nquads) return;
  int cur[4], end[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 4 * Q + i;
    cur[i] = row < nb ? row_ptr[row] : 0;
    end[i] = row < nb ? row_ptr[row + 1] : 0;
  }
  const int out = row_ptr[4 * Q];
  int k = 0;
  while (true) {
    int jc = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (cur[i] < end[i]) jc = min(jc, col[cur[i]] >> 1);
    if (jc == 0x7fffffff) break;
    int sub = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // row i = 2t + a holds bit 4t + 2a + b = 2i + b for key block 2jc + b
      while (cur[i] < end[i] && (col[cur[i]] >> 1) == jc) {
        sub |= 1 << (2 * i + (col[cur[i]] & 1));
        ++cur[i];
      }
    }
    const int tiles = ((sub & 0x0f) ? 1 : 0) | ((sub & 0xf0) ? 2 : 0);
    qcol[out + k] = (jc << 10) | (sub << 2) | tiles;
    ++k;
  }
  qlen[Q] = k;
}

// Coarse pairs for the backward on 64-token blocks: row R of the coarse list
// merges rows 2R and 2R + 1 of a block list (the CSR, or the transposed lists)
// by coarse index c = idx >> 1; entry = c << 4 | sub, sub bit 2a + b meaning
// that row 2R + a lists block 2c + b. Row R's entries start at ptr[2R]. One
// thread per coarse row.
__global__ void coarse_pair_merge_kernel(int nb, const int* __restrict__ ptr,
                                         const int* __restrict__ idx, int* __restrict__ ccol,
                                         int* __restrict__ clen) {
  const int R = blockIdx.x * blockDim.x + threadIdx.x;
  const int ncoarse = (nb + 1) / 2;
  if (R >= ncoarse) return;
  int cur[2], end[2];
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int row = 2 * R + a;
    cur[a] = row < nb ? ptr[row] : 0;
    end[a] = row < nb ? ptr[row + 1] : 0;
  }
  const int out = ptr[2 * R];
  int k = 0;
  while (true) {
    int c = 0x7fffffff;
#pragma unroll
    for (int a = 0; a < 2; ++a)
      if (cur[a] < end[a]) c = min(c, idx[cur[a]] >> 1);
    if (c == 0x7fffffff) break;
    int sub = 0;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      while (cur[a] < end[a] && (idx[cur[a]] >> 1) == c) {
        sub |= 1 << (2 * a + (idx[cur[a]] & 1));
        ++cur[a];
      }
    }
    ccol[out + k] = (c << 4) | sub;
    ++k;
  }
  clen[R] = k;
}

// Single thread: quads ordered by descending summed length of their four rows
// (stable counting sort; lengths are 0..4*nb). hist must hold 4*nb + 2 ints.
__global__ void quad_order_kernel(int nb, const int* __restrict__ row_ptr,
                                  int* __restrict__ qorder, int* __restrict__ hist) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const int nquads = (nb + 3) / 4;
  const int top = 4 * nb + 1;
  for (int i = 0; i <= top; ++i) hist[i] = 0;
  for (int Q = 0; Q < nquads; ++Q) {
    const int e = min(4 * Q + 4, nb);
    hist[top - (row_ptr[e] - row_ptr[4 * Q])]++;
  }
  int acc = 0;
  for (int i = 0; i <= top; ++i) {
    const int v = hist[i];
    hist[i] = acc;
    acc += v;
  }
  for (int Q = 0; Q < nquads; ++Q) {
    const int e = min(4 * Q + 4, nb);
    qorder[hist[top - (row_ptr[e] - row_ptr[4 * Q])]++] = Q;
  }
}

// Single thread: pairs ordered by descending summed row length (stable
// counting sort; lengths are 0..2*nb). hist must hold 2*nb + 2 ints.
__global__ void pair_order_kernel(int nb, const int* __restrict__ row_ptr,
                                  int* __restrict__ porder, int* __restrict__ hist) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const int npairs = (nb + 1) / 2;
  const int top = 2 * nb + 1;
  for (int i = 0; i <= top; ++i) hist[i] = 0;
  for (int P = 0; P < npairs; ++P) {
    const int e = min(2 * P + 2, nb);
    hist[top - (row_ptr[e] - row_ptr[2 * P])]++;
  }
  int acc = 0;
  for (int i = 0; i <= top; ++i) {
    const int v = hist[i];
    hist[i] = acc;
    acc += v;
  }
  for (int P = 0; P < npairs; ++P) {
    const int e = min(2 * P + 2, nb);
    porder[hist[top - (row_ptr[e] - row_ptr[2 * P])]++] = P;
  }
}

}  // namespace va
