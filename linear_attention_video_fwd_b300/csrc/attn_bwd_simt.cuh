// Block-sparse attention backward: the row preprocess and the float32 FMA
// kernels (fp32 inputs, and any case the tensor-core kernels do not take).
//
// Gradients of o_i = sum_j p_ij v_j, p_ij = exp(scale q_i.k_j - lse_i) on the
// live blocks, for an upstream gradient g = dL/do (the chain rule; Radial
// Attention's LoRA fine-tuning under its static mask trains through it):
//   delta_i = g_i . o_i,  dp_ij = g_i . v_j,  ds_ij = p_ij (dp_ij - delta_i)
//   dv_j = sum_i p_ij g_i,  dq_i = scale sum_j ds_ij k_j,  dk_j = scale sum_i ds_ij q_i
// p is recomputed from the forward's lse. The query side walks the CSR rows;
// the key side walks the transposed CSR (for key block J, the query blocks
// that see it), so neither needs atomics and the results are deterministic.
#pragma once

#include "common.cuh"

namespace va {

// Per row of a [BH, N] grid padded to Np rows per head, both negated so the
// kernels add them: ndelta = -(g . o) in float32 and nlse2 = -lse * log2(e).
// Padding rows, and rows that saw no key (lse = -inf), get nlse2 = -inf (so
// every recomputed p is 0) and ndelta = 0.
// One warp per row; grid (ceil(Np / 8), BH), 256 threads.
template <typename T>
__global__ void bwd_prep_kernel(const T* __restrict__ o, const T* __restrict__ g,
                                const float* __restrict__ lse, int N, int Np, int D,
                                float* __restrict__ ndelta, float* __restrict__ nlse2) {
  const int bh = blockIdx.y;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= Np) return;
  const long long out = static_cast<long long>(bh) * Np + n;
  if (n >= N) {
    if (lane == 0) {
      ndelta[out] = 0.f;
      nlse2[out] = -INFINITY;
    }
    return;
  }
  const long long row = (static_cast<long long>(bh) * N + n) * D;
  float acc = 0.f;
  for (int c = lane; c < D; c += 32) acc = fmaf(to_f32(g[row + c]), to_f32(o[row + c]), acc);
#pragma unroll
  for (int s = 16; s; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) {
    const float l = lse[static_cast<long long>(bh) * N + n];
    const bool dead = l == -INFINITY;
    ndelta[out] = dead ? 0.f : -acc;
    nlse2[out] = dead ? -INFINITY : -l * 1.4426950408889634f;
  }
}

// Rows per CTA of the float32 kernels: 64 rows of four threads, so the
// per-row registers (three or four vectors of d / 4 floats) fit without spills.
constexpr int BWS_ROWS = 64;

// dq for 64 rows of query block I of head bh (blockIdx = (I * BLK / 64 +
// part, bh)). Four threads share a query row, thread u owning dims
// {4 i + u}; keys are staged 32 at a time.
template <typename T, int D, int BLK>
__global__ void __launch_bounds__(BWS_ROWS * 4)
    bwd_dq_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                       const T* __restrict__ g, const float* __restrict__ ndelta,
                       const float* __restrict__ nlse2, const int* __restrict__ row_ptr,
                       const int* __restrict__ col, T* __restrict__ dq, int N, int Np,
                       float scale, float scale_log2) {
  constexpr int TPR = 4, DQ = D / TPR, BN = 32, NT = BWS_ROWS * TPR;
  __shared__ float ks[BN][D];
  __shared__ float vs[BN][D];
  const int I = blockIdx.x / (BLK / BWS_ROWS);
  const long long bh = blockIdx.y;
  const int tid = threadIdx.x, r = tid / TPR, u = tid % TPR;
  const int row = blockIdx.x * BWS_ROWS + r;
  const bool row_ok = row < N;
  const T* kb = k + bh * N * D;
  const T* vb = v + bh * N * D;
  float qr[DQ], gr[DQ], acc[DQ];
#pragma unroll
  for (int i = 0; i < DQ; ++i) {
    const long long at = (bh * N + row) * D + TPR * i + u;
    qr[i] = row_ok ? to_f32(q[at]) : 0.f;
    gr[i] = row_ok ? to_f32(g[at]) : 0.f;
    acc[i] = 0.f;
  }
  const float nl2 = nlse2[bh * Np + row];   // -inf on padding rows
  const float ndl = ndelta[bh * Np + row];
  for (int e = row_ptr[I]; e < row_ptr[I + 1]; ++e) {
    const int kstart = col[e] * BLK;
    const int kcount = min(BLK, N - kstart);
    for (int s0 = 0; s0 < kcount; s0 += BN) {
      __syncthreads();
      for (int idx = tid; idx < BN * D; idx += NT) {
        const int jj = idx / D, c = idx % D;
        const bool ok = s0 + jj < kcount;
        const long long at = static_cast<long long>(kstart + s0 + jj) * D + c;
        ks[jj][c] = ok ? to_f32(kb[at]) : 0.f;
        vs[jj][c] = ok ? to_f32(vb[at]) : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int j = 0; j < BN; ++j) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int i = 0; i < DQ; ++i) {
          s = fmaf(qr[i], ks[j][TPR * i + u], s);
          dp = fmaf(gr[i], vs[j][TPR * i + u], dp);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        dp += __shfl_xor_sync(0xffffffffu, dp, 1);
        dp += __shfl_xor_sync(0xffffffffu, dp, 2);
        const float p = (s0 + j < kcount) ? exp2f(fmaf(s, scale_log2, nl2)) : 0.f;
        const float ds = p * (dp + ndl);
#pragma unroll
        for (int i = 0; i < DQ; ++i) acc[i] = fmaf(ds, ks[j][TPR * i + u], acc[i]);
      }
    }
  }
  if (row_ok) {
    T* out = dq + (bh * N + row) * D;
#pragma unroll
    for (int i = 0; i < DQ; ++i) out[TPR * i + u] = from_f32<T>(acc[i] * scale);
  }
}

// dk and dv for 64 rows of key block J of head bh (blockIdx = (J * BLK / 64
// + part, bh)), walking the query blocks of the transposed CSR. Four threads
// share a key row; queries, their upstream gradients, nlse2 and ndelta are
// staged 32 at a time.
template <typename T, int D, int BLK>
__global__ void __launch_bounds__(BWS_ROWS * 4)
    bwd_dkdv_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                         const T* __restrict__ v, const T* __restrict__ g,
                         const float* __restrict__ ndelta, const float* __restrict__ nlse2,
                         const int* __restrict__ t_ptr, const int* __restrict__ t_row,
                         T* __restrict__ dk, T* __restrict__ dv, int N, int Np, float scale,
                         float scale_log2) {
  constexpr int TPR = 4, DQ = D / TPR, BN = 32, NT = BWS_ROWS * TPR;
  __shared__ float qs[BN][D];
  __shared__ float gs[BN][D];
  __shared__ float ls[BN], dls[BN];
  const int J = blockIdx.x / (BLK / BWS_ROWS);
  const long long bh = blockIdx.y;
  const int tid = threadIdx.x, r = tid / TPR, u = tid % TPR;
  const int key = blockIdx.x * BWS_ROWS + r;
  const bool key_ok = key < N;
  const T* qb = q + bh * N * D;
  const T* gb = g + bh * N * D;
  float kr[DQ], vr[DQ], ak[DQ], av[DQ];
#pragma unroll
  for (int i = 0; i < DQ; ++i) {
    const long long at = (bh * N + key) * D + TPR * i + u;
    kr[i] = key_ok ? to_f32(k[at]) : 0.f;
    vr[i] = key_ok ? to_f32(v[at]) : 0.f;
    ak[i] = 0.f;
    av[i] = 0.f;
  }
  for (int e = t_ptr[J]; e < t_ptr[J + 1]; ++e) {
    const int qstart = t_row[e] * BLK;
    const int qcount = min(BLK, N - qstart);
    for (int s0 = 0; s0 < qcount; s0 += BN) {
      __syncthreads();
      for (int idx = tid; idx < BN * D; idx += NT) {
        const int ii = idx / D, c = idx % D;
        const bool ok = s0 + ii < qcount;
        const long long at = static_cast<long long>(qstart + s0 + ii) * D + c;
        qs[ii][c] = ok ? to_f32(qb[at]) : 0.f;
        gs[ii][c] = ok ? to_f32(gb[at]) : 0.f;
      }
      if (tid < BN) {
        // padded rows hold nlse2 = -inf and ndelta = 0
        ls[tid] = nlse2[bh * Np + qstart + s0 + tid];
        dls[tid] = ndelta[bh * Np + qstart + s0 + tid];
      }
      __syncthreads();
#pragma unroll 4
      for (int ii = 0; ii < BN; ++ii) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int i = 0; i < DQ; ++i) {
          s = fmaf(kr[i], qs[ii][TPR * i + u], s);
          dp = fmaf(vr[i], gs[ii][TPR * i + u], dp);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        dp += __shfl_xor_sync(0xffffffffu, dp, 1);
        dp += __shfl_xor_sync(0xffffffffu, dp, 2);
        const float p = exp2f(fmaf(s, scale_log2, ls[ii]));
        const float ds = p * (dp + dls[ii]);
#pragma unroll
        for (int i = 0; i < DQ; ++i) {
          av[i] = fmaf(p, gs[ii][TPR * i + u], av[i]);
          ak[i] = fmaf(ds, qs[ii][TPR * i + u], ak[i]);
        }
      }
    }
  }
  if (key_ok) {
    const long long at = (bh * N + key) * D;
#pragma unroll
    for (int i = 0; i < DQ; ++i) {
      dk[at + TPR * i + u] = from_f32<T>(ak[i] * scale);
      dv[at + TPR * i + u] = from_f32<T>(av[i]);
    }
  }
}

}  // namespace va
