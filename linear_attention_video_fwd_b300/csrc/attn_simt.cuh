// Block-sparse attention forward on the float32 FMA pipes.
//
// One CTA per (query block I, batch*head). Four threads share a query row;
// thread u of the row owns dims {4 i + u}, so the four threads read
// consecutive floats of a staged key/value row (no bank conflicts) and the
// eight rows of a warp read the same row (broadcast). Keys are streamed in
// sub-tiles of 32 through shared memory, in the order of the CSR row, with an
// online (running-max) softmax in float32 and exp2 of log2e-scaled logits.
// Keys j >= N of the last block are excluded.
#pragma once

#include "common.cuh"

namespace va {


template <typename T, int D, int BLK>
__global__ void __launch_bounds__(BLK * 4)
    attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const int* __restrict__ row_ptr, const int* __restrict__ col,
                     T* __restrict__ out, float* __restrict__ lse, int N, float scale_log2) {
  constexpr int TPR = 4;
  constexpr int DQ = D / TPR;
  constexpr int BN = 32;
  constexpr int NT = BLK * TPR;
  __shared__ float ks[BN][D];
  __shared__ float vs[BN][D];

  const int I = blockIdx.x;
  const long long bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int r = tid / TPR, u = tid % TPR;
  const int row = I * BLK + r;
  const bool row_ok = row < N;
  const T* qb = q + bh * N * D;
  const T* kb = k + bh * N * D;
  const T* vb = v + bh * N * D;

  float qr[DQ], o[DQ];
#pragma unroll
  for (int i = 0; i < DQ; ++i) {
    qr[i] = row_ok ? to_f32(qb[static_cast<long long>(row) * D + TPR * i + u]) : 0.f;
    o[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;

  const int beg = row_ptr[I], end = row_ptr[I + 1];
  for (int e = beg; e < end; ++e) {
    const int J = col[e];
    const int kstart = J * BLK;
    const int kcount = min(BLK, N - kstart);
    for (int s0 = 0; s0 < kcount; s0 += BN) {
      __syncthreads();
      for (int idx = tid; idx < BN * D; idx += NT) {
        const int jj = idx / D, c = idx % D;
        const int key = kstart + s0 + jj;
        const bool ok = s0 + jj < kcount;
        ks[jj][c] = ok ? to_f32(kb[static_cast<long long>(key) * D + c]) : 0.f;
        vs[jj][c] = ok ? to_f32(vb[static_cast<long long>(key) * D + c]) : 0.f;
      }
      __syncthreads();
      float s[BN];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < DQ; ++i) acc = fmaf(qr[i], ks[j][TPR * i + u], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        s[j] = (s0 + j < kcount) ? acc * scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
      const float m_new = fmaxf(m, mx);
      if (m_new == -INFINITY) continue;
      const float alpha = exp2f(m - m_new);  // 0 when m == -inf
      l *= alpha;
#pragma unroll
      for (int i = 0; i < DQ; ++i) o[i] *= alpha;
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        const float p = exp2f(s[j] - m_new);
        l += p;
#pragma unroll
        for (int i = 0; i < DQ; ++i) o[i] = fmaf(p, vs[j][TPR * i + u], o[i]);
      }
      m = m_new;
    }
  }

  if (row_ok) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T* ob = out + bh * N * D + static_cast<long long>(row) * D;
#pragma unroll
    for (int i = 0; i < DQ; ++i) ob[TPR * i + u] = from_f32<T>(o[i] * inv);
    if (lse != nullptr && u == 0) {
      lse[bh * N + row] = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    }
  }
}

}  // namespace va
