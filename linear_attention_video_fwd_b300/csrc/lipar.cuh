// LIPAR inter-frame pruning and restoration (LIPAR summary, sec. 2 B):
// tokens whose latent patch barely differs from the same patch of the previous
// frame are dropped before attention and restored afterwards by duplicating
// the previous frame's result. Readings (the page gives no formulas), per
// batch of a latent x[b, t, h, w, :]:
//   changed(t, h, w) = t == 0 or max_c |x[t, h, w, c] - x[t-1, h, w, c]| >= tau
//   keep(t, h, w)    = t == 0 or changed somewhere in the 3 x 3 spatial
//                      neighbourhood of (h, w) in frame t (motion check)
//   order            = kept tokens in token order (the compacted sequence)
//   src(t, h, w)     = slot of (t, h, w) if kept, else src(t - 1, h, w)
// The largest channel difference is exact in float32, so the decisions do not
// depend on the order of any arithmetic. Every kernel is memory bound.
#pragma once

#include "common.cuh"

namespace va {

// changed[b][n]: one warp per token, the largest |x_t - x_{t-1}| over C
// channels against tau. Grid (ceil(N / 8), B), 256 threads.
template <typename T>
__global__ void lp_changed_kernel(const T* __restrict__ x, int N, int F, int C, float tau,
                                  uint8_t* __restrict__ changed) {
  const int b = blockIdx.y;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  uint8_t* ch = changed + static_cast<long long>(b) * N;
  if (n < F) {  // frame 0
    if (lane == 0) ch[n] = 1;
    return;
  }
  const T* cur = x + (static_cast<long long>(b) * N + n) * C;
  const T* prev = cur - static_cast<long long>(F) * C;
  float m = 0.f;
  for (int c = lane; c < C; c += 32) m = fmaxf(m, fabsf(to_f32(cur[c]) - to_f32(prev[c])));
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) ch[n] = m >= tau ? 1 : 0;
}

// keep[b][n] = frame 0, or a changed token in the 3 x 3 neighbourhood.
// Grid (ceil(N / 256), B), 256 threads.
__global__ void lp_keep_kernel(const uint8_t* __restrict__ changed, int N, int H, int W,
                               uint8_t* __restrict__ keep) {
  const int b = blockIdx.y;
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const int F = H * W;
  const uint8_t* ch = changed + static_cast<long long>(b) * N;
  uint8_t k = 1;
  if (n >= F) {
    const int s = n % F, h = s / W, w = s % W;
    const int base = n - s;
    k = 0;
    for (int dh = -1; dh <= 1; ++dh)
      for (int dw = -1; dw <= 1; ++dw) {
        const int hh = h + dh, ww = w + dw;
        if (hh >= 0 && hh < H && ww >= 0 && ww < W && ch[base + hh * W + ww]) k = 1;
      }
  }
  keep[static_cast<long long>(b) * N + n] = k;
}

// Compaction of one batch (one CTA of 1024 threads per batch): slot[n] = rank
// of n among the kept tokens (-1 if pruned), order[slot] = n, count[b].
__global__ void lp_compact_kernel(const uint8_t* __restrict__ keep, int N, int* __restrict__ slot,
                                  int* __restrict__ order, int* __restrict__ count) {
  __shared__ int part[1024];
  const int b = blockIdx.x, tid = threadIdx.x;
  const uint8_t* kp = keep + static_cast<long long>(b) * N;
  const int per = (N + 1023) / 1024;
  const int lo = min(N, tid * per), hi = min(N, lo + per);
  int c = 0;
  for (int n = lo; n < hi; ++n) c += kp[n];
  part[tid] = c;
  __syncthreads();
  for (int stride = 1; stride < 1024; stride <<= 1) {
    const int v = tid >= stride ? part[tid - stride] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int r = tid > 0 ? part[tid - 1] : 0;
  int* sl = slot + static_cast<long long>(b) * N;
  int* od = order + static_cast<long long>(b) * N;
  for (int n = lo; n < hi; ++n) {
    if (kp[n]) {
      sl[n] = r;
      od[r] = n;
      ++r;
    } else {
      sl[n] = -1;
    }
  }
  if (tid == 1023) count[b] = part[1023];
}

// src[b][n]: one thread per in-frame position walks the frames in order.
// Grid (ceil(F / 256), B), 256 threads.
__global__ void lp_src_kernel(const int* __restrict__ slot, int T, int F,
                              int* __restrict__ src) {
  const int b = blockIdx.y;
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= F) return;
  const long long base = static_cast<long long>(b) * T * F;
  int cur = 0;
  for (int t = 0; t < T; ++t) {
    const int sl = slot[base + static_cast<long long>(t) * F + s];
    if (sl >= 0) cur = sl;  // frame 0 is always kept, so cur is set at t = 0
    src[base + static_cast<long long>(t) * F + s] = cur;
  }
}

// out[b][h][k] = x[b][h][order[b][k]] for k < count[b]; rows of `row16`
// 16-byte words, one warp per row. Grid (ceil(N / 8), B * heads), 256 threads.
__global__ void lp_gather_kernel(const uint4* __restrict__ x, const int* __restrict__ order,
                                 const int* __restrict__ count, int heads, int N, int row16,
                                 uint4* __restrict__ out) {
  const int bh = blockIdx.y, b = bh / heads;
  const int k = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (k >= count[b]) return;
  const int n = order[static_cast<long long>(b) * N + k];
  const uint4* s = x + (static_cast<long long>(bh) * N + n) * row16;
  uint4* d = out + (static_cast<long long>(bh) * N + k) * row16;
  for (int i = lane; i < row16; i += 32) d[i] = s[i];
}

// out[b][h][n] = y[b][h][src[b][n]]; one warp per row.
// Grid (ceil(N / 8), B * heads), 256 threads.
__global__ void lp_restore_kernel(const uint4* __restrict__ y, const int* __restrict__ src,
                                  int heads, int N, int row16, uint4* __restrict__ out) {
  const int bh = blockIdx.y, b = bh / heads;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  const int k = src[static_cast<long long>(b) * N + n];
  const uint4* s = y + (static_cast<long long>(bh) * N + k) * row16;
  uint4* d = out + (static_cast<long long>(bh) * N + n) * row16;
  for (int i = lane; i < row16; i += 32) d[i] = s[i];
}

}  // namespace va
