// Lloyd k-means per (batch, head) and per-cluster statistics, the clustering
// step of SVG-EAR's parameter-free linear compensation (SVG-EAR, gist.science
// 2603.08982, technical summary sec. 2, idea 1: queries and keys are grouped
// by semantic similarity; the page names no algorithm, Lloyd iteration on the
// raw head vectors with squared Euclidean distance is the reading used).
//
// One iteration: assign (nearest centroid, ties to the lowest index) ->
// counts -> offsets -> member lists -> means. The member sums are exact
// (64-bit fixed point for bf16 inputs, float64 for float32), so the centroids
// do not depend on the (atomic, unordered) member order.
#pragma once

#include "common.cuh"

namespace va {

// 16-byte load of CH = 16 / sizeof(T) consecutive elements, as floats.
template <typename T>
struct Chunk16 {
  static constexpr int CH = 16 / static_cast<int>(sizeof(T));
  __device__ __forceinline__ static void load(const T* src, float (&out)[16 / sizeof(T)]) {
    const uint4 raw = *reinterpret_cast<const uint4*>(src);
    if constexpr (sizeof(T) == 4) {
      out[0] = __uint_as_float(raw.x);
      out[1] = __uint_as_float(raw.y);
      out[2] = __uint_as_float(raw.z);
      out[3] = __uint_as_float(raw.w);
    } else {
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  }
};

// dstT[d * R + r] = row(r)[d] for r < R, d < D (zeros where row(r) is null).
// Consecutive threads take consecutive rows, so the shared-memory writes are
// conflict-free; each thread reads 16 bytes of one row.
template <typename T, int D, int R, int NT, typename RowFn>
__device__ __forceinline__ void stage_transposed(float* dstT, RowFn row) {
  constexpr int CH = Chunk16<T>::CH;
  for (int e = threadIdx.x; e < R * (D / CH); e += NT) {
    const int r = e % R, ch = e / R;
    const T* src = row(r);
    float f[CH];
    if (src != nullptr) {
      Chunk16<T>::load(src + ch * CH, f);
    } else {
#pragma unroll
      for (int i = 0; i < CH; ++i) f[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) dstT[(ch * CH + i) * R + r] = f[i];
  }
}

// dst[r * D + d] = row(r)[d] (row-major, zeros where row(r) is null).
template <typename T, int D, int R, int NT, typename RowFn>
__device__ __forceinline__ void stage_rows(float* dst, RowFn row) {
  constexpr int CH = Chunk16<T>::CH;
  for (int e = threadIdx.x; e < R * (D / CH); e += NT) {
    const int r = e / (D / CH), ch = e % (D / CH);
    const T* src = row(r);
    float f[CH];
    if (src != nullptr) {
      Chunk16<T>::load(src + ch * CH, f);
    } else {
#pragma unroll
      for (int i = 0; i < CH; ++i) f[i] = 0.f;
    }
    float4* d4 = reinterpret_cast<float4*>(dst + r * D + ch * CH);
#pragma unroll
    for (int i = 0; i < CH / 4; ++i)
      d4[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
  }
}

constexpr int KM_THREADS = 256;
constexpr int KM_PT = 64;  // points per CTA
constexpr int KM_CT = 64;  // centroids per inner tile

// assign[i] = argmin_c (|c|^2 - 2 x_i . c) over c < C (|x_i|^2 is common to
// all c); ties -> lowest c. count[assign[i]] += 1 (count zeroed by the caller).
// Grid: (ceil(N / KM_PT), BH). x: [BH, N, D], cent: [BH, C, D] fp32,
// cnorm: [BH, C] fp32 (|c|^2).
template <typename T, int D>
__global__ void __launch_bounds__(KM_THREADS)
    km_assign_kernel(const T* __restrict__ x, const float* __restrict__ cent,
                     const float* __restrict__ cnorm, int N, int C, int* __restrict__ assign,
                     int* __restrict__ count) {
  extern __shared__ float km_smem[];
  float* xT = km_smem;                 // [D][KM_PT]
  float* cT = km_smem + D * KM_PT;     // [D][KM_CT]
  const int bh = blockIdx.y;
  const int i0 = blockIdx.x * KM_PT;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const T* xb = x + static_cast<long long>(bh) * N * D;
  const float* cb = cent + static_cast<long long>(bh) * C * D;
  const float* nb = cnorm + static_cast<long long>(bh) * C;

  // stage the point tile transposed: xT[d][p]
  stage_transposed<T, D, KM_PT, KM_THREADS>(xT, [&](int p) -> const T* {
    return i0 + p < N ? xb + static_cast<long long>(i0 + p) * D : nullptr;
  });
  float best[4];
  int besti[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    best[a] = INFINITY;
    besti[a] = 0x7fffffff;
  }
  for (int c0 = 0; c0 < C; c0 += KM_CT) {
    __syncthreads();
    stage_transposed<float, D, KM_CT, KM_THREADS>(cT, [&](int c) -> const float* {
      return c0 + c < C ? cb + static_cast<long long>(c0 + c) * D : nullptr;
    });
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
    for (int dd = 0; dd < D; ++dd) {
      const float4 xv = *reinterpret_cast<const float4*>(&xT[dd * KM_PT + ty * 4]);
      const float4 cv = *reinterpret_cast<const float4*>(&cT[dd * KM_CT + tx * 4]);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
      const float ca[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xa[a], ca[b], acc[a][b]);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int c = c0 + tx * 4 + b;
      if (c < C) {
        const float cn = nb[c];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float dist = fmaf(-2.f, acc[a][b], cn);
          if (dist < best[a]) {  // clusters visited in ascending order per thread
            best[a] = dist;
            besti[a] = c;
          }
        }
      }
    }
  }
  // reduce over the 16 threads (tx) that share these 4 points
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    float bv = best[a];
    int bi = besti[a];
#pragma unroll
    for (int o = 8; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov < bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    const int i = i0 + ty * 4 + a;
    if (tx == 0 && i < N) {
      assign[static_cast<long long>(bh) * N + i] = bi;
      atomicAdd(&count[static_cast<long long>(bh) * C + bi], 1);
    }
  }
}

// Exclusive scan of count[bh][0..C) into off[bh][0..C] (off[C] = N) and a
// zeroed fill cursor. One CTA per bh, 1024 threads.
__global__ void km_offsets_kernel(const int* __restrict__ count, int C, int* __restrict__ off,
                                  int* __restrict__ fill) {
  __shared__ int part[1024];
  const int bh = blockIdx.x, tid = threadIdx.x;
  const int* cnt = count + static_cast<long long>(bh) * C;
  int* o = off + static_cast<long long>(bh) * (C + 1);
  const int per = (C + 1023) / 1024;
  const int lo = min(C, tid * per), hi = min(C, lo + per);
  int s = 0;
  for (int c = lo; c < hi; ++c) s += cnt[c];
  part[tid] = s;
  __syncthreads();
  for (int stride = 1; stride < 1024; stride <<= 1) {
    const int v = tid >= stride ? part[tid - stride] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int base = tid > 0 ? part[tid - 1] : 0;
  for (int c = lo; c < hi; ++c) {
    o[c] = base;
    base += cnt[c];
    fill[static_cast<long long>(bh) * C + c] = 0;
  }
  if (tid == 1023) o[C] = part[1023];
}

// perm[off[a_i] + k] = i (member lists; order within a cluster unspecified).
// Assignment values outside [0, C) are reported as VA_ERR_DEVICE and skipped.
// Lanes of a warp with the same cluster take their slots with one atomic
// (neighbouring tokens often share a cluster). Whole warps: blockDim is a
// multiple of 32.
__global__ void km_scatter_kernel(const int* __restrict__ assign, int N, int C,
                                  const int* __restrict__ off, int* __restrict__ fill,
                                  int* __restrict__ perm) {
  const int bh = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool inr = i < N;
  const int a = inr ? assign[static_cast<long long>(bh) * N + i] : -1;
  const bool valid = inr && a >= 0 && a < C;
  if (inr && !valid) raise_error(VA_ERR_DEVICE);
  const unsigned grp = __match_any_sync(0xffffffffu, valid ? a : -1);
  if (!valid) return;
  const int leader = __ffs(grp) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(&fill[static_cast<long long>(bh) * C + a], __popc(grp));
  base = __shfl_sync(grp, base, leader);
  const int pos = off[static_cast<long long>(bh) * (C + 1) + a] + base +
                  __popc(grp & ((1u << lane) - 1u));
  perm[static_cast<long long>(bh) * N + pos] = i;
}

// Stable member lists: perm[off[a] + k] = the k-th member of cluster a in
// ascending token order, so that everything summed over a member list (fp32
// means, probe and attention accumulations) is the same on every call. Tiles
// of KS_TILE tokens: per-tile member counts, a scan of those counts down the
// tiles of each cluster, then one warp per tile placing its tokens in order.
// base is [BH][ntiles][C]. Assignment values outside [0, C) are reported as
// VA_ERR_DEVICE and skipped.
constexpr int KS_TILE = 1024;

__global__ void __launch_bounds__(256) km_tile_count_kernel(const int* __restrict__ assign, int N,
                                                            int C, int* __restrict__ base) {
  extern __shared__ int hist[];  // [C]
  const int bh = blockIdx.y, tile = blockIdx.x, ntiles = gridDim.x;
  for (int c = threadIdx.x; c < C; c += blockDim.x) hist[c] = 0;
  __syncthreads();
  const int i0 = tile * KS_TILE, i1 = min(N, i0 + KS_TILE);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const int a = assign[static_cast<long long>(bh) * N + i];
    if (a >= 0 && a < C) {
      atomicAdd(&hist[a], 1);
    } else {
      raise_error(VA_ERR_DEVICE);
    }
  }
  __syncthreads();
  int* row = base + (static_cast<long long>(bh) * ntiles + tile) * C;
  for (int c = threadIdx.x; c < C; c += blockDim.x) row[c] = hist[c];
}

// In place: base[t][c] <- off[c] + sum over tiles t' < t of count[t'][c].
__global__ void km_tile_scan_kernel(const int* __restrict__ off, int C, int ntiles,
                                    int* __restrict__ base) {
  const int bh = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  int run = off[static_cast<long long>(bh) * (C + 1) + c];
  int* col = base + static_cast<long long>(bh) * ntiles * C + c;
  for (int t0 = 0; t0 < ntiles; t0 += 8) {
    int v[8];  // eight loads in flight before the stores
#pragma unroll
    for (int j = 0; j < 8; ++j)
      v[j] = t0 + j < ntiles ? col[static_cast<long long>(t0 + j) * C] : 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (t0 + j < ntiles) col[static_cast<long long>(t0 + j) * C] = run;
      run += v[j];
    }
  }
}

__global__ void __launch_bounds__(128) km_tile_place_kernel(const int* __restrict__ assign, int N,
                                                            int C,
                                                            const int* __restrict__ base,
                                                            int* __restrict__ perm) {
  extern __shared__ int next[];  // [C]: next free slot of each cluster
  const int bh = blockIdx.y, tile = blockIdx.x, ntiles = gridDim.x;
  const int* row = base + (static_cast<long long>(bh) * ntiles + tile) * C;
  for (int c = threadIdx.x; c < C; c += blockDim.x) next[c] = row[c];
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int i0 = tile * KS_TILE, i1 = min(N, i0 + KS_TILE);
  for (int i = i0 + lane; i - lane < i1; i += 32) {
    const bool inr = i < i1;
    const int a = inr ? assign[static_cast<long long>(bh) * N + i] : -1;
    const bool valid = inr && a >= 0 && a < C;
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? a : -1);
    const int leader = __ffs(grp) - 1;
    int pos = 0;
    if (valid) {
      pos = next[a] + __popc(grp & ((1u << lane) - 1u));
      perm[static_cast<long long>(bh) * N + pos] = i;
    }
    __syncwarp();
    if (valid && lane == leader) next[a] += __popc(grp);
    __syncwarp();
  }
}

// Histogram of an externally supplied assignment (range-checked).
__global__ void km_count_kernel(const int* __restrict__ assign, int N, int C,
                                int* __restrict__ count) {
  const int bh = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool inr = i < N;
  const int a = inr ? assign[static_cast<long long>(bh) * N + i] : -1;
  const bool valid = inr && a >= 0 && a < C;
  if (inr && !valid) raise_error(VA_ERR_DEVICE);
  const unsigned grp = __match_any_sync(0xffffffffu, valid ? a : -1);
  if (valid && lane == __ffs(grp) - 1)
    atomicAdd(&count[static_cast<long long>(bh) * C + a], __popc(grp));
}

// A bf16 value as a signed fixed-point integer with 32 fraction bits: exact
// for |x| >= 2^-25, truncated toward zero (error < 2^-32) below, for
// |x| < 2^31. value = mant * 2^(e - 134), so the magnitude is mant shifted
// by e - 102; PTX shifts clamp counts past the width, so a tiny value shifts
// out to 0 and zero / subnormal inputs (e = 0) are masked to 0.
__device__ __forceinline__ long long bf16_fixed32(uint32_t bits16) {
  const uint32_t e = (bits16 >> 7) & 0xFFu;
  const uint32_t mant = ((bits16 & 0x7Fu) | 0x80u) & (e != 0 ? 0xFFu : 0u);
  const int sh = static_cast<int>(e) - 102;
  unsigned long long mag;
  if (sh >= 0) {
    asm("shl.b64 %0, %1, %2;" : "=l"(mag) : "l"(static_cast<unsigned long long>(mant)), "r"(sh));
  } else {
    uint32_t m32;
    asm("shr.u32 %0, %1, %2;" : "=r"(m32) : "r"(mant), "r"(-sh));
    mag = m32;
  }
  const long long sg = static_cast<long long>(static_cast<int>(bits16 << 16) >> 31);  // 0 or -1
  return (static_cast<long long>(mag) ^ sg) - sg;
}

// One warp per cluster: mean of its members, written as fp32 to mean[bh][c];
// |mean|^2 (fp32) to norm[bh][c] if norm != nullptr. An empty cluster keeps
// mean[bh][c] when keep_empty, else gets zeros. Sums are exact and
// order-independent: 64-bit fixed point for bf16 (members with |x| < 2^-25
// contribute with an error below 2^-32; |sum| must stay below 2^31), float64
// for float32. The bf16 mean is the fp32 sum divided in fp32 (within one ulp
// of the exact mean). Member indices are fetched 32 at a time so the row loads of a
// cluster are independent. Grid: (ceil(C / 8), BH), 256 threads.
template <typename T, int D>
__global__ void km_means_kernel(const T* __restrict__ x, int N, int C,
                                const int* __restrict__ off, const int* __restrict__ perm,
                                float* __restrict__ mean, float* __restrict__ norm,
                                int keep_empty) {
  constexpr int PER = D / 32;
  constexpr bool kFixed = sizeof(T) == 2;
  const int bh = blockIdx.y;
  const int c = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (c >= C) return;
  const int* o = off + static_cast<long long>(bh) * (C + 1);
  const int beg = o[c], end = o[c + 1];
  const int* pm = perm + static_cast<long long>(bh) * N;
  const T* xb = x + static_cast<long long>(bh) * N * D;
  float* m = mean + (static_cast<long long>(bh) * C + c) * D;
  long long iacc[PER];
  double dacc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    iacc[e] = 0;
    dacc[e] = 0.0;
  }
  for (int t0 = beg; t0 < end; t0 += 32) {
    const int my = (t0 + lane < end) ? pm[t0 + lane] : 0;
    const int cnt = min(32, end - t0);
#pragma unroll 4
    for (int q = 0; q < cnt; ++q) {
      const int idx = __shfl_sync(0xffffffffu, my, q);
      const T* row = xb + static_cast<long long>(idx) * D + lane * PER;
      if constexpr (kFixed) {
        const uint16_t* r16 = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
        for (int e = 0; e < PER; ++e) iacc[e] += bf16_fixed32(r16[e]);
      } else {
#pragma unroll
        for (int e = 0; e < PER; ++e) dacc[e] += static_cast<double>(to_f32(row[e]));
      }
    }
  }
  float nrm = 0.f;
  if (end > beg) {
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      // fixed point: the exact sum rounded to fp32, then an IEEE fp32 division
      // (at most one ulp from the exact mean; no fp64 on the bf16 path, whose
      // rate is a small fraction of fp32's on this part)
      const float mv =
          kFixed ? __fdiv_rn(static_cast<float>(iacc[e]) * 0x1p-32f, static_cast<float>(end - beg))
                 : static_cast<float>(dacc[e] / static_cast<double>(end - beg));
      m[lane * PER + e] = mv;
      nrm = fmaf(mv, mv, nrm);
    }
  } else {
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      float mv = keep_empty ? m[lane * PER + e] : 0.f;
      if (!keep_empty) m[lane * PER + e] = 0.f;
      nrm = fmaf(mv, mv, nrm);
    }
  }
  if (norm != nullptr) {
#pragma unroll
    for (int o2 = 16; o2; o2 >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, o2);
    if (lane == 0) norm[static_cast<long long>(bh) * C + c] = nrm;
  }
}

// Member sums of bf16 points as 64-bit fixed point (bf16_fixed32), balanced:
// warp g sums the 32 cluster-ordered points perm[32g .. 32g + 31] of its
// (batch, head), splitting at cluster changes, and adds each run into
// sums[bh][c][0..D) with 64-bit integer atomics (exact, so the result does not
// depend on the order). sums must be zeroed. Grid (ceil(N / 256), BH), 256
// threads.
template <int D>
__global__ void km_sum_kernel(const __nv_bfloat16* __restrict__ x, int N, int C,
                              const int* __restrict__ perm, const int* __restrict__ assign,
                              unsigned long long* __restrict__ sums) {
  constexpr int PER = D / 32;
  const int bh = blockIdx.y;
  const int t0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * 32;
  const int lane = threadIdx.x & 31;
  if (t0 >= N) return;
  const long long nb = static_cast<long long>(bh) * N;
  const int my = t0 + lane < N ? perm[nb + t0 + lane] : 0;
  const int myc = t0 + lane < N ? assign[nb + my] : -1;
  const int cnt = min(32, N - t0);
  const uint16_t* xb = reinterpret_cast<const uint16_t*>(x) + nb * D + lane * PER;
  long long acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0;
  int cur = __shfl_sync(0xffffffffu, myc, 0);
  for (int q = 0; q < cnt; ++q) {
    const int idx = __shfl_sync(0xffffffffu, my, q);
    const int c = __shfl_sync(0xffffffffu, myc, q);
    if (c != cur) {
      if (cur >= 0 && cur < C) {
        unsigned long long* dst = sums + (static_cast<long long>(bh) * C + cur) * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) atomicAdd(dst + e, static_cast<unsigned long long>(acc[e]));
      }
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = 0;
      cur = c;
    }
    // the lane's PER consecutive bf16 values in one 4- or 8-byte load
    const uint32_t* row = reinterpret_cast<const uint32_t*>(xb + static_cast<long long>(idx) * D);
    uint32_t w[PER / 2];
    if constexpr (PER == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(row);
      w[0] = v.x;
      w[1] = v.y;
    } else {
#pragma unroll
      for (int i = 0; i < PER / 2; ++i) w[i] = row[i];
    }
#pragma unroll
    for (int i = 0; i < PER / 2; ++i) {
      acc[2 * i] += bf16_fixed32(w[i] & 0xffffu);
      acc[2 * i + 1] += bf16_fixed32(w[i] >> 16);
    }
  }
  if (cur >= 0 && cur < C) {
    unsigned long long* dst = sums + (static_cast<long long>(bh) * C + cur) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) atomicAdd(dst + e, static_cast<unsigned long long>(acc[e]));
  }
}

// Incremental member sums: for every point whose cluster changed from prev to
// assign, its 64-bit fixed-point row (bf16_fixed32) is added to the new
// cluster's sum and subtracted from the old one, and prev takes the new
// cluster. Integer arithmetic keeps the sums exactly equal to a full
// recomputation, in any order. Warp g handles points 32g .. 32g + 31 of its
// (batch, head) in token order. Grid (ceil(N / 256), BH), 256 threads.
template <int D>
__global__ void km_delta_kernel(const __nv_bfloat16* __restrict__ x, int N, int C,
                                int* __restrict__ prev, const int* __restrict__ assign,
                                unsigned long long* __restrict__ sums) {
  constexpr int PER = D / 32;
  const int bh = blockIdx.y;
  const int t0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * 32;
  const int lane = threadIdx.x & 31;
  if (t0 >= N) return;
  const long long nb = static_cast<long long>(bh) * N;
  const int i = t0 + lane;
  int an = 0, ao = 0;
  bool moved = false;
  if (i < N) {
    an = assign[nb + i];
    ao = prev[nb + i];
    moved = an != ao;
    if (moved && (an < 0 || an >= C || ao < 0 || ao >= C)) {
      raise_error(VA_ERR_DEVICE);
      moved = false;
    }
    if (moved) prev[nb + i] = an;
  }
  const uint16_t* xb = reinterpret_cast<const uint16_t*>(x) + nb * D + lane * PER;
  for (unsigned m = __ballot_sync(0xffffffffu, moved); m; m &= m - 1) {
    const int q = __ffs(m) - 1;
    const int cn = __shfl_sync(0xffffffffu, an, q), co = __shfl_sync(0xffffffffu, ao, q);
    const uint32_t* row = reinterpret_cast<const uint32_t*>(xb + static_cast<long long>(t0 + q) * D);
    unsigned long long* dn = sums + (static_cast<long long>(bh) * C + cn) * D + lane * PER;
    unsigned long long* dold = sums + (static_cast<long long>(bh) * C + co) * D + lane * PER;
#pragma unroll
    for (int w = 0; w < PER / 2; ++w) {
      const uint32_t v = row[w];
      const long long lo = bf16_fixed32(v & 0xffffu), hi = bf16_fixed32(v >> 16);
      atomicAdd(dn + 2 * w, static_cast<unsigned long long>(lo));
      atomicAdd(dn + 2 * w + 1, static_cast<unsigned long long>(hi));
      atomicAdd(dold + 2 * w, static_cast<unsigned long long>(-lo));
      atomicAdd(dold + 2 * w + 1, static_cast<unsigned long long>(-hi));
    }
  }
}

// mean[bh][c] = sums / count (fp32), |mean|^2 to norm (if non-null), and the
// bf16 split hi = bf16(mean), lo = bf16(mean - hi) (if non-null). An empty
// cluster keeps mean (and its split) when keep_empty, else gets zeros.
// One warp per cluster; grid (ceil(C / 8), BH), 256 threads.
template <int D>
__global__ void km_finalize_kernel(const unsigned long long* __restrict__ sums,
                                   const int* __restrict__ count, int C, float* __restrict__ mean,
                                   float* __restrict__ norm, __nv_bfloat16* __restrict__ hi,
                                   __nv_bfloat16* __restrict__ lo, int keep_empty) {
  constexpr int PER = D / 32;
  const int bh = blockIdx.y;
  const int c = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (c >= C) return;
  const long long row = (static_cast<long long>(bh) * C + c) * D + lane * PER;
  const int n = count[static_cast<long long>(bh) * C + c];
  float nrm = 0.f;
  if (n > 0 || !keep_empty) {
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      // exact fixed-point sum rounded to fp32, then an IEEE fp32 division
      const float mv =
          n > 0 ? __fdiv_rn(static_cast<float>(static_cast<long long>(sums[row + e])) * 0x1p-32f,
                            static_cast<float>(n))
                : 0.f;
      mean[row + e] = mv;
      nrm = fmaf(mv, mv, nrm);
      if (hi != nullptr) {
        const __nv_bfloat16 h = __float2bfloat16_rn(mv);
        hi[row + e] = h;
        lo[row + e] = __float2bfloat16_rn(mv - __bfloat162float(h));
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < PER; ++e) nrm = fmaf(mean[row + e], mean[row + e], nrm);
  }
  if (norm != nullptr) {
#pragma unroll
    for (int o2 = 16; o2; o2 >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, o2);
    if (lane == 0) norm[static_cast<long long>(bh) * C + c] = nrm;
  }
}

// Initial centroids: cent[bh][c] = x[bh][init[bh][c]] (fp32), |c|^2 to cnorm.
// Indices outside [0, N) are reported as VA_ERR_DEVICE (the row is zeroed).
// One warp per centroid; grid (ceil(C / 8), BH).
// Warm start: cent = c0 (skipped when they alias) and cnorm = |c0|^2, with
// the same per-lane order of accumulation as km_init_kernel, so a warm start
// from the float copies of the seed rows reproduces a seeded run exactly.
// Grid (ceil(C / 8), BH), 256 threads.
template <int D>
__global__ void km_warm_kernel(const float* __restrict__ c0, int C, float* __restrict__ cent,
                               float* __restrict__ cnorm) {
  constexpr int PER = D / 32;
  const int bh = blockIdx.y;
  const int c = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (c >= C) return;
  const long long row = (static_cast<long long>(bh) * C + c) * D + lane * PER;
  float nrm = 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const float v = c0[row + e];
    if (c0 != cent) cent[row + e] = v;
    nrm = fmaf(v, v, nrm);
  }
#pragma unroll
  for (int o2 = 16; o2; o2 >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, o2);
  if (lane == 0) cnorm[static_cast<long long>(bh) * C + c] = nrm;
}

template <typename T, int D>
__global__ void km_init_kernel(const T* __restrict__ x, const int* __restrict__ init, int N,
                               int C, float* __restrict__ cent, float* __restrict__ cnorm) {
  constexpr int PER = D / 32;
  const int bh = blockIdx.y;
  const int c = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (c >= C) return;
  const int idx = init[static_cast<long long>(bh) * C + c];
  const bool ok = idx >= 0 && idx < N;
  if (!ok && lane == 0) raise_error(VA_ERR_DEVICE);
  float* m = cent + (static_cast<long long>(bh) * C + c) * D;
  const T* row = x + (static_cast<long long>(bh) * N + (ok ? idx : 0)) * D;
  float nrm = 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const float v = ok ? to_f32(row[lane * PER + e]) : 0.f;
    m[lane * PER + e] = v;
    nrm = fmaf(v, v, nrm);
  }
#pragma unroll
  for (int o2 = 16; o2; o2 >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, o2);
  if (lane == 0) cnorm[static_cast<long long>(bh) * C + c] = nrm;
}

}  // namespace va
