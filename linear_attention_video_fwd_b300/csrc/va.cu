// libva: C ABI of the block-sparse video attention library (see include/va.h).
// One translation unit: the kernels live in the headers included below.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>
#include <type_traits>
#include <vector>
#include <utility>

#include "va.h"
#include "common.cuh"
#include "mask.cuh"
#include "attn_simt.cuh"
#include "attn_tc.cuh"
#include "svgear.cuh"
#include "kmeans_tc.cuh"
#include "comp_tc.cuh"
#include "probe_tc.cuh"
#include "linear_tc.cuh"
#include "lipar.cuh"
#include "attn_bwd_simt.cuh"
#include "attn_bwd_tc.cuh"

#define VA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

int64_t g_wait_limit = 4000000000LL;

// Scratch memory pool of the library, one per device: stream-ordered, and
// with no release threshold, so memory freed at the end of a call stays
// mapped for the next one instead of going back to the driver at every
// synchronisation (the pool keeps the peak scratch of the process).
cudaMemPool_t scratch_pool() {
  static cudaMemPool_t pools[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (pools[dev] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    uint64_t keep = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    pools[dev] = pool;
  }
  return pools[dev];
}

struct Scoped {
  // Stream-ordered scratch allocations released at scope exit.
  cudaStream_t s;
  static constexpr int kCap = 64;
  void* ptrs[kCap];
  int n = 0;
  explicit Scoped(cudaStream_t st) : s(st) {}
  ~Scoped() {
    for (int i = 0; i < n; ++i) cudaFreeAsync(ptrs[i], s);
  }
  template <typename T>
  int alloc(T** p, size_t count) {
    *p = nullptr;
    if (count == 0) count = 1;
    if (fault_injected()) return VA_ERR_OOM;
    if (n >= kCap) return VA_ERR_OOM;
    void* raw = nullptr;
    cudaMemPool_t pool = scratch_pool();
    cudaError_t e = pool != nullptr ? cudaMallocFromPoolAsync(&raw, count * sizeof(T), pool, s)
                                    : cudaMallocAsync(&raw, count * sizeof(T), s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? VA_ERR_OOM : VA_ERR_CUDA;
    }
    ptrs[n++] = raw;
    *p = static_cast<T*>(raw);
    return VA_OK;
  }
  // VA_FAULT_INJECT=alloc makes every scratch allocation fail (host-side
  // fault injection for the error paths).
  static bool fault_injected() {
    const char* f = std::getenv("VA_FAULT_INJECT");
    return f != nullptr && std::strstr(f, "alloc") != nullptr;
  }
};

// One-time configuration of a device (kernel attributes, SM counts), run
// under a lock so that host threads calling concurrently neither race on the
// flags nor launch before the attributes are set. A failed configuration is
// retried on the next call.
struct DeviceOnce {
  std::mutex mu;
  std::atomic<bool> done[64];
};

template <typename Fn>
int device_once(DeviceOnce& once, int dev, Fn&& fn) {
  if (dev < 0 || dev >= 64) return VA_ERR_UNSUPPORTED;
  if (once.done[dev].load(std::memory_order_acquire)) return VA_OK;
  std::lock_guard<std::mutex> lock(once.mu);
  if (once.done[dev].load(std::memory_order_relaxed)) return VA_OK;
  const int st = fn();
  if (st == VA_OK) once.done[dev].store(true, std::memory_order_release);
  return st;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return VA_OK;
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? VA_ERR_OOM : VA_ERR_CUDA;
}

int launch_status() { return cuda_status(cudaGetLastError()); }

// Launch `kernel` as a programmatic dependent of the previous kernel on `s`:
// it may be scheduled before that kernel completes, and must itself execute
// griddepcontrol.wait before touching that kernel's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  }
  return fn;
}

// 3-D map over a [BH, N, D] bf16 tensor: box of 64 dims x box_rows rows x 1
// head, 128-byte swizzle; rows beyond N read as zeros.
int encode_bf16_rows_box(CUtensorMap* map, const void* base, int BH, int N, int D, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return VA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VA_OK : VA_ERR_CUDA;
}

// 3-D map over a [BH, N, D] bf16 tensor: box of 64 dims x 128 rows x 1 head,
// 128-byte swizzle; rows beyond N read as zeros.
int encode_bf16_rows(CUtensorMap* map, const void* base, int BH, int N, int D) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return VA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VA_OK : VA_ERR_CUDA;
}

}  // namespace

struct va_mask {
  int kind, T, H, W, N, step;
  va_mask_params p;
  int nqb;
  int64_t nnz, live_pairs;
  int32_t* row_ptr = nullptr;  // device [nqb + 1]
  int32_t* col = nullptr;      // device [nnz]
  int32_t* order = nullptr;    // device [nqb]: rows by descending length
  // query-block pairs {2P, 2P+1} for the two-tile tensor-core kernel
  int npairs = 0;
  int32_t* pcol = nullptr;     // device [nnz]: merged rows, entry J << 2 | live bits
  int32_t* plen = nullptr;     // device [npairs]: merged length per pair
  int32_t* porder = nullptr;   // device [npairs]: pairs by descending work
  // 64-token blocks only: quads of query blocks {4Q .. 4Q + 3} over pairs of
  // key blocks for the two-tile tensor-core kernel (quad_merge_kernel)
  int nquads = 0;
  int32_t* qcol = nullptr;     // device [nnz]: entry J' << 10 | sub bits << 2 | tile bits
  int32_t* qlen = nullptr;     // device [nquads]
  int32_t* qorder = nullptr;   // device [nquads]: quads by descending work
  // transposed lists for the backward: for key block J, the query blocks
  // that see it (ascending), and key blocks by descending list length
  int32_t* t_ptr = nullptr;    // device [nqb + 1]
  int32_t* t_row = nullptr;    // device [nnz]
  int32_t* t_order = nullptr;  // device [nqb]
  // 64-token blocks only: coarse pairs for the tensor-core backward
  // (coarse_pair_merge_kernel): query-block pairs over key-block pairs (dq)
  // and key-block pairs over query-block pairs (dk, dv); entry c << 4 | sub
  int32_t* cq_col = nullptr;   // device [nnz], rows start at row_ptr[2R]
  int32_t* cq_len = nullptr;   // device [ceil(nqb / 2)]
  int32_t* cq_order = nullptr;
  int32_t* ck_col = nullptr;   // device [nnz], rows start at t_ptr[2R]
  int32_t* ck_len = nullptr;
  int32_t* ck_order = nullptr;
  int device = 0;
};

namespace {

// A mask's arrays live on the device it was built on: a kernel running on
// another device must not be handed them.
int check_mask_device(const va_mask* m) {
  int dev = 0;
  const int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  return dev == m->device ? VA_OK : VA_ERR_INVALID;
}

// Mask limits shared by both builds: at most VA_MASK_MAX_BLOCKS blocks per
// side (the count and fill kernels test every block pair), and int32 CSR
// offsets, so at most INT32_MAX live block pairs.
constexpr int64_t kMaxMaskNnz = 0x7fffffffLL;

}  // namespace

VA_EXPORT int va_version(void) { return 100; }

VA_EXPORT int va_csr_validate(const int32_t* row_ptr, const int32_t* col_idx, int nqb, int64_t nnz,
                              int require_diagonal) {
  if (row_ptr == nullptr || nqb < 1 || nnz < 0 || (nnz > 0 && col_idx == nullptr))
    return VA_ERR_INVALID;
  if (row_ptr[0] != 0 || static_cast<int64_t>(row_ptr[nqb]) != nnz) return VA_ERR_DEVICE;
  for (int i = 0; i < nqb; ++i) {
    const int32_t b = row_ptr[i], e = row_ptr[i + 1];
    if (e < b || static_cast<int64_t>(e) > nnz) return VA_ERR_DEVICE;
    bool diag = false;
    for (int32_t p = b; p < e; ++p) {
      const int32_t c = col_idx[p];
      if (c < 0 || c >= nqb || (p > b && c <= col_idx[p - 1])) return VA_ERR_DEVICE;
      diag = diag || c == i;
    }
    if (require_diagonal && !diag) return VA_ERR_DEVICE;
  }
  return VA_OK;
}

namespace {

// VA_CHECKED=1 makes every mask build copy its lists back and validate them
// on the host: the rows and the transposed lists as CSR (with the diagonal,
// which every rule of the library keeps), and the transposed lists as the
// exact transpose of the rows.
bool checked_mode() {
  const char* f = std::getenv("VA_CHECKED");
  return f != nullptr && f[0] != '\0' && f[0] != '0';
}

int validate_mask(const va_mask* m) {
  const int nb = m->nqb;
  const int64_t nnz = m->nnz;
  std::vector<int32_t> rp(nb + 1), col(nnz > 0 ? nnz : 1), tp(nb + 1), tr(nnz > 0 ? nnz : 1);
  int st;
  if ((st = cuda_status(cudaMemcpy(rp.data(), m->row_ptr, sizeof(int32_t) * (nb + 1),
                                   cudaMemcpyDeviceToHost))) ||
      (st = cuda_status(cudaMemcpy(tp.data(), m->t_ptr, sizeof(int32_t) * (nb + 1),
                                   cudaMemcpyDeviceToHost))))
    return st;
  if (nnz > 0 &&
      ((st = cuda_status(cudaMemcpy(col.data(), m->col, sizeof(int32_t) * nnz,
                                    cudaMemcpyDeviceToHost))) ||
       (st = cuda_status(cudaMemcpy(tr.data(), m->t_row, sizeof(int32_t) * nnz,
                                    cudaMemcpyDeviceToHost)))))
    return st;
  if ((st = va_csr_validate(rp.data(), col.data(), nb, nnz, 1)) ||
      (st = va_csr_validate(tp.data(), tr.data(), nb, nnz, 1)))
    return st;
  // transpose check: count of (i, j) in rows == count of (j, i) in columns
  std::vector<int32_t> fill(tp.begin(), tp.end() - 1);
  for (int i = 0; i < nb; ++i)
    for (int32_t p = rp[i]; p < rp[i + 1]; ++p) {
      const int32_t j = col[p];
      if (fill[j] >= tp[j + 1] || tr[fill[j]] != i) return VA_ERR_DEVICE;
      ++fill[j];
    }
  return VA_OK;
}

}  // namespace

VA_EXPORT const char* va_status_string(int status) {
  switch (status) {
    case VA_OK: return "ok";
    case VA_ERR_INVALID: return "invalid argument";
    case VA_ERR_UNSUPPORTED: return "unsupported configuration";
    case VA_ERR_CUDA: return "CUDA runtime error";
    case VA_ERR_OOM: return "device allocation failed";
    case VA_ERR_TIMEOUT: return "device-side wait timed out";
    case VA_ERR_DEVICE: return "device-side bounds check failed";
    default: return "unknown status";
  }
}

VA_EXPORT int va_set_wait_limit(int64_t cycles) {
  if (cycles < 1000) return VA_ERR_INVALID;
  g_wait_limit = cycles;
  return VA_OK;
}

VA_EXPORT int va_device_error(va_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  int word = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&word, va::g_err_word, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaMemcpyToSymbol(va::g_err_word, &zero, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  return word;
}

VA_EXPORT int va_selftest_wait_timeout(int64_t cycles, va_stream_t stream) {
  if (cycles < 1000 || cycles > 10000000000LL) return VA_ERR_INVALID;
  va::wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(cycles);
  return launch_status();
}

// ------------------------------------------------------------------ masks --

namespace {

// Host checks shared by the mask entries: kind, grid and parameters. Sets the
// token count N and the block count nb; the callers apply their block limits.
int mask_grid_args(int kind, int T, int H, int W, const va_mask_params& p, int64_t* N64,
                   int64_t* nb64) {
  if (kind != VA_MASK_DENSE && kind != VA_MASK_RADIAL && kind != VA_MASK_LVSA)
    return VA_ERR_INVALID;
  if (T < 1 || H < 1 || W < 1) return VA_ERR_INVALID;
  const int64_t n = static_cast<int64_t>(H) * W * T;
  if (n >= (1LL << 30)) return VA_ERR_INVALID;
  if (p.block < 1 || p.block > 4096) return VA_ERR_INVALID;
  if (p.w0 < 0 || p.local < 0 || p.period < 0) return VA_ERR_INVALID;
  *N64 = n;
  *nb64 = (n + p.block - 1) / p.block;
  return VA_OK;
}

}  // namespace

VA_EXPORT int va_mask_build(int kind, int T, int H, int W, const va_mask_params* params,
                            int step, va_mask** out, va_stream_t stream) {
  if (out == nullptr || params == nullptr) return VA_ERR_INVALID;
  *out = nullptr;
  const va_mask_params p = *params;
  int64_t N64 = 0, nb64 = 0;
  if (int st0 = mask_grid_args(kind, T, H, W, p, &N64, &nb64)) return st0;
  const int64_t F64 = static_cast<int64_t>(H) * W;
  if (nb64 > VA_MASK_MAX_BLOCKS) return VA_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  va::MaskDesc md;
  md.kind = kind;
  md.T = T;
  md.F = static_cast<int>(F64);
  md.N = static_cast<int>(N64);
  md.block = p.block;
  md.nb = static_cast<int>((N64 + p.block - 1) / p.block);
  md.w0 = (kind == VA_MASK_RADIAL && p.w0 == 0) ? md.F : p.w0;
  md.local = p.local;
  md.period = p.period;
  md.anchor0 = p.anchor0;
  md.rot_stride = p.rot_stride;
  md.step = step;

  va_mask* m = new va_mask();
  m->kind = kind;
  m->T = T;
  m->H = H;
  m->W = W;
  m->N = md.N;
  m->step = step;
  m->p = p;
  m->nqb = md.nb;
  cudaGetDevice(&m->device);

  int st = VA_OK;
  {
    Scoped scratch(s);
    int* cnt = nullptr;
    long long* keytok = nullptr;
    long long* summary = nullptr;
    int* hist = nullptr;
    if ((st = scratch.alloc(&cnt, md.nb)) || (st = scratch.alloc(&keytok, md.nb)) ||
        (st = scratch.alloc(&summary, 2)) || (st = scratch.alloc(&hist, md.nb + 1))) {
      delete m;
      return st;
    }
    if (Scoped::fault_injected()) {
      delete m;
      return VA_ERR_OOM;
    }
    if ((st = cuda_status(cudaMalloc(&m->row_ptr, sizeof(int32_t) * (md.nb + 1)))) ||
        (st = cuda_status(cudaMalloc(&m->order, sizeof(int32_t) * md.nb)))) {
      va_mask_free(m);
      return st;
    }
    const int threads = 256;
    const int blocks = static_cast<int>((static_cast<int64_t>(md.nb) * 32 + threads - 1) / threads);
    va::mask_count_kernel<<<blocks, threads, 0, s>>>(md, cnt, keytok);
    va::mask_scan_kernel<<<1, 1024, 0, s>>>(md, cnt, keytok, m->row_ptr, summary, m->order, hist);
    if ((st = launch_status())) {
      va_mask_free(m);
      return st;
    }
    long long host_summary[2] = {0, 0};
    if ((st = cuda_status(cudaMemcpyAsync(host_summary, summary, sizeof(host_summary),
                                          cudaMemcpyDeviceToHost, s))) ||
        (st = cuda_status(cudaStreamSynchronize(s)))) {
      va_mask_free(m);
      return st;
    }
    m->nnz = host_summary[0];
    m->live_pairs = host_summary[1];
    if (m->nnz > kMaxMaskNnz) {
      // int32 row offsets cannot index the list: stop before any fill
      va_mask_free(m);
      return VA_ERR_UNSUPPORTED;
    }
    if ((st = cuda_status(cudaMalloc(&m->col, sizeof(int32_t) * (m->nnz > 0 ? m->nnz : 1))))) {
      va_mask_free(m);
      return st;
    }
    va::mask_fill_kernel<<<blocks, threads, 0, s>>>(md, m->row_ptr, m->col);
    if ((st = launch_status())) {
      va_mask_free(m);
      return st;
    }
    m->npairs = (md.nb + 1) / 2;
    int* phist = nullptr;
    if ((st = scratch.alloc(&phist, 2 * static_cast<size_t>(md.nb) + 2)) ||
        (st = cuda_status(cudaMalloc(&m->pcol, sizeof(int32_t) * (m->nnz > 0 ? m->nnz : 1)))) ||
        (st = cuda_status(cudaMalloc(&m->plen, sizeof(int32_t) * m->npairs))) ||
        (st = cuda_status(cudaMalloc(&m->porder, sizeof(int32_t) * m->npairs)))) {
      va_mask_free(m);
      return st;
    }
    va::pair_merge_kernel<<<(m->npairs + 127) / 128, 128, 0, s>>>(md.nb, m->row_ptr, m->col,
                                                                   m->pcol, m->plen);
    va::pair_order_kernel<<<1, 1, 0, s>>>(md.nb, m->row_ptr, m->porder, phist);
    if ((st = launch_status())) {
      va_mask_free(m);
      return st;
    }
    if (m->p.block == 64) {
      m->nquads = (md.nb + 3) / 4;
      int* qhist = nullptr;
      if ((st = scratch.alloc(&qhist, 4 * static_cast<size_t>(md.nb) + 2)) ||
          (st = cuda_status(cudaMalloc(&m->qcol, sizeof(int32_t) * (m->nnz > 0 ? m->nnz : 1)))) ||
          (st = cuda_status(cudaMalloc(&m->qlen, sizeof(int32_t) * m->nquads))) ||
          (st = cuda_status(cudaMalloc(&m->qorder, sizeof(int32_t) * m->nquads)))) {
        va_mask_free(m);
        return st;
      }
      va::quad_merge_kernel<<<(m->nquads + 127) / 128, 128, 0, s>>>(md.nb, m->row_ptr, m->col,
                                                                     m->qcol, m->qlen);
      va::quad_order_kernel<<<1, 1, 0, s>>>(md.nb, m->row_ptr, m->qorder, qhist);
      if ((st = launch_status())) {
        va_mask_free(m);
        return st;
      }
    }
    // The transposed lists reuse the count / scan / fill kernels with the
    // roles of query and key blocks swapped; the live pairs are the same, so
    // their number is already known.
    if ((st = cuda_status(cudaMalloc(&m->t_ptr, sizeof(int32_t) * (md.nb + 1)))) ||
        (st = cuda_status(cudaMalloc(&m->t_order, sizeof(int32_t) * md.nb))) ||
        (st = cuda_status(cudaMalloc(&m->t_row, sizeof(int32_t) * (m->nnz > 0 ? m->nnz : 1))))) {
      va_mask_free(m);
      return st;
    }
    va::MaskDesc mt = md;
    mt.transpose = 1;
    va::mask_count_kernel<<<blocks, threads, 0, s>>>(mt, cnt, keytok);
    va::mask_scan_kernel<<<1, 1024, 0, s>>>(mt, cnt, keytok, m->t_ptr, summary, m->t_order, hist);
    va::mask_fill_kernel<<<blocks, threads, 0, s>>>(mt, m->t_ptr, m->t_row);
    if ((st = launch_status())) {
      va_mask_free(m);
      return st;
    }
    if (m->p.block == 64) {
      // coarse pairs of both lists for the tensor-core backward
      const int nc = (md.nb + 1) / 2;
      const size_t nn = static_cast<size_t>(m->nnz > 0 ? m->nnz : 1);
      int* chist = nullptr;
      if ((st = scratch.alloc(&chist, 2 * static_cast<size_t>(md.nb) + 2)) ||
          (st = cuda_status(cudaMalloc(&m->cq_col, sizeof(int32_t) * nn))) ||
          (st = cuda_status(cudaMalloc(&m->cq_len, sizeof(int32_t) * nc))) ||
          (st = cuda_status(cudaMalloc(&m->cq_order, sizeof(int32_t) * nc))) ||
          (st = cuda_status(cudaMalloc(&m->ck_col, sizeof(int32_t) * nn))) ||
          (st = cuda_status(cudaMalloc(&m->ck_len, sizeof(int32_t) * nc))) ||
          (st = cuda_status(cudaMalloc(&m->ck_order, sizeof(int32_t) * nc)))) {
        va_mask_free(m);
        return st;
      }
      va::coarse_pair_merge_kernel<<<(nc + 127) / 128, 128, 0, s>>>(md.nb, m->row_ptr, m->col,
                                                                     m->cq_col, m->cq_len);
      va::coarse_pair_merge_kernel<<<(nc + 127) / 128, 128, 0, s>>>(md.nb, m->t_ptr, m->t_row,
                                                                     m->ck_col, m->ck_len);
      va::pair_order_kernel<<<1, 1, 0, s>>>(md.nb, m->row_ptr, m->cq_order, chist);
      va::pair_order_kernel<<<1, 1, 0, s>>>(md.nb, m->t_ptr, m->ck_order, chist);
      if ((st = launch_status())) {
        va_mask_free(m);
        return st;
      }
    }
  }
  if ((st = cuda_status(cudaStreamSynchronize(s)))) {
    va_mask_free(m);
    return st;
  }
  if (checked_mode() && (st = validate_mask(m))) {
    va_mask_free(m);
    return st;
  }
  *out = m;
  return VA_OK;
}

VA_EXPORT int va_mask_csr(const va_mask* m, const int32_t** row_ptr_dev,
                          const int32_t** col_idx_dev, int* nqb, int64_t* nnz) {
  if (m == nullptr) return VA_ERR_INVALID;
  if (row_ptr_dev) *row_ptr_dev = m->row_ptr;
  if (col_idx_dev) *col_idx_dev = m->col;
  if (nqb) *nqb = m->nqb;
  if (nnz) *nnz = m->nnz;
  return VA_OK;
}

VA_EXPORT int va_mask_info(const va_mask* m, int* N, int* block, int64_t* live_pairs) {
  if (m == nullptr) return VA_ERR_INVALID;
  if (N) *N = m->N;
  if (block) *block = m->p.block;
  if (live_pairs) *live_pairs = m->live_pairs;
  return VA_OK;
}

VA_EXPORT int va_mask_to_host(const va_mask* m, int32_t* row_ptr, int32_t* col_idx) {
  if (m == nullptr || row_ptr == nullptr || (col_idx == nullptr && m->nnz > 0))
    return VA_ERR_INVALID;
  int st = cuda_status(
      cudaMemcpy(row_ptr, m->row_ptr, sizeof(int32_t) * (m->nqb + 1), cudaMemcpyDeviceToHost));
  if (st) return st;
  if (m->nnz > 0)
    st = cuda_status(
        cudaMemcpy(col_idx, m->col, sizeof(int32_t) * m->nnz, cudaMemcpyDeviceToHost));
  return st;
}

VA_EXPORT int va_mask_free(va_mask* m) {
  if (m == nullptr) return VA_OK;
  if (m->row_ptr) cudaFree(m->row_ptr);
  if (m->col) cudaFree(m->col);
  if (m->order) cudaFree(m->order);
  if (m->pcol) cudaFree(m->pcol);
  if (m->plen) cudaFree(m->plen);
  if (m->porder) cudaFree(m->porder);
  if (m->qcol) cudaFree(m->qcol);
  if (m->qlen) cudaFree(m->qlen);
  if (m->qorder) cudaFree(m->qorder);
  for (int32_t* pp : {m->cq_col, m->cq_len, m->cq_order, m->ck_col, m->ck_len, m->ck_order})
    if (pp) cudaFree(pp);
  if (m->t_ptr) cudaFree(m->t_ptr);
  if (m->t_row) cudaFree(m->t_row);
  if (m->t_order) cudaFree(m->t_order);
  delete m;
  return VA_OK;
}

// ------------------------------------------------------------ mask cache --
// Masks are reused across the denoising steps of one video (the radial mask
// is static; LVSA's anchors rotate with the step, so its mask repeats with the
// rotation's period): the cache keys a mask by what its CSR depends on.

namespace {

// Everything a mask's CSR depends on. For a radial mask that is the grid, the
// block and the effective w0 (0 means the frame size); for LVSA the grid, the
// block, the local window and the anchor rule, where with period > 0 only the
// phase (anchor0 + rot_stride * step) mod period matters; a dense mask
// depends on the grid and the block alone.
struct MaskKey {
  int dev, kind, T, H, W, block, w0, local, period, anchor;
  bool operator==(const MaskKey& o) const {
    return dev == o.dev && kind == o.kind && T == o.T && H == o.H && W == o.W &&
           block == o.block && w0 == o.w0 && local == o.local && period == o.period &&
           anchor == o.anchor;
  }
};

int mask_key(int kind, int T, int H, int W, const va_mask_params& p, int step, int dev,
             MaskKey* k) {
  int64_t N64 = 0, nb64 = 0;
  if (int st = mask_grid_args(kind, T, H, W, p, &N64, &nb64)) return st;
  if (nb64 > VA_MASK_MAX_BLOCKS) return VA_ERR_UNSUPPORTED;
  *k = MaskKey{dev, kind, T, H, W, p.block, 0, 0, 0, 0};
  if (kind == VA_MASK_RADIAL) {
    k->w0 = p.w0 == 0 ? H * W : p.w0;
  } else if (kind == VA_MASK_LVSA) {
    k->local = p.local;
    k->period = p.period;
    if (p.period > 0) {
      int64_t r = (static_cast<int64_t>(p.anchor0) +
                   static_cast<int64_t>(p.rot_stride) * step) % p.period;
      if (r < 0) r += p.period;
      k->anchor = static_cast<int>(r);
    } else {
      k->anchor = p.anchor0;
    }
  }
  return VA_OK;
}

// Frees a mask with its own device current (a cache may hold masks of
// several devices).
void free_on_device(va_mask* m) {
  const int dev = m->device;
  int cur = 0;
  const bool have = cudaGetDevice(&cur) == cudaSuccess;
  if (have && cur != dev) cudaSetDevice(dev);
  va_mask_free(m);
  if (have && cur != dev) cudaSetDevice(cur);
}

}  // namespace

struct va_mask_cache {
  std::mutex mu;
  int capacity = 0;
  std::vector<std::pair<MaskKey, va_mask*>> entries;
  int64_t hits = 0, misses = 0;
};

VA_EXPORT int va_mask_cache_create(int capacity, va_mask_cache** out) {
  if (out == nullptr) return VA_ERR_INVALID;
  *out = nullptr;
  if (capacity < 1 || capacity > VA_MASK_CACHE_MAX) return VA_ERR_INVALID;
  va_mask_cache* c = new (std::nothrow) va_mask_cache();
  if (c == nullptr) return VA_ERR_OOM;
  c->capacity = capacity;
  c->entries.reserve(static_cast<size_t>(capacity));
  *out = c;
  return VA_OK;
}

VA_EXPORT int va_mask_cache_get(va_mask_cache* cache, int kind, int T, int H, int W,
                                const va_mask_params* params, int step, const va_mask** out,
                                va_stream_t stream) {
  if (out == nullptr) return VA_ERR_INVALID;
  *out = nullptr;
  if (cache == nullptr || params == nullptr) return VA_ERR_INVALID;
  int dev = 0;
  if (int st = cuda_status(cudaGetDevice(&dev))) return st;
  MaskKey key;
  if (int st = mask_key(kind, T, H, W, *params, step, dev, &key)) return st;
  std::lock_guard<std::mutex> lock(cache->mu);
  for (auto& e : cache->entries) {
    if (e.first == key) {
      ++cache->hits;
      *out = e.second;
      return VA_OK;
    }
  }
  if (static_cast<int>(cache->entries.size()) >= cache->capacity) return VA_ERR_UNSUPPORTED;
  va_mask* m = nullptr;
  if (int st = va_mask_build(kind, T, H, W, params, step, &m, stream)) return st;
  cache->entries.emplace_back(key, m);
  ++cache->misses;
  *out = m;
  return VA_OK;
}

VA_EXPORT int va_mask_cache_stats(va_mask_cache* cache, int64_t* hits, int64_t* misses,
                                  int* entries) {
  if (cache == nullptr) return VA_ERR_INVALID;
  std::lock_guard<std::mutex> lock(cache->mu);
  if (hits) *hits = cache->hits;
  if (misses) *misses = cache->misses;
  if (entries) *entries = static_cast<int>(cache->entries.size());
  return VA_OK;
}

VA_EXPORT int va_mask_cache_clear(va_mask_cache* cache) {
  if (cache == nullptr) return VA_ERR_INVALID;
  std::lock_guard<std::mutex> lock(cache->mu);
  for (auto& e : cache->entries) free_on_device(e.second);
  cache->entries.clear();
  return VA_OK;
}

VA_EXPORT int va_mask_cache_destroy(va_mask_cache* cache) {
  if (cache == nullptr) return VA_OK;
  va_mask_cache_clear(cache);
  delete cache;
  return VA_OK;
}

VA_EXPORT int va_mask_same(int kind, int T, int H, int W, const va_mask_params* params,
                           int step_a, int step_b, int* same) {
  if (params == nullptr || same == nullptr) return VA_ERR_INVALID;
  *same = 0;
  MaskKey ka, kb;
  if (int st = mask_key(kind, T, H, W, *params, step_a, 0, &ka)) return st;
  if (int st = mask_key(kind, T, H, W, *params, step_b, 0, &kb)) return st;
  *same = ka == kb ? 1 : 0;
  return VA_OK;
}

// -------------------------------------------------------------- attention --

namespace {

template <typename T, int D, int BLK>
int launch_simt(const void* q, const void* k, const void* v, const va_mask* m, void* out,
                float* lse, int BH, int N, float scale, cudaStream_t s) {
  dim3 grid(m->nqb, BH);
  va::attn_simt_kernel<T, D, BLK><<<grid, BLK * 4, 0, s>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), m->row_ptr,
      m->col, static_cast<T*>(out), lse, N, scale * 1.4426950408889634f);
  return launch_status();
}

// SUB: a mask of 64-token blocks, run as 128-row tiles over the mask's quads.
template <int D, bool SUB = false>
int launch_tc(const void* q, const void* k, const void* v, const va_mask* m, void* out, float* lse,
              int BH, int N, float scale, cudaStream_t s) {
  static DeviceOnce once;
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  st = device_once(once, dev, [] {
    // The kernel's setmaxnreg split assumes this exact per-thread register
    // count at launch; anything else could leave the increase waiting.
    cudaFuncAttributes fa;
    int r = cuda_status(cudaFuncGetAttributes(&fa, va::attn_tc_kernel<D, SUB>));
    if (r) return r;
    if (fa.numRegs != va::TC_LAUNCH_REGS) return VA_ERR_UNSUPPORTED;
    return cuda_status(cudaFuncSetAttribute(va::attn_tc_kernel<D, SUB>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            va::TcDim<D>::kSmemBytes));
  });
  if (st) return st;
  CUtensorMap mq, mk, mv;
  if ((st = encode_bf16_rows(&mq, q, BH, N, D)) || (st = encode_bf16_rows(&mk, k, BH, N, D)) ||
      (st = encode_bf16_rows(&mv, v, BH, N, D)))
    return st;
  va::TcArgs a;
  a.row_ptr = m->row_ptr;
  a.col = m->col;
  a.pcol = SUB ? m->qcol : m->pcol;
  a.plen = SUB ? m->qlen : m->plen;
  a.porder = SUB ? m->qorder : m->porder;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.N = N;
  a.nqb = SUB ? (m->nqb + 1) / 2 : m->nqb;   // 128-row tiles
  a.npairs = SUB ? m->nquads : m->npairs;
  if (SUB && a.pcol == nullptr) return VA_ERR_UNSUPPORTED;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit = g_wait_limit;
  const long long grid = static_cast<long long>(a.npairs) * BH;
  if (grid > 0x7fffffffLL) return VA_ERR_UNSUPPORTED;
  va::attn_tc_kernel<D, SUB><<<static_cast<unsigned>(grid), va::TC_THREADS,
                               va::TcDim<D>::kSmemBytes, s>>>(mq, mk, mv, a);
  return launch_status();
}

}  // namespace

VA_EXPORT int va_sparse_attn_fwd(const void* q, const void* k, const void* v, const va_mask* m,
                                 void* out, float* lse, int B, int heads, int N, int d,
                                 float scale, int dtype, va_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || m == nullptr || out == nullptr)
    return VA_ERR_INVALID;
  if (B < 1 || heads < 1 || N != m->N) return VA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return VA_ERR_INVALID;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return VA_ERR_INVALID;
  if (int dst = check_mask_device(m)) return dst;
  if (!std::isfinite(scale)) return VA_ERR_INVALID;
  const int64_t BH64 = static_cast<int64_t>(B) * heads;
  if (BH64 > 65535 && dtype == VA_F32) return VA_ERR_UNSUPPORTED;
  if (BH64 * N >= (1LL << 31)) return VA_ERR_UNSUPPORTED;
  const int BH = static_cast<int>(BH64);
  const int blk = m->p.block;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == VA_F32) {
    if (d == 64 && blk == 64) return launch_simt<float, 64, 64>(q, k, v, m, out, lse, BH, N, scale, s);
    if (d == 64 && blk == 128) return launch_simt<float, 64, 128>(q, k, v, m, out, lse, BH, N, scale, s);
    if (d == 128 && blk == 64) return launch_simt<float, 128, 64>(q, k, v, m, out, lse, BH, N, scale, s);
    if (d == 128 && blk == 128) return launch_simt<float, 128, 128>(q, k, v, m, out, lse, BH, N, scale, s);
    return VA_ERR_UNSUPPORTED;
  }
  if (dtype == VA_BF16) {
    if (d == 128 && blk == 128) return launch_tc<128>(q, k, v, m, out, lse, BH, N, scale, s);
    if (d == 64 && blk == 128) return launch_tc<64>(q, k, v, m, out, lse, BH, N, scale, s);
    if (d == 128 && blk == 64) return launch_tc<128, true>(q, k, v, m, out, lse, BH, N, scale, s);
    if (d == 64 && blk == 64) return launch_tc<64, true>(q, k, v, m, out, lse, BH, N, scale, s);
    return VA_ERR_UNSUPPORTED;
  }
  return VA_ERR_UNSUPPORTED;
}

// --------------------------------------------------------------- backward --

namespace {

template <typename T, int D, int BLK>
int launch_bwd_simt(const void* q, const void* k, const void* v, const void* g, const va_mask* m,
                    const float* ndelta, const float* nlse2, void* dq, void* dk, void* dv, int BH,
                    int N, int Np, float scale, cudaStream_t s) {
  dim3 grid(m->nqb * (BLK / va::BWS_ROWS), BH);
  const float sl2 = scale * 1.4426950408889634f;
  va::bwd_dq_simt_kernel<T, D, BLK><<<grid, va::BWS_ROWS * 4, 0, s>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
      static_cast<const T*>(g), ndelta, nlse2, m->row_ptr, m->col, static_cast<T*>(dq), N, Np,
      scale, sl2);
  va::bwd_dkdv_simt_kernel<T, D, BLK><<<grid, va::BWS_ROWS * 4, 0, s>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
      static_cast<const T*>(g), ndelta, nlse2, m->t_ptr, m->t_row, static_cast<T*>(dk),
      static_cast<T*>(dv), N, Np, scale, sl2);
  return launch_status();
}

// SUB: a mask of 64-token blocks, run on its coarse pairs (128-token tiles).
template <int D, bool SUB = false>
int launch_bwd_tc(const void* q, const void* k, const void* v, const void* g, const va_mask* m,
                  const float* ndelta, const float* nlse2, void* dq, void* dk, void* dv, int BH,
                  int N, int Np, float scale, cudaStream_t s) {
  static DeviceOnce once;
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  st = device_once(once, dev, [] {
    int r;
    if ((r = cuda_status(cudaFuncSetAttribute(va::bwd_dkdv_tc_kernel<D, SUB>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              va::BwDim<D>::kSmemBytes))) ||
        (r = cuda_status(cudaFuncSetAttribute(va::bwd_dq_tc_kernel<D, SUB>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              va::BwDim<D>::kSmemBytes))))
      return r;
    return VA_OK;
  });
  if (st) return st;
  CUtensorMap mq, mk, mv, mg;
  if ((st = encode_bf16_rows(&mq, q, BH, N, D)) || (st = encode_bf16_rows(&mk, k, BH, N, D)) ||
      (st = encode_bf16_rows(&mv, v, BH, N, D)) || (st = encode_bf16_rows(&mg, g, BH, N, D)))
    return st;
  if (SUB && (m->cq_col == nullptr || m->ck_col == nullptr)) return VA_ERR_UNSUPPORTED;
  const int nb = SUB ? (m->nqb + 1) / 2 : m->nqb;  // 128-token tiles
  const long long grid = static_cast<long long>(nb) * BH;
  if (grid > 0x7fffffffLL) return VA_ERR_UNSUPPORTED;
  va::BwArgs a;
  a.ndelta = ndelta;
  a.nlse2 = nlse2;
  a.N = N;
  a.Np = Np;
  a.nb = nb;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit = g_wait_limit;
  a.ptr = m->t_ptr;
  a.idx = SUB ? m->ck_col : m->t_row;
  a.order = SUB ? m->ck_order : m->t_order;
  a.len = SUB ? m->ck_len : nullptr;
  a.d0 = static_cast<__nv_bfloat16*>(dv);
  a.d1 = static_cast<__nv_bfloat16*>(dk);
  va::bwd_dkdv_tc_kernel<D, SUB>
      <<<static_cast<unsigned>(grid), va::BW_THREADS, va::BwDim<D>::kSmemBytes, s>>>(mq, mk, mv,
                                                                                  mg, a);
  a.ptr = m->row_ptr;
  a.idx = SUB ? m->cq_col : m->col;
  a.order = SUB ? m->cq_order : m->order;
  a.len = SUB ? m->cq_len : nullptr;
  a.d0 = static_cast<__nv_bfloat16*>(dq);
  a.d1 = nullptr;
  va::bwd_dq_tc_kernel<D, SUB>
      <<<static_cast<unsigned>(grid), va::BW_THREADS, va::BwDim<D>::kSmemBytes, s>>>(mq, mk, mv,
                                                                                mg, a);
  return launch_status();
}

}  // namespace

VA_EXPORT int va_sparse_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                                 const void* dout, const float* lse, const va_mask* m, void* dq,
                                 void* dk, void* dv, int B, int heads, int N, int d, float scale,
                                 int dtype, va_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || dout == nullptr ||
      lse == nullptr || m == nullptr || dq == nullptr || dk == nullptr || dv == nullptr)
    return VA_ERR_INVALID;
  if (B < 1 || heads < 1 || N != m->N || m->t_ptr == nullptr) return VA_ERR_INVALID;
  if (int dst = check_mask_device(m)) return dst;
  for (const void* p : {q, k, v, out, dout, static_cast<const void*>(dq),
                        static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (!aligned16(p)) return VA_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return VA_ERR_INVALID;
  if (!std::isfinite(scale)) return VA_ERR_INVALID;
  const int64_t BH64 = static_cast<int64_t>(B) * heads;
  if (BH64 > 65535) return VA_ERR_UNSUPPORTED;
  if (BH64 * N >= (1LL << 31)) return VA_ERR_UNSUPPORTED;
  const int BH = static_cast<int>(BH64);
  const int blk = m->p.block;
  const bool tc = dtype == VA_BF16 && (d == 64 || d == 128) && (blk == 64 || blk == 128);
  // rows of the per-row scratch, whole blocks (whole 128-token tiles on the
  // tensor-core path with 64-token blocks)
  const int Np = tc && blk == 64 ? (m->nqb + 1) / 2 * 128 : m->nqb * blk;
  const bool simt = dtype == VA_F32 && (d == 64 || d == 128) && (blk == 64 || blk == 128);
  if (!tc && !simt) return VA_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Scoped scratch(s);
  float* ndelta = nullptr;
  float* nlse2 = nullptr;
  int st;
  const size_t rows = static_cast<size_t>(BH) * Np;
  if ((st = scratch.alloc(&ndelta, rows)) || (st = scratch.alloc(&nlse2, rows))) return st;
  dim3 pgrid((Np + 7) / 8, BH);
  if (tc) {
    va::bwd_prep_kernel<__nv_bfloat16><<<pgrid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse, N,
        Np, d, ndelta, nlse2);
    if ((st = launch_status())) return st;
    if (blk == 64)
      return d == 64 ? launch_bwd_tc<64, true>(q, k, v, dout, m, ndelta, nlse2, dq, dk, dv, BH,
                                               N, Np, scale, s)
                     : launch_bwd_tc<128, true>(q, k, v, dout, m, ndelta, nlse2, dq, dk, dv, BH,
                                                N, Np, scale, s);
    if (d == 64)
      return launch_bwd_tc<64>(q, k, v, dout, m, ndelta, nlse2, dq, dk, dv, BH, N, Np, scale, s);
    return launch_bwd_tc<128>(q, k, v, dout, m, ndelta, nlse2, dq, dk, dv, BH, N, Np, scale, s);
  }
  va::bwd_prep_kernel<float><<<pgrid, 256, 0, s>>>(static_cast<const float*>(out),
                                                   static_cast<const float*>(dout), lse, N, Np,
                                                   d, ndelta, nlse2);
  if ((st = launch_status())) return st;
  if (d == 64 && blk == 64)
    return launch_bwd_simt<float, 64, 64>(q, k, v, dout, m, ndelta, nlse2, dq, dk, dv, BH, N, Np, scale, s);
  if (d == 64 && blk == 128)
    return launch_bwd_simt<float, 64, 128>(q, k, v, dout, m, ndelta, nlse2, dq, dk, dv, BH, N, Np, scale, s);
  if (d == 128 && blk == 64)
    return launch_bwd_simt<float, 128, 64>(q, k, v, dout, m, ndelta, nlse2, dq, dk, dv, BH, N, Np, scale, s);
  return launch_bwd_simt<float, 128, 128>(q, k, v, dout, m, ndelta, nlse2, dq, dk, dv, BH, N, Np, scale, s);
}

// Host-buffer attention: (batch*head) chunks move through a ring of device
// buffers; host->device copies, the attention kernel and device->host copies
// run on three streams ordered by events, so the transfers of one chunk
// overlap the attention of another.
namespace {

constexpr int kHostRing = 3;

struct HostStreams {
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, in_ready[kHostRing] = {}, in_free[kHostRing] = {},
              out_free[kHostRing] = {}, done[3] = {};
  std::mutex enqueue;  // one call at a time enqueues on these streams
};

// Streams and events of the current device, created on first use.
int host_streams(HostStreams** out) {
  static HostStreams per_dev[64];
  static bool ready[64] = {false};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return VA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  HostStreams& h = per_dev[dev];
  if (!ready[dev]) {
    int st;
    const unsigned fl = cudaEventDisableTiming;
    if ((st = cuda_status(cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking))) ||
        (st = cuda_status(cudaStreamCreateWithFlags(&h.comp, cudaStreamNonBlocking))) ||
        (st = cuda_status(cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking))) ||
        (st = cuda_status(cudaEventCreateWithFlags(&h.start, fl))))
      return st;
    for (int t = 0; t < 3; ++t)
      if ((st = cuda_status(cudaEventCreateWithFlags(&h.done[t], fl)))) return st;
    for (int j = 0; j < kHostRing; ++j)
      if ((st = cuda_status(cudaEventCreateWithFlags(&h.in_ready[j], fl))) ||
          (st = cuda_status(cudaEventCreateWithFlags(&h.in_free[j], fl))) ||
          (st = cuda_status(cudaEventCreateWithFlags(&h.out_free[j], fl))))
        return st;
    ready[dev] = true;
  }
  *out = &h;
  return VA_OK;
}

}  // namespace

VA_EXPORT int va_sparse_attn_fwd_host(const void* q, const void* k, const void* v,
                                      const va_mask* m, void* out, float* lse, int B, int heads,
                                      int N, int d, float scale, int dtype, va_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || m == nullptr || out == nullptr)
    return VA_ERR_INVALID;
  if (B < 1 || heads < 1 || N != m->N || N < 1 || d < 1) return VA_ERR_INVALID;
  if (!std::isfinite(scale)) return VA_ERR_INVALID;
  if (int dst = check_mask_device(m)) return dst;
  if (dtype != VA_BF16 && dtype != VA_F32) return VA_ERR_UNSUPPORTED;
  const int64_t BH64 = static_cast<int64_t>(B) * heads;
  if (BH64 * N >= (1LL << 31)) return VA_ERR_UNSUPPORTED;
  const int BH = static_cast<int>(BH64);
  HostStreams* h = nullptr;
  int st;
  if ((st = host_streams(&h))) return st;
  std::lock_guard<std::mutex> lock(h->enqueue);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // chunks of `hc` (batch*head) slices: about 12 chunks, at least one slice
  const int hc = BH >= 12 ? BH / 12 : 1;
  const int nch = (BH + hc - 1) / hc;
  const size_t esz = dtype == VA_BF16 ? 2 : 4;
  const size_t slice = static_cast<size_t>(N) * d * esz;   // one (b, h) of q, k, v or out
  const size_t lslice = static_cast<size_t>(N) * sizeof(float);
  Scoped scratch(s);
  uint8_t* buf[kHostRing][4];
  float* lbuf[kHostRing] = {};
  for (int j = 0; j < kHostRing; ++j) {
    for (int t = 0; t < 4; ++t)
      if ((st = scratch.alloc(&buf[j][t], slice * hc))) return st;
    if (lse != nullptr && (st = scratch.alloc(&lbuf[j], lslice * hc / sizeof(float)))) return st;
  }
  // fork from the caller's stream (the scratch is allocated there) ...
  if ((st = cuda_status(cudaEventRecord(h->start, s))) ||
      (st = cuda_status(cudaStreamWaitEvent(h->h2d, h->start, 0))) ||
      (st = cuda_status(cudaStreamWaitEvent(h->comp, h->start, 0))) ||
      (st = cuda_status(cudaStreamWaitEvent(h->d2h, h->start, 0))))
    return st;
  // ... and join back on every exit, so the scratch is released on the
  // caller's stream only after all three streams are done with it
  auto join = [&](int status) -> int {
    cudaStream_t side[3] = {h->h2d, h->comp, h->d2h};
    for (int t = 0; t < 3; ++t) {
      const int js = cuda_status(cudaEventRecord(h->done[t], side[t]));
      const int ws = js ? js : cuda_status(cudaStreamWaitEvent(s, h->done[t], 0));
      if (status == VA_OK) status = ws;
    }
    return status;
  };
  const uint8_t* hin[3] = {static_cast<const uint8_t*>(q), static_cast<const uint8_t*>(k),
                           static_cast<const uint8_t*>(v)};
  for (int i = 0; i < nch; ++i) {
    const int j = i % kHostRing;
    const int b0 = i * hc, nb = std::min(hc, BH - b0);
    const size_t off = static_cast<size_t>(b0) * slice, bytes = static_cast<size_t>(nb) * slice;
    // inputs of slot j are free once the attention of chunk i - ring finished
    if (i >= kHostRing && (st = cuda_status(cudaStreamWaitEvent(h->h2d, h->in_free[j], 0))))
      return join(st);
    for (int t = 0; t < 3; ++t)
      if ((st = cuda_status(cudaMemcpyAsync(buf[j][t], hin[t] + off, bytes,
                                            cudaMemcpyHostToDevice, h->h2d))))
        return join(st);
    if ((st = cuda_status(cudaEventRecord(h->in_ready[j], h->h2d))) ||
        (st = cuda_status(cudaStreamWaitEvent(h->comp, h->in_ready[j], 0))))
      return join(st);
    // output of slot j is free once the copy-out of chunk i - ring finished
    if (i >= kHostRing && (st = cuda_status(cudaStreamWaitEvent(h->comp, h->out_free[j], 0))))
      return join(st);
    if ((st = va_sparse_attn_fwd(buf[j][0], buf[j][1], buf[j][2], m, buf[j][3],
                                 lse != nullptr ? lbuf[j] : nullptr, 1, nb, N, d, scale, dtype,
                                 reinterpret_cast<va_stream_t>(h->comp))))
      return join(st);
    if ((st = cuda_status(cudaEventRecord(h->in_free[j], h->comp))) ||
        (st = cuda_status(cudaStreamWaitEvent(h->d2h, h->in_free[j], 0))) ||
        (st = cuda_status(cudaMemcpyAsync(static_cast<uint8_t*>(out) + off, buf[j][3], bytes,
                                          cudaMemcpyDeviceToHost, h->d2h))))
      return join(st);
    if (lse != nullptr &&
        (st = cuda_status(cudaMemcpyAsync(lse + static_cast<size_t>(b0) * N, lbuf[j],
                                          static_cast<size_t>(nb) * lslice,
                                          cudaMemcpyDeviceToHost, h->d2h))))
      return join(st);
    if ((st = cuda_status(cudaEventRecord(h->out_free[j], h->d2h)))) return join(st);
  }
  return join(VA_OK);
}

// ------------------------------------------------- linear / mixed attention --

namespace {

// Linear attention (bf16, d = D) of every (batch, head): split state sums,
// their merge into bf16 pieces of [S | z]^T, then the output; with mix != 0
// the output kernel blends r * out (the attention already there) with the
// linear result.
template <int D>
int run_linear(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
               __nv_bfloat16* out, int BH, int N, int mix, float r, cudaStream_t s) {
  using Dm = va::LnDim<D>;
  static DeviceOnce once;
  static int num_sms[64] = {0};
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  st = device_once(once, dev, [dev] {
    int r;
    if ((r = cuda_status(cudaFuncSetAttribute(va::lin_state_kernel<D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              Dm::kStateSmem))) ||
        (r = cuda_status(cudaFuncSetAttribute(va::lin_out_kernel<D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              Dm::kOutSmem))) ||
        (r = cuda_status(cudaDeviceGetAttribute(&num_sms[dev], cudaDevAttrMultiProcessorCount,
                                                dev))))
      return r;
    return VA_OK;
  });
  if (st) return st;
  const int ntiles = (N + 127) / 128;
  const int nsplit = std::max(1, std::min(ntiles, num_sms[dev] / BH));
  Scoped scratch(s);
  float* part;
  __nv_bfloat16* piece;
  const size_t bh = static_cast<size_t>(BH);
  if ((st = scratch.alloc(&part, bh * nsplit * D * Dm::kRow)) ||
      (st = scratch.alloc(&piece, bh * 2 * Dm::kNext * D)))
    return st;
  CUtensorMap mk, mv, mq, mp, mo;
  if ((st = encode_bf16_rows(&mk, k, BH, N, D)) || (st = encode_bf16_rows(&mv, v, BH, N, D)) ||
      (st = encode_bf16_rows(&mq, q, BH, N, D)) || (st = encode_bf16_rows(&mo, out, BH, N, D)) ||
      (st = encode_bf16_rows_box(&mp, piece, BH, 2 * Dm::kNext, D, Dm::kNext)))
    return st;
  va::lin_state_kernel<D><<<dim3(nsplit, BH), va::LN_STATE_THREADS, Dm::kStateSmem, s>>>(
      mk, mv, N, part, g_wait_limit);
  // prep and out are programmatic dependents: each starts while its
  // predecessor drains and waits (griddepcontrol.wait) before reading its output.
  if ((st = cuda_status(launch_dependent(va::lin_prep_kernel<D>, dim3(Dm::kNext, BH), D, 0, s,
                                         static_cast<const float*>(part), nsplit, piece))) ||
      (st = cuda_status(launch_dependent(va::lin_out_kernel<D>, dim3(nsplit, BH),
                                         va::LN_OUT_THREADS, Dm::kOutSmem, s, mq, mp, mo, N, out,
                                         mix, r, static_cast<long long>(g_wait_limit)))))
    return st;
  return launch_status();
}

int run_linear_d(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                 __nv_bfloat16* out, int BH, int N, int d, int mix, float r, cudaStream_t s) {
  return d == 64 ? run_linear<64>(q, k, v, out, BH, N, mix, r, s)
                 : run_linear<128>(q, k, v, out, BH, N, mix, r, s);
}

int check_linear_args(const void* q, const void* k, const void* v, const void* out, int B,
                      int heads, int N, int d, int dtype, int* BH) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return VA_ERR_INVALID;
  if (B < 1 || heads < 1 || N < 1) return VA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return VA_ERR_INVALID;
  if (dtype != VA_BF16 || (d != 64 && d != 128)) return VA_ERR_UNSUPPORTED;
  const int64_t BH64 = static_cast<int64_t>(B) * heads;
  if (BH64 > 65535 || BH64 * N >= (1LL << 31)) return VA_ERR_UNSUPPORTED;
  *BH = static_cast<int>(BH64);
  return VA_OK;
}

}  // namespace

VA_EXPORT int va_linear_attn_fwd(const void* q, const void* k, const void* v, void* out, int B,
                                 int heads, int N, int d, int dtype, va_stream_t stream) {
  int BH = 0;
  const int st = check_linear_args(q, k, v, out, B, heads, N, d, dtype, &BH);
  if (st) return st;
  using T = __nv_bfloat16;
  return run_linear_d(static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
                      static_cast<T*>(out), BH, N, d, 0, 0.f, reinterpret_cast<cudaStream_t>(stream));
}

VA_EXPORT int va_mixed_attn_fwd(const void* q, const void* k, const void* v, const va_mask* m,
                                float r, void* out, int B, int heads, int N, int d, float scale,
                                int dtype, va_stream_t stream) {
  int BH = 0;
  int st = check_linear_args(q, k, v, out, B, heads, N, d, dtype, &BH);
  if (st) return st;
  if (m == nullptr || N != m->N) return VA_ERR_INVALID;
  if (!(r >= 0.f && r <= 1.f)) return VA_ERR_INVALID;
  if ((st = check_mask_device(m))) return st;
  using T = __nv_bfloat16;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (r > 0.f &&
      (st = va_sparse_attn_fwd(q, k, v, m, out, nullptr, B, heads, N, d, scale, dtype, stream)))
    return st;
  if (r == 1.f) return VA_OK;
  return run_linear_d(static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
                      static_cast<T*>(out), BH, N, d, r > 0.f ? 1 : 0, r, s);
}

// ------------------------------------------------------------------ LIPAR --

VA_EXPORT int va_lipar_prune(const void* x, int B, int T, int H, int W, int C, float tau,
                             int dtype, uint8_t* keep, int32_t* order, int32_t* src,
                             int32_t* count, va_stream_t stream) {
  if (x == nullptr || keep == nullptr || order == nullptr || src == nullptr || count == nullptr)
    return VA_ERR_INVALID;
  if (B < 1 || T < 1 || H < 1 || W < 1 || C < 1 || std::isnan(tau)) return VA_ERR_INVALID;
  if (dtype != VA_BF16 && dtype != VA_F32) return VA_ERR_UNSUPPORTED;
  const int64_t N64 = static_cast<int64_t>(T) * H * W;
  if (N64 >= (1LL << 31) || static_cast<int64_t>(B) * N64 * C >= (1LL << 40) || B > 65535)
    return VA_ERR_UNSUPPORTED;
  const size_t esz = dtype == VA_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(x) & (esz - 1)) ||
      (reinterpret_cast<uintptr_t>(order) & 3u) || (reinterpret_cast<uintptr_t>(src) & 3u) ||
      (reinterpret_cast<uintptr_t>(count) & 3u))
    return VA_ERR_INVALID;
  const int N = static_cast<int>(N64), F = H * W;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Scoped scratch(s);
  uint8_t* changed;
  int* slot;
  int st;
  if ((st = scratch.alloc(&changed, static_cast<size_t>(B) * N)) ||
      (st = scratch.alloc(&slot, static_cast<size_t>(B) * N)))
    return st;
  const dim3 gw((N + 7) / 8, B), gt((N + 255) / 256, B);
  if (dtype == VA_BF16)
    va::lp_changed_kernel<__nv_bfloat16><<<gw, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(x), N, F, C, tau, changed);
  else
    va::lp_changed_kernel<float><<<gw, 256, 0, s>>>(static_cast<const float*>(x), N, F, C, tau,
                                                    changed);
  va::lp_keep_kernel<<<gt, 256, 0, s>>>(changed, N, H, W, keep);
  va::lp_compact_kernel<<<B, 1024, 0, s>>>(keep, N, slot, order, count);
  va::lp_src_kernel<<<dim3((F + 255) / 256, B), 256, 0, s>>>(slot, T, F, src);
  return launch_status();
}

namespace {

int lipar_rows_check(const void* a, const void* b, int B, int heads, int N, int d, int dtype,
                     int* row16) {
  if (a == nullptr || b == nullptr) return VA_ERR_INVALID;
  if (B < 1 || heads < 1 || N < 1 || d < 1) return VA_ERR_INVALID;
  if (dtype != VA_BF16 && dtype != VA_F32) return VA_ERR_UNSUPPORTED;
  const int64_t bytes = static_cast<int64_t>(d) * (dtype == VA_BF16 ? 2 : 4);
  if (bytes % 16 != 0) return VA_ERR_UNSUPPORTED;
  if (!aligned16(a) || !aligned16(b)) return VA_ERR_INVALID;
  const int64_t BH = static_cast<int64_t>(B) * heads;
  if (BH > 65535 || BH * N >= (1LL << 40)) return VA_ERR_UNSUPPORTED;
  *row16 = static_cast<int>(bytes / 16);
  return VA_OK;
}

}  // namespace

VA_EXPORT int va_lipar_gather(const void* x, const int32_t* order, const int32_t* count, int B,
                              int heads, int N, int d, int dtype, void* out,
                              va_stream_t stream) {
  int row16 = 0;
  int st = lipar_rows_check(x, out, B, heads, N, d, dtype, &row16);
  if (st) return st;
  if (order == nullptr || count == nullptr) return VA_ERR_INVALID;
  va::lp_gather_kernel<<<dim3((N + 7) / 8, B * heads), 256, 0,
                         reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(x), order, count, heads, N, row16, static_cast<uint4*>(out));
  return launch_status();
}

VA_EXPORT int va_lipar_restore(const void* y, const int32_t* src, int B, int heads, int N, int d,
                               int dtype, void* out, va_stream_t stream) {
  int row16 = 0;
  int st = lipar_rows_check(y, out, B, heads, N, d, dtype, &row16);
  if (st) return st;
  if (src == nullptr) return VA_ERR_INVALID;
  va::lp_restore_kernel<<<dim3((N + 7) / 8, B * heads), 256, 0,
                          reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(y), src, heads, N, row16, static_cast<uint4*>(out));
  return launch_status();
}

// ------------------------------------------------------------ clustering --

namespace {

constexpr int kMaxClusters = 4096;

template <typename T, int D>
int set_smem_attrs() {
  static DeviceOnce once;
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  return device_once(once, dev, [] {
    int r;
    if ((r = cuda_status(cudaFuncSetAttribute(va::km_assign_kernel<T, D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              2 * D * va::KM_PT * 4))) ||
        (r = cuda_status(cudaFuncSetAttribute(va::probe_pass1_kernel<T, D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              va::probe_smem_bytes<D>(kMaxClusters)))) ||
        (r = cuda_status(cudaFuncSetAttribute(va::probe_pass2_kernel<T, D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              va::probe_smem_bytes<D>(kMaxClusters)))) ||
        (r = cuda_status(cudaFuncSetAttribute(va::comp_attn_kernel<T, D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              va::comp_smem_bytes<D>(kMaxClusters)))))
      return r;
    return VA_OK;
  });
}

// Member lists in ascending token order from counts and offsets: per-tile
// counts, their scan down the tiles, then the placement (deterministic).
int stable_lists(const int* assign, int BH, int N, int C, const int* off, int* perm,
                 cudaStream_t s) {
  const int ntiles = (N + va::KS_TILE - 1) / va::KS_TILE;
  Scoped scratch(s);
  int* tbase = nullptr;
  if (int st = scratch.alloc(&tbase, static_cast<size_t>(BH) * ntiles * C)) return st;
  const size_t hist = sizeof(int) * static_cast<size_t>(C);
  va::km_tile_count_kernel<<<dim3(ntiles, BH), 256, hist, s>>>(assign, N, C, tbase);
  va::km_tile_scan_kernel<<<dim3((C + 255) / 256, BH), 256, 0, s>>>(off, C, ntiles, tbase);
  va::km_tile_place_kernel<<<dim3(ntiles, BH), 128, hist, s>>>(assign, N, C, tbase, perm);
  return launch_status();
}

// Member lists of an assignment: count -> offsets -> perm, each cluster's
// members in ascending token order. count must be zeroed by the caller.
int cluster_lists(const int* assign, int BH, int N, int C, int* count, int* off, int* fill,
                  int* perm, cudaStream_t s) {
  const dim3 g((N + 255) / 256, BH);
  va::km_count_kernel<<<g, 256, 0, s>>>(assign, N, C, count);
  va::km_offsets_kernel<<<BH, 1024, 0, s>>>(count, C, off, fill);
  if (int st = launch_status()) return st;
  return stable_lists(assign, BH, N, C, off, perm, s);
}

// bf16, d = D: distances on the tensor cores (split-bf16 centroids).
template <int D>
int run_cluster_tc(const __nv_bfloat16* x, const int* init, const float* c0, int BH, int N, int C,
                   int iters, int* assign, float* cent, int* count, cudaStream_t s) {
  static DeviceOnce once;
  static int num_sms[64] = {0};
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  st = device_once(once, dev, [dev] {
    int r;
    if ((r = set_smem_attrs<__nv_bfloat16, D>()) ||
        (r = cuda_status(cudaFuncSetAttribute(va::km_assign_tc_kernel<D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              va::KaDim<D>::kSmemBytes))) ||
        (r = cuda_status(cudaDeviceGetAttribute(&num_sms[dev], cudaDevAttrMultiProcessorCount,
                                                dev))))
      return r;
    return VA_OK;
  });
  if (st) return st;
  // assignment grid: resident chunks of 256 clusters, point tiles split so
  // that the persistent CTAs fill about one wave
  const int nchunks = (C + va::KA_CHUNK - 1) / va::KA_CHUNK;
  const int ntiles = (N + 127) / 128;
  const long long per_wave = static_cast<long long>(BH) * nchunks;
  const int nsplit = static_cast<int>(
      std::max(1LL, std::min(static_cast<long long>(ntiles), num_sms[dev] / per_wave)));
  if (nchunks > 65535) return VA_ERR_UNSUPPORTED;
  Scoped scratch(s);
  float* cnorm = nullptr;
  int *off = nullptr, *fill = nullptr, *perm = nullptr, *prev = nullptr;
  __nv_bfloat16 *hi = nullptr, *lo = nullptr;
  unsigned long long* sums = nullptr;
  const size_t nc = static_cast<size_t>(BH) * C * D;
  if ((st = scratch.alloc(&cnorm, static_cast<size_t>(BH) * C)) ||
      (st = scratch.alloc(&off, static_cast<size_t>(BH) * (C + 1))) ||
      (st = scratch.alloc(&fill, static_cast<size_t>(BH) * C)) ||
      (st = scratch.alloc(&perm, static_cast<size_t>(BH) * N)) ||
      (st = scratch.alloc(&prev, static_cast<size_t>(BH) * N)) ||
      (st = scratch.alloc(&hi, nc)) || (st = scratch.alloc(&lo, nc)) ||
      (st = scratch.alloc(&sums, nc)))
    return st;
  float* pdist = nullptr;
  int* pidx = nullptr;
  if (nchunks > 1) {
    const size_t np = static_cast<size_t>(BH) * nchunks * N;
    if ((st = scratch.alloc(&pdist, np)) || (st = scratch.alloc(&pidx, np))) return st;
  }
  CUtensorMap mx, mh, ml;
  if ((st = encode_bf16_rows(&mx, x, BH, N, D)) || (st = encode_bf16_rows(&mh, hi, BH, C, D)) ||
      (st = encode_bf16_rows(&ml, lo, BH, C, D)))
    return st;
  const dim3 gc((C + 7) / 8, BH);
  const dim3 ga(nsplit, nchunks, BH);
  const dim3 gn((N + 255) / 256, BH);
  const unsigned gs = static_cast<unsigned>((nc + 255) / 256);
  if (c0 != nullptr)
    va::km_warm_kernel<D><<<gc, 256, 0, s>>>(c0, C, cent, cnorm);
  else
    va::km_init_kernel<__nv_bfloat16, D><<<gc, 256, 0, s>>>(x, init, N, C, cent, cnorm);
  va::km_split_kernel<<<gs, 256, 0, s>>>(cent, static_cast<long long>(nc), hi, lo);
  const int rounds = iters > 0 ? iters : 1;
  for (int it = 0; it < rounds; ++it) {
    if ((st = cuda_status(cudaMemsetAsync(count, 0, sizeof(int) * BH * C, s)))) return st;
    va::km_assign_tc_kernel<D><<<ga, va::KA_THREADS, va::KaDim<D>::kSmemBytes, s>>>(
        mx, mh, ml, cnorm, N, C, assign, count, pdist, pidx, g_wait_limit);
    if (nchunks > 1)
      va::ka_merge_kernel<<<dim3((N + 255) / 256, BH), 256, 0, s>>>(pdist, pidx, N, C, nchunks,
                                                                   assign, count);
    if (iters == 0) break;
    if (it <= 1) {
      // member sums from scratch (cluster-ordered runs) while many points still
      // move: at the Wan shape a third of them do after the first update, where
      // the moves alone cost more than the full sum
      va::km_offsets_kernel<<<BH, 1024, 0, s>>>(count, C, off, fill);
      va::km_scatter_kernel<<<gn, 256, 0, s>>>(assign, N, C, off, fill, perm);
      if ((st = cuda_status(cudaMemsetAsync(sums, 0, sizeof(unsigned long long) * nc, s))) ||
          (st = cuda_status(cudaMemcpyAsync(prev, assign, sizeof(int) * BH * N,
                                            cudaMemcpyDeviceToDevice, s))))
        return st;
      va::km_sum_kernel<D><<<gn, 256, 0, s>>>(x, N, C, perm, assign, sums);
    } else {
      // later iterations move the points that changed cluster (a few percent,
      // as the clustering settles); the sums stay exact
      va::km_delta_kernel<D><<<gn, 256, 0, s>>>(x, N, C, prev, assign, sums);
    }
    va::km_finalize_kernel<D><<<gc, 256, 0, s>>>(sums, count, C, cent, cnorm, hi, lo, 1);
  }
  return launch_status();
}

template <typename T, int D>
int run_cluster(const T* x, const int* init, const float* c0, int BH, int N, int C, int iters,
                int* assign, float* cent, int* count, cudaStream_t s) {
  int st = set_smem_attrs<T, D>();
  if (st) return st;
  Scoped scratch(s);
  float* cnorm = nullptr;
  int *off = nullptr, *fill = nullptr, *perm = nullptr;
  if ((st = scratch.alloc(&cnorm, static_cast<size_t>(BH) * C)) ||
      (st = scratch.alloc(&off, static_cast<size_t>(BH) * (C + 1))) ||
      (st = scratch.alloc(&fill, static_cast<size_t>(BH) * C)) ||
      (st = scratch.alloc(&perm, static_cast<size_t>(BH) * N)))
    return st;
  const dim3 gc((C + 7) / 8, BH);
  const dim3 ga((N + va::KM_PT - 1) / va::KM_PT, BH);
  const dim3 gn((N + 255) / 256, BH);
  if (c0 != nullptr)
    va::km_warm_kernel<D><<<gc, 256, 0, s>>>(c0, C, cent, cnorm);
  else
    va::km_init_kernel<T, D><<<gc, 256, 0, s>>>(x, init, N, C, cent, cnorm);
  const int rounds = iters > 0 ? iters : 1;
  for (int it = 0; it < rounds; ++it) {
    if ((st = cuda_status(cudaMemsetAsync(count, 0, sizeof(int) * BH * C, s)))) return st;
    va::km_assign_kernel<T, D><<<ga, va::KM_THREADS, 2 * D * va::KM_PT * 4, s>>>(
        x, cent, cnorm, N, C, assign, count);
    if (iters == 0) break;
    va::km_offsets_kernel<<<BH, 1024, 0, s>>>(count, C, off, fill);
    if ((st = stable_lists(assign, BH, N, C, off, perm, s))) return st;
    va::km_means_kernel<T, D><<<gc, 256, 0, s>>>(x, N, C, off, perm, cent, cnorm, 1);
  }
  return launch_status();
}

}  // namespace

namespace {

// Seeded (init_idx) or warm-started (c0) Lloyd k-means; exactly one is set.
int cluster_entry(const void* x, const int32_t* init_idx, const float* c0, int B, int heads,
                  int N, int d, int C, int iters, int dtype, int32_t* assign, float* centroid,
                  int32_t* count, va_stream_t stream) {
  if (x == nullptr || assign == nullptr || centroid == nullptr || count == nullptr)
    return VA_ERR_INVALID;
  if (B < 1 || heads < 1 || N < 1 || C < 1 || C > N || iters < 0) return VA_ERR_INVALID;
  if (!aligned16(x) || !aligned16(centroid) || (reinterpret_cast<uintptr_t>(assign) & 3u) ||
      (reinterpret_cast<uintptr_t>(count) & 3u) || (reinterpret_cast<uintptr_t>(init_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(c0) & 15u))
    return VA_ERR_INVALID;
  if (C > kMaxClusters || (d != 64 && d != 128)) return VA_ERR_UNSUPPORTED;
  const int64_t BH64 = static_cast<int64_t>(B) * heads;
  if (BH64 > 65535 || BH64 * N * d >= (1LL << 40)) return VA_ERR_UNSUPPORTED;
  const int BH = static_cast<int>(BH64);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int* ii = init_idx;
  if (dtype == VA_BF16) {
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    return d == 128 ? run_cluster_tc<128>(xb, ii, c0, BH, N, C, iters, assign, centroid, count, s)
                    : run_cluster_tc<64>(xb, ii, c0, BH, N, C, iters, assign, centroid, count, s);
  }
  if (dtype == VA_F32) {
    const float* xf = static_cast<const float*>(x);
    return d == 128 ? run_cluster<float, 128>(xf, ii, c0, BH, N, C, iters, assign, centroid,
                                              count, s)
                    : run_cluster<float, 64>(xf, ii, c0, BH, N, C, iters, assign, centroid,
                                             count, s);
  }
  return VA_ERR_UNSUPPORTED;
}

}  // namespace

VA_EXPORT int va_cluster(const void* x, const int32_t* init_idx, int B, int heads, int N, int d,
                         int C, int iters, int dtype, int32_t* assign, float* centroid,
                         int32_t* count, va_stream_t stream) {
  if (init_idx == nullptr) return VA_ERR_INVALID;
  return cluster_entry(x, init_idx, nullptr, B, heads, N, d, C, iters, dtype, assign, centroid,
                       count, stream);
}

VA_EXPORT int va_cluster_from(const void* x, const float* centroid_init, int B, int heads, int N,
                              int d, int C, int iters, int dtype, int32_t* assign,
                              float* centroid, int32_t* count, va_stream_t stream) {
  if (centroid_init == nullptr) return VA_ERR_INVALID;
  return cluster_entry(x, nullptr, centroid_init, B, heads, N, d, C, iters, dtype, assign,
                       centroid, count, stream);
}
// -------------------------------------------- compensation and routing --

namespace {

// Compensated attention on the tensor cores (bf16, d = D): cluster-ordered
// copies of Q, K, V, bf16 centroids, per-cluster slot prefixes and virtual
// biases, then comp_tc_kernel over pairs of 128-row query chunks.
template <int D>
int comp_tensor_cores(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                      int Cq, int Ck, int BH, int N, const int* nq, const int* qoff,
                      const int* qperm, const int* nk, const int* koff, const int* kperm,
                      const float* kc, const float* vc, const int* seln, const int* selc,
                      const uint8_t* sel, float scale, __nv_bfloat16* out, Scoped& scratch,
                      cudaStream_t s) {
  static DeviceOnce once;
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  st = device_once(once, dev, [] {
    cudaFuncAttributes fa;
    int r = cuda_status(cudaFuncGetAttributes(&fa, va::comp_tc_kernel<D>));
    if (r) return r;
    if (fa.numRegs != va::TC_LAUNCH_REGS) return VA_ERR_UNSUPPORTED;
    return cuda_status(cudaFuncSetAttribute(va::comp_tc_kernel<D>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            va::ct_smem_bytes<D>()));
  });
  if (st) return st;
  const size_t bh = static_cast<size_t>(BH);
  const int nv = (Ck + 127) / 128;
  __nv_bfloat16 *qs, *ks, *vs, *kcb, *vcb;
  int *selbox, *nch, *choff, *chfill;
  float* vbias;
  if ((st = scratch.alloc(&qs, bh * N * D)) || (st = scratch.alloc(&ks, bh * N * D)) ||
      (st = scratch.alloc(&vs, bh * N * D)) || (st = scratch.alloc(&kcb, bh * Ck * D)) ||
      (st = scratch.alloc(&vcb, bh * Ck * D)) ||
      (st = scratch.alloc(&selbox, bh * Cq * (Ck + 1))) ||
      (st = scratch.alloc(&vbias, bh * Cq * nv * 128)) || (st = scratch.alloc(&nch, bh * Cq)) ||
      (st = scratch.alloc(&choff, bh * (Cq + 1))) || (st = scratch.alloc(&chfill, bh * Cq)))
    return st;
  const dim3 gg((N + va::GR_ROWS<D> - 1) / va::GR_ROWS<D>, BH);
  va::gather_rows_kernel<D><<<gg, 128, 0, s>>>(q, qperm, N, qs);
  va::gather_rows_kernel<D><<<gg, 128, 0, s>>>(k, kperm, N, ks);
  va::gather_rows_kernel<D><<<gg, 128, 0, s>>>(v, kperm, N, vs);
  const long long ncen = static_cast<long long>(bh) * Ck * D;
  va::f32_to_bf16_kernel<<<static_cast<unsigned>((ncen + 255) / 256), 256, 0, s>>>(kc, ncen, kcb);
  va::f32_to_bf16_kernel<<<static_cast<unsigned>((ncen + 255) / 256), 256, 0, s>>>(vc, ncen, vcb);
  va::comp_prep_kernel<<<dim3((Cq + 7) / 8, BH), 256, 0, s>>>(nk, seln, selc, sel, Cq, Ck, nv,
                                                             selbox, vbias);
  va::chunk_count_kernel<<<dim3((Cq + 255) / 256, BH), 256, 0, s>>>(nq, Cq, 128, nch);
  va::km_offsets_kernel<<<BH, 1024, 0, s>>>(nch, Cq, choff, chfill);
  // slot table: per query cluster, its selected clusters' 8-row slots padded
  // to whole 16-slot tiles. Its size is only known on the device; it is
  // allocated for the bound sum_c ceil(n_c / 8) + 15 <= N / 8 + Ck + 16 slots
  // per query cluster, so no synchronisation is needed.
  int *slcnt, *sloff, *slfill, *slots;
  long long* slbase;
  if ((st = scratch.alloc(&slcnt, bh * Cq)) || (st = scratch.alloc(&sloff, bh * (Cq + 1))) ||
      (st = scratch.alloc(&slfill, bh * Cq)) || (st = scratch.alloc(&slbase, bh + 1)))
    return st;
  va::slot_count_kernel<<<dim3((Cq + 255) / 256, BH), 256, 0, s>>>(seln, selbox, Cq, Ck, slcnt);
  va::km_offsets_kernel<<<BH, 1024, 0, s>>>(slcnt, Cq, sloff, slfill);
  va::slot_base_kernel<<<1, 1, 0, s>>>(sloff, Cq, BH, slbase);
  if ((st = launch_status())) return st;
  const size_t slot_bound =
      bh * static_cast<size_t>(Cq) * (static_cast<size_t>(N) / 8 + static_cast<size_t>(Ck) + 16);
  if ((st = scratch.alloc(&slots, slot_bound))) return st;
  va::slot_fill_kernel<<<dim3(Cq, BH), 256, 0, s>>>(koff, seln, selc, selbox, Cq, Ck, slbase,
                                                   sloff, slots);
  if ((st = launch_status())) return st;
  CUtensorMap mq, mkc, mvc;
  va::CompSlotMaps slot_maps;
  if ((st = encode_bf16_rows_box(&mq, qs, BH, N, D, 128)) ||
      (st = encode_bf16_rows_box(&mkc, kcb, BH, Ck, D, 128)) ||
      (st = encode_bf16_rows_box(&mvc, vcb, BH, Ck, D, 128)))
    return st;
  for (int i = 0; i < va::CT_NBOX; ++i)
    if ((st = encode_bf16_rows_box(&slot_maps.k[i], ks, BH, N, D, 8 << i)) ||
        (st = encode_bf16_rows_box(&slot_maps.v[i], vs, BH, N, D, 8 << i)))
      return st;
  va::CompArgs a;
  a.choff = choff;
  a.qoff = qoff;
  a.qperm = qperm;
  a.koff = koff;
  a.nk = nk;
  a.seln = seln;
  a.selc = selc;
  a.selbox = selbox;
  a.vbias = vbias;
  a.slots = slots;
  a.slotbase = slbase;
  a.slotoff = sloff;
  a.out = out;
  a.N = N;
  a.Cq = Cq;
  a.Ck = Ck;
  a.nv = nv;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit = g_wait_limit;
  const int max_chunks = (N + 127) / 128 + Cq;
  va::comp_tc_kernel<D><<<dim3((max_chunks + 1) / 2, BH), va::TC_THREADS, va::ct_smem_bytes<D>(),
                          s>>>(mq, mkc, mvc, slot_maps, a);
  return launch_status();
}

// Error probe on the tensor cores (bf16, d = D): padded cluster-ordered
// K/V with group metadata, three bf16 pieces of the proxies, then pass 1
// (split partials of m2, Z, O), their merge and pass 2 (err).
template <int D>
int probe_tensor_cores(const __nv_bfloat16* k, const __nv_bfloat16* v, int Cq, int Ck, int BH,
                       int N, const int* nq, const int* nk, const int* koff, const int* kperm,
                       const float* qc, const float* vc, float scale, float* err,
                       Scoped& scratch, cudaStream_t s) {
  static DeviceOnce once;
  static int num_sms[64] = {0};
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  st = device_once(once, dev, [dev] {
    cudaFuncAttributes fa1, fa2;
    int r;
    if ((r = cuda_status(cudaFuncGetAttributes(&fa1, va::probe_tc_kernel<1, D>))) ||
        (r = cuda_status(cudaFuncGetAttributes(&fa2, va::probe_tc_kernel<2, D>))))
      return r;
    if (fa1.numRegs != va::PT_LAUNCH_REGS || fa2.numRegs != va::PT_LAUNCH_REGS)
      return VA_ERR_UNSUPPORTED;
    if ((r = cuda_status(cudaFuncSetAttribute(va::probe_tc_kernel<1, D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              va::PtDim<D>::kSmem))) ||
        (r = cuda_status(cudaFuncSetAttribute(va::probe_tc_kernel<2, D>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              va::PtDim<D>::kSmem))) ||
        (r = cuda_status(cudaDeviceGetAttribute(&num_sms[dev], cudaDevAttrMultiProcessorCount,
                                                dev))))
      return r;
    return VA_OK;
  });
  if (st) return st;
  const size_t bh = static_cast<size_t>(BH);
  const int Cqp = (Cq + 127) / 128 * 128;
  const int ntiles = Cqp / 128;
  // rows per head: every cluster padded to 16, plus 64 zero rows after them
  const long long Npad = (static_cast<long long>(N) + 15LL * Ck + 64 + 15) / 16 * 16;
  if (Npad > (1LL << 30) || static_cast<long long>(BH) * ntiles > 65535)
    return VA_ERR_UNSUPPORTED;
  const int G = static_cast<int>(Npad / 16);
  const long long per_head = static_cast<long long>(BH) * ntiles;
  const int NS = static_cast<int>(
      std::max(1LL, std::min(static_cast<long long>(Ck), num_sms[dev] / per_head)));
  int *cnt16, *kpoff, *kpfill, *gmeta;
  __nv_bfloat16 *kpad, *vpad, *qp;
  float *part, *mzo;
  if ((st = scratch.alloc(&cnt16, bh * Ck)) || (st = scratch.alloc(&kpoff, bh * (Ck + 1))) ||
      (st = scratch.alloc(&kpfill, bh * Ck)) ||
      (st = scratch.alloc(&gmeta, bh * static_cast<size_t>(G))) ||
      (st = scratch.alloc(&kpad, bh * static_cast<size_t>(Npad) * D)) ||
      (st = scratch.alloc(&vpad, bh * static_cast<size_t>(Npad) * D)) ||
      (st = scratch.alloc(&qp, bh * 3 * Cqp * D)) ||
      (st = scratch.alloc(&part, bh * Cq * NS * va::PtDim<D>::kRow)) ||
      (st = scratch.alloc(&mzo, bh * Cq * va::PtDim<D>::kRow)))
    return st;
  const long long nbk = static_cast<long long>(bh) * Ck;
  va::pad16_count_kernel<<<static_cast<unsigned>((nbk + 255) / 256), 256, 0, s>>>(
      nk, static_cast<int>(nbk), cnt16);
  va::km_offsets_kernel<<<BH, 1024, 0, s>>>(cnt16, Ck, kpoff, kpfill);
  va::pad_gather_kernel<D><<<dim3(Ck + 1, BH), 128, 0, s>>>(k, v, N, Ck, nk, koff, kperm, kpoff,
                                                           Npad, G, kpad, vpad, gmeta);
  va::proxy_pieces_kernel<D><<<dim3(Cqp, BH), D, 0, s>>>(qc, Cq, Cqp, qp);
  if ((st = launch_status())) return st;
  CUtensorMap mq, mk, mv;
  if ((st = encode_bf16_rows_box(&mq, qp, BH, 3 * Cqp, D, 128)) ||
      (st = encode_bf16_rows_box(&mk, kpad, BH, static_cast<int>(Npad), D, va::PT_KT)) ||
      (st = encode_bf16_rows_box(&mv, vpad, BH, static_cast<int>(Npad), D, va::PT_KT)))
    return st;
  va::ProbeArgs a;
  a.gmeta = gmeta;
  a.kpoff = kpoff;
  a.nq = nq;
  a.mzo = mzo;
  a.vc = vc;
  a.part = part;
  a.err = err;
  a.Cq = Cq;
  a.Ck = Ck;
  a.Cqp = Cqp;
  a.G = G;
  a.NS = NS;
  a.sl2 = scale * 1.4426950408889634f;
  a.wait_limit = g_wait_limit;
  const dim3 grid(NS, ntiles, BH);
  va::probe_tc_kernel<1, D><<<grid, va::PT_THREADS, va::PtDim<D>::kSmem, s>>>(mq, mk, mv, a);
  va::probe_tc_combine_kernel<D><<<dim3(Cq, BH), D, 0, s>>>(part, Cq, NS, mzo);
  va::probe_tc_kernel<2, D><<<grid, va::PT_THREADS, va::PtDim<D>::kSmem, s>>>(mq, mk, mv, a);
  return launch_status();
}

// Error probe on the FP32 pipe (fp32 inputs or d = 64): pass 1 split
// partials of m, Z, O, their merge, pass 2 err.
template <typename T, int D>
int probe_simt(const T* k, const T* v, int Cq, int Ck, int BH, int N, const int* nq,
               const int* nk, const int* koff, const int* kperm, const int* kassign,
               const float* qc, const float* kc, const float* vc, float scale, float* err,
               Scoped& scratch, cudaStream_t s) {
  const size_t bh = static_cast<size_t>(BH);
  float *part, *mzo;
  int st;
  if ((st = scratch.alloc(&part, bh * Cq * va::PR_SPLIT * (D + 2))) ||
      (st = scratch.alloc(&mzo, bh * Cq * (D + 2))))
    return st;
  const int pg = (Cq + va::PR_PG - 1) / va::PR_PG;
  va::probe_pass1_kernel<T, D><<<dim3(pg, va::PR_SPLIT, BH), va::PR_THREADS,
                                 va::probe_smem_bytes<D>(0), s>>>(k, v, N, Cq, qc, scale, part);
  va::probe_combine_kernel<D><<<dim3(Cq, BH), D, 0, s>>>(part, Cq, mzo);
  va::probe_pass2_kernel<T, D><<<dim3(pg, va::PR_CSPLIT, BH), va::PR_THREADS,
                                 va::probe_smem_bytes<D>(Ck), s>>>(
      k, v, N, Cq, Ck, qc, nq, kc, vc, nk, koff, kperm, kassign, mzo, scale, err);
  return launch_status();
}

template <typename T, int D>
int run_compensate(const T* q, const T* k, const T* v, const int* qassign, int Cq,
                   const int* kassign, int Ck, long long budget, float scale, int BH, int N,
                   T* out, float* err_out, uint8_t* sel_out, cudaStream_t s) {
  int st = set_smem_attrs<T, D>();
  if (st) return st;
  Scoped scratch(s);
  int *nq, *qoff, *qfill, *qperm, *nk, *koff, *kfill, *kperm, *seln, *selc, *nch, *choff, *chfill;
  float *qc, *kc, *vc, *err;
  unsigned long long* cut;
  const size_t bh = static_cast<size_t>(BH);
  if ((st = scratch.alloc(&nq, bh * Cq)) || (st = scratch.alloc(&qoff, bh * (Cq + 1))) ||
      (st = scratch.alloc(&qfill, bh * Cq)) || (st = scratch.alloc(&qperm, bh * N)) ||
      (st = scratch.alloc(&nk, bh * Ck)) || (st = scratch.alloc(&koff, bh * (Ck + 1))) ||
      (st = scratch.alloc(&kfill, bh * Ck)) || (st = scratch.alloc(&kperm, bh * N)) ||
      (st = scratch.alloc(&qc, bh * Cq * D)) || (st = scratch.alloc(&kc, bh * Ck * D)) ||
      (st = scratch.alloc(&vc, bh * Ck * D)) || (st = scratch.alloc(&seln, bh * Cq)) ||
      (st = scratch.alloc(&selc, bh * Cq * Ck)) || (st = scratch.alloc(&cut, bh)) ||
      (st = scratch.alloc(&nch, bh * Cq)) || (st = scratch.alloc(&choff, bh * (Cq + 1))) ||
      (st = scratch.alloc(&chfill, bh * Cq)))
    return st;
  err = err_out;
  if (err == nullptr && (st = scratch.alloc(&err, bh * Cq * Ck))) return st;

  // cluster sizes, member lists and member means of q (per query cluster) and
  // of k, v (per key cluster); empty clusters get zero means
  if ((st = cuda_status(cudaMemsetAsync(nq, 0, sizeof(int) * bh * Cq, s))) ||
      (st = cuda_status(cudaMemsetAsync(nk, 0, sizeof(int) * bh * Ck, s))))
    return st;
  if ((st = cluster_lists(qassign, BH, N, Cq, nq, qoff, qfill, qperm, s)) ||
      (st = cluster_lists(kassign, BH, N, Ck, nk, koff, kfill, kperm, s)))
    return st;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    // balanced exact sums over the cluster-ordered members, then the means
    unsigned long long* sums;
    const size_t cmax = static_cast<size_t>(Cq > Ck ? Cq : Ck);
    if ((st = scratch.alloc(&sums, bh * cmax * D))) return st;
    struct MeanJob { const T* x; const int* perm; const int* assign; const int* count; int C;
                     float* mean; };
    const MeanJob jobs[3] = {{q, qperm, qassign, nq, Cq, qc}, {k, kperm, kassign, nk, Ck, kc},
                             {v, kperm, kassign, nk, Ck, vc}};
    for (const MeanJob& jb : jobs) {
      if ((st = cuda_status(
               cudaMemsetAsync(sums, 0, sizeof(unsigned long long) * bh * jb.C * D, s))))
        return st;
      va::km_sum_kernel<D><<<dim3((N + 255) / 256, BH), 256, 0, s>>>(jb.x, N, jb.C, jb.perm,
                                                                     jb.assign, sums);
      va::km_finalize_kernel<D><<<dim3((jb.C + 7) / 8, BH), 256, 0, s>>>(
          sums, jb.count, jb.C, jb.mean, nullptr, nullptr, nullptr, 0);
    }
  } else {
    va::km_means_kernel<T, D><<<dim3((Cq + 7) / 8, BH), 256, 0, s>>>(q, N, Cq, qoff, qperm, qc,
                                                                    nullptr, 0);
    va::km_means_kernel<T, D><<<dim3((Ck + 7) / 8, BH), 256, 0, s>>>(k, N, Ck, koff, kperm, kc,
                                                                    nullptr, 0);
    va::km_means_kernel<T, D><<<dim3((Ck + 7) / 8, BH), 256, 0, s>>>(v, N, Ck, koff, kperm, vc,
                                                                    nullptr, 0);
  }
  if ((st = launch_status())) return st;

  // probe: err = NaN where a cluster is empty, else the proxy error
  if ((st = cuda_status(cudaMemsetAsync(err, 0xFF, sizeof(float) * bh * Cq * Ck, s)))) return st;
  if constexpr (std::is_same<T, __nv_bfloat16>::value)
    st = probe_tensor_cores<D>(k, v, Cq, Ck, BH, N, nq, nk, koff, kperm, qc, vc, scale, err,
                               scratch, s);
  else
    st = probe_simt<T, D>(k, v, Cq, Ck, BH, N, nq, nk, koff, kperm, kassign, qc, kc, vc, scale,
                          err, scratch, s);
  if (st) return st;

  // routing
  uint8_t* sel = sel_out;
  if (sel == nullptr && (st = scratch.alloc(&sel, bh * Cq * Ck))) return st;
  unsigned long long *rkeys, *rcosts;
  if ((st = scratch.alloc(&rkeys, bh * Cq * Ck)) || (st = scratch.alloc(&rcosts, bh * Cq * Ck)))
    return st;
  va::route_keys_kernel<<<dim3((Cq * Ck + 255) / 256, BH), 256, 0, s>>>(err, nq, nk, Cq, Ck,
                                                                       rkeys, rcosts);
  unsigned long long *rstate, *rhist;
  unsigned int* rcount;
  if ((st = scratch.alloc(&rstate, bh * 4)) || (st = scratch.alloc(&rhist, bh * 256)) ||
      (st = scratch.alloc(&rcount, bh)))
    return st;
  va::route_init_kernel<<<(BH * 256 + 255) / 256, 256, 0, s>>>(budget, BH, rstate, rhist, rcount);
  const dim3 gsel((Cq * Ck + va::RS_PER_CTA - 1) / va::RS_PER_CTA, BH);
  // The low 32 bits of a key are the block index p * Ck + c: digits above its
  // bit length are 0 in every valid key, so those passes would only append
  // zero digits to the prefix (the mass under the prefix always exceeds the
  // remaining budget after the first pass) and are skipped.
  int idx_bits = 0;
  while (idx_bits < 32 && (static_cast<long long>(Cq) * Ck - 1) >> idx_bits) ++idx_bits;
  for (int shift = 56; shift >= 0; shift -= 8) {
    if (shift < 32 && shift >= idx_bits) continue;
    va::route_pass_kernel<<<gsel, va::RS_THREADS, 0, s>>>(rkeys, rcosts, Cq * Ck, shift, rstate,
                                                           rhist, rcount);
  }
  va::route_cut_kernel<<<(BH + 255) / 256, 256, 0, s>>>(rstate, BH, cut);
  va::route_mark_kernel<<<dim3(Cq, BH), 256, 0, s>>>(err, nq, nk, Cq, Ck, cut, sel, seln, selc);
  if ((st = launch_status())) return st;

  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    return comp_tensor_cores<D>(q, k, v, Cq, Ck, BH, N, nq, qoff, qperm, nk, koff, kperm, kc, vc,
                             seln, selc, sel, scale, out, scratch, s);
  }

  // compensated attention: chunks of up to 64 queries of one query cluster
  va::comp_chunks_kernel<<<dim3((Cq + 255) / 256, BH), 256, 0, s>>>(nq, Cq, nch);
  va::km_offsets_kernel<<<BH, 1024, 0, s>>>(nch, Cq, choff, chfill);
  const int max_chunks = (N + va::CA_QT - 1) / va::CA_QT + Cq;
  va::comp_attn_kernel<T, D><<<dim3(max_chunks, BH), va::CA_THREADS, va::comp_smem_bytes<D>(Ck),
                               s>>>(q, k, v, N, Cq, Ck, choff, qoff, qperm, koff, kperm, kc, vc,
                                    nk, seln, selc, scale * 1.4426950408889634f, out);
  return launch_status();
}

}  // namespace

VA_EXPORT int va_compensate_route(const void* q, const void* k, const void* v,
                                  const int32_t* qassign, int Cq, const int32_t* kassign, int Ck,
                                  double density, float scale, int B, int heads, int N, int d,
                                  int dtype, void* out, float* err_out, uint8_t* sel_out,
                                  va_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || qassign == nullptr ||
      kassign == nullptr || out == nullptr)
    return VA_ERR_INVALID;
  if (B < 1 || heads < 1 || N < 1 || Cq < 1 || Ck < 1 || Cq > N || Ck > N) return VA_ERR_INVALID;
  if (!(density >= 0.0 && density <= 1.0) || !std::isfinite(scale)) return VA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(qassign) & 3u) || (reinterpret_cast<uintptr_t>(kassign) & 3u) ||
      (reinterpret_cast<uintptr_t>(err_out) & 3u))
    return VA_ERR_INVALID;
  if (Cq > kMaxClusters || Ck > kMaxClusters || (d != 64 && d != 128)) return VA_ERR_UNSUPPORTED;
  const int64_t BH64 = static_cast<int64_t>(B) * heads;
  if (BH64 > 65535 || BH64 * N * d >= (1LL << 40)) return VA_ERR_UNSUPPORTED;
  const int BH = static_cast<int>(BH64);
  const long long budget =
      static_cast<long long>(std::floor(density * static_cast<double>(N) * static_cast<double>(N)));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == VA_BF16) {
    using T = __nv_bfloat16;
    const T *qt = static_cast<const T*>(q), *kt = static_cast<const T*>(k),
            *vt = static_cast<const T*>(v);
    T* ot = static_cast<T*>(out);
    return d == 128 ? run_compensate<T, 128>(qt, kt, vt, qassign, Cq, kassign, Ck, budget, scale,
                                             BH, N, ot, err_out, sel_out, s)
                    : run_compensate<T, 64>(qt, kt, vt, qassign, Cq, kassign, Ck, budget, scale,
                                            BH, N, ot, err_out, sel_out, s);
  }
  if (dtype == VA_F32) {
    using T = float;
    const T *qt = static_cast<const T*>(q), *kt = static_cast<const T*>(k),
            *vt = static_cast<const T*>(v);
    T* ot = static_cast<T*>(out);
    return d == 128 ? run_compensate<T, 128>(qt, kt, vt, qassign, Cq, kassign, Ck, budget, scale,
                                             BH, N, ot, err_out, sel_out, s)
                    : run_compensate<T, 64>(qt, kt, vt, qassign, Cq, kassign, Ck, budget, scale,
                                            BH, N, ot, err_out, sel_out, s);
  }
  return VA_ERR_UNSUPPORTED;
}

// ------------------------------------------------- allocation-free masks --
//
// va_mask_build_static: the mask build of va_mask_build for callers that must
// not allocate device memory. Its scratch lives in one statically sized
// device array (every GPU that loads the library holds it until exit); the
// caller passes the CSR output arrays.

namespace {

constexpr size_t kStaticMaxBlocks = VA_STATIC_MAX_BLOCKS;
// layout: summary (2 x int64, padded to 256 B) | key tokens (int64 x max) |
// counts (int32 x max) | histogram (int32 x (max + 1), padded to 8 B) |
// row order (int32 x max)
constexpr size_t kScrSummary = 0;
constexpr size_t kScrKeyTok = 256;
constexpr size_t kScrCnt = kScrKeyTok + 8 * kStaticMaxBlocks;
constexpr size_t kScrHist = kScrCnt + 4 * kStaticMaxBlocks;
constexpr size_t kScrOrder = kScrHist + ((4 * (kStaticMaxBlocks + 1) + 7) & ~size_t(7));
constexpr size_t kScrBytes = kScrOrder + 4 * kStaticMaxBlocks;

}  // namespace

static __device__ __align__(256) unsigned char g_static_scratch[kScrBytes];

namespace {

std::mutex g_static_mu;
void* g_static_addr[64] = {nullptr};

// Device address of g_static_scratch on the current device (looked up once
// per device; the host-side symbol itself is not a device address).
int static_scratch(void** out) {
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st) return st;
  if (dev < 0 || dev >= 64) return VA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void* p = nullptr;
    st = cuda_status(cudaGetSymbolAddress(&p, g_static_scratch));
    if (st) return st;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return VA_OK;
}

}  // namespace

VA_EXPORT int va_mask_build_static(int kind, int T, int H, int W, const va_mask_params* params,
                                   int step, int32_t* row_ptr, int32_t* col_idx,
                                   int64_t col_capacity, int64_t* nnz, va_stream_t stream) {
  if (params == nullptr || row_ptr == nullptr || nnz == nullptr) return VA_ERR_INVALID;
  if (col_capacity < 0 || (col_idx == nullptr && col_capacity > 0)) return VA_ERR_INVALID;
  const va_mask_params p = *params;
  int64_t N64 = 0, nb64 = 0;
  if (int st0 = mask_grid_args(kind, T, H, W, p, &N64, &nb64)) return st0;
  const int64_t F64 = static_cast<int64_t>(H) * W;
  if (nb64 > static_cast<int64_t>(kStaticMaxBlocks)) return VA_ERR_UNSUPPORTED;
  *nnz = 0;

  va::MaskDesc md;
  md.kind = kind;
  md.T = T;
  md.F = static_cast<int>(F64);
  md.N = static_cast<int>(N64);
  md.block = p.block;
  md.nb = static_cast<int>(nb64);
  md.w0 = (kind == VA_MASK_RADIAL && p.w0 == 0) ? md.F : p.w0;
  md.local = p.local;
  md.period = p.period;
  md.anchor0 = p.anchor0;
  md.rot_stride = p.rot_stride;
  md.step = step;

  void* base = nullptr;
  int st = static_scratch(&base);
  if (st) return st;
  unsigned char* b = static_cast<unsigned char*>(base);
  long long* summary = reinterpret_cast<long long*>(b + kScrSummary);
  long long* keytok = reinterpret_cast<long long*>(b + kScrKeyTok);
  int* cnt = reinterpret_cast<int*>(b + kScrCnt);
  int* hist = reinterpret_cast<int*>(b + kScrHist);
  int* order = reinterpret_cast<int*>(b + kScrOrder);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // The previous call's contents stay in the array: start the summary at zero.
  if ((st = cuda_status(cudaMemsetAsync(summary, 0, 2 * sizeof(long long), s)))) return st;
  const int threads = 256;
  const int blocks = static_cast<int>((static_cast<int64_t>(md.nb) * 32 + threads - 1) / threads);
  va::mask_count_kernel<<<blocks, threads, 0, s>>>(md, cnt, keytok);
  va::mask_scan_kernel<<<1, 1024, 0, s>>>(md, cnt, keytok, row_ptr, summary, order, hist);
  if ((st = launch_status())) return st;
  long long host_summary[2] = {0, 0};
  if ((st = cuda_status(cudaMemcpyAsync(host_summary, summary, sizeof(host_summary),
                                        cudaMemcpyDeviceToHost, s))) ||
      (st = cuda_status(cudaStreamSynchronize(s))))
    return st;
  *nnz = host_summary[0];
  // int32 row offsets cannot index more live pairs: row_ptr is not usable
  if (host_summary[0] > kMaxMaskNnz) return VA_ERR_UNSUPPORTED;
  if (host_summary[0] > col_capacity) return VA_ERR_INVALID;
  if (host_summary[0] > 0) {
    va::mask_fill_kernel<<<blocks, threads, 0, s>>>(md, row_ptr, col_idx);
    if ((st = launch_status())) return st;
  }
  return VA_OK;
}
