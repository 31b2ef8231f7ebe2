// C ABI of the library (declared in include/nm.h): argument validation,
// status codes, plans and dispatch to the kernels.  Nothing here allocates
// device memory; every launch goes to the caller's stream.
#include <cstdint>
#include <cstring>
#include <new>

#include "nm_internal.h"

namespace {

bool is_elem(nm_dtype_t t) { return t == NM_F16 || t == NM_BF16 || t == NM_I8; }
int64_t elem_size(nm_dtype_t t) {
  switch (t) {
    case NM_F16:
    case NM_BF16: return 2;
    case NM_I8: return 1;
    case NM_F32:
    case NM_I32: return 4;
  }
  return 0;
}
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
// The CUDA error behind the calling thread's last NM_ERR_CUDA.
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

nm_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return NM_OK;
  g_last_cuda_error = e;
  return NM_ERR_CUDA;
}

nm_status_t check_nm(int n, int m) {
  if (m < 2 || m > 32 || n < 1 || n >= m) return NM_ERR_INVALID_ARG;
  return NM_OK;
}

// Validates a rows x cols matrix with leading dimension ld.
nm_status_t check_matrix(const void* p, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t t, bool nullable) {
  if (rows < 0 || cols < 0) return NM_ERR_INVALID_ARG;
  if (p == nullptr) return (nullable || rows == 0 || cols == 0) ? NM_OK : NM_ERR_INVALID_ARG;
  if (ld < cols || ld < 1) return NM_ERR_INVALID_ARG;
  if (!aligned(p, (uintptr_t)elem_size(t))) return NM_ERR_MISALIGNED;
  return NM_OK;
}

size_t tc_meta_bytes(int64_t rows, int64_t cols) {
  return (size_t)((cols / 32) * (((rows + 127) / 128) * 128) * 4);
}

}  // namespace

struct nm_spmm_plan_s {
  nm_spmm_desc_t d;
  int kind;  // 0 tc sparse, 1 tc dense masked, 2 gather n:m, 3 int8 mma.sp, 4 vector/block units
  int split_k;
  size_t ws_bytes;
  bool searchable;  // created with NM_ALGO_DEFAULT and not yet searched
};

extern "C" {

const char* nm_status_string(nm_status_t s) {
  switch (s) {
    case NM_OK: return "NM_OK";
    case NM_ERR_INVALID_ARG: return "NM_ERR_INVALID_ARG";
    case NM_ERR_UNSUPPORTED: return "NM_ERR_UNSUPPORTED";
    case NM_ERR_MISALIGNED: return "NM_ERR_MISALIGNED";
    case NM_ERR_CUDA: return "NM_ERR_CUDA";
    case NM_ERR_TIMEOUT: return "NM_ERR_TIMEOUT";
  }
  return "NM_ERR_UNKNOWN";
}

int nm_version(void) { return 1; }

const char* nm_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda_error);
}

nm_status_t nm_compressed_size(int64_t rows, int64_t cols, nm_dtype_t dtype, int n, int m, nm_meta_layout_t layout,
                               size_t* vals_bytes, size_t* meta_bytes) {
  if (vals_bytes == nullptr || meta_bytes == nullptr || rows < 0 || cols < 0 || !is_elem(dtype))
    return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_nm(n, m)) return st;
  if (cols % m) return NM_ERR_INVALID_ARG;
  if (layout != NM_META_CANONICAL && layout != NM_META_TC) return NM_ERR_INVALID_ARG;
  *vals_bytes = (size_t)(rows * (cols / m) * n * elem_size(dtype));
  if (n == 2 && m == 4) {
    if (layout == NM_META_TC) {
      if (dtype == NM_I8 || cols % 32) return NM_ERR_UNSUPPORTED;
      *meta_bytes = tc_meta_bytes(rows, cols);
    } else {
      *meta_bytes = (size_t)(rows * ((cols / 4 + 3) / 4) * 2);
    }
  } else {
    if (layout == NM_META_TC) return NM_ERR_UNSUPPORTED;
    *meta_bytes = (size_t)(rows * (cols / m) * n);
  }
  return NM_OK;
}

nm_status_t nm_prune(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int n, int m,
                     void* W_out, int64_t ld_out, uint32_t* mask_bits, nm_stream_t stream) {
  if (!is_elem(dtype)) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_nm(n, m)) return st;
  if (cols % m) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_matrix(W, rows, cols, ld, dtype, false)) return st;
  if (nm_status_t st = check_matrix(W_out, rows, cols, ld_out, dtype, true)) return st;
  if (W_out == W && W != nullptr && ld_out != ld) return NM_ERR_INVALID_ARG;
  if (mask_bits != nullptr && !aligned(mask_bits, 4)) return NM_ERR_MISALIGNED;
  nmk::PruneLaunch a{};
  a.dt = (int)dtype;
  a.W = W;
  a.rowsL = rows;
  a.colsL = cols;
  a.ld = ld;
  a.trans = 0;
  a.n = n;
  a.m = m;
  a.W_out = W_out;
  a.ld_out = ld_out;
  a.mask_bits = mask_bits;
  return from_cuda(nmk::launch_prune(a, (cudaStream_t)stream));
}

nm_status_t nm_compress(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int n, int m,
                        int transpose, nm_meta_layout_t layout, void* vals, void* meta, nm_stream_t stream) {
  if (!is_elem(dtype) || (transpose != 0 && transpose != 1)) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_nm(n, m)) return st;
  if (nm_status_t st = check_matrix(W, rows, cols, ld, dtype, false)) return st;
  const int64_t rowsL = transpose ? cols : rows, colsL = transpose ? rows : cols;
  size_t vb = 0, mb = 0;
  if (nm_status_t st = nm_compressed_size(rowsL, colsL, dtype, n, m, layout, &vb, &mb)) return st;
  if (vals != nullptr && !aligned(vals, (uintptr_t)elem_size(dtype))) return NM_ERR_MISALIGNED;
  if (meta != nullptr && !aligned(meta, 4)) return NM_ERR_MISALIGNED;
  nmk::PruneLaunch a{};
  a.dt = (int)dtype;
  a.W = W;
  a.rowsL = rowsL;
  a.colsL = colsL;
  a.ld = ld;
  a.trans = transpose;
  a.n = n;
  a.m = m;
  a.vals = vals;
  a.meta = meta;
  a.meta_tc = layout == NM_META_TC;
  return from_cuda(nmk::launch_prune(a, (cudaStream_t)stream));
}

nm_status_t nm_prune_compress(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int n, int m,
                              void* W_out, int64_t ld_out, uint32_t* mask_bits, nm_meta_layout_t layout, void* vals,
                              void* meta, nm_stream_t stream) {
  if (!is_elem(dtype)) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_nm(n, m)) return st;
  if (cols % m) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_matrix(W, rows, cols, ld, dtype, false)) return st;
  if (nm_status_t st = check_matrix(W_out, rows, cols, ld_out, dtype, true)) return st;
  if (W_out == W && W != nullptr) return NM_ERR_INVALID_ARG;
  size_t vb = 0, mb = 0;
  if (nm_status_t st = nm_compressed_size(rows, cols, dtype, n, m, layout, &vb, &mb)) return st;
  if (mask_bits != nullptr && !aligned(mask_bits, 4)) return NM_ERR_MISALIGNED;
  if (vals != nullptr && !aligned(vals, (uintptr_t)elem_size(dtype))) return NM_ERR_MISALIGNED;
  if (meta != nullptr && !aligned(meta, 4)) return NM_ERR_MISALIGNED;
  nmk::PruneLaunch a{};
  a.dt = (int)dtype;
  a.W = W;
  a.rowsL = rows;
  a.colsL = cols;
  a.ld = ld;
  a.trans = 0;
  a.n = n;
  a.m = m;
  a.W_out = W_out;
  a.ld_out = ld_out;
  a.mask_bits = mask_bits;
  a.vals = vals;
  a.meta = meta;
  a.meta_tc = layout == NM_META_TC;
  return from_cuda(nmk::launch_prune(a, (cudaStream_t)stream));
}

nm_status_t nm_decompress(const void* vals, const void* meta, int64_t rows, int64_t cols, nm_dtype_t dtype, int n,
                          int m, nm_meta_layout_t layout, void* W_out, int64_t ld_out, nm_stream_t stream) {
  if (!is_elem(dtype)) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_nm(n, m)) return st;
  size_t vb = 0, mb = 0;
  if (nm_status_t st = nm_compressed_size(rows, cols, dtype, n, m, layout, &vb, &mb)) return st;
  if (rows > 0 && cols > 0 && (vals == nullptr || meta == nullptr)) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_matrix(W_out, rows, cols, ld_out, dtype, false)) return st;
  if (vals != nullptr && !aligned(vals, (uintptr_t)elem_size(dtype))) return NM_ERR_MISALIGNED;
  if (meta != nullptr && !aligned(meta, 4)) return NM_ERR_MISALIGNED;
  nmk::DecompressLaunch a{};
  a.dt = (int)dtype;
  a.vals = vals;
  a.meta = meta;
  a.rows = rows;
  a.cols = cols;
  a.n = n;
  a.m = m;
  a.meta_tc = layout == NM_META_TC;
  a.W_out = W_out;
  a.ld_out = ld_out;
  return from_cuda(nmk::launch_decompress(a, (cudaStream_t)stream));
}

nm_status_t nm_check(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int n, int m,
                     int transposable, int32_t* d_violations, nm_stream_t stream) {
  if (!is_elem(dtype) || d_violations == nullptr) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_nm(n, m)) return st;
  if (cols % m) return NM_ERR_INVALID_ARG;
  if (transposable && (n != 2 || m != 4 || rows % 4)) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_matrix(W, rows, cols, ld, dtype, false)) return st;
  if (!aligned(d_violations, 4)) return NM_ERR_MISALIGNED;
  return from_cuda(nmk::launch_check((int)dtype, W, rows, cols, ld, n, m, transposable ? 1 : 0, d_violations,
                                     (cudaStream_t)stream));
}

nm_status_t nm_prune_transposable(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype,
                                  void* W_out, int64_t ld_out, uint32_t* mask_bits, void* vals, void* meta,
                                  void* valsT, void* metaT, nm_meta_layout_t layout, nm_stream_t stream) {
  if (!is_elem(dtype)) return NM_ERR_INVALID_ARG;
  if (layout != NM_META_CANONICAL && layout != NM_META_TC) return NM_ERR_INVALID_ARG;
  if (rows % 4 || cols % 4) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_matrix(W, rows, cols, ld, dtype, false)) return st;
  if (nm_status_t st = check_matrix(W_out, rows, cols, ld_out, dtype, true)) return st;
  if (W_out == W && W != nullptr && ld_out != ld) return NM_ERR_INVALID_ARG;
  if (layout == NM_META_TC) {
    if (dtype == NM_I8) return NM_ERR_UNSUPPORTED;
    if (meta != nullptr && cols % 32) return NM_ERR_UNSUPPORTED;
    if (metaT != nullptr && rows % 32) return NM_ERR_UNSUPPORTED;
  }
  const uintptr_t es = (uintptr_t)elem_size(dtype);
  if ((vals && !aligned(vals, es)) || (valsT && !aligned(valsT, es)) || (meta && !aligned(meta, 4)) ||
      (metaT && !aligned(metaT, 4)) || (mask_bits && !aligned(mask_bits, 4)))
    return NM_ERR_MISALIGNED;
  nmk::TransposableLaunch a{};
  a.dt = (int)dtype;
  a.W = W;
  a.rows = rows;
  a.cols = cols;
  a.ld = ld;
  a.W_out = W_out;
  a.ld_out = ld_out;
  a.mask_bits = mask_bits;
  a.vals = vals;
  a.meta = meta;
  a.valsT = valsT;
  a.metaT = metaT;
  a.meta_tc = layout == NM_META_TC;
  return from_cuda(nmk::launch_transposable(a, (cudaStream_t)stream));
}

nm_status_t nm_sgd_prune_transposable(void* W, const void* dW, float lr, int64_t rows, int64_t cols, int64_t ld,
                                      int64_t ld_grad, nm_dtype_t dtype, uint32_t* mask_bits, void* vals, void* meta,
                                      void* valsT, void* metaT, nm_meta_layout_t layout, nm_stream_t stream) {
  if (!is_elem(dtype)) return NM_ERR_INVALID_ARG;
  if (dtype == NM_I8) return NM_ERR_UNSUPPORTED;
  if (layout != NM_META_CANONICAL && layout != NM_META_TC) return NM_ERR_INVALID_ARG;
  if (rows % 4 || cols % 4) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_matrix(W, rows, cols, ld, dtype, false)) return st;
  if (nm_status_t st = check_matrix(dW, rows, cols, ld_grad, dtype, false)) return st;
  if (dW == W && W != nullptr) return NM_ERR_INVALID_ARG;
  if (layout == NM_META_TC) {
    if (meta != nullptr && cols % 32) return NM_ERR_UNSUPPORTED;
    if (metaT != nullptr && rows % 32) return NM_ERR_UNSUPPORTED;
  }
  const uintptr_t es = (uintptr_t)elem_size(dtype);
  if ((vals && !aligned(vals, es)) || (valsT && !aligned(valsT, es)) || (meta && !aligned(meta, 4)) ||
      (metaT && !aligned(metaT, 4)) || (mask_bits && !aligned(mask_bits, 4)) || !aligned(dW, 4 * es) ||
      ld_grad % 4)
    return NM_ERR_MISALIGNED;
  nmk::TransposableLaunch a{};
  a.dt = (int)dtype;
  a.W = W;
  a.rows = rows;
  a.cols = cols;
  a.ld = ld;
  a.mask_bits = mask_bits;
  a.vals = vals;
  a.meta = meta;
  a.valsT = valsT;
  a.metaT = metaT;
  a.meta_tc = layout == NM_META_TC;
  a.grad = dW;
  a.ld_grad = ld_grad;
  a.lr = lr;
  a.W_upd = W;
  return from_cuda(nmk::launch_transposable(a, (cudaStream_t)stream));
}

// ------------------------------------------------------- vector/block units
}  // extern "C"

namespace {
nm_status_t units_shape(int64_t rows, int64_t cols, int bh, int bw, int64_t* units) {
  if (rows < 0 || cols < 0 || bh < 1 || bw < 1) return NM_ERR_INVALID_ARG;
  if (bw != 32 || (bh != 1 && bh != 32)) return NM_ERR_UNSUPPORTED;
  if (cols % bw || rows % bh) return NM_ERR_INVALID_ARG;
  *units = (rows / bh) * (cols / bw);
  if (*units >= (int64_t(1) << 31)) return NM_ERR_UNSUPPORTED;
  return NM_OK;
}

// Every check of a unit selection's arguments except the workspace's; touches no CUDA state.
nm_status_t check_units_args(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int bh, int bw,
                             int64_t keep, const void* W_out, int64_t ld_out, const uint32_t* mask_bits,
                             const int32_t* csr, const void* vals, int64_t* units) {
  if (!is_elem(dtype)) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = units_shape(rows, cols, bh, bw, units)) return st;
  if (dtype == NM_BF16) return NM_ERR_UNSUPPORTED;
  if (keep < 0 || keep > *units) return NM_ERR_INVALID_ARG;
  if (nm_status_t st = check_matrix(W, rows, cols, ld, dtype, false)) return st;
  if (nm_status_t st = check_matrix(W_out, rows, cols, ld_out, dtype, true)) return st;
  if (W_out == W && W != nullptr && ld_out != ld) return NM_ERR_INVALID_ARG;
  const int64_t es = elem_size(dtype);
  if (!aligned(W, 16) || (ld * es) % 16 || !aligned(W_out, 16) || (W_out != nullptr && (ld_out * es) % 16) ||
      !aligned(vals, 16) || !aligned(csr, 4) || !aligned(mask_bits, 4))
    return NM_ERR_MISALIGNED;
  return NM_OK;
}

nm_status_t prune_units(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int bh, int bw,
                        int64_t keep, int abs_of_sum, void* W_out, int64_t ld_out, uint32_t* mask_bits,
                        int32_t* csr, void* vals, void* workspace, size_t workspace_bytes, nm_stream_t stream) {
  int64_t units = 0;
  if (nm_status_t st = check_units_args(W, rows, cols, ld, dtype, bh, bw, keep, W_out, ld_out, mask_bits, csr, vals,
                                        &units))
    return st;
  if (!aligned(workspace, 16)) return NM_ERR_MISALIGNED;
  if (units > 0 && (workspace == nullptr || workspace_bytes < nmk::blocks_workspace(units))) return NM_ERR_INVALID_ARG;
  nmk::BlocksLaunch a{};
  a.dt = (int)dtype;
  a.W = W;
  a.rows = rows;
  a.cols = cols;
  a.ld = ld;
  a.bh = bh;
  a.units = units;
  a.unit_rows = rows / bh;
  a.keep = keep;
  a.abs_of_sum = abs_of_sum;
  a.W_out = W_out;
  a.ld_out = ld_out;
  a.mask_bits = mask_bits;
  a.csr = csr;
  a.vals = vals;
  a.ws = workspace;
  return from_cuda(nmk::launch_blocks(a, (cudaStream_t)stream));
}
}  // namespace

extern "C" {

nm_status_t nm_prune_units_workspace(int64_t rows, int64_t cols, int bh, int bw, size_t* bytes) {
  if (bytes == nullptr) return NM_ERR_INVALID_ARG;
  int64_t units = 0;
  if (nm_status_t st = units_shape(rows, cols, bh, bw, &units)) return st;
  *bytes = units > 0 ? nmk::blocks_workspace(units) : 0;
  return NM_OK;
}

nm_status_t nm_prune_vector_wise(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int v,
                                 int64_t keep, nm_score_t score, void* W_out, int64_t ld_out, uint32_t* mask_bits,
                                 int32_t* csr, void* vals, void* workspace, size_t workspace_bytes,
                                 nm_stream_t stream) {
  if (score != NM_SCORE_ABS_OF_SUM && score != NM_SCORE_SUM_OF_ABS) return NM_ERR_INVALID_ARG;
  return prune_units(W, rows, cols, ld, dtype, 1, v, keep, score == NM_SCORE_ABS_OF_SUM, W_out, ld_out, mask_bits,
                     csr, vals, workspace, workspace_bytes, stream);
}

nm_status_t nm_prune_block_wise(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int bh,
                                int bw, int64_t keep, void* W_out, int64_t ld_out, uint32_t* mask_bits, int32_t* csr,
                                void* vals, void* workspace, size_t workspace_bytes, nm_stream_t stream) {
  if (bh == 1) return NM_ERR_UNSUPPORTED;  // 1 x bw blocks are vectors: nm_prune_vector_wise
  return prune_units(W, rows, cols, ld, dtype, bh, bw, keep, 0, W_out, ld_out, mask_bits, csr, vals, workspace,
                     workspace_bytes, stream);
}

nm_status_t nm_prune_vector_wise_noalloc(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype,
                                         int v, int64_t keep, nm_score_t score, void* W_out, int64_t ld_out,
                                         uint32_t* mask_bits, int32_t* csr, void* vals, nm_stream_t stream) {
  if (score != NM_SCORE_ABS_OF_SUM && score != NM_SCORE_SUM_OF_ABS) return NM_ERR_INVALID_ARG;
  int64_t units = 0;
  if (nm_status_t st = units_shape(rows, cols, 1, v, &units)) return st;
  if (units > nmk::fixed_scratch_units()) return NM_ERR_UNSUPPORTED;
  // every argument is checked before the one-time address lookup, so that a rejected call touches no
  // CUDA state
  if (nm_status_t st = check_units_args(W, rows, cols, ld, dtype, 1, v, keep, W_out, ld_out, mask_bits, csr, vals,
                                        &units))
    return st;
  void* scratch = nullptr;
  size_t bytes = 0;
  if (units > 0) {
    if (nm_status_t st = from_cuda(nmk::fixed_scratch(&scratch, &bytes))) return st;
  }
  return prune_units(W, rows, cols, ld, dtype, 1, v, keep, score == NM_SCORE_ABS_OF_SUM, W_out, ld_out, mask_bits,
                     csr, vals, scratch, bytes, stream);
}

// ------------------------------------------------------------------ products
nm_status_t nm_spmm_plan(nm_spmm_plan_t* plan, const nm_spmm_desc_t* desc) {
  if (plan == nullptr || desc == nullptr) return NM_ERR_INVALID_ARG;
  *plan = nullptr;
  const nm_spmm_desc_t& d = *desc;
  if (d.M < 0 || d.N < 0 || d.K < 0) return NM_ERR_INVALID_ARG;
  if (d.algo != NM_ALGO_DEFAULT && d.algo != NM_ALGO_PAIRED && d.algo != NM_ALGO_SINGLE) return NM_ERR_INVALID_ARG;
  if (!is_elem(d.ab_type)) return NM_ERR_INVALID_ARG;
  const bool fp = d.ab_type != NM_I8;
  if (fp ? (d.cd_type != d.ab_type && d.cd_type != NM_F32) : (d.cd_type != NM_I32 && d.cd_type != NM_I8))
    return NM_ERR_UNSUPPORTED;
  if ((d.order_a != NM_ROW && d.order_a != NM_COL) || (d.order_b != NM_ROW && d.order_b != NM_COL) ||
      (d.order_cd != NM_ROW && d.order_cd != NM_COL))
    return NM_ERR_INVALID_ARG;
  // leading dimensions
  const int64_t es = elem_size(d.ab_type), eo = elem_size(d.cd_type);
  const int64_t b_inner = d.order_b == NM_COL ? d.K : d.N;
  const int64_t cd_inner = d.order_cd == NM_ROW ? d.N : d.M;
  if (d.ldb < b_inner || d.ldb < 1 || d.ldc < 0 || d.ldd < cd_inner || d.ldd < 1) return NM_ERR_INVALID_ARG;
  if (d.ldc != 0 && d.ldc < cd_inner) return NM_ERR_INVALID_ARG;
  if ((d.ldb * es) % 16) return NM_ERR_MISALIGNED;
  int kind = -1;
  if (d.mode == NM_SPMM_SPARSE_A) {
    if (nm_status_t st = check_nm(d.n, d.m)) return st;
    if (d.K % d.m) return NM_ERR_INVALID_ARG;
    if (d.order_b != NM_COL) return NM_ERR_UNSUPPORTED;
    if (d.n == 2 && d.m == 4) {
      if (fp) {
        if (d.meta_layout != NM_META_TC) return NM_ERR_UNSUPPORTED;
        if (d.K % 32) return NM_ERR_UNSUPPORTED;
        kind = 0;
      } else {
        if (d.meta_layout != NM_META_CANONICAL) return NM_ERR_UNSUPPORTED;
        if (d.K % 64) return NM_ERR_UNSUPPORTED;
        if (d.K == 0) return NM_ERR_UNSUPPORTED;
        kind = 3;
      }
    } else {
      if (d.meta_layout != NM_META_CANONICAL || !fp) return NM_ERR_UNSUPPORTED;
      // kept-value indices of a row are 32-bit; a batch of B is staged in shared memory
      if (d.K > 2147483647LL || (d.N > 1 && d.K > 12800)) return NM_ERR_UNSUPPORTED;
      kind = 2;
    }
  } else if (d.mode == NM_SPMM_DENSE_MASKED) {
    if (!fp) return NM_ERR_UNSUPPORTED;
    const int64_t a_inner = d.order_a == NM_ROW ? d.K : d.M;
    if (d.lda < a_inner || d.lda < 1) return NM_ERR_INVALID_ARG;
    if ((d.lda * es) % 16) return NM_ERR_MISALIGNED;
    kind = 1;
  } else if (d.mode == NM_SPMM_BLOCK_SPARSE_A) {
    if (!fp || d.order_b != NM_COL) return NM_ERR_UNSUPPORTED;
    if (d.m != 32 || (d.n != 1 && d.n != 32)) return NM_ERR_UNSUPPORTED;
    if (d.K % 32 || d.M % d.n) return NM_ERR_INVALID_ARG;
    kind = 4;
  } else {
    return NM_ERR_INVALID_ARG;
  }
  // an fp32 C/D only on the tensor-core products, an int8 C/D only on the int8 sparse product
  if (fp && d.cd_type == NM_F32 && kind != 0 && kind != 1) return NM_ERR_UNSUPPORTED;
  if (!fp && d.cd_type == NM_I8 && kind != 3) return NM_ERR_UNSUPPORTED;
  // The tensor-core and int8 kernels write D (and read C) in 16-byte pieces;
  // the CUDA-core GEMV kernels (kinds 2 and 4) access them element by element.
  const bool cd_wide = kind != 2 && kind != 4;
  if (cd_wide && ((d.ldd * eo) % 16 || (d.ldc * eo) % 16)) return NM_ERR_MISALIGNED;
  nm_spmm_plan_s* p = new (std::nothrow) nm_spmm_plan_s;
  if (p == nullptr) return NM_ERR_INVALID_ARG;
  p->d = d;
  p->kind = kind;
  p->split_k = kind == 1 ? nmk::spmm_tc_dense_masked_split(d) : 1;
  p->ws_bytes = kind == 1 ? nmk::spmm_tc_dense_masked_workspace(d, p->split_k) : 0;
  p->searchable = d.algo == NM_ALGO_DEFAULT;
  *plan = p;
  return NM_OK;
}

nm_status_t nm_spmm_plan_workspace(nm_spmm_plan_t plan, size_t* bytes) {
  if (plan == nullptr || bytes == nullptr) return NM_ERR_INVALID_ARG;
  *bytes = plan->ws_bytes;
  return NM_OK;
}

nm_status_t nm_spmm_plan_split_k(nm_spmm_plan_t plan, int* split_k) {
  if (plan == nullptr || split_k == nullptr) return NM_ERR_INVALID_ARG;
  *split_k = plan->kind == 1 ? plan->split_k : 1;
  return NM_OK;
}

nm_status_t nm_spmm_plan_launches(nm_spmm_plan_t plan, int* launches) {
  if (plan == nullptr || launches == nullptr) return NM_ERR_INVALID_ARG;
  const nm_spmm_desc_t& d = plan->d;
  *launches = (d.M == 0 || d.N == 0) ? 0 : plan->kind == 1 ? nmk::spmm_tc_dense_masked_launches(d, plan->split_k) : 1;
  return NM_OK;
}

nm_status_t nm_spmm_plan_destroy(nm_spmm_plan_t plan) {
  delete plan;
  return NM_OK;
}

nm_status_t nm_spmm(nm_spmm_plan_t plan, const void* alpha, const void* A, const void* A_meta, const void* B,
                    const void* beta, const void* C, void* D, void* workspace, size_t workspace_bytes,
                    int32_t* d_status, nm_stream_t stream) {
  if (plan == nullptr || alpha == nullptr || beta == nullptr) return NM_ERR_INVALID_ARG;
  const nm_spmm_desc_t& d = plan->d;
  nmk::SpmmLaunch a{};
  a.d = d;
  const bool int_scalars = d.ab_type == NM_I8 && d.cd_type == NM_I32;
  if (int_scalars) {
    std::memcpy(&a.alpha_i, alpha, 4);
    std::memcpy(&a.beta_i, beta, 4);
  } else {
    std::memcpy(&a.alpha_f, alpha, 4);
    std::memcpy(&a.beta_f, beta, 4);
  }
  const bool beta_zero = int_scalars ? a.beta_i == 0 : a.beta_f == 0.0f;
  if (d.M == 0 || d.N == 0) return NM_OK;
  // DENSE_MASKED may run without a mask (a plain dense product)
  const bool meta_optional = plan->kind == 1;
  if (A == nullptr || (A_meta == nullptr && !meta_optional) || B == nullptr || D == nullptr) {
    if (d.K > 0 || D == nullptr) return NM_ERR_INVALID_ARG;
  }
  if (plan->kind == 4 && A_meta == nullptr) return NM_ERR_INVALID_ARG;
  if (!beta_zero && (C == nullptr || d.ldc == 0)) return NM_ERR_INVALID_ARG;
  const uintptr_t cd_align = (plan->kind == 2 || plan->kind == 4) ? (uintptr_t)elem_size(d.cd_type) : 16;
  if (!aligned(A, 16) || !aligned(A_meta, 16) || !aligned(B, 16) || !aligned(D, cd_align) ||
      (!beta_zero && !aligned(C, cd_align)) || (d_status && !aligned(d_status, 4)))
    return NM_ERR_MISALIGNED;
  if (workspace_bytes < plan->ws_bytes || (plan->ws_bytes > 0 && workspace == nullptr)) return NM_ERR_INVALID_ARG;
  if (workspace != nullptr && !aligned(workspace, 16)) return NM_ERR_MISALIGNED;
  a.A = A;
  a.A_meta = A_meta;
  a.B = B;
  a.C = beta_zero ? nullptr : C;
  a.D = D;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  a.d_status = d_status;
  cudaStream_t s = (cudaStream_t)stream;
  switch (plan->kind) {
    case 0: return from_cuda(nmk::launch_spmm_tc_sparse(a, s));
    case 1: return from_cuda(nmk::launch_spmm_tc_dense_masked(a, plan->split_k, s));
    case 2: return from_cuda(nmk::launch_spmm_nm_gather(a, s));
    case 3: return from_cuda(nmk::launch_spmm_i8(a, s));
    case 4: return from_cuda(nmk::launch_spmm_blocks(a, s));
  }
  return NM_ERR_INVALID_ARG;
}

nm_status_t nm_spmm_search(nm_spmm_plan_t plan, const void* alpha, const void* A, const void* A_meta, const void* B,
                           const void* beta, const void* C, void* D, void* workspace, size_t workspace_bytes,
                           int repeats, int* chosen_algo, nm_stream_t stream) {
  if (plan == nullptr || alpha == nullptr || beta == nullptr || repeats < 1 || repeats > 1000)
    return NM_ERR_INVALID_ARG;
  nm_spmm_desc_t& d = plan->d;
  const bool tc = plan->kind == 0 || plan->kind == 1;
  const bool even_blocks = ((d.M + 127) / 128) % 2 == 0;
  if (!tc || !plan->searchable || d.M == 0 || d.N == 0 || d.K == 0) {
    if (chosen_algo != nullptr) *chosen_algo = d.algo;
    return NM_OK;
  }
  // Candidates (algorithm, K split): the paired and the single-CTA kernel (paired only when M
  // spans an even number of 128-row blocks); for DENSE_MASKED also the plan's split's
  // neighbours h - 1, h - 2 and h + 1 whose workspace fits in the caller's.  Candidate 0,
  // the plan's default, stays unless another is at least 2% faster.
  struct Cand {
    int algo, split;
  };
  Cand cand[8];
  int nc = 0;
  const int h = plan->split_k;
  int splits[4] = {h, 0, 0, 0}, ns = 1;
  if (plan->kind == 1) {
    for (int sk : {h - 1, h - 2, h + 1})
      if (nmk::spmm_tc_dense_masked_split_ok(d, sk) && nmk::spmm_tc_dense_masked_workspace(d, sk) <= workspace_bytes)
        splits[ns++] = sk;
  }
  for (int j = 0; j < ns; ++j) {
    if (even_blocks) {
      cand[nc++] = {NM_ALGO_PAIRED, splits[j]};
      cand[nc++] = {NM_ALGO_SINGLE, splits[j]};
    } else {
      cand[nc++] = {NM_ALGO_DEFAULT, splits[j]};  // the single-CTA kernel
    }
  }
  if (nc == 1) {
    if (chosen_algo != nullptr) *chosen_algo = d.algo;
    return NM_OK;
  }
  float beta_f = 0.0f;
  std::memcpy(&beta_f, beta, 4);
  if (beta_f != 0.0f && C == D) return NM_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  cudaEvent_t ev[2] = {nullptr, nullptr};
  nm_status_t st = NM_OK;
  auto use = [&](const Cand& c) {
    d.algo = c.algo;
    plan->split_k = c.split;
    plan->ws_bytes = plan->kind == 1 ? nmk::spmm_tc_dense_masked_workspace(d, c.split) : 0;
  };
  // Three rounds, the candidates alternating within each, keep each candidate's fastest round:
  // one sample per candidate moved with the clock (power capping) and with the event timer's
  // granularity.
  constexpr int kRounds = 3;
  float best_ms[8] = {};
  for (int round = 0; round < kRounds && st == NM_OK; ++round) {
    for (int i = 0; i < nc && st == NM_OK; ++i) {
      if (ev[0] == nullptr) {
        if ((st = from_cuda(cudaEventCreate(&ev[0]))) != NM_OK) break;
        if ((st = from_cuda(cudaEventCreate(&ev[1]))) != NM_OK) break;
      }
      use(cand[i]);
      // one untimed run, then the timed ones
      if ((st = nm_spmm(plan, alpha, A, A_meta, B, beta, C, D, workspace, workspace_bytes, nullptr, stream)) != NM_OK)
        break;
      if ((st = from_cuda(cudaEventRecord(ev[0], s))) != NM_OK) break;
      for (int r = 0; r < repeats && st == NM_OK; ++r)
        st = nm_spmm(plan, alpha, A, A_meta, B, beta, C, D, workspace, workspace_bytes, nullptr, stream);
      if (st != NM_OK) break;
      if ((st = from_cuda(cudaEventRecord(ev[1], s))) != NM_OK) break;
      if ((st = from_cuda(cudaEventSynchronize(ev[1]))) != NM_OK) break;
      float ms = 0.0f;
      if ((st = from_cuda(cudaEventElapsedTime(&ms, ev[0], ev[1]))) != NM_OK) break;
      if (round == 0 || ms < best_ms[i]) best_ms[i] = ms;
    }
  }
  int best = 0;
  for (int i = 1; i < nc; ++i)
    if (best_ms[i] < best_ms[best]) best = i;
  if (!(best_ms[best] < 0.98f * best_ms[0])) best = 0;
  for (cudaEvent_t e : ev)
    if (e != nullptr) cudaEventDestroy(e);
  if (st == NM_OK) {
    use(cand[best]);
    plan->searchable = false;
  } else {
    use(Cand{NM_ALGO_DEFAULT, h});
  }
  if (chosen_algo != nullptr) *chosen_algo = d.algo;
  return st;
}

}  // extern "C"
