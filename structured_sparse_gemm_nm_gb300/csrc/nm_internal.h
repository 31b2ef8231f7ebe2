// Internal launch interface between the C-ABI layer (nm_api.cu) and the kernels.
// Every launcher only enqueues work; argument checking happens in nm_api.cu.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/nm.h"

namespace nmk {

// ---- pruning / compression (nm_prune.cu) -------------------------------
// The "logical" matrix L has rowsL x colsL elements; its groups run along rows.
// trans = 0: L = W (L[r][c] = W[r*ld + c]); trans = 1: L = W^T (L[r][c] = W[c*ld + r]).
struct PruneLaunch {
  int dt;
  const void* W;
  int64_t rowsL, colsL, ld;
  int trans;
  int n, m;
  void* W_out;          // only with trans = 0
  int64_t ld_out;
  uint32_t* mask_bits;  // only with trans = 0
  void* vals;
  void* meta;
  int meta_tc;          // 2:4 only: 1 = tensor-core order
};
cudaError_t launch_prune(const PruneLaunch& a, cudaStream_t s);

struct DecompressLaunch {
  int dt;
  const void* vals;
  const void* meta;
  int64_t rows, cols;
  int n, m;
  int meta_tc;
  void* W_out;
  int64_t ld_out;
};
cudaError_t launch_decompress(const DecompressLaunch& a, cudaStream_t s);

cudaError_t launch_check(int dt, const void* W, int64_t rows, int64_t cols, int64_t ld, int n, int m,
                         int transposable, int32_t* d_violations, cudaStream_t s);

// ---- transposable 4x4 (nm_transposable.cu) ------------------------------
struct TransposableLaunch {
  int dt;
  const void* W;
  int64_t rows, cols, ld;
  void* W_out;
  int64_t ld_out;
  uint32_t* mask_bits;
  void* vals;
  void* meta;
  void* valsT;
  void* metaT;
  int meta_tc;
  // optional SGD update before the prune: W <- round(W - lr * grad), written back to W_upd (= W)
  const void* grad;
  int64_t ld_grad;
  float lr;
  void* W_upd;
};
cudaError_t launch_transposable(const TransposableLaunch& a, cudaStream_t s);

// ---- vector-wise / block-wise selection (nm_blocks.cu) -------------------
// Units are 1 x 32 vectors (bh = 1) or 32 x 32 blocks (bh = 32) in row-major order.
struct BlocksLaunch {
  int dt;  // kF16 or kI8
  const void* W;
  int64_t rows, cols, ld;
  int bh;
  int64_t units, unit_rows;  // unit_rows = rows / bh
  int64_t keep;
  int abs_of_sum;  // vector-wise score: 1 = |sum w|, 0 = sum |w|
  void* W_out;
  int64_t ld_out;
  uint32_t* mask_bits;
  int32_t* csr;
  void* vals;
  void* ws;
};
size_t blocks_workspace(int64_t units);
cudaError_t launch_blocks(const BlocksLaunch& a, cudaStream_t s);
// Device address and size of the library's own fixed scratch for the selection
// (looked up once per device, on the current device).
int64_t fixed_scratch_units();
cudaError_t fixed_scratch(void** ptr, size_t* bytes);

// ---- products (nm_spmm_tc.cu, nm_spmm_cc.cu, nm_blocks.cu) ---------------
struct SpmmLaunch {
  nm_spmm_desc_t d;
  const void* A;
  const void* A_meta;
  const void* B;
  const void* C;
  void* D;
  float alpha_f, beta_f;
  int32_t alpha_i, beta_i;
  void* ws;
  size_t ws_bytes;
  int32_t* d_status;
};

// Tensor-core paths (tcgen05).  `split_k` is the plan's K split for DENSE_MASKED.
cudaError_t launch_spmm_tc_sparse(const SpmmLaunch& a, cudaStream_t s);
cudaError_t launch_spmm_tc_dense_masked(const SpmmLaunch& a, int split_k, cudaStream_t s);
size_t spmm_tc_dense_masked_workspace(const nm_spmm_desc_t& d, int split_k);
// Kernels one call of the masked dense product launches: the product, and the finalize
// when it splits K and does not sum the splits itself.
int spmm_tc_dense_masked_launches(const nm_spmm_desc_t& d, int split_k);
int spmm_tc_dense_masked_split(const nm_spmm_desc_t& d);
// A K split the masked dense product accepts: 1, or up to 16 splits of at least 8 stages each.
bool spmm_tc_dense_masked_split_ok(const nm_spmm_desc_t& d, int split_k);

// CUDA-core paths: n:m gather (any m <= 32) and 2:4 int8 (mma.sp).
cudaError_t launch_spmm_nm_gather(const SpmmLaunch& a, cudaStream_t s);
cudaError_t launch_spmm_i8(const SpmmLaunch& a, cudaStream_t s);
// CUDA-core product over kept 1 x 32 vectors (n = 1) or 32 x 32 blocks (n = 32).
cudaError_t launch_spmm_blocks(const SpmmLaunch& a, cudaStream_t s);

namespace tc {
// A 2-D tiled tensor map (the driver's encoder; false if it rejects the arguments) and the
// binding of the current device's primary context that encoding needs.
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
              uint64_t pitch_bytes, uint32_t inner_box, uint32_t outer_box, CUtensorMapSwizzle sw);
cudaError_t bind_context();
}  // namespace tc

}  // namespace nmk
