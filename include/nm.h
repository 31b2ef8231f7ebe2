/*
 * nm.h - C ABI of the N:M structured-sparsity library for NVIDIA GB300 (sm_103a).
 *
 * The calls follow the workflow of the cuSPARSELt blog ("Exploiting NVIDIA
 * Ampere Structured Sparsity with cuSPARSELt", the workflow list and the
 * "Structured sparse matrix-matrix multiplication code example"): describe
 * the product once (nm_spmm_plan), prune (nm_prune / nm_prune_transposable),
 * check the pattern (nm_check), compress (nm_compress), then multiply
 * (nm_spmm) as often as needed.
 *
 * Conventions shared by every call
 *   - Matrices are dense row-major arrays with a leading dimension `ld`
 *     counted in elements (ld >= cols).  Sizes are int64_t element counts.
 *   - Every pointer argument that names matrix data is a DEVICE pointer owned
 *     by the caller; the library never allocates, frees or keeps it.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream).  Arguments are validated on the host before anything is
 *     enqueued; on an error nothing is launched and the stream is untouched.
 *     No call synchronises the stream.
 *   - A launch failure reported by the CUDA runtime returns NM_ERR_CUDA.
 *     Results that depend on data (a violation count, a wait that gave up)
 *     are written to caller-owned device int32 words.
 *   - Element types: NM_F16 / NM_BF16 are IEEE binary16 / bfloat16 bit
 *     patterns, NM_I8 is two's-complement int8.
 *   - Magnitude order: |w| by value, NaN above every number (several NaNs
 *     tie), int8 -128 has magnitude 128.  Equal magnitudes: lower position
 *     wins.  Pruned slots of a dense output are written as +0.
 *
 * Storage formats
 *   - 2:4 canonical metadata (NM_META_CANONICAL): per group of 4 consecutive
 *     elements of a row one 4-bit code i0 | i1 << 2 (i0 < i1 the kept
 *     positions).  Group g of a row is at bits 4*(g % 4) of uint16 word
 *     g / 4; a row has ceil(cols/16) words; rows are packed back to back.
 *   - 2:4 tensor-core metadata (NM_META_TC): the order in which the sparse
 *     tensor core reads metadata for 128-row tiles of 16-bit operands, one
 *     block per k-step of 32 columns.  It is a uint32 array of shape
 *     [cols/32][S], S = ceil(rows/128)*128 slots.  Word [s][16b + 8h + i]
 *     holds, in its low 16 bits, the four codes of row 16b+i for columns
 *     32s+16h .. 32s+16h+15 and, in its high 16 bits, the same codes of row
 *     16b+8+i.  Codes of rows past `rows` are 0x4 (positions 0 and 1), so the
 *     tensor core only ever reads valid codes.  Same size as the canonical
 *     layout (up to the row padding).  Needs cols % 32 == 0.
 *   - N:M metadata for (n, m) != (2, 4): one uint8 position (0..m-1) per kept
 *     value, in the same order as the values (NM_META_CANONICAL only).
 *   - Compressed values: rows x (cols/m*n) elements, packed, kept entries in
 *     ascending position order with their original bits.
 *   - Bit masks: row-major, ceil(cols/32) uint32 words per row, bit c % 32 of
 *     word c / 32 is element c.
 */
#ifndef NM_H_
#define NM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* nm_stream_t;

typedef enum {
  NM_OK = 0,
  NM_ERR_INVALID_ARG = 1, /* a size, pointer or enum is out of range            */
  NM_ERR_UNSUPPORTED = 2, /* valid request this build has no kernel for         */
  NM_ERR_MISALIGNED = 3,  /* a pointer or leading dimension breaks an alignment */
  NM_ERR_CUDA = 4,        /* the CUDA runtime reported an error                  */
  NM_ERR_TIMEOUT = 5      /* written to a status word: a bounded wait gave up    */
} nm_status_t;

typedef enum { NM_F16 = 0, NM_BF16 = 1, NM_I8 = 2, NM_F32 = 3, NM_I32 = 4 } nm_dtype_t;

typedef enum { NM_META_CANONICAL = 0, NM_META_TC = 1 } nm_meta_layout_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* nm_status_string(nm_status_t status);

/* Library ABI version, currently 1. */
int nm_version(void);

/* Text of the CUDA runtime error behind the calling thread's most recent
 * NM_ERR_CUDA (static string, never NULL; "no CUDA error" if there was none). */
const char* nm_last_cuda_error(void);

/*
 * nm_compressed_size - host-only size query (cuSPARSELt blog, code example,
 * cusparseLtSpMMACompressedSize before the compressed buffer is allocated).
 * Writes the byte sizes of the compressed values and of the metadata of a
 * rows x cols matrix pruned n:m with the given metadata layout.
 * Errors: NM_ERR_INVALID_ARG for bad sizes/NULL outputs, NM_ERR_UNSUPPORTED
 * for NM_META_TC with (n,m) != (2,4) or a non-16-bit type or cols % 32 != 0.
 */
nm_status_t nm_compressed_size(int64_t rows, int64_t cols, nm_dtype_t dtype, int n, int m,
                               nm_meta_layout_t layout, size_t* vals_bytes, size_t* meta_bytes);

/*
 * nm_prune - greedy N:M magnitude pruning along rows (apex PR #1631
 * "[sparse] update support for arbitrary N:M settings sparse", extension 1,
 * mn_1d_greedy; cuSPARSELt blog, cusparseLtSpMMAPrune in the code example).
 * In every group of m consecutive elements of a row the n largest |w| are
 * kept.  W: rows x cols, leading dimension ld.  W_out (nullable): pruned
 * copy with leading dimension ld_out; it may be W itself (in-place, then
 * ld_out == ld).  mask_bits (nullable): bit mask of the kept entries.
 * Requires 1 <= n < m <= 32, cols % m == 0, dtype F16/BF16/I8.
 */
nm_status_t nm_prune(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int n, int m,
                     void* W_out, int64_t ld_out, uint32_t* mask_bits, nm_stream_t stream);

/*
 * nm_compress - select and pack in one pass (cuSPARSELt blog, Figure 2 text
 * and cusparseLtSpMMACompress).  The selection is nm_prune's rule applied to
 * W itself, so an already pruned W keeps its nonzeros.  transpose = 0
 * compresses W (groups along rows); transpose = 1 compresses W^T, i.e. the
 * groups run down the columns of W and the outputs describe a cols x rows
 * matrix.  vals and meta (either nullable) receive the compressed values and
 * the metadata in `layout`.  Sizes come from nm_compressed_size for the
 * compressed matrix's (rows, cols).
 */
nm_status_t nm_compress(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int n, int m,
                        int transpose, nm_meta_layout_t layout, void* vals, void* meta, nm_stream_t stream);

/*
 * nm_prune_compress - nm_prune and nm_compress (transpose = 0) in one pass
 * over W: every output of either, each nullable (W_out, ld_out, mask_bits;
 * vals, meta in `layout`), from a single read of W.  Meant for operands pruned
 * at run time, such as activations (PyTorch issue #126420, maintainer reply:
 * activation sparsity), where a second pass would double the traffic.
 * Requirements and errors are those of the two calls; W_out may not alias W
 * here (NM_ERR_INVALID_ARG).
 */
nm_status_t nm_prune_compress(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int n, int m,
                              void* W_out, int64_t ld_out, uint32_t* mask_bits, nm_meta_layout_t layout, void* vals,
                              void* meta, nm_stream_t stream);

/*
 * nm_decompress - inverse of nm_compress: scatter the values back to their
 * positions, +0 everywhere else.  rows x cols is the dense shape; W_out has
 * leading dimension ld_out.
 */
nm_status_t nm_decompress(const void* vals, const void* meta, int64_t rows, int64_t cols, nm_dtype_t dtype, int n,
                          int m, nm_meta_layout_t layout, void* W_out, int64_t ld_out, nm_stream_t stream);

/*
 * nm_check - pattern check (cuSPARSELt blog, cusparseLtSpMMAPruneCheck):
 * *d_violations (device int32, caller-owned) is set to the number of groups
 * of m consecutive row elements holding more than n nonzeros (NaN counts as
 * nonzero, -0 does not).  With transposable != 0 (2:4 only, rows % 4 == 0)
 * the groups of 4 consecutive rows of every column, aligned to multiples of
 * 4, are counted as well.  Zero means the matrix conforms.
 */
nm_status_t nm_check(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int n, int m,
                     int transposable, int32_t* d_violations, nm_stream_t stream);

/*
 * nm_prune_transposable - 2:4 mask on 4x4 tiles that is 2:4 along rows and
 * along columns (PyTorch issue #126420, maintainer reply: the forward W x
 * and the backward W^T dL/dy both need 2:4), computed at run time.  Per tile
 * the kept pattern is, among the 90 with two entries in every row and every
 * column, the one with the largest float32 score ((p0+p1)+p2)+p3 where p_r
 * is the float32 sum of row r's two kept magnitudes; ties go to the earliest
 * pattern when row 0's pair is the outermost loop over the pairs
 * (0,1),(0,2),(0,3),(1,2),(1,3),(2,3).  NaN magnitudes score +Inf.
 * Outputs, each nullable: W_out (pruned copy, may alias W with ld_out == ld),
 * mask_bits, vals/meta (compressed W, groups along rows, rows x cols/2) and
 * valsT/metaT (compressed W^T, cols x rows/2), metadata in `layout`.
 * Requires rows % 4 == 0 and cols % 4 == 0; NM_META_TC needs cols % 32 == 0
 * for meta and rows % 32 == 0 for metaT.
 */
nm_status_t nm_prune_transposable(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype,
                                  void* W_out, int64_t ld_out, uint32_t* mask_bits, void* vals, void* meta,
                                  void* valsT, void* metaT, nm_meta_layout_t layout, nm_stream_t stream);

/*
 * nm_sgd_prune_transposable - the optimizer's weight write fused with the
 * run-time re-prune of a 2:4 training layer (PyTorch issue #126420,
 * maintainer reply: fast sparsification kernels do run-time sparsity for
 * training, with the 4x4-tile mask that serves W x and W^T dL/dy).  In one
 * pass over W (rows x cols, leading dimension ld, F16 or BF16, updated in
 * place) and its gradient dW (leading dimension ld_grad, same type):
 *   W[i][j] <- round(W[i][j] + round(round(-lr * dW[i][j])))
 * where the product and the sum are each rounded to float32 (no fused
 * multiply-add) and the result is rounded to W's type (round to nearest
 * even); then the updated W is pruned and compressed exactly as
 * nm_prune_transposable does (mask_bits, vals/meta, valsT/metaT, each
 * nullable; W itself stays dense: it is the master copy the next step
 * updates).  Requirements as nm_prune_transposable, plus dW 4-element
 * aligned (NM_ERR_MISALIGNED); I8 is NM_ERR_UNSUPPORTED; dW must not alias W.
 */
nm_status_t nm_sgd_prune_transposable(void* W, const void* dW, float lr, int64_t rows, int64_t cols, int64_t ld,
                                      int64_t ld_grad, nm_dtype_t dtype, uint32_t* mask_bits, void* vals, void* meta,
                                      void* valsT, void* metaT, nm_meta_layout_t layout, nm_stream_t stream);

/* ------------------------------------------------------------------------
 * Vector-wise and block-wise pruning (apex PR #1631 "[sparse] update support
 * for arbitrary N:M settings sparse", extension 2: unstructured_vector_wise
 * and unstructured_block_wise).  A unit is a 1 x v vector (v consecutive
 * elements of a row) or a bh x bw block; units are numbered in row-major
 * order of their top-left element.  The `keep` units with the largest score
 * are kept, equal scores going to the lower unit index; everything else is
 * pruned.  Callers derive keep from a density as floor(units * density).
 *
 * Scores are computed exactly (f16 and int8 only): vector-wise by |sum w|
 * (NM_SCORE_ABS_OF_SUM, the page's rule) or sum |w| (NM_SCORE_SUM_OF_ABS);
 * block-wise always by sum |w|.  An infinite score ranks above every number,
 * a NaN score (a NaN element, or +Inf and -Inf in one signed sum) below
 * every number.
 *
 * Outputs, each nullable:
 *   W_out      pruned copy (kept units copied, the rest +0); may alias W
 *              with ld_out == ld.
 *   mask_bits  bit mask of the kept elements (format above).
 *   csr        int32: unit-row pointers (rows/bh + 1 entries, entry r = kept
 *              units before unit row r), then one unit-column index per kept
 *              unit (column c covers W columns bw*c .. bw*c + bw - 1), in
 *              ascending order within each unit row.  rows/bh + 1 + keep
 *              entries in all.
 *   vals       the kept units' elements, unit after unit in the csr order,
 *              each unit row-major (bh * bw elements); keep * bh * bw
 *              elements in all.
 * workspace: device scratch of nm_prune_units_workspace bytes, 16-byte
 * aligned; its contents are not needed between calls.  Calls that share a
 * workspace must not overlap on the GPU.
 * Requirements: dtype NM_F16 or NM_I8 (NM_ERR_UNSUPPORTED otherwise);
 * v == 32, bh == bw == 32 (NM_ERR_UNSUPPORTED otherwise); cols % bw == 0 and
 * rows % bh == 0; 0 <= keep <= units < 2^31; W, W_out and vals 16-byte
 * aligned and ld, ld_out multiples of 16 bytes (NM_ERR_MISALIGNED).
 * ---------------------------------------------------------------------- */
typedef enum { NM_SCORE_ABS_OF_SUM = 0, NM_SCORE_SUM_OF_ABS = 1 } nm_score_t;

/* Host-only: workspace bytes for a rows x cols matrix cut into bh x bw units. */
nm_status_t nm_prune_units_workspace(int64_t rows, int64_t cols, int bh, int bw, size_t* bytes);

/* Vector-wise pruning: units are 1 x v vectors. */
nm_status_t nm_prune_vector_wise(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int v,
                                 int64_t keep, nm_score_t score, void* W_out, int64_t ld_out, uint32_t* mask_bits,
                                 int32_t* csr, void* vals, void* workspace, size_t workspace_bytes,
                                 nm_stream_t stream);

/* Block-wise pruning: units are bh x bw blocks, scored by sum |w|. */
nm_status_t nm_prune_block_wise(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype, int bh,
                                int bw, int64_t keep, void* W_out, int64_t ld_out, uint32_t* mask_bits, int32_t* csr,
                                void* vals, void* workspace, size_t workspace_bytes, nm_stream_t stream);

/*
 * nm_prune_vector_wise_noalloc - nm_prune_vector_wise without a workspace
 * argument, for callers that cannot allocate device memory at the time of the
 * call: code whose device memory is owned and accounted by someone else (a
 * framework's caching allocator, an inference server that forbids new
 * allocations once it has started), and latency-critical loops that cannot
 * afford cudaMalloc's implicit synchronisation or an out-of-memory failure
 * at run time.  The pages have no counterpart; it is an addition of this
 * library.
 *
 * The scratch lives in a fixed array of device memory inside the library
 * (about 8 MiB, held on every device that loads the library until the
 * process exits), so the call allocates nothing.  It handles at most
 * NM_NOALLOC_MAX_UNITS vectors (rows * cols / v); larger matrices are
 * rejected with NM_ERR_UNSUPPORTED before anything runs.  Every other
 * argument, requirement and output is that of nm_prune_vector_wise.
 *
 * The first call on a device does a one-time set-up on the current device
 * (it looks up the array's device address, which may load the library's
 * device code); make that first call before any stream capture.  The address
 * is kept for the rest of the process, so the device (or its primary context)
 * must not be reset after the first call.  Every argument is checked before
 * that set-up: a rejected call touches no CUDA state.  All calls on
 * a device share the one array and each call clears what must start at zero,
 * so calls must not overlap on the GPU: two calls in flight at the same time
 * (on different streams, or from different host threads) race on the
 * scratch and give wrong results.
 */
#define NM_NOALLOC_MAX_UNITS 524288
nm_status_t nm_prune_vector_wise_noalloc(const void* W, int64_t rows, int64_t cols, int64_t ld, nm_dtype_t dtype,
                                         int v, int64_t keep, nm_score_t score, void* W_out, int64_t ld_out,
                                         uint32_t* mask_bits, int32_t* csr, void* vals, nm_stream_t stream);

/* ------------------------------------------------------------------------
 * The product D = alpha * op(A) * op(B) + beta * C  (cuSPARSELt blog, the
 * GEMM paragraph: A is M x K, B is K x N, C and D are M x N; "N" layout =
 * column-major, "T" = row-major; FP16/BF16 inputs accumulate in FP32, INT8
 * inputs in INT32).
 * ---------------------------------------------------------------------- */
typedef enum {
  NM_SPMM_SPARSE_A = 0,       /* A is N:M sparse, given compressed (values + metadata)                */
  NM_SPMM_DENSE_MASKED = 1,   /* A and B dense; the product is multiplied by a bit mask of D's shape  */
  NM_SPMM_BLOCK_SPARSE_A = 2  /* A is given as its kept n x m units: values + CSR (see below)         */
} nm_spmm_mode_t;

typedef enum {
  NM_ROW = 0, /* row-major: the second index is contiguous */
  NM_COL = 1  /* column-major: the first index is contiguous */
} nm_order_t;

/*
 * Algorithm selection for the tensor-core products (SPARSE_A 2:4 F16/BF16 and
 * DENSE_MASKED), after the algorithm-selection step of the cuSPARSELt blog's
 * code example.  Other products have one kernel and ignore the choice.
 *   NM_ALGO_DEFAULT  the library's choice: paired CTAs when M spans an even
 *                    number of 128-row blocks, single CTAs otherwise.
 *   NM_ALGO_PAIRED   two CTAs of a cluster run one M256 x N256 tile with
 *                    tcgen05 cta_group::2 (each holds 128 rows of A and half
 *                    of B); falls back to single CTAs for an odd block count.
 *   NM_ALGO_SINGLE   one CTA per M128 x N256 tile (tcgen05 cta_group::1).
 */
typedef enum { NM_ALGO_DEFAULT = 0, NM_ALGO_PAIRED = 1, NM_ALGO_SINGLE = 2 } nm_algo_t;

typedef struct {
  int64_t M, N, K;
  nm_spmm_mode_t mode;
  int n, m;                     /* sparsity of A (SPARSE_A)                                   */
  nm_dtype_t ab_type;           /* F16, BF16 or I8                                            */
  nm_dtype_t cd_type;           /* F16/BF16 in: ab_type, or F32 (tensor-core products);       */
                                /* I8 in (2:4 sparse product): I32, or I8 (see nm_spmm)       */
  nm_order_t order_a;           /* DENSE_MASKED: ROW = A stored M x K, COL = stored K x M     */
  nm_order_t order_b;           /* ROW = B stored K x N, COL = B stored N x K                 */
  nm_order_t order_cd;          /* ROW = C, D stored M x N, COL = stored N x M                */
  int64_t lda, ldb, ldc, ldd;   /* leading dimensions in elements (lda: DENSE_MASKED only)    */
  nm_meta_layout_t meta_layout; /* SPARSE_A 2:4 with F16/BF16 needs NM_META_TC                */
  int algo;                     /* an nm_algo_t                                               */
} nm_spmm_desc_t;

typedef struct nm_spmm_plan_s* nm_spmm_plan_t;

/*
 * nm_spmm_plan - validate a product description and choose its kernel and
 * tile configuration once (cuSPARSELt blog, code example: matrix and matmul
 * descriptors, algorithm selection, plan).  *plan is a host object owned by
 * the caller until nm_spmm_plan_destroy; it is read-only afterwards and may
 * be used from several host threads.
 * Supported: SPARSE_A 2:4 F16/BF16 (tensor cores, B in NM_COL), SPARSE_A 2:4
 * I8 -> I32 (canonical metadata, B in NM_COL), SPARSE_A n:m with m <= 32 and
 * canonical metadata (CUDA-core gather, B in NM_COL, K < 2^31; with N > 1
 * also K <= 12800, the batch staged in shared memory), DENSE_MASKED F16/BF16
 * (tensor cores, any orders), BLOCK_SPARSE_A F16/BF16 with units of n x m =
 * 1 x 32 or 32 x 32 (CUDA cores, B in NM_COL; A = the vals and A_meta = the
 * csr that nm_prune_vector_wise / nm_prune_block_wise write; K % 32 == 0 and,
 * for 32 x 32, M % 32 == 0).
 */
nm_status_t nm_spmm_plan(nm_spmm_plan_t* plan, const nm_spmm_desc_t* desc);

/* Device workspace bytes nm_spmm needs with this plan (may be 0).  After
 * nm_spmm_search the size of the K split it chose, which never exceeds the
 * workspace_bytes given to the search. */
nm_status_t nm_spmm_plan_workspace(nm_spmm_plan_t plan, size_t* bytes);

/*
 * Host-only: the number of kernels one nm_spmm call with this plan launches on
 * its stream (*launches, host): 0 for an empty D, else 1, or 2 for a
 * DENSE_MASKED product split along K whose splits a separate kernel sums (the
 * paired kernel sums two splits itself).  Reflects the plan's algorithm as
 * chosen by nm_spmm_search when that has run.
 */
nm_status_t nm_spmm_plan_launches(nm_spmm_plan_t plan, int* launches);

/*
 * nm_spmm_plan_split_k - the number of parts a DENSE_MASKED plan splits K into
 * (*split_k, host; 1 = not split), as planned or as nm_spmm_search chose; 1
 * for every other product.  Splits hold whole 64-K stages; the last may be
 * shorter.
 */
nm_status_t nm_spmm_plan_split_k(nm_spmm_plan_t plan, int* split_k);

nm_status_t nm_spmm_plan_destroy(nm_spmm_plan_t plan);

/*
 * nm_spmm - run a planned product (cuSPARSELt blog, cusparseLtMatmul).
 * alpha, beta: HOST pointers to float (F16/BF16 inputs, or I8 inputs with an I8
 * output) or int32 (I8 inputs with an I32 output).  With an I8 output the
 * scales are float: D = saturate(round(alpha * acc + beta * C)) where acc is
 * the exact int32 accumulation, the int32 -> float conversion, each product
 * and the sum are rounded to float32, the result is rounded to the nearest
 * integer (ties to even) and clamped to [-128, 127] (cuSPARSELt blog, key
 * features: INT8 inputs and output; the pages give no scale, this is the
 * library's definition).  beta == 0
 * means C is not read (it may be NULL).  A: compressed values (SPARSE_A) or
 * dense A (DENSE_MASKED).  A_meta: metadata (SPARSE_A) or the bit mask of
 * D's M x N shape in row-major order (DENSE_MASKED; NULL = no mask, a plain
 * dense product).  C may alias D.
 * workspace: device buffer of at least nm_spmm_plan_workspace bytes (NULL if
 * 0); its contents need no initialisation (a DENSE_MASKED product split
 * along K keeps fp32 partials there and, with two splits on paired CTAs,
 * per-launch arrival words through which the product sums the splits
 * itself); calls that may run at the same time must not share one.  d_status (nullable, device int32): set to NM_ERR_TIMEOUT if a bounded
 * pipeline wait gave up; it is not cleared by the call.
 * Base pointers must be 16-byte aligned and leading dimensions multiples of
 * 16 bytes (NM_ERR_MISALIGNED); for the CUDA-core products (SPARSE_A with
 * (n, m) != (2, 4), BLOCK_SPARSE_A) C and D need only element alignment.
 */
nm_status_t nm_spmm(nm_spmm_plan_t plan, const void* alpha, const void* A, const void* A_meta, const void* B,
                    const void* beta, const void* C, void* D, void* workspace, size_t workspace_bytes,
                    int32_t* d_status, nm_stream_t stream);

/*
 * nm_spmm_search - algorithm search at plan time (cuSPARSELt blog, code
 * example: the algorithm-selection step, and the closing paragraph's
 * performance auto-tuning, cusparseLtMatmulSearch).  For a plan whose
 * description asked for NM_ALGO_DEFAULT on a tensor-core product (SPARSE_A
 * 2:4 F16/BF16 or DENSE_MASKED), the candidates are NM_ALGO_PAIRED and
 * NM_ALGO_SINGLE when M spans an even number of 128-row blocks (else the
 * single-CTA kernel alone) and, for DENSE_MASKED, the plan's K split s and the
 * splits s - 1, s - 2 and s + 1 that keep at least 8 stages of 64 K per split
 * and whose workspace fits in workspace_bytes.  It runs every candidate on the
 * given operands in three rounds that alternate them, each round `repeats`
 * timed runs per candidate (after one untimed run), timed with CUDA events on
 * `stream`, and keeps the fastest candidate's best round if it is at least 2%
 * faster than the default's (paired where possible, split s); else the
 * default.  Results of different K splits differ by float32 rounding only.
 * Other plans keep their kernel and only report it.  *chosen_algo (nullable,
 * host) receives the algorithm the plan now uses.
 * Arguments are those of nm_spmm; D (and the workspace) are overwritten with
 * the product, and with beta != 0 C must not alias D (NM_ERR_INVALID_ARG).
 * The call synchronises `stream`.  It changes the plan: do not run it while
 * another thread uses the same plan.  repeats must be 1..1000.
 */
nm_status_t nm_spmm_search(nm_spmm_plan_t plan, const void* alpha, const void* A, const void* A_meta, const void* B,
                           const void* beta, const void* C, void* D, void* workspace, size_t workspace_bytes,
                           int repeats, int* chosen_algo, nm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NM_H_ */
