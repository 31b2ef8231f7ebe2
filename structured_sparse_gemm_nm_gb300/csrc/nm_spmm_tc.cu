// Tensor-core products on Blackwell (sm_103a): D = alpha * A * B + beta * C.
//
//  * SPARSE:        A is 2:4 sparse (cuSPARSELt blog, Figure 2 text: half-size
//                   values plus metadata; the sparse tensor core skips the
//                   zeros), F16/BF16 with F32 accumulation.  Issued as
//                   tcgen05.mma.sp with the metadata in tensor memory.
//  * DENSE_MASKED:  A and B dense, D = alpha * (mask .* (A B)) + beta * C, the
//                   weight gradient of a layer whose weight keeps a fixed
//                   sparsity pattern.  Issued as dense tcgen05.mma; K may be
//                   split across CTAs (fp32 partials in the workspace, summed
//                   by a finalize kernel) when the output has few tiles.
//
// Pairs of CTAs.  A single CTA's M128 x N256 sparse MMA reads its A and B
// operands from shared memory at 128 bytes per clock (20 KB per K32 step: 160
// cycles, measured on GB300), more than the 2:4 tensor rate needs.  With
// cta_group::2 the two CTAs of a cluster run M256 MMAs over both CTAs' shared
// memory: each CTA stages its own 128 rows of A and one 128-row block of B
// (tile columns 128 r .. 128 r + 127 for rank r), and a paired sparse K32 step
// reads 12 KB per SM: measured at 128 cycles for M256 x N256, twice the dense
// rate.  Every CTA loads only the tiles it holds; no TMA load delivers to
// more than one CTA.
//
// Paired kernel (default when M spans an even number of 128-row blocks),
// warp roles per CTA:
//   warp 0       TMA producer (SPARSE: one lane per box): A, then B in 64-K
//                boxes of 16 KB, all on the even CTA's `full` barrier (a warp streams
//                large boxes grouped per barrier far faster than one box per
//                barrier); SPARSE stages hold 128 K, DENSE 64 K
//   warps 1, 14  even CTA: the two MMA issuers, columns 0..127 and 128..255
//                of the tile as M256 x N128 MMAs.  An MMA holds its issuing
//                thread until it has nearly completed, so every barrier wait,
//                commit or loop step of one issuer would leave the tensor pipe
//                idle; two issuers overlap each other's.  Issuer h reads rows
//                64 h .. 64 h + 63 of each CTA's B block.
//                (odd CTA: no issuer; its copies complete on the even CTA's
//                `full` barrier)
//   warps 2..5   SPARSE metadata: per pair of k-steps, each warp writes one
//                32-bit code word per lane (row) and k-step with tcgen05.st
//                into a pair of the four 64-column-aligned tensor-memory slots
//                of its own CTA (the sparse MMA reads metadata only there);
//                the two slot pairs alternate, each with a full/empty barrier
//                pair shared by both CTAs
//   warps 6..13  epilogue: drain this CTA's 128 accumulator rows with
//                tcgen05.ld, first half first, hand each half back to its
//                issuer, then write D straight from registers (no shared-
//                memory staging)
// The accumulator holds 256 columns (SPARSE: one buffer, the metadata slots
// use the other half of tensor memory; DENSE: two buffers).
//
// Single-CTA kernel (an odd number of row blocks, or algo NM_ALGO_SINGLE):
// M128 x N256 tiles, two MMA issuers of 128 columns each, metadata slot pairs
// per stage on the stage's `full` barrier, and an epilogue that stages 32 x 32
// blocks for TMA bulk stores.
//
// Every mbarrier wait is bounded; a wait that gives up sets an abort flag and
// NM_ERR_TIMEOUT in the caller's status word, the roles drain their
// outstanding asynchronous work and the CTA frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <chrono>
#include <mutex>

#include "nm_device.cuh"
#include "nm_internal.h"
#include "../../include/nm_testing.h"

namespace nmk {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int kKPerStage = 64;  // dense-equivalent K per stage
constexpr int kMetaWarp0 = 2, kMetaWarps = 4;
constexpr int kEpiWarp0 = kMetaWarp0 + kMetaWarps, kEpiWarps = 8;
constexpr int kMmaWarpB = kEpiWarp0 + kEpiWarps;  // single CTA: second MMA issuer (columns 128..255)
constexpr int kTmemCols = 512;
constexpr int kMetaCol = 256, kMetaColStride = 64;  // four metadata slots: columns 256, 320, 384, 448
constexpr int kEpiBufBytes = 32 * 32 * 2;  // single CTA: one 32 x 32 16-bit output block

// Output element kinds of C and D.
constexpr int kCdF16 = 0, kCdBF16 = 1, kCdF32 = 2;


template <bool SPARSE, bool PAIR>
struct Cfg {
  static constexpr int kWarps = kMmaWarpB + 1;
  static constexpr int kThreads = 32 * kWarps;
  // dense-equivalent K per stage: paired SPARSE stages hold 128 K (A 16 KB + B 2 x 16 KB, in large
  // TMA boxes), the others 64
  static constexpr int kKStage = (SPARSE && PAIR) ? 128 : kKPerStage;
  static constexpr int kSubs = kKStage / 64;  // SPARSE: pairs of k-steps per stage
  // A: SPARSE 128 rows x kKStage / 2 compressed values (64 B rows with the 64B swizzle, 128 B rows
  // with the 128B swizzle); dense 128 x 64 (128B swizzle)
  static constexpr int kATileBytes = SPARSE ? BM * kKStage : BM * 128;
  // B: rows x kKStage (boxes of 64 K with the 128B swizzle); a pair holds one 128-row half of the 256 rows
  static constexpr int kBRows = PAIR ? BN / 2 : BN;
  static constexpr int kBTileBytes = kBRows * 2 * kKStage;
  static constexpr int kTxBytes = kATileBytes + kBTileBytes;  // TMA bytes per stage
  static constexpr int kStageBytes = kTxBytes;
  static constexpr int kStages = PAIR ? (SPARSE ? 4 : 6) : (SPARSE ? 5 : 4);
  static constexpr int kAcc = SPARSE ? 1 : 2;  // 256-column accumulator buffers
  static constexpr int kEpiOffset = kStages * kStageBytes;
  // 16-bit D staging for the TMA stores: one 32 x 32 block per epilogue warp (two, alternating,
  // in the paired kernel)
  static constexpr int kEpiBufs = PAIR ? 2 : 1;
  static constexpr int kBarOffset = kEpiOffset + kEpiWarps * kEpiBufs * kEpiBufBytes;
  static constexpr int kSmemBytes = 1024 + kBarOffset + 512;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct Params {
  int M, N, K;
  int num_m_blk, num_n_blk;
  int k_stages;          // stages over the whole K
  int split_k;           // DENSE: number of K splits (1 = direct epilogue)
  int stages_per_split;
  int num_units;         // (pair-)tiles x splits
  int num_k_steps;       // SPARSE: K / 32
  const uint32_t* meta;  // SPARSE: tensor-core metadata [K/32][meta_slots]
  int64_t meta_slots;
  int a_mn, b_mn;        // DENSE operand majors (1 = M/N contiguous)
  int bf16;              // A, B element type
  int cd_kind;           // kCdF16, kCdBF16 or kCdF32
  float alpha, beta;
  const void* C;
  void* D;
  int64_t ldc, ldd;
  int cd_col;     // 1: D[n * ldd + m]; 0: D[m * ldd + n]
  int tma_store;  // single CTA: 1 = D written by TMA bulk stores (16-bit D, C not read)
  const uint32_t* mask;
  int64_t mask_words;
  float* partial;  // DENSE split-K: tiled fp32 partials
  // DENSE split-K summed in the product (paired, two splits): per epilogue warp and tile, a
  // 64-bit word (launch token << 32 | arrivals); the warp that arrives last sums the splits
  int fuse_split;
  uint32_t split_token;
  unsigned long long* split_cnt;
  int32_t* status;
  long long wait_budget;  // cycles
  int fault_test;         // 1: the MMA lane waits on a barrier nothing arrives at
};

// ----------------------------------------------------------------- PTX glue
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// CLUSTER: acquire at cluster scope, for barriers the other CTA of the pair arrives on.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (CLUSTER)
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  return ok != 0;
}

// Bounded wait: false if the budget ran out (then the status word and the
// CTA's abort flag are set) or another role already aborted.
template <bool CLUSTER = false>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, long long budget,
                                            int32_t* status) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try<CLUSTER>(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      if (status != nullptr) atomicExch(status, (int)NM_ERR_TIMEOUT);
      return false;
    }
  }
}
// The phase is usually complete already: test it inline and only call out to
// the bounded loop when it is not.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, long long budget,
                                          int32_t* status) {
  if (mbar_try<CLUSTER>(bar, parity)) return true;
  return mbar_wait_slow<CLUSTER>(bar, parity, abort_flag, budget, status);
}
// Drain wait at the end of a role: bounded, no status (the role already reported any timeout).
template <bool CLUSTER = false>
__device__ __forceinline__ void mbar_wait_quiet(uint32_t bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  while (!mbar_try<CLUSTER>(bar, parity) && clock64() - t0 < budget) {
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Paired form: the copy lands in this CTA's shared memory and completes its bytes on a
// barrier that may sit in the other CTA of the pair (here: the even CTA's `full` barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cluster_bar, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
               "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
// Relaxed remote arrive.  Used where what it announces was completed by the
// arriving thread itself and is read only through the arriving CTA's own
// shared or tensor memory (TMA bytes whose completion this thread observed,
// metadata written with tcgen05.st and waited for, accumulator columns read
// with tcgen05.ld and waited for).  A release at cluster scope costs over a
// thousand cycles per arrive on GB300.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start, leading/stride byte
// offsets (16-byte units), fixed version bit 46, swizzle mode in bits 61..63.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}
constexpr uint32_t kSwizzle128 = 2, kSwizzle64 = 4;

// Instruction descriptor for kind::f16: D = F32, A/B = F16 or BF16, shape M x N.
__device__ __forceinline__ uint32_t idesc_f16(int bf16, int a_mn, int b_mn, bool sparse, int m, int n) {
  uint32_t d = (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) | ((uint32_t)a_mn << 15) |
               ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
  if (sparse) d |= 1u << 2;
  return d;
}

__device__ __forceinline__ void mma_dense(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_sparse(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t tmem_meta, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\ntcgen05.mma.sp.cta_group::1.kind::f16 [%0], %1, %2, [%3], %4, p;\n}" ::
          "r"(tmem_d),
      "l"(a), "l"(b), "r"(tmem_meta), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// cta_group::2 forms: the MMA is issued by the even CTA of the pair and reads
// the operands of both CTAs at the same shared-memory offsets (and the
// metadata of both at the same tensor-memory column); a commit arrives on one
// barrier, in either CTA, once the prior MMAs of the issuing thread complete.
__device__ __forceinline__ void mma_dense_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_sparse_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t tmem_meta,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\ntcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n}" ::
          "r"(tmem_d),
      "l"(a), "l"(b), "r"(tmem_meta), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit_pair(uint32_t cluster_bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(cluster_bar)
               : "memory");
}
// The same barrier offset in both CTAs of the pair.
__device__ __forceinline__ void tc_commit_both(uint32_t bar) {
  tc_commit_pair(bar);
  tc_commit_pair(peer_addr(bar, 1));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Loads and the wait for them sit in one asm statement: the registers are
// defined only once the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// Two 32-column loads in flight at once.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// C and D elements: f16, bf16 or f32 (cd_kind).
__device__ __forceinline__ float load_cd(const void* base, int64_t off, int cd_kind) {
  if (cd_kind == kCdF32) return reinterpret_cast<const float*>(base)[off];
  const uint16_t b = reinterpret_cast<const uint16_t*>(base)[off];
  return cd_kind == kCdBF16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
}
__device__ __forceinline__ void store_cd(void* base, int64_t off, float x, int cd_kind) {
  if (cd_kind == kCdF32) {
    reinterpret_cast<float*>(base)[off] = x;
    return;
  }
  reinterpret_cast<uint16_t*>(base)[off] = cd_kind == kCdBF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x))
                                                              : __half_as_ushort(__float2half_rn(x));
}
// Compile-time form for the drain: one conversion instruction per pair.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2t(float lo, float hi) {
  if constexpr (BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
  // one round-to-nearest conversion of the pair; `lo` lands in the low 16 bits
  return bf16 ? pack2t<true>(lo, hi) : pack2t<false>(lo, hi);
}
// One warp's 32 lanes x 64 accumulator columns (two 32-column loads in flight)
// into packed pairs: alpha applied when SCALE, masked columns zeroed when
// MASKED (mask words ma, mb for the two 32-column halves).
template <bool BF16, bool SCALE, bool MASKED>
__device__ __forceinline__ void pack64(const uint32_t (&va)[32], const uint32_t (&vb)[32], float alpha, uint32_t ma,
                                       uint32_t mb, uint32_t (&pa)[16], uint32_t (&pb)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float a0 = __uint_as_float(va[2 * j]), a1 = __uint_as_float(va[2 * j + 1]);
    float b0 = __uint_as_float(vb[2 * j]), b1 = __uint_as_float(vb[2 * j + 1]);
    if constexpr (SCALE) {
      a0 *= alpha;
      a1 *= alpha;
      b0 *= alpha;
      b1 *= alpha;
    }
    if constexpr (MASKED) {
      a0 = ((ma >> (2 * j)) & 1u) ? a0 : 0.0f;
      a1 = ((ma >> (2 * j + 1)) & 1u) ? a1 : 0.0f;
      b0 = ((mb >> (2 * j)) & 1u) ? b0 : 0.0f;
      b1 = ((mb >> (2 * j + 1)) & 1u) ? b1 : 0.0f;
    }
    pa[j] = pack2t<BF16>(a0, a1);
    pb[j] = pack2t<BF16>(b0, b1);
  }
}
template <bool MASKED>
__device__ __forceinline__ void pack64_any(int bf16, bool scale, const uint32_t (&va)[32], const uint32_t (&vb)[32],
                                           float alpha, uint32_t ma, uint32_t mb, uint32_t (&pa)[16],
                                           uint32_t (&pb)[16]) {
  if (bf16) {
    if (scale)
      pack64<true, true, MASKED>(va, vb, alpha, ma, mb, pa, pb);
    else
      pack64<true, false, MASKED>(va, vb, alpha, ma, mb, pa, pb);
  } else {
    if (scale)
      pack64<false, true, MASKED>(va, vb, alpha, ma, mb, pa, pb);
    else
      pack64<false, false, MASKED>(va, vb, alpha, ma, mb, pa, pb);
  }
}
template <bool MASKED>
__device__ __forceinline__ void drain64_any(int bf16, bool scale, uint32_t taddr, float alpha, uint32_t ma,
                                            uint32_t mb, uint32_t (&pa)[16], uint32_t (&pb)[16]) {
  uint32_t va[32], vb[32];
  tmem_ld32x2(taddr, taddr + 32, va, vb);
  pack64_any<MASKED>(bf16, scale, va, vb, alpha, ma, mb, pa, pb);
}
// Work unit u -> 128-row block of this CTA, 256-column block and K split.
// Paired: the pair's 256 rows are row blocks 2 * (pair index) and
// 2 * (pair index) + 1, the CTA of rank r taking the second index r.
struct Unit {
  int m0, n0, kbeg, kend, split;
};
__device__ __forceinline__ Unit decode_unit(const Params& p, int u, int cl, int rank) {
  Unit t;
  const int mcount = p.num_m_blk / cl;
  const int mi = u % mcount;
  const int rest = u / mcount;
  t.n0 = (rest % p.num_n_blk) * BN;
  t.split = rest / p.num_n_blk;
  t.m0 = (mi * cl + rank) * BM;
  t.kbeg = t.split * p.stages_per_split;
  t.kend = min(p.k_stages, t.kbeg + p.stages_per_split);
  return t;
}

// fp32 partial of one K split, in the tiled order
// [split][m block][n block][col / 4][128 rows][4]: for each group of four
// columns the 32 lanes of a warp write 512 contiguous bytes.
__device__ __forceinline__ void store_partial_chunk(const Params& p, const Unit& t, int col, int q, int lane,
                                                    const uint32_t (&v)[32], uint32_t mword) {
  float4* tile = reinterpret_cast<float4*>(p.partial) +
                 ((int64_t)(t.split * p.num_m_blk + t.m0 / BM) * p.num_n_blk + t.n0 / BN) * (BM * BN / 4);
  const int c4_0 = col / 4;
#pragma unroll
  for (int j4 = 0; j4 < 8; ++j4) {
    float4 w;
    w.x = ((mword >> (4 * j4)) & 1u) ? __uint_as_float(v[4 * j4]) * p.alpha : 0.0f;
    w.y = ((mword >> (4 * j4 + 1)) & 1u) ? __uint_as_float(v[4 * j4 + 1]) * p.alpha : 0.0f;
    w.z = ((mword >> (4 * j4 + 2)) & 1u) ? __uint_as_float(v[4 * j4 + 2]) * p.alpha : 0.0f;
    w.w = ((mword >> (4 * j4 + 3)) & 1u) ? __uint_as_float(v[4 * j4 + 3]) * p.alpha : 0.0f;
    tile[(c4_0 + j4) * BM + 32 * q + lane] = w;
  }
}
// Element-wise D of one row's 32 columns starting at nb: alpha, mask, beta * C.
__device__ __forceinline__ void store_chunk_generic(const Params& p, int row, int nb, const uint32_t (&v)[32],
                                                    uint32_t mword) {
  const int cnt = min(32, p.N - nb);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j >= cnt) break;
    float x = ((mword >> j) & 1u) ? __uint_as_float(v[j]) * p.alpha : 0.0f;
    const int64_t doff = p.cd_col ? (int64_t)(nb + j) * p.ldd + row : (int64_t)row * p.ldd + nb + j;
    const int64_t coff = p.cd_col ? (int64_t)(nb + j) * p.ldc + row : (int64_t)row * p.ldc + nb + j;
    if (p.C != nullptr) x = fmaf(p.beta, load_cd(p.C, coff, p.cd_kind), x);
    store_cd(p.D, doff, x, p.cd_kind);
  }
}

// Split-K summed in the product: the arrival of one epilogue warp at its region of a tile, after
// its partial stores (this launch's token in the high word; a stale token restarts the count).
// Returns true for the warp that arrives last (which resets the word); its later reads of the
// other splits' partials are ordered after their writers' fences by the atomic and the fence
// that follows it.
__device__ __forceinline__ bool split_arrive_last(const Params& p, int64_t idx, int lane) {
  __threadfence();  // this lane's partial stores before the arrival
  __syncwarp();
  uint32_t last = 0;
  if (lane == 0) {
    unsigned long long* w = p.split_cnt + idx;
    const unsigned long long tok = (unsigned long long)p.split_token << 32;
    unsigned long long old = atomicAdd(w, 0ull), nw;
    while (true) {
      nw = (old & 0xFFFFFFFF00000000ull) == tok ? old + 1ull : tok | 1ull;
      const unsigned long long prev = atomicCAS(w, old, nw);
      if (prev == old) break;
      old = prev;
    }
    last = (uint32_t)nw == (uint32_t)p.split_k ? 1u : 0u;
    // every split has arrived: the word returns to 0, which no launch's token equals, so a
    // workspace that outlives this launch (or this process) holds no count of it
    if (last) atomicExch(w, 0ull);
    __threadfence();
  }
  return __shfl_sync(0xFFFFFFFFu, last, 0) != 0;
}
// The sum over the splits (in split order) of one row's 32 columns of a tile's partials, then
// beta * C, stored to D; the same arithmetic as the separate finalize.
__device__ __forceinline__ void store_split_sum_chunk(const Params& p, const Unit& t, int col, int q, int lane,
                                                      int row, int nb) {
  const int64_t per_split = (int64_t)p.num_m_blk * p.num_n_blk * (BM * BN / 4);
  const float4* src = reinterpret_cast<const float4*>(p.partial) +
                      ((int64_t)(t.m0 / BM) * p.num_n_blk + t.n0 / BN) * (BM * BN / 4) + (col / 4) * BM + 32 * q + lane;
  float x[32];
#pragma unroll
  for (int j4 = 0; j4 < 8; ++j4) {
    const float4 w = __ldcg(src + j4 * BM);
    x[4 * j4] = w.x, x[4 * j4 + 1] = w.y, x[4 * j4 + 2] = w.z, x[4 * j4 + 3] = w.w;
  }
  for (int sp = 1; sp < p.split_k; ++sp) {
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
      const float4 w = __ldcg(src + sp * per_split + j4 * BM);
      x[4 * j4] += w.x, x[4 * j4 + 1] += w.y, x[4 * j4 + 2] += w.z, x[4 * j4 + 3] += w.w;
    }
  }
  if (row >= p.M || nb >= p.N) return;
  const int cnt = min(32, p.N - nb);
  if (p.C != nullptr) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j >= cnt) break;
      const int64_t coff = p.cd_col ? (int64_t)(nb + j) * p.ldc + row : (int64_t)row * p.ldc + nb + j;
      x[j] = fmaf(p.beta, load_cd(p.C, coff, p.cd_kind), x[j]);
    }
  }
  if (!p.cd_col && cnt == 32 && p.cd_kind != kCdF32) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.D) + (int64_t)row * p.ldd + nb;
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = pack2(x[2 * j], x[2 * j + 1], p.cd_kind == kCdBF16);
#pragma unroll
      for (int k = 0; k < 4; ++k) reinterpret_cast<uint4*>(dst)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
      return;
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j >= cnt) break;
    const int64_t doff = p.cd_col ? (int64_t)(nb + j) * p.ldd + row : (int64_t)row * p.ldd + nb + j;
    store_cd(p.D, doff, x[j], p.cd_kind);
  }
}

// fp32 D of one row's 32 columns starting at nb (no C, no K split): alpha and the mask applied;
// column-major D: 32 lanes (rows) write 128 contiguous bytes per column; row-major: 16-byte stores.
__device__ __forceinline__ void store_chunk_f32(const Params& p, int row, int nb, const uint32_t (&v)[32],
                                                uint32_t mword, bool scale) {
  const int cnt = min(32, p.N - nb);
  float* D32 = reinterpret_cast<float*>(p.D);
  auto val = [&](int j) -> float {
    const float x = __uint_as_float(v[j]);
    return ((mword >> j) & 1u) ? (scale ? x * p.alpha : x) : 0.0f;
  };
  if (p.cd_col) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < cnt) D32[(int64_t)(nb + j) * p.ldd + row] = val(j);
  } else if (cnt == 32) {
    float4* dst = reinterpret_cast<float4*>(D32 + (int64_t)row * p.ldd + nb);
#pragma unroll
    for (int k = 0; k < 8; ++k) dst[k] = make_float4(val(4 * k), val(4 * k + 1), val(4 * k + 2), val(4 * k + 3));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < cnt) D32[(int64_t)row * p.ldd + nb + j] = val(j);
  }
}

// ----------------------------------------------------------------- kernel
// The warps of a CTA are spread over the SM's four sub-partitions, each with a
// quarter of the register file: 14 or 15 warps put four on one of them, so
// 128 registers per thread is the most that fits.
template <bool SPARSE, bool PAIR>
__global__ void __maxnreg__(128)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const Params p) {
  using C = Cfg<SPARSE, PAIR>;
  constexpr int CL = PAIR ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  // bars: full[S], empty[S], tfull[2], tempty[4] (single: 2 buffers x 2 column halves; paired: one per
  // buffer), drain, mfull[2], mempty[2] (paired SPARSE: one pair per metadata slot pair)
  const uint32_t bar_full = smem_u32(bars), bar_empty = smem_u32(bars + C::kStages);
  const uint32_t bar_tfull = smem_u32(bars + 2 * C::kStages), bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 32;
  const uint32_t bar_mfull = bar_drain + 8, bar_mempty = bar_mfull + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x / CL, num_clusters = gridDim.x / CL;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      uint32_t full_count;
      // single CTA: the producer's expect_tx arrival and (SPARSE) one arrival per metadata warp
      // once it has written the stage's metadata slot pair; paired: the even CTA's producer arms
      // its barrier with both CTAs' bytes, and both CTAs' copies complete on it (the odd CTA's
      // `full` barriers stay unused)
      if constexpr (PAIR)
        full_count = 1;
      else
        full_count = 1 + (SPARSE ? kMetaWarps : 0);
      mbar_init(bar_full + 8 * s, full_count);
      // released by the commits of the two issuers that read the stage
      mbar_init(bar_empty + 8 * s, 2);
    }
    for (int a = 0; a < 2; ++a) mbar_init(bar_tfull + 8 * a, 2);
    // one arrival per epilogue warp once it has read its columns of that half (paired: from both CTAs)
    for (int a = 0; a < 4; ++a) mbar_init(bar_tempty + 8 * a, PAIR ? 2 * kEpiWarps : kEpiWarps);
    mbar_init(bar_drain, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_mfull + 8 * i, 2 * kMetaWarps);  // paired SPARSE: the metadata warps of both CTAs
      mbar_init(bar_mempty + 8 * i, 2);              // the commits of the two paired issuers
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (PAIR) {  // collective across the pair: both CTAs allocate
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // set-up done: from here on global memory may hold the previous grid's results
  pdl_trigger();
  pdl_wait();

  if (PAIR && warp == 0) {
    // ------------------------------------------------------- paired TMA producer
    // This CTA holds 128 rows of A and the 128-row block 128 r .. 128 r + 127 of the
    // tile's B (r = this CTA's rank).  The stage's copies, A then B in 64-K boxes of 16 KB,
    // complete on one barrier: measured on GB300, one warp streams large boxes grouped per
    // barrier at about the L2's rate.  Both CTAs' copies complete on the even
    // CTA's `full` barrier, which its producer arms with the bytes of both; the odd CTA's
    // bytes may land before that arming, which only makes the transaction count
    // transiently negative within the phase.  The odd CTA issues a stage only after its
    // `empty` barrier shows the previous phase consumed, so its bytes never reach an
    // earlier phase.
    // A bulk tensor copy holds the thread that issues it for a few hundred cycles.  SPARSE:
    // each of the stage's three boxes (A, B's two 64-K halves) is issued by its own lane of
    // a warp that runs the loop together, which measured 3-4% faster than one lane issuing
    // all three.  DENSE: one lane runs the loop and issues the stage's boxes (A: one, or two
    // 64-row boxes when M-major; B: likewise); the warp-wide form measured 20-25% slower
    // there.
    const uint32_t lead_full = peer_addr(bar_full, 0);
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    }
    if constexpr (SPARSE) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_parity = 0;  // per-stage bits for the drain at the end
      bool ok = true;
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
        const Unit t = decode_unit(p, u, CL, rank);
        const int nb = t.n0 + C::kBRows * (int)rank;  // first column of D this CTA's B block holds
        for (int ks = t.kbeg; ks < t.kend; ++ks) {
          if (lane == 0)
            ok = mbar_wait<true>(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.wait_budget, p.status);
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) break;
          const uint32_t fb = lead_full + 8 * stage;
          const uint32_t sA = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sB = sA + C::kATileBytes;
          if (leader && lane == 0) mbar_expect_tx(bar_full + 8 * stage, 2 * C::kTxBytes);
          if (lane == 0)
            tma_load_2d_pair(sA, &tmA, fb, ks * (C::kKStage / 2), t.m0);
          else if (lane <= C::kKStage / 64)  // 128 rows x 64 K per box
            tma_load_2d_pair(sB + 16384u * (uint32_t)(lane - 1), &tmB, fb, ks * C::kKStage + 64 * (lane - 1), nb);
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: every copy into this CTA must have landed before the CTA may exit.  The even
      // CTA waits for its `full` barriers (both CTAs' bytes); the odd CTA, whose copies
      // complete there, for its `empty` barriers: a stage is released only after the MMAs
      // that read it, which waited for all its bytes.
      if (lane == 0)
        for (int s = 0; s < C::kStages; ++s)
          if ((issued >> s) & 1u)
            mbar_wait_quiet<true>((leader ? bar_full : bar_empty) + 8 * s, (last_parity >> s) & 1u, p.wait_budget);
    } else if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_parity = 0;
      bool ok = true;
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
        const Unit t = decode_unit(p, u, CL, rank);
        const int nb = t.n0 + C::kBRows * (int)rank;
        for (int ks = t.kbeg; ks < t.kend; ++ks) {
          if (!mbar_wait<true>(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.wait_budget, p.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = lead_full + 8 * stage;
          const uint32_t sA = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sB = sA + C::kATileBytes;
          if (leader) mbar_expect_tx(bar_full + 8 * stage, 2 * C::kTxBytes);
          if (p.a_mn) {  // two 64-row (M) boxes of 64 K
            tma_load_2d_pair(sA, &tmA, fb, t.m0, ks * 64);
            tma_load_2d_pair(sA + C::kATileBytes / 2, &tmA, fb, t.m0 + 64, ks * 64);
          } else {
            tma_load_2d_pair(sA, &tmA, fb, ks * 64, t.m0);
          }
          if (p.b_mn) {  // two 64-row (N) boxes of 64 K
            tma_load_2d_pair(sB, &tmB, fb, nb, ks * 64);
            tma_load_2d_pair(sB + 8192, &tmB, fb, nb + 64, ks * 64);
          } else {
            tma_load_2d_pair(sB, &tmB, fb, ks * 64, nb);  // 128 rows x 64 K
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      for (int s = 0; s < C::kStages; ++s)
        if ((issued >> s) & 1u)
          mbar_wait_quiet<true>((leader ? bar_full : bar_empty) + 8 * s, (last_parity >> s) & 1u, p.wait_budget);
    }
  } else if (!PAIR && warp == 0) {
    // ------------------------------------------------------- TMA producer
    // A bulk tensor copy holds the thread that issues it for several hundred cycles
    // whatever its size, so the stage's copies (A, and B or this CTA's half of it) are
    // issued by one lane each, in one instruction.
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    }
    const int na = (!SPARSE && p.a_mn) ? 2 : 1;                    // copies of A per stage
    const int nbc = (!SPARSE && p.b_mn) ? C::kBRows / 64 : 1;       // copies of B per stage
    const bool copier = lane < na + nbc;
    const bool is_a = lane < na;
    const int h = is_a ? lane : lane - na;  // which copy of its operand this lane issues
    const CUtensorMap* map = is_a ? &tmA : &tmB;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, last_parity = 0;  // per-stage bits for the drain at the end
    bool ok = true;
    for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
      const Unit t = decode_unit(p, u, CL, rank);
      const int nb = t.n0 + C::kBRows * (int)rank;  // B: the tile's 256 rows, or this CTA's half of them
      for (int ks = t.kbeg; ks < t.kend; ++ks) {
        if (lane == 0) ok = mbar_wait<PAIR>(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.wait_budget, p.status);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        const uint32_t fb = bar_full + 8 * stage;
        const uint32_t sA = smem_u32(smem + stage * C::kStageBytes);
        const uint32_t sB = sA + C::kATileBytes;
        if (lane == 0) mbar_expect_tx(fb, C::kTxBytes);
        __syncwarp();
        if (copier) {
          uint32_t dst;
          int x, y;
          if (is_a) {
            if (SPARSE) {
              dst = sA, x = ks * (kKPerStage / 2), y = t.m0;
            } else if (p.a_mn) {  // two 64-row (M) boxes of 64 K
              dst = sA + (uint32_t)(C::kATileBytes / 2) * (uint32_t)h, x = t.m0 + 64 * h, y = ks * 64;
            } else {
              dst = sA, x = ks * 64, y = t.m0;
            }
          } else if (!SPARSE && p.b_mn) {  // 64-row (N) boxes of 64 K
            dst = sB + 8192 * h, x = nb + 64 * h, y = ks * 64;
          } else {
            dst = sB, x = ks * 64, y = nb;
          }
          tma_load_2d(dst, map, fb, x, y);
        }
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // Drain: every copy into this CTA must have landed before the CTA may exit.  (The full
    // barrier also counts the metadata warps' arrivals; those all come before the stage's
    // MMAs, so a consumed stage is complete, and an abort ends within the budget.)
    if (lane == 0)
      for (int s = 0; s < C::kStages; ++s)
        if ((issued >> s) & 1u) mbar_wait_quiet<PAIR>(bar_full + 8 * s, (last_parity >> s) & 1u, p.wait_budget);
  } else if (warp == 1 || warp == kMmaWarpB) {
    if constexpr (PAIR) {
      if (lane == 0 && leader) {
        // ----------------------------------------------- paired MMA issuers
        // An MMA holds its issuing thread until it has nearly completed, so every
        // instruction a single issuer runs between MMAs (barrier waits, commits,
        // loop work) would leave the tensor pipe idle.  Two issuers, warp 1 for
        // columns 0..127 of the tile and warp 14 for columns 128..255 (M256 x N128
        // MMAs), overlap each other's bookkeeping with MMAs.
        const int h = warp == 1 ? 0 : 1;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        const uint32_t idesc = idesc_f16(p.bf16, SPARSE ? 0 : p.a_mn, SPARSE ? 0 : p.b_mn, SPARSE, 2 * BM, BN / 2);
        constexpr uint32_t kStageUnits = C::kStageBytes >> 4;
        // Issuer h reads rows 64 h .. 64 h + 63 of each CTA's B block: its accumulator columns
        // 128 h .. 128 h + 63 are tile columns 64 h .. 64 h + 63 (the even CTA's block) and
        // 128 h + 64 .. 128 h + 127 are tile columns 128 + 64 h .. 128 + 64 h + 63 (the odd CTA's).
        const uint32_t sA0 = smem_u32(smem), sB0 = sA0 + C::kATileBytes + 8192u * (uint32_t)h;
        // Stage-0 descriptors; advancing the 14-bit start field by offset >> 4 moves them.
        //   SPARSE A: 128 rows x 128 B (128B swizzle), 32 B per k-step;
        //   SPARSE B: 128 rows x 128 B per 64-K box (boxes 16 KB apart), 64 B per k-step in a box
        //   DENSE K-major: 128B swizzle, 32 B per K16 step; M/N-major: 64-wide atoms 8 KB apart,
        //   2048 B per K16 step
        // SPARSE A rows hold kKStage / 2 compressed values: 64 B (64B swizzle, 8-row groups 512 B
        // apart) or 128 B (128B swizzle)
        const uint64_t a_desc0 = (!SPARSE && p.a_mn) ? sdesc(sA0, 8192, 1024, kSwizzle128)
                                 : (SPARSE && C::kKStage == 64) ? sdesc(sA0, 16, 512, kSwizzle64)
                                                                : sdesc(sA0, 16, 1024, kSwizzle128);
        const uint64_t b_desc0 = (!SPARSE && p.b_mn) ? sdesc(sB0, 8192, 1024, kSwizzle128)
                                                     : sdesc(sB0, 16, 1024, kSwizzle128);
        const uint32_t a_step = (!SPARSE && p.a_mn) ? (2048 >> 4) : (32 >> 4);
        const uint32_t b_step = SPARSE ? (64 >> 4) : (p.b_mn ? (2048 >> 4) : (32 >> 4));
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t g2 = 0;  // SPARSE: pairs of k-steps issued; pair g2 reads metadata slot pair g2 % 2
        if (p.fault_test && h == 0)  // the drain barrier cannot complete before this issuer commits: runs out
          ok = mbar_wait(bar_drain, 0, abort_flag, p.wait_budget, p.status);
        for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
          const Unit t = decode_unit(p, u, CL, rank);
          // both CTAs' epilogues have read this issuer's column half of the buffer
          if (!mbar_wait<true>(bar_tempty + 8 * (2 * acc + h), acc_phase ^ 1, abort_flag, p.wait_budget, p.status))
            break;
          tc_fence_after();
          const uint32_t tacc = tmem + acc * BN + (BN / 2) * h;
          int kstep = 0;
          for (int ks = t.kbeg; ks < t.kend; ++ks) {
            if (!mbar_wait<true>(bar_full + 8 * stage, phase, abort_flag, p.wait_budget, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = a_desc0 + (uint64_t)(stage * kStageUnits);
            const uint64_t bd = b_desc0 + (uint64_t)(stage * kStageUnits);
            if constexpr (SPARSE) {
              // four k-steps per stage, in two pairs; each pair waits for its metadata slot pair
              // (written by both CTAs' metadata warps) and its completion frees the pair
              for (int sub = 0; sub < C::kSubs; ++sub, ++g2) {
                const int k0 = 2 * C::kSubs * ks + 2 * sub;
                if (k0 >= p.num_k_steps) break;  // no MMA past K
                if (!mbar_wait<true>(bar_mfull + 8 * (g2 & 1u), (g2 >> 1) & 1u, abort_flag, p.wait_budget,
                                     p.status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint32_t tmeta = tmem + kMetaCol + kMetaColStride * 2 * (g2 & 1u);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  const int i = 2 * sub + j;  // k-step within the stage
                  if (j == 1 && k0 + 1 >= p.num_k_steps) break;
                  mma_sparse_pair(tacc, ad + (uint64_t)(i * a_step),
                                  bd + (uint64_t)(((16384 >> 4) * (i >> 1)) + b_step * (i & 1)),
                                  tmeta + kMetaColStride * j, idesc, (kstep > 0 || i > 0) ? 1u : 0u);
                }
                tc_commit_both(bar_mempty + 8 * (g2 & 1u));
              }
              if (!ok) break;
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_dense_pair(tacc, ad + (uint64_t)(j * a_step), bd + (uint64_t)(j * b_step), idesc,
                               (kstep > 0 || j > 0) ? 1u : 0u);
            }
            ++kstep;
            tc_commit_both(bar_empty + 8 * stage);
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          tc_commit_both(bar_tfull + 8 * acc);
          if (++acc == C::kAcc) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
        tc_commit_both(bar_drain);
      }
      // all paired MMAs have completed before either CTA frees its tensor memory
      if (lane == 0 && warp == 1) mbar_wait_quiet<true>(bar_drain, 0u, p.wait_budget);
    } else {
      // ----------------------------------------------------- single-CTA MMA issuers
      // Two single-thread issuers share every stage: warp 1 computes columns
      // 0..127 and warp kMmaWarpB columns 128..255 of the tile.  An MMA holds
      // its issuing thread for about its execution time, so while one issuer
      // waits, commits and loops, the other one keeps the tensor pipe busy.
      if (lane == 0) {
        const uint32_t nhalf = warp == 1 ? 0u : 1u;
        const uint32_t idesc = idesc_f16(p.bf16, SPARSE ? 0 : p.a_mn, SPARSE ? 0 : p.b_mn, SPARSE, BM, BN / 2);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t mpair = 0;  // SPARSE: metadata slot pair of the current stage (alternates every stage)
        constexpr uint32_t kStageUnits = C::kStageBytes >> 4;
        // B's second 128 rows (K-major) or second two 64-column atoms (MN-major) start 16 KB in
        const uint32_t sA0 = smem_u32(smem), sB0 = sA0 + C::kATileBytes + 16384u * nhalf;
        uint64_t a_desc0, b_desc0;
        uint32_t a_step = 0, b_step = 0;
        if constexpr (SPARSE) {
          a_desc0 = sdesc(sA0, 16, 512, kSwizzle64);
          b_desc0 = sdesc(sB0, 16, 1024, kSwizzle128);
        } else {
          a_desc0 = p.a_mn ? sdesc(sA0, C::kATileBytes / 2, 1024, kSwizzle128) : sdesc(sA0, 16, 1024, kSwizzle128);
          b_desc0 = p.b_mn ? sdesc(sB0, 8192, 1024, kSwizzle128) : sdesc(sB0, 16, 1024, kSwizzle128);
          a_step = p.a_mn ? (2048 >> 4) : (32 >> 4);
          b_step = p.b_mn ? (2048 >> 4) : (32 >> 4);
        }
        bool ok = true;
        if (p.fault_test && nhalf == 0)  // the drain barrier cannot complete before this issuer commits: runs out
          ok = mbar_wait(bar_drain, 0, abort_flag, p.wait_budget, p.status);
        for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
          const Unit t = decode_unit(p, u, CL, rank);
          // this issuer's column half of the buffer has been read by the epilogue
          if (!mbar_wait(bar_tempty + 8 * (2 * acc + (int)nhalf), acc_phase ^ 1, abort_flag, p.wait_budget, p.status))
            break;
          tc_fence_after();
          const uint32_t tacc = tmem + acc * BN + (BN / 2) * nhalf;
          int kstep = 0;  // MMA k-steps issued for this tile
          for (int ks = t.kbeg; ks < t.kend; ++ks) {
            if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.wait_budget, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = a_desc0 + (uint64_t)(stage * kStageUnits);
            const uint64_t bd = b_desc0 + (uint64_t)(stage * kStageUnits);
            if constexpr (SPARSE) {
              // the full barrier also covers this stage's metadata (slots 2 * mpair + j)
              const uint32_t tmeta = tmem + kMetaCol + kMetaColStride * 2 * mpair;
              mma_sparse(tacc, ad, bd, tmeta, idesc, kstep > 0 ? 1u : 0u);
              if (2 * ks + 1 < p.num_k_steps)  // no MMA past K
                mma_sparse(tacc, ad + (32 >> 4), bd + (64 >> 4), tmeta + kMetaColStride, idesc, 1u);
              ++kstep;
              mpair ^= 1u;
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_dense(tacc, ad + (uint64_t)(j * a_step), bd + (uint64_t)(j * b_step), idesc,
                          (kstep > 0 || j > 0) ? 1u : 0u);
              ++kstep;
            }
            tc_commit(bar_empty + 8 * stage);
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          tc_commit(bar_tfull + 8 * acc);
          if (++acc == C::kAcc) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
        // Drain: all issued tensor-core work completes before TMEM is freed.
        tc_commit(bar_drain);
        mbar_wait_quiet(bar_drain, 0u, p.wait_budget);
      }
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------- SPARSE metadata
    if constexpr (SPARSE && PAIR) {
      // Paired: k-steps in pairs.  Pair g2 goes to slot pair g2 % 2 once the MMAs of pair
      // g2 - 2 (the last to read it) have completed; this CTA's 128 rows are written with
      // tcgen05.st and announced on the even CTA's mfull barrier of the slot pair.
      const int q = warp & 3;  // TMEM lane quarter this warp may access
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + kMetaCol;
      const uint32_t lead_mfull = peer_addr(bar_mfull, 0);
      const int S = p.num_k_steps;
      uint32_t g2 = 0;
      bool ok = true;
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
        const Unit t = decode_unit(p, u, CL, rank);
        const uint32_t* src = p.meta + t.m0 + 32 * q + lane;
        auto word = [&](int kstep) -> uint32_t {
          return kstep < S ? __ldg(src + (int64_t)kstep * p.meta_slots) : 0x44444444u;  // 0x4: a valid code
        };
        const int pb = C::kSubs * t.kbeg, pe = min(C::kSubs * t.kend, (S + 1) / 2);  // pairs of k-steps of this unit
        uint32_t ring[4][2];  // the words of the next four pairs, loaded ahead of their use
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ring[i][0] = pb + i < pe ? word(2 * (pb + i)) : 0u;
          ring[i][1] = pb + i < pe ? word(2 * (pb + i) + 1) : 0u;
        }
        for (int p0 = pb; ok && p0 < pe; p0 += 4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int pi = p0 + i;
            if (pi >= pe) break;
            const uint32_t w0 = ring[i][0], w1 = ring[i][1];
            if (pi + 4 < pe) {
              ring[i][0] = word(2 * (pi + 4));
              ring[i][1] = word(2 * (pi + 4) + 1);
            }
            if (!mbar_wait<true>(bar_mempty + 8 * (g2 & 1u), ((g2 >> 1) & 1u) ^ 1u, abort_flag, p.wait_budget,
                                 p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t ta = tq + kMetaColStride * 2 * (g2 & 1u);
            tmem_st1(ta, w0);
            tmem_st1(ta + kMetaColStride, w1);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (leader)
                mbar_arrive(bar_mfull + 8 * (g2 & 1u));
              else
                mbar_arrive_remote_relaxed(lead_mfull + 8 * (g2 & 1u));
            }
            ++g2;
          }
        }
      }
    } else if constexpr (SPARSE) {
      const int q = warp & 3;  // TMEM lane quarter this warp may access
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + kMetaCol;
      const int S = p.num_k_steps;
      int g = 0;  // stages handed to the MMA so far, in the order the MMA consumes them
      bool ok = true;
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
        const Unit t = decode_unit(p, u, CL, rank);
        const uint32_t* src = p.meta + t.m0 + 32 * q + lane;
        auto word = [&](int kstep) -> uint32_t {
          return kstep < S ? __ldg(src + (int64_t)kstep * p.meta_slots) : 0x44444444u;  // 0x4: a valid code
        };
        // the words of the next four stages are loaded ahead of their use
        uint32_t ring[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ks = t.kbeg + i;
#pragma unroll
          for (int j = 0; j < 2; ++j) ring[i][j] = ks < t.kend ? word(2 * ks + j) : 0u;
        }
        for (int ks0 = t.kbeg; ok && ks0 < t.kend; ks0 += 4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int ks = ks0 + i;
            if (ks >= t.kend) break;
            const uint32_t w0 = ring[i][0], w1 = ring[i][1];
            if (ks + 4 < t.kend) {
              ring[i][0] = word(2 * (ks + 4));
              ring[i][1] = word(2 * (ks + 4) + 1);
            }
            // slot pair g & 1 was last read by the MMAs of stage g - 2: wait until that stage is released
            if (g >= 2) {
              const int h = g - 2;
              if (!mbar_wait(bar_empty + 8 * (h % C::kStages), (uint32_t)((h / C::kStages) & 1), abort_flag,
                             p.wait_budget, p.status)) {
                ok = false;
                break;
              }
            }
            tc_fence_after();
            const uint32_t ta = tq + kMetaColStride * 2 * (g & 1);
            tmem_st1(ta, w0);
            tmem_st1(ta + kMetaColStride, w1);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_full + 8 * (g % C::kStages));
            ++g;
          }
        }
      }
    }
  } else if (warp >= kEpiWarp0 + kEpiWarps) {
    // (every warp above the epilogue's has a role above)
  } else if constexpr (PAIR) {
    // ------------------------------------------------------- paired epilogue
    // Warp ew reads TMEM lane quarter q (its 32 rows of this CTA's 128) and, of
    // each 128-column half, the 64 columns 64 hw .. 64 hw + 63.  Half 0 is read
    // first and handed back to its issuer, which starts the next tile while
    // half 1 is read.  Common case (16-bit D, C not read, no K split): all four
    // 32-column chunks are packed in registers before D is written, so the
    // accumulator is free after the reads alone; each chunk is then staged as a
    // 32 x 32 block in shared memory (two per warp, alternating) and written by
    // one TMA store.  Column-major D is staged [n][m]: lane pairs swap halves
    // so that each lane writes 4 bytes (rows 2i, 2i + 1 of one column), an even
    // lane's column 2j and an odd lane's column 2j + 1 filling one 128-byte line
    // per instruction; row-major D is staged [m][n] in the 64-byte swizzle.
    const int ew = warp - kEpiWarp0;
    const int q = warp & 3;
    const int hw = ew >> 2;
    const uint32_t lead_tempty = peer_addr(bar_tempty, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    const bool scale = p.alpha != 1.0f;
    const bool fast = p.split_k == 1 && p.C == nullptr && p.cd_kind != kCdF32;
    const bool fast32 = p.split_k == 1 && p.C == nullptr && p.cd_kind == kCdF32;
    // chunk c (32 columns): accumulator column 128 (c / 2) + 64 hw + 32 (c % 2), which holds tile
    // column 128 hw + 32 c (see the issuers); chunks 0, 1 lie in the first issuer's half
    auto chunk_col = [&](int c) { return 128 * (c >> 1) + 64 * hw + 32 * (c & 1); };
    auto tile_col = [&](int c) { return 128 * hw + 32 * c; };
    uint8_t* const stage0 = smem + C::kEpiOffset + ew * (2 * kEpiBufBytes);
    int n_stored = 0;  // TMA stores this warp has issued (lane 0 commits each as a group)
    for (int u = cluster_id; u < p.num_units; u += num_clusters) {
      const Unit t = decode_unit(p, u, CL, rank);
      if (!mbar_wait<true>(bar_tfull + 8 * acc, acc_phase, abort_flag, p.wait_budget, p.status)) break;
      tc_fence_after();
      const int mq = t.m0 + 32 * q;
      const int row = mq + lane;
      const bool row_ok = row < p.M;
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + acc * BN;
      auto mask_word = [&](int c) -> uint32_t {
        const int nb = t.n0 + tile_col(c);
        return (!SPARSE && p.mask != nullptr && row_ok && nb < p.N) ? p.mask[(int64_t)row * p.mask_words + nb / 32]
                                                                      : 0xFFFFFFFFu;
      };
      // hands column half h of the current buffer back to its issuer (on the even CTA)
      auto release = [&](int h) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(bar_tempty + 8 * (2 * acc + h));
          else
            mbar_arrive_remote_relaxed(lead_tempty + 8 * (2 * acc + h));
        }
      };
      if (fast) {
        uint32_t pk[4][16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // two 32-column loads in flight; the half is handed back as
                                       // soon as they have landed, then packed
          uint32_t va[32], vb[32];
          tmem_ld32x2(tq + chunk_col(2 * h), tq + chunk_col(2 * h) + 32, va, vb);
          release(h);
          pack64_any<!SPARSE>(p.bf16, scale, va, vb, p.alpha, mask_word(2 * h), mask_word(2 * h + 1), pk[2 * h],
                              pk[2 * h + 1]);
        }
        if (mq < p.M) {
          const bool odd = lane & 1;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int nb = t.n0 + tile_col(c);
            if (nb >= p.N) continue;
            uint8_t* buf = stage0 + (n_stored & 1) * kEpiBufBytes;
            if (n_stored >= 2) {
              if (lane == 0) bulk_wait_read1();  // the store before last has read this block
              __syncwarp();
            }
            if (p.cd_col) {
              // block [32 n][32 m], 64-byte rows: element (n, m) at (n * 32 + m) * 2
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const uint32_t own = pk[c][j];
                const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, own, 1);
                // even lane: column 2j of rows lane, lane + 1; odd lane: column 2j + 1 of rows lane - 1, lane
                const uint32_t w = odd ? __byte_perm(other, own, 0x7632) : __byte_perm(own, other, 0x5410);
                *reinterpret_cast<uint32_t*>(buf + (2 * j + (odd ? 1 : 0)) * 64 + (lane & ~1) * 2) = w;
              }
            } else {
              // block [32 m][32 n], 64-byte rows in the 64B-swizzled order of the store map:
              // 16-byte chunk k of row r sits at chunk k ^ ((r >> 1) & 3)
              uint4* b4 = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                b4[k ^ ((lane >> 1) & 3)] =
                    make_uint4(pk[c][4 * k], pk[c][4 * k + 1], pk[c][4 * k + 2], pk[c][4 * k + 3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              if (p.cd_col)
                tma_store_2d(&tmD, smem_u32(buf), mq, nb);
              else
                tma_store_2d(&tmD, smem_u32(buf), nb, mq);
              bulk_commit();
            }
            ++n_stored;
          }
        }
      } else if (fast32) {
        // fp32 D: a half's two chunks are loaded, the half is handed back, then stored
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t va[32], vb[32];
          tmem_ld32x2(tq + chunk_col(2 * h), tq + chunk_col(2 * h) + 32, va, vb);
          release(h);
          const int nba = t.n0 + tile_col(2 * h), nbb = t.n0 + tile_col(2 * h + 1);
          if (row_ok && nba < p.N) store_chunk_f32(p, row, nba, va, mask_word(2 * h), scale);
          if (row_ok && nbb < p.N) store_chunk_f32(p, row, nbb, vb, mask_word(2 * h + 1), scale);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tq + chunk_col(c), v);
          const uint32_t mword = mask_word(c);
          const int nb = t.n0 + tile_col(c);
          if (p.split_k > 1)
            store_partial_chunk(p, t, tile_col(c), q, lane, v, mword);
          else if (row_ok && nb < p.N)
            store_chunk_generic(p, row, nb, v, mword);
          if (c & 1) release(c >> 1);
        }
        if (!SPARSE && p.fuse_split) {  // the split that arrives last at this warp's region sums them
          const int64_t idx = ((int64_t)(t.m0 / BM) * p.num_n_blk + t.n0 / BN) * kEpiWarps + ew;
          if (split_arrive_last(p, idx, lane)) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) store_split_sum_chunk(p, t, tile_col(c), q, lane, row, t.n0 + tile_col(c));
          }
        }
      }
      if (++acc == C::kAcc) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait_all();  // staging blocks stay valid until the stores are done
    __syncwarp();
  } else {
    // ------------------------------------------------------- single-CTA epilogue
    const int ew = warp - kEpiWarp0;
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const int hw = ew / 4;  // which 64 columns of each 128-column half
    uint8_t* buf = smem + C::kEpiOffset + ew * kEpiBufBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool stored = false;
    // Hands column half h of the current buffer back to the issuers once this warp has read it.
    auto release = [&](int h) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * (2 * acc + h));
    };
    for (int u = cluster_id; u < p.num_units; u += num_clusters) {
      const Unit t = decode_unit(p, u, CL, rank);
      if (!mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag, p.wait_budget, p.status)) break;
      tc_fence_after();
      const int mq = t.m0 + 32 * q;
      const int row = mq + lane;
      const bool row_ok = row < p.M;
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + acc * BN;
      // packed chunk c (32 columns) of this warp: tile column 128 * (c / 2) + 64 * hw + 32 * (c % 2)
      uint32_t pk[4][16];
      auto chunk_col = [&](int c) { return 128 * (c >> 1) + 64 * hw + 32 * (c & 1); };
      if (p.split_k == 1 && p.tma_store) {
        // half 0 first: once every warp has read its 64 columns of it, the first issuer can
        // start the next tile while the second half is read
        const bool scale = p.alpha != 1.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t ma = 0xFFFFFFFFu, mb = 0xFFFFFFFFu;
          if (!SPARSE && p.mask != nullptr && row_ok) {
            const int na = t.n0 + chunk_col(2 * h), nbb = na + 32;
            if (na < p.N) ma = p.mask[(int64_t)row * p.mask_words + na / 32];
            if (nbb < p.N) mb = p.mask[(int64_t)row * p.mask_words + nbb / 32];
          }
          drain64_any<!SPARSE>(p.bf16, scale, tq + chunk_col(2 * h), p.alpha, ma, mb, pk[2 * h], pk[2 * h + 1]);
          release(h);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tq + chunk_col(c), v);
          const int nb = t.n0 + chunk_col(c);
          uint32_t mword = 0xFFFFFFFFu;
          if (!SPARSE && p.mask != nullptr && row_ok && nb < p.N) mword = p.mask[(int64_t)row * p.mask_words + nb / 32];
          if (p.split_k > 1)
            store_partial_chunk(p, t, chunk_col(c), q, lane, v, mword);
          else if (row_ok && nb < p.N)
            store_chunk_generic(p, row, nb, v, mword);
          if (c & 1) release(c >> 1);  // chunks 0, 1 are this warp's columns of half 0
        }
      }
      if (++acc == C::kAcc) {
        acc = 0;
        acc_phase ^= 1;
      }
      if (p.split_k == 1 && p.tma_store && mq < p.M) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int nb = t.n0 + chunk_col(c);
          if (nb >= p.N) continue;
          if (stored) {
            if (lane == 0) bulk_wait_read0();  // the previous store has read the staging block
            __syncwarp();
          }
          if (p.cd_col) {
            // block [32 n][32 m], 64-byte rows: element (n, m) at (n * 32 + m) * 2
            uint16_t* b16 = reinterpret_cast<uint16_t*>(buf);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              b16[(2 * j) * 32 + lane] = (uint16_t)(pk[c][j] & 0xFFFFu);
              b16[(2 * j + 1) * 32 + lane] = (uint16_t)(pk[c][j] >> 16);
            }
          } else {
            // block [32 m][32 n], 64-byte rows in the 64B-swizzled order of the store map:
            // 16-byte chunk k of row r sits at chunk k ^ ((r >> 1) & 3)
            uint4* b4 = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              b4[k ^ ((lane >> 1) & 3)] = make_uint4(pk[c][4 * k], pk[c][4 * k + 1], pk[c][4 * k + 2], pk[c][4 * k + 3]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            if (p.cd_col)
              tma_store_2d(&tmD, smem_u32(buf), mq, nb);
            else
              tma_store_2d(&tmD, smem_u32(buf), nb, mq);
            bulk_commit();
          }
          stored = true;
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // staging blocks stay valid until the stores are done
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
  if constexpr (PAIR) cluster_sync();  // no CTA leaves while the other may still signal it
}

// D = beta * C (or 0) when K == 0: no product to accumulate.
__global__ void scale_c_kernel(const void* C, void* D, int64_t rows, int64_t cols, int64_t ldc, int64_t ldd,
                               float beta, int cd_kind) {
  const int64_t total = rows * cols;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / cols, c = i - r * cols;
    const float x = C != nullptr ? beta * load_cd(C, r * ldc + c, cd_kind) : 0.0f;
    store_cd(D, r * ldd + c, x, cd_kind);
  }
}

// Sum of the K splits' fp32 partials (alpha and mask already applied), plus
// beta * C, converted to D.
__global__ void finalize_split_kernel(const float4* __restrict__ part, int splits, int num_m_blk, int num_n_blk,
                                      int64_t M, int64_t N, const void* __restrict__ C, void* __restrict__ D,
                                      int64_t ldc, int64_t ldd, int cd_col, float beta, int cd_kind) {
  // one thread per four columns of one row, in the tiled order the product wrote
  pdl_trigger();
  pdl_wait();
  const int64_t per_split = (int64_t)num_m_blk * num_n_blk * (BM * BN / 4);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < per_split;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = i / (BM * BN / 4);
    const int rem = (int)(i - tile * (BM * BN / 4));
    const int c4 = rem / BM, r = rem - c4 * BM;
    const int64_t m = (tile / num_n_blk) * BM + r, n0 = (tile % num_n_blk) * BN + 4 * c4;
    if (m >= M || n0 >= N) continue;
    float4 x = part[i];
    for (int s = 1; s < splits; ++s) {
      const float4 y = part[(int64_t)s * per_split + i];
      x.x += y.x, x.y += y.y, x.z += y.z, x.w += y.w;
    }
    const float v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + j;
      if (n >= N) break;
      float o = v[j];
      if (C != nullptr) o = fmaf(beta, load_cd(C, cd_col ? n * ldc + m : m * ldc + n, cd_kind), o);
      store_cd(D, cd_col ? n * ldd + m : m * ldd + n, o, cd_kind);
    }
  }
}

// Row-major D from the tiled partials: one CTA per 128-row x 32-column slab of
// a tile.  The partials are read in their stored order (consecutive rows for
// each group of four columns), summed over the splits in split order, turned
// through shared memory and written along D's rows, eight values per store.
__global__ void __launch_bounds__(256) finalize_split_rows_kernel(const float4* __restrict__ part, int splits,
                                                                  int num_m_blk, int num_n_blk, int64_t M, int64_t N,
                                                                  const void* __restrict__ C, void* __restrict__ D,
                                                                  int64_t ldc, int64_t ldd, float beta, int cd_kind) {
  __shared__ float sm[BM][33];
  pdl_trigger();
  pdl_wait();
  const int64_t tile = blockIdx.x / (BN / 32);
  const int slab = blockIdx.x - (int)tile * (BN / 32);
  const int64_t per_split = (int64_t)num_m_blk * num_n_blk * (BM * BN / 4);
  const float4* src = part + tile * (BM * BN / 4) + (int64_t)slab * 8 * BM;  // column groups 8 slab .. 8 slab + 7
  // each element summed in split order; the loads of up to five splits (four float4 each per
  // thread) are issued before their adds, so five splits cost one round trip to memory
  constexpr int kChunk = 5;
  float4 x[4];
  for (int c0 = 0; c0 < splits; c0 += kChunk) {
    float4 y[kChunk][4];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      if (c0 + j >= splits) break;
      const float4* ps = src + (int64_t)(c0 + j) * per_split;
#pragma unroll
      for (int k = 0; k < 4; ++k) y[j][k] = ps[threadIdx.x + 256 * k];
    }
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      if (c0 + j >= splits) break;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (c0 + j == 0) {
          x[k] = y[j][k];
        } else {
          x[k].x += y[j][k].x, x[k].y += y[j][k].y, x[k].z += y[j][k].z, x[k].w += y[j][k].w;
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = threadIdx.x + 256 * k;  // (column group g, row r) = (e / 128, e % 128)
    const int g = e / BM, r = e - g * BM;
    sm[r][4 * g] = x[k].x, sm[r][4 * g + 1] = x[k].y, sm[r][4 * g + 2] = x[k].z, sm[r][4 * g + 3] = x[k].w;
  }
  __syncthreads();
  const int64_t m0 = (tile / num_n_blk) * BM, n0 = (tile % num_n_blk) * BN + 32 * slab;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int e = threadIdx.x + 256 * k;  // (row r, eight columns q) = (e / 4, e % 4)
    const int r = e >> 2, q = e & 3;
    const int64_t m = m0 + r, n = n0 + 8 * q;
    if (m >= M || n >= N) continue;
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j] = sm[r][8 * q + j];
      if (C != nullptr && n + j < N) o[j] = fmaf(beta, load_cd(C, m * ldc + n + j, cd_kind), o[j]);
    }
    if (cd_kind == kCdF32) {
      float* dst = reinterpret_cast<float*>(D) + m * ldd + n;
      if (n + 8 <= N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
        reinterpret_cast<float4*>(dst)[0] = make_float4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(o[4], o[5], o[6], o[7]);
      } else {
        for (int j = 0; j < 8 && n + j < N; ++j) dst[j] = o[j];
      }
      continue;
    }
    const int bf16 = cd_kind == kCdBF16;
    uint16_t* dst = reinterpret_cast<uint16_t*>(D) + m * ldd + n;
    if (n + 8 <= N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
      uint4 w;
      w.x = pack2(o[0], o[1], bf16), w.y = pack2(o[2], o[3], bf16), w.z = pack2(o[4], o[5], bf16),
      w.w = pack2(o[6], o[7], bf16);
      *reinterpret_cast<uint4*>(dst) = w;
    } else {
      for (int j = 0; j < 8 && n + j < N; ++j) store_cd(D, m * ldd + n + j, o[j], cd_kind);
    }
  }
}

// ----------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D tensor map over a row-major array: inner extent `inner` (contiguous),
// `outer` rows `pitch_bytes` apart, box inner_box x outer_box.
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
              uint64_t pitch_bytes, uint32_t inner_box, uint32_t outer_box, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {inner_box, outer_box};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps are encoded through the driver entry point, which needs a context bound to the
// calling thread.  A thread that has not yet made a runtime call needing one (a framework's
// worker thread, for example) has none, so the current device's primary context is bound first.
cudaError_t bind_context() {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  return cudaSetDevice(dev);
}

int num_sms() {
  static std::atomic<int> cached{0};
  int v = cached.load();
  if (v == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (v <= 0) v = 152;  // no device visible: GB300's count
    cached.store(v);
  }
  return v;
}

// The shared-memory opt-in is set once per device (and so never during a
// stream capture that replays the launches later).
template <bool SPARSE, bool PAIR>
cudaError_t set_smem_attr() {
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done_mask.load() & bit) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(spmm_tc_kernel<SPARSE, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<SPARSE, PAIR>::kSmemBytes);
  if (e == cudaSuccess) done_mask.fetch_or(bit);
  return e;
}

long long default_budget() { return 1ll << 32; }  // about two seconds at 2 GHz

int cd_kind_of(nm_dtype_t t) { return t == NM_F32 ? kCdF32 : (t == NM_BF16 ? kCdBF16 : kCdF16); }

cudaError_t launch_k0(const SpmmLaunch& a, cudaStream_t s) {
  const nm_spmm_desc_t& d = a.d;
  const int64_t rows = d.order_cd == NM_ROW ? d.M : d.N, cols = d.order_cd == NM_ROW ? d.N : d.M;
  scale_c_kernel<<<grid_for(rows * cols, 256), 256, 0, s>>>(a.C, a.D, rows, cols, d.ldc, d.ldd, a.beta_f,
                                                            cd_kind_of(d.cd_type));
  return cudaGetLastError();
}

Params base_params(const SpmmLaunch& a) {
  const nm_spmm_desc_t& d = a.d;
  Params p{};
  p.M = (int)d.M;
  p.N = (int)d.N;
  p.K = (int)d.K;
  p.num_m_blk = (int)((d.M + BM - 1) / BM);
  p.num_n_blk = (int)((d.N + BN - 1) / BN);
  p.k_stages = (int)((d.K + kKPerStage - 1) / kKPerStage);
  p.split_k = 1;
  p.stages_per_split = p.k_stages;
  p.bf16 = d.ab_type == NM_BF16;
  p.cd_kind = cd_kind_of(d.cd_type);
  p.alpha = a.alpha_f;
  p.beta = a.beta_f;
  p.C = a.C;
  p.D = a.D;
  p.ldc = d.ldc;
  p.ldd = d.ldd;
  p.cd_col = d.order_cd == NM_COL;
  p.tma_store = a.C == nullptr && p.cd_kind != kCdF32;
  p.status = a.d_status;
  p.wait_budget = default_budget();
  return p;
}

// Store map over D in 32 x 32 blocks (single-CTA kernel): column-major D (m
// contiguous) is staged [n][m] unswizzled; row-major D (n contiguous) is
// staged [m][n] with the 64-byte swizzle so that each lane's 64-byte row write
// is bank-conflict free.  Not used (and not encoded) for an fp32 D.
bool make_store_map(CUtensorMap* map, const nm_spmm_desc_t& d, void* D) {
  if (d.cd_type == NM_F32) {
    *map = CUtensorMap{};
    return true;
  }
  if (d.order_cd == NM_COL)
    return make_map(map, D, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)d.M, (uint64_t)d.N, (uint64_t)(d.ldd * 2), 32, 32,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  return make_map(map, D, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)d.N, (uint64_t)d.M, (uint64_t)(d.ldd * 2), 32, 32,
                  CU_TENSOR_MAP_SWIZZLE_64B);
}

template <bool SPARSE, bool PAIR>
cudaError_t launch_kernel(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mD, Params p,
                          cudaStream_t s) {
  using C = Cfg<SPARSE, PAIR>;
  constexpr int CL = PAIR ? 2 : 1;
  if (cudaError_t e = set_smem_attr<SPARSE, PAIR>()) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 1 : 0;
  // persistent grid: as many clusters as can be resident at once (queried once per device)
  static std::atomic<int> resident{0};
  int max_clusters = resident.load();
  if (max_clusters == 0) {
    cfg.gridDim = dim3((unsigned)(num_sms() / CL * CL));
    int n = 0;
    if (PAIR) {
      if (cudaOccupancyMaxActiveClusters(&n, spmm_tc_kernel<SPARSE, PAIR>, &cfg) != cudaSuccess) n = 0;
      cudaGetLastError();
    }
    max_clusters = n > 0 ? n : num_sms() / CL;
    resident.store(max_clusters);
  }
  const int clusters = p.num_units < max_clusters ? p.num_units : max_clusters;
  cfg.gridDim = dim3((unsigned)(clusters * CL));
  // programmatic dependent launch (the kernel waits for the previous grid after its set-up)
  attr[PAIR ? 1 : 0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[PAIR ? 1 : 0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = PAIR ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, spmm_tc_kernel<SPARSE, PAIR>, mA, mB, mD, p);
}

// Pairs of CTAs when the row blocks come in pairs, unless the plan asks for
// single CTAs (algo NM_ALGO_SINGLE).
bool use_pair(int num_m_blk, int algo) { return num_m_blk % 2 == 0 && algo != NM_ALGO_SINGLE; }

}  // namespace tc

cudaError_t spmm_tc_sparse_impl(const SpmmLaunch& a, cudaStream_t s, int fault_test, long long budget) {
  using namespace tc;
  const nm_spmm_desc_t& d = a.d;
  if (d.K == 0) return launch_k0(a, s);
  if (cudaError_t e = bind_context()) return e;
  Params p = base_params(a);
  p.fault_test = fault_test;
  if (budget > 0) p.wait_budget = budget;
  const bool pair = use_pair(p.num_m_blk, d.algo);
  const int cl = pair ? 2 : 1;
  p.num_units = (p.num_m_blk / cl) * p.num_n_blk;
  p.num_k_steps = (int)(d.K / 32);
  p.meta = static_cast<const uint32_t*>(a.A_meta);
  p.meta_slots = tc_slots(d.M);
  const CUtensorMapDataType u16 = CU_TENSOR_MAP_DATA_TYPE_UINT16;
  CUtensorMap mA, mB, mD;
  const int64_t kc = d.K / 2;  // compressed values per row, packed
  if (pair) {  // 128 dense K per stage: A boxes of 64 compressed values (128 B rows, 128B swizzle)
    p.k_stages = (int)((d.K + Cfg<true, true>::kKStage - 1) / Cfg<true, true>::kKStage);
    p.stages_per_split = p.k_stages;
  }
  constexpr int kPairAStride = Cfg<true, true>::kKStage / 2;  // compressed values per A row and stage (paired)
  const int a_box = pair ? kPairAStride : 32;
  if (!make_map(&mA, a.A, u16, (uint64_t)kc, (uint64_t)d.M, (uint64_t)(kc * 2), (uint32_t)a_box, BM,
                a_box == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&mB, a.B, u16, (uint64_t)d.K, (uint64_t)d.N, (uint64_t)(d.ldb * 2), 64, (uint32_t)(BN / cl),
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_store_map(&mD, d, a.D))
    return cudaErrorInvalidValue;
  if (pair) return launch_kernel<true, true>(mA, mB, mD, p, s);
  return launch_kernel<true, false>(mA, mB, mD, p, s);
}

cudaError_t launch_spmm_tc_sparse(const SpmmLaunch& a, cudaStream_t s) { return spmm_tc_sparse_impl(a, s, 0, 0); }

// K split of the masked dense product: the number of splits that best fills
// the SMs (fewest waves per unit of K), each split keeping at least 8 stages.
int spmm_tc_dense_masked_split(const nm_spmm_desc_t& d) {
  using namespace tc;
  if (d.K <= 0 || d.M <= 0 || d.N <= 0) return 1;
  const int64_t tiles = ((d.M + BM - 1) / BM) * ((d.N + BN - 1) / BN);
  const int64_t stages = (d.K + kKPerStage - 1) / kKPerStage;
  const int sms = num_sms();
  int best = 1;
  double best_cost = 1e30;
  for (int sk = 1; sk <= 16; ++sk) {
    if (sk > 1 && stages / sk < 8) break;
    const int64_t units = tiles * sk;
    const double waves = (double)((units + sms - 1) / sms);
    const double cost = waves / sk + 0.02 * (sk - 1);  // partial traffic penalty
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = sk;
    }
  }
  return best;
}
bool spmm_tc_dense_masked_split_ok(const nm_spmm_desc_t& d, int split_k) {
  using namespace tc;
  const int64_t stages = (d.K + kKPerStage - 1) / kKPerStage;
  return split_k == 1 || (split_k > 1 && split_k <= 16 && stages / split_k >= 8);
}
size_t spmm_tc_dense_masked_workspace(const nm_spmm_desc_t& d, int split_k) {
  // whole 128 x 256 tiles per split (the tiled partial order of the product's epilogue), then
  // one 64-bit arrival word per tile and epilogue warp (splits summed in the product)
  const size_t tiles = (size_t)((d.M + tc::BM - 1) / tc::BM) * (size_t)((d.N + tc::BN - 1) / tc::BN);
  return split_k > 1 ? (size_t)split_k * tiles * tc::BM * tc::BN * sizeof(float) + tiles * tc::kEpiWarps * 8 : 0;
}

int spmm_tc_dense_masked_launches(const nm_spmm_desc_t& d, int split_k) {
  using namespace tc;
  if (d.K == 0 || d.M == 0 || d.N == 0 || split_k <= 1) return 1;
  // the launch's own reduction to the splits that are not empty, and its pairing rule
  const int64_t k_stages = (d.K + kKPerStage - 1) / kKPerStage;
  const int64_t per = (k_stages + split_k - 1) / split_k;
  const int64_t splits = (k_stages + per - 1) / per;
  if (splits <= 1) return 1;
  const bool pair = use_pair((int)((d.M + BM - 1) / BM), d.algo);
  return pair && splits == 2 ? 1 : 2;
}

cudaError_t launch_spmm_tc_dense_masked(const SpmmLaunch& a, int split_k, cudaStream_t s) {
  using namespace tc;
  const nm_spmm_desc_t& d = a.d;
  if (d.K == 0) return launch_k0(a, s);
  if (cudaError_t e = bind_context()) return e;
  Params p = base_params(a);
  p.a_mn = d.order_a == NM_COL;
  p.b_mn = d.order_b == NM_ROW;
  p.mask = static_cast<const uint32_t*>(a.A_meta);
  p.mask_words = (d.N + 31) / 32;
  if (split_k > 1) {
    if (a.ws == nullptr || a.ws_bytes < spmm_tc_dense_masked_workspace(d, split_k)) return cudaErrorInvalidValue;
    p.stages_per_split = (p.k_stages + split_k - 1) / split_k;
    p.split_k = (p.k_stages + p.stages_per_split - 1) / p.stages_per_split;  // splits that are not empty
    p.partial = static_cast<float*>(a.ws);
    p.tma_store = 0;
  }
  const bool pair = use_pair(p.num_m_blk, d.algo);
  if (pair && p.split_k == 2) {
    // two splits are summed by the paired product itself: the warp that finishes a tile's region
    // last adds the other split's partial (in split order, as the finalize would) and writes D
    // tokens differ between launches of this process and, from a per-process start, most
    // likely from those of another process that used the same memory; never 0
    static std::atomic<uint32_t> launches{(uint32_t)std::chrono::steady_clock::now().time_since_epoch().count() *
                                          2654435761u};
    uint32_t token = ++launches;
    if (token == 0) token = ++launches;
    const size_t tiles = (size_t)p.num_m_blk * (size_t)p.num_n_blk;
    p.fuse_split = 1;
    p.split_token = token;
    p.split_cnt = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(a.ws) +
                                                       (size_t)split_k * tiles * BM * BN * sizeof(float));
  }
  const int cl = pair ? 2 : 1;
  p.num_units = (p.num_m_blk / cl) * p.num_n_blk * p.split_k;
  const uint32_t b_rows = (uint32_t)(BN / cl);  // paired: this CTA's 128-row block of B
  const CUtensorMapDataType u16 = CU_TENSOR_MAP_DATA_TYPE_UINT16;
  CUtensorMap mA, mB, mD;
  bool ok;
  if (p.a_mn)
    ok = make_map(&mA, a.A, u16, (uint64_t)d.M, (uint64_t)d.K, (uint64_t)(d.lda * 2), 64, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok = make_map(&mA, a.A, u16, (uint64_t)d.K, (uint64_t)d.M, (uint64_t)(d.lda * 2), 64, BM,
                  CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok) {
    if (p.b_mn)
      ok = make_map(&mB, a.B, u16, (uint64_t)d.N, (uint64_t)d.K, (uint64_t)(d.ldb * 2), 64, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    else
      ok = make_map(&mB, a.B, u16, (uint64_t)d.K, (uint64_t)d.N, (uint64_t)(d.ldb * 2), 64, b_rows,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (ok) ok = make_store_map(&mD, d, a.D);
  if (!ok) return cudaErrorInvalidValue;
  cudaError_t e = pair ? launch_kernel<false, true>(mA, mB, mD, p, s) : launch_kernel<false, false>(mA, mB, mD, p, s);
  if (e != cudaSuccess || p.split_k == 1 || p.fuse_split) return e;
  const int cdk = cd_kind_of(d.cd_type);
  if (d.order_cd == NM_ROW) {
    return launch_pdl(finalize_split_rows_kernel, dim3((unsigned)((int64_t)p.num_m_blk * p.num_n_blk * (BN / 32))),
                      dim3(256), 0, s, reinterpret_cast<const float4*>(p.partial), p.split_k, p.num_m_blk,
                      p.num_n_blk, d.M, d.N, a.C, a.D, d.ldc, d.ldd, a.beta_f, cdk);
  }
  // column-major D: the stored order already runs along D's columns
  const int64_t groups = (int64_t)p.num_m_blk * p.num_n_blk * (BM * BN / 4);
  finalize_split_kernel<<<grid_for(groups, 256), 256, 0, s>>>(reinterpret_cast<const float4*>(p.partial), p.split_k,
                                                              p.num_m_blk, p.num_n_blk, d.M, d.N, a.C, a.D, d.ldc,
                                                              d.ldd, d.order_cd == NM_COL, a.beta_f, cdk);
  return cudaGetLastError();
}

}  // namespace nmk

// Test entry point (declared in include/nm_testing.h): runs the sparse kernel
// with the MMA lane waiting on a barrier nothing arrives at and a short wait
// budget, so the bounded-wait path can be exercised without hanging or
// faulting the GPU.
extern "C" nm_status_t nm_test_spmm_wait_timeout(nm_spmm_plan_t plan_unused, const nm_spmm_desc_t* desc,
                                                 const void* A, const void* A_meta, const void* B, void* D,
                                                 int32_t* d_status, long long budget_cycles, nm_stream_t stream) {
  (void)plan_unused;
  if (desc == nullptr || desc->mode != NM_SPMM_SPARSE_A || desc->K <= 0) return NM_ERR_INVALID_ARG;
  nmk::SpmmLaunch a{};
  a.d = *desc;
  a.A = A;
  a.A_meta = A_meta;
  a.B = B;
  a.D = D;
  a.alpha_f = 1.0f;
  a.d_status = d_status;
  return nmk::spmm_tc_sparse_impl(a, (cudaStream_t)stream, 1, budget_cycles) == cudaSuccess ? NM_OK : NM_ERR_CUDA;
}
