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
// A persistent CTA per SM computes 128 x 256 output tiles.  Two CTAs of a
// cluster work on neighbouring 128-row blocks of the same 256-column block:
// each fetches half of the shared B tile and multicasts it to both, which
// halves the L2 traffic of B.  Warp roles per CTA:
//   warp 0       TMA producer: A and (its half of) B for stages of 64 dense K
//   warp 1       owns tensor memory; one lane issues the tcgen05.mma of
//                columns 0..127 of the tile (M128 N128 per instruction)
//   warps 2..5   SPARSE metadata: each warp loads one 32-bit code word per
//                lane (row slot) and k-step from global memory and writes it
//                with tcgen05.st into one of four 64-column-aligned TMEM
//                slots (the sparse MMA accepts its metadata only there); this
//                keeps metadata movement out of the tensor pipe.  The slots
//                form two pairs used by alternate stages: the metadata warps
//                refill a pair once the stage that last used it is released
//                (its `empty` barrier) and then arrive on the new stage's
//                `full` barrier, so the MMA issuer waits on one barrier per
//                stage and commits once per stage.
//   warps 6..13  epilogue: drain the FP32 accumulator (alpha, mask) into
//                packed registers, release it, then stage 32 x 32 blocks in
//                shared memory and write them with TMA bulk stores
//   warp 14      one lane issues the tcgen05.mma of columns 128..255; an MMA
//                holds its issuing thread for about its execution time, so two
//                issuers keep the tensor pipe busy through each other's
//                barrier waits, commits and loop overhead
// Every mbarrier wait is bounded; a wait that gives up sets an abort flag
// and NM_ERR_TIMEOUT in the caller's status word, the roles drain their
// outstanding asynchronous work and the CTA frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "nm_device.cuh"
#include "nm_internal.h"

namespace nmk {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int kKPerStage = 64;  // dense-equivalent K per stage
constexpr int kMetaWarp0 = 2, kMetaWarps = 4;
constexpr int kEpiWarp0 = kMetaWarp0 + kMetaWarps, kEpiWarps = 8;
constexpr int kMmaWarpB = kEpiWarp0 + kEpiWarps;  // second MMA issuer (columns 128..255)
constexpr int kThreads = 32 * (kMmaWarpB + 1);
constexpr int kTmemCols = 512;
constexpr int kMetaCol = 256, kMetaColStride = 64;  // four metadata slots: columns 256, 320, 384, 448
constexpr int kEpiBufBytes = 32 * 32 * 2;  // one 32 x 32 output block

// PAIR: the two CTAs of a cluster run one M256 x N256 product (tcgen05 with
// cta_group::2); each holds its 128 rows of A and one 128-row half of B.
template <bool SPARSE, bool PAIR = false>
struct Cfg {
  // dense-equivalent K per stage: 64, or 128 for the paired product (four k-steps per
  // barrier wait and commit of its single issuer)
  static constexpr int kKStage = PAIR ? 128 : kKPerStage;
  static constexpr int kSteps = kKStage / 32;  // SPARSE k-steps per stage
  // SPARSE A: 128 rows x kKStage/2 compressed values (64B swizzle for 64 B rows, 128B for
  // 128 B rows); dense A: 128 x 64 (128B swizzle).
  static constexpr int kATileBytes = SPARSE ? BM * kKStage : BM * 128;
  // B: rows x 64 elements per 128B-swizzled box; PAIR holds 128 rows and two boxes along K
  static constexpr int kBTileBytes = PAIR ? (BN / 2) * 256 : BN * 128;
  // PAIR: the stage also carries its k-steps' metadata, one 16-byte row per row of A
  static constexpr int kMetaBytes = PAIR ? kSteps * BM * 16 : 0;
  static constexpr int kStageBytes = kATileBytes + kBTileBytes + kMetaBytes;
  static constexpr int kStages = PAIR ? 3 : (SPARSE ? 5 : 4);
  static constexpr int kAcc = SPARSE ? 1 : 2;  // 256-column accumulator buffers
  static constexpr int kEpiOffset = kStages * kStageBytes;
  static constexpr int kBarOffset = kEpiOffset + kEpiWarps * kEpiBufBytes;
  static constexpr int kSmemBytes = 1024 + kBarOffset + 512;
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
  int bf16;
  float alpha, beta;
  const void* C;
  void* D;
  int64_t ldc, ldd;
  int cd_col;     // 1: D[n * ldd + m]; 0: D[m * ldd + n]
  int tma_store;  // 1: D written by TMA bulk stores (C not read)
  const uint32_t* mask;
  int64_t mask_words;
  float* partial;  // DENSE split-K: [split][M][N]
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
// CLUSTER: acquire at cluster scope, for barriers the peer CTA arrives on.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (CLUSTER)
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
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

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// The same box lands at the same offset in the shared memory of every CTA in
// `mask`, each completing bytes on its own barrier at offset `bar`.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
               "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory matrix descriptor (tcgen05): start, leading/stride byte
// offsets (16-byte units), fixed version bit 46, swizzle mode in bits 61..63.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}
constexpr uint32_t kSwizzle128 = 2, kSwizzle64 = 4;

// Instruction descriptor for kind::f16: D = F32, A/B = F16 or BF16, M = 128, N = 128
// (each of the two issuers computes one 128-column half of the tile).
__device__ __forceinline__ uint32_t idesc_f16(int bf16, int a_mn, int b_mn, bool sparse) {
  uint32_t d = (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) | ((uint32_t)a_mn << 15) |
               ((uint32_t)b_mn << 16) | ((uint32_t)((BN / 2) >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
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
// Arrives on the barrier at the same offset in every CTA of `mask` once the prior MMAs complete.
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// cta_group::2 forms: the MMA is issued by the even CTA of the pair and reads
// the operands of both CTAs at the same shared-memory offsets; the commit
// arrives on the barrier at the same offset in both CTAs.
__device__ __forceinline__ void mma_sparse_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t tmem_meta,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\ntcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n}" ::
          "r"(tmem_d),
      "l"(a), "l"(b), "r"(tmem_meta), "r"(idesc), "r"(acc));
}
// Copies 128 rows x 16 bytes of each CTA's shared memory into its own tensor
// memory (four columns at `taddr`), in order with the MMAs this thread issues.
__device__ __forceinline__ void tc_cp_pair(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.128x128b [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
// Address of the same shared-memory location in the even CTA of the pair.
__device__ __forceinline__ uint32_t pair_leader_addr(uint32_t a) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Relaxed remote arrive for "stage ready": the data it announces was written
// into this CTA's shared memory (TMA, and metadata rows already fenced to the
// async proxy), completion was observed here, and it is read only through
// this CTA's shared memory by the paired tensor-core instructions.  A release
// at cluster scope costs over a thousand cycles per arrive, which would limit
// the pair to one stage per relay round trip.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
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

__device__ __forceinline__ float load_cd(const void* base, int64_t off, int bf16) {
  const uint16_t b = reinterpret_cast<const uint16_t*>(base)[off];
  return bf16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
}
__device__ __forceinline__ uint16_t to_cd(float x, int bf16) {
  return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
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
// One warp's 32 lanes x 64 accumulator columns (two 32-column loads in flight)
// into packed pairs: alpha applied when SCALE, masked columns zeroed when
// MASKED (mask words ma, mb for the two 32-column halves).
template <bool BF16, bool SCALE, bool MASKED>
__device__ __forceinline__ void drain64(uint32_t taddr, float alpha, uint32_t ma, uint32_t mb, uint32_t (&pa)[16],
                                        uint32_t (&pb)[16]) {
  uint32_t va[32], vb[32];
  tmem_ld32x2(taddr, taddr + 32, va, vb);
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
__device__ __forceinline__ void drain64_any(int bf16, bool scale, uint32_t taddr, float alpha, uint32_t ma,
                                            uint32_t mb, uint32_t (&pa)[16], uint32_t (&pb)[16]) {
  if (bf16) {
    if (scale)
      drain64<true, true, MASKED>(taddr, alpha, ma, mb, pa, pb);
    else
      drain64<true, false, MASKED>(taddr, alpha, ma, mb, pa, pb);
  } else {
    if (scale)
      drain64<false, true, MASKED>(taddr, alpha, ma, mb, pa, pb);
    else
      drain64<false, false, MASKED>(taddr, alpha, ma, mb, pa, pb);
  }
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
  // one round-to-nearest conversion of the pair; `lo` lands in the low 16 bits
  if (bf16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Work unit u -> 128-row block, 256-column block and K split.  In a cluster
// of two, CTA rank r takes row block 2 * (pair index) + r.
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

// ----------------------------------------------------------------- kernel
// 15 warps are resident as 16 for register allocation (warps are allocated in
// groups of four), so 128 registers per thread is the most that still fits
// the 64K-register file.
template <bool SPARSE, int CL, bool PAIR>
__global__ void __maxnreg__(128)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const Params p) {
  static_assert(!PAIR || (SPARSE && CL == 2), "the paired product is the sparse one on clusters of two");
  using C = Cfg<SPARSE, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  // bars: full[S], empty[S], tfull[2], tempty[2 buffers][2 column halves], drain
  const uint32_t bar_full = smem_u32(bars), bar_empty = smem_u32(bars + C::kStages);
  const uint32_t bar_tfull = smem_u32(bars + 2 * C::kStages), bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 7);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
  const int cluster_id = blockIdx.x / CL, num_clusters = gridDim.x / CL;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      // SPARSE: the producer's expect_tx arrival and one arrival per metadata warp;
      // PAIR: the leader's barrier also takes the peer's relayed arrival
      mbar_init(bar_full + 8 * s, (SPARSE ? 1 + kMetaWarps : 1) + (PAIR && rank == 0 ? 1 : 0));
      // released by both issuers of every CTA that reads the stage (PAIR: the one paired issuer)
      mbar_init(bar_empty + 8 * s, PAIR ? 1 : 2 * CL);
    }
    for (int a = 0; a < 2; ++a) mbar_init(bar_tfull + 8 * a, PAIR ? 1 : 2);
    // one arrival per epilogue warp once it has read its columns of that half
    // (PAIR: a single barrier per buffer, after both halves, from both CTAs' epilogues)
    for (int a = 0; a < 4; ++a) mbar_init(bar_tempty + 8 * a, PAIR ? 2 * kEpiWarps : kEpiWarps);
    mbar_init(bar_drain, PAIR ? 1 : 2);
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
  if (CL > 1) cluster_sync();  // the peer's barriers exist before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // set-up done: from here on global memory may hold the previous grid's results
  pdl_trigger();
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_parity = 0;  // per-stage bits for the drain at the end
      bool ok = true;
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
        const Unit t = decode_unit(p, u, CL, rank);
        for (int ks = t.kbeg; ks < t.kend; ++ks) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.wait_budget, p.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t sA = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sB = sA + C::kATileBytes;
          mbar_expect_tx(fb, C::kATileBytes + C::kBTileBytes);  // PAIR's metadata rows come from the metadata warps
          if constexpr (SPARSE) {
            tma_load_2d(sA, &tmA, fb, ks * (C::kKStage / 2), t.m0);
          } else if (p.a_mn) {
            tma_load_2d(sA, &tmA, fb, t.m0, ks * 64);
            tma_load_2d(sA + C::kATileBytes / 2, &tmA, fb, t.m0 + 64, ks * 64);
          } else {
            tma_load_2d(sA, &tmA, fb, ks * 64, t.m0);
          }
          // B: this CTA fetches 256 / CL rows (columns of D) and, in a cluster, multicasts them;
          // PAIR: each CTA keeps its own half, which the paired MMA reads in place
          const int nb = t.n0 + (BN / CL) * (int)rank;
          const uint32_t sBh = sB + (C::kBTileBytes / CL) * rank;
          if constexpr (PAIR) {
            tma_load_2d(sB, &tmB, fb, ks * 128, nb);
            tma_load_2d(sB + C::kBTileBytes / 2, &tmB, fb, ks * 128 + 64, nb);
          } else if (!SPARSE && p.b_mn) {
#pragma unroll
            for (int h = 0; h < 4 / CL; ++h) {
              if (CL > 1)
                tma_load_2d_mc(sBh + 8192 * h, &tmB, fb, nb + 64 * h, ks * 64, (uint16_t)((1u << CL) - 1));
              else
                tma_load_2d(sBh + 8192 * h, &tmB, fb, nb + 64 * h, ks * 64);
            }
          } else {
            if (CL > 1)
              tma_load_2d_mc(sBh, &tmB, fb, ks * 64, nb, (uint16_t)((1u << CL) - 1));
            else
              tma_load_2d(sBh, &tmB, fb, ks * 64, nb);
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: every copy into this CTA must have landed before the CTA may exit.
      for (int s = 0; s < C::kStages; ++s)
        if ((issued >> s) & 1u) {
          const uint32_t par = (last_parity >> s) & 1u;
          const long long t0 = clock64();
          while (!mbar_try(bar_full + 8 * s, par) && clock64() - t0 < p.wait_budget) {
          }
        }
    }
  } else if (warp == 1 || warp == kMmaWarpB) {
    if constexpr (PAIR) {
      // ----------------------------------------------------- paired issuer / relay
      // The even CTA issues M256 x N256 MMAs over both CTAs' operands and
      // commits to both CTAs' barriers; the odd CTA's warp 1 relays "stage
      // ready" (its own TMA bytes and metadata) to the even CTA's full barrier.
      if (warp == 1 && lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        if (rank == 0) {
          const uint32_t idesc = (1u << 4) | ((uint32_t)p.bf16 << 7) | ((uint32_t)p.bf16 << 10) | (1u << 2) |
                                 ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);
          constexpr uint32_t kStageUnits = C::kStageBytes >> 4;
          const uint32_t sA0 = smem_u32(smem);
          // A: 128 rows x 128 B (128B swizzle), 32 B per k-step; B: two boxes of 128 rows x 128 B,
          // 64 B per k-step within a box; metadata: 16-byte rows, one block of 128 rows per k-step
          const uint64_t a_desc0 = sdesc(sA0, 16, 1024, kSwizzle128);
          const uint64_t b_desc0 = sdesc(sA0 + C::kATileBytes, 16, 1024, kSwizzle128);
          const uint64_t m_desc0 = sdesc(sA0 + C::kATileBytes + C::kBTileBytes, 16, 128, 0);
          uint32_t mslot = 0, acc_phase = 0;
          if (p.fault_test) ok = mbar_wait(bar_drain, 0, abort_flag, p.wait_budget, p.status);  // runs out
          for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
            const Unit t = decode_unit(p, u, CL, rank);
            if (!mbar_wait<true>(bar_tempty, acc_phase ^ 1, abort_flag, p.wait_budget, p.status)) break;
            tc_fence_after();
            int kstep = 0;
            for (int ks = t.kbeg; ks < t.kend; ++ks) {
              if (!mbar_wait<true>(bar_full + 8 * stage, phase, abort_flag, p.wait_budget, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t ad = a_desc0 + (uint64_t)(stage * kStageUnits);
              const uint64_t bd = b_desc0 + (uint64_t)(stage * kStageUnits);
              const uint64_t md = m_desc0 + (uint64_t)(stage * kStageUnits);
              // metadata into the next of four 64-column-aligned slots, then the MMA that reads it
              const int left = p.num_k_steps - C::kSteps * ks;  // no MMA past K
              const int steps = left < C::kSteps ? left : C::kSteps;
              for (int j = 0; j < steps; ++j) {
                const uint32_t tmeta = tmem + kMetaCol + kMetaColStride * mslot;
                tc_cp_pair(tmeta, md + (uint64_t)((BM * 16 * j) >> 4));
                const uint64_t bj = bd + (uint64_t)(((C::kBTileBytes / 2) * (j / 2) + 64 * (j % 2)) >> 4);
                mma_sparse_pair(tmem, ad + (uint64_t)((32 * j) >> 4), bj, tmeta, idesc, (kstep > 0 || j > 0) ? 1u : 0u);
                mslot = (mslot + 1) & 3u;
              }
              ++kstep;
              tc_commit_pair(bar_empty + 8 * stage);
              if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1;
              }
            }
            if (!ok) break;
            tc_commit_pair(bar_tfull);
            acc_phase ^= 1;
          }
          tc_commit_pair(bar_drain);
        } else {
          for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
            const Unit t = decode_unit(p, u, CL, rank);
            for (int ks = t.kbeg; ks < t.kend; ++ks) {
              if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.wait_budget, p.status)) {
                ok = false;
                break;
              }
              mbar_arrive_remote_relaxed(pair_leader_addr(bar_full + 8 * stage));
              if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
        }
        // all paired MMAs have completed before either CTA frees its tensor memory
        const long long t0 = clock64();
        while (!mbar_try(bar_drain, 0u) && clock64() - t0 < p.wait_budget) {
        }
      }
    } else {
    // ------------------------------------------------------- MMA issuers
    // Two single-thread issuers share every stage: warp 1 computes columns
    // 0..127 and warp kMmaWarpB columns 128..255 of the tile.  An MMA holds
    // its issuing thread for about its execution time, so while one issuer
    // waits, commits and loops, the other one keeps the tensor pipe busy.
    if (lane == 0) {
      const uint32_t nhalf = warp == 1 ? 0u : 1u;
      const uint32_t idesc = idesc_f16(p.bf16, SPARSE ? 0 : p.a_mn, SPARSE ? 0 : p.b_mn, SPARSE);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      uint32_t mpair = 0;  // SPARSE: metadata slot pair of the current stage (alternates every stage)
      // Shared-memory descriptors of stage 0.  Advancing a descriptor's start address
      // (bits 0-13, in 16-byte units) by an offset is adding offset >> 4, since every
      // shared address fits the 14-bit field.
      //   SPARSE A: 128 rows x 64 B (64B swizzle, 8-row groups 512 B apart), 32 B per k-step
      //   SPARSE B: 256 rows x 128 B (128B swizzle), 64 B per k-step
      //   DENSE A/B K-major: 128B swizzle, 32 B per K16 step; MN-major: 2048 B per K16 step
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
          // descriptors of this stage: the stage-0 descriptors with the start address advanced
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
          if (CL > 1)
            tc_commit_mc(bar_empty + 8 * stage, (uint16_t)((1u << CL) - 1));
          else
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
      const long long t0 = clock64();
      while (!mbar_try(bar_drain, 0u) && clock64() - t0 < p.wait_budget) {
      }
    }
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------- SPARSE metadata
    if constexpr (SPARSE) {
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
        constexpr int KS = C::kSteps;
        uint32_t ring[4][KS];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ks = t.kbeg + i;
#pragma unroll
          for (int j = 0; j < KS; ++j) ring[i][j] = ks < t.kend ? word(KS * ks + j) : 0u;
        }
        for (int ks0 = t.kbeg; ok && ks0 < t.kend; ks0 += 4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int ks = ks0 + i;
            if (ks >= t.kend) break;
            uint32_t w[KS];
#pragma unroll
            for (int j = 0; j < KS; ++j) w[j] = ring[i][j];
            if (ks + 4 < t.kend) {
#pragma unroll
              for (int j = 0; j < KS; ++j) ring[i][j] = word(KS * (ks + 4) + j);
            }
            if constexpr (PAIR) {
              // the words go to the stage's metadata rows (copied to tensor memory by the
              // paired issuer); the stage buffer was last read by the MMAs of stage g - kStages
              if (g >= C::kStages) {
                const int h = g - C::kStages;
                if (!mbar_wait(bar_empty + 8 * (h % C::kStages), (uint32_t)((h / C::kStages) & 1), abort_flag,
                               p.wait_budget, p.status)) {
                  ok = false;
                  break;
                }
              }
              uint8_t* mrow = smem + (g % C::kStages) * C::kStageBytes + C::kATileBytes + C::kBTileBytes +
                              (32 * q + lane) * 16;
#pragma unroll
              for (int j = 0; j < KS; ++j) *reinterpret_cast<uint32_t*>(mrow + BM * 16 * j) = w[j];
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_full + 8 * (g % C::kStages));
              ++g;
              continue;
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
            tmem_st1(ta, w[0]);
            tmem_st1(ta + kMetaColStride, w[1]);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_full + 8 * (g % C::kStages));
            ++g;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------- epilogue
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
      if (lane == 0) {
        if constexpr (PAIR) {
          if (h == 1) {  // the paired issuer needs both halves: one arrival, after the second
            if (rank == 1)  // the accumulator reads completed (wait::ld) before this arrive
              mbar_arrive_remote_relaxed(pair_leader_addr(bar_tempty + 8 * 2 * acc));
            else
              mbar_arrive(bar_tempty + 8 * 2 * acc);
          }
        } else {
          mbar_arrive(bar_tempty + 8 * (2 * acc + h));
        }
      }
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
          if (p.split_k > 1) {
            // fp32 partial of this K split in the tiled order [split][m block][n block][col / 4][128 rows][4]:
            // for each group of four columns the 32 lanes write 512 contiguous bytes
            float4* tile = reinterpret_cast<float4*>(p.partial) +
                           ((int64_t)(t.split * p.num_m_blk + t.m0 / BM) * p.num_n_blk + t.n0 / BN) * (BM * BN / 4);
            const int c4_0 = chunk_col(c) / 4;
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              float4 w;
              w.x = ((mword >> (4 * j4)) & 1u) ? __uint_as_float(v[4 * j4]) * p.alpha : 0.0f;
              w.y = ((mword >> (4 * j4 + 1)) & 1u) ? __uint_as_float(v[4 * j4 + 1]) * p.alpha : 0.0f;
              w.z = ((mword >> (4 * j4 + 2)) & 1u) ? __uint_as_float(v[4 * j4 + 2]) * p.alpha : 0.0f;
              w.w = ((mword >> (4 * j4 + 3)) & 1u) ? __uint_as_float(v[4 * j4 + 3]) * p.alpha : 0.0f;
              tile[(c4_0 + j4) * BM + 32 * q + lane] = w;
            }
          } else if (row_ok && nb < p.N) {
            const int cnt = min(32, p.N - nb);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (j >= cnt) break;
              float x = ((mword >> j) & 1u) ? __uint_as_float(v[j]) * p.alpha : 0.0f;
              const int64_t doff = p.cd_col ? (int64_t)(nb + j) * p.ldd + row : (int64_t)row * p.ldd + nb + j;
              const int64_t coff = p.cd_col ? (int64_t)(nb + j) * p.ldc + row : (int64_t)row * p.ldc + nb + j;
              if (p.C != nullptr) x = fmaf(p.beta, load_cd(p.C, coff, p.bf16), x);
              reinterpret_cast<uint16_t*>(p.D)[doff] = to_cd(x, p.bf16);
            }
          }
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
  if (CL > 1) cluster_sync();  // no CTA leaves while its peer may still signal it
}

// D = beta * C (or 0) when K == 0: no product to accumulate.
__global__ void scale_c_kernel(const uint16_t* C, uint16_t* D, int64_t rows, int64_t cols, int64_t ldc, int64_t ldd,
                               float beta, int bf16) {
  const int64_t total = rows * cols;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / cols, c = i - r * cols;
    const float x = C != nullptr ? beta * load_cd(C, r * ldc + c, bf16) : 0.0f;
    D[r * ldd + c] = to_cd(x, bf16);
  }
}

// Sum of the K splits' fp32 partials (alpha and mask already applied), plus
// beta * C, converted to D.
__global__ void finalize_split_kernel(const float4* __restrict__ part, int splits, int num_m_blk, int num_n_blk,
                                      int64_t M, int64_t N, const uint16_t* __restrict__ C, uint16_t* __restrict__ D,
                                      int64_t ldc, int64_t ldd, int cd_col, float beta, int bf16) {
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
      if (C != nullptr) o = fmaf(beta, load_cd(C, cd_col ? n * ldc + m : m * ldc + n, bf16), o);
      D[cd_col ? n * ldd + m : m * ldd + n] = to_cd(o, bf16);
    }
  }
}

// Row-major D from the tiled partials: one CTA per 128-row x 32-column slab of
// a tile.  The partials are read in their stored order (consecutive rows for
// each group of four columns), summed over the splits in split order, turned
// through shared memory and written along D's rows, eight values per store.
__global__ void __launch_bounds__(256) finalize_split_rows_kernel(const float4* __restrict__ part, int splits,
                                                                  int num_m_blk, int num_n_blk, int64_t M, int64_t N,
                                                                  const uint16_t* __restrict__ C,
                                                                  uint16_t* __restrict__ D, int64_t ldc, int64_t ldd,
                                                                  float beta, int bf16) {
  __shared__ float sm[BM][33];
  pdl_trigger();
  pdl_wait();
  const int64_t tile = blockIdx.x / (BN / 32);
  const int slab = blockIdx.x - (int)tile * (BN / 32);
  const int64_t per_split = (int64_t)num_m_blk * num_n_blk * (BM * BN / 4);
  const float4* src = part + tile * (BM * BN / 4) + (int64_t)slab * 8 * BM;  // column groups 8 slab .. 8 slab + 7
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = threadIdx.x + 256 * k;  // (column group g, row r) = (e / 128, e % 128)
    float4 x = src[e];
    for (int sp = 1; sp < splits; ++sp) {
      const float4 y = src[(int64_t)sp * per_split + e];
      x.x += y.x, x.y += y.y, x.z += y.z, x.w += y.w;
    }
    const int g = e / BM, r = e - g * BM;
    sm[r][4 * g] = x.x, sm[r][4 * g + 1] = x.y, sm[r][4 * g + 2] = x.z, sm[r][4 * g + 3] = x.w;
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
      if (C != nullptr && n + j < N) o[j] = fmaf(beta, load_cd(C, m * ldc + n + j, bf16), o[j]);
    }
    uint16_t* dst = D + m * ldd + n;
    if (n + 8 <= N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
      uint4 w;
      w.x = pack2(o[0], o[1], bf16), w.y = pack2(o[2], o[3], bf16), w.z = pack2(o[4], o[5], bf16),
      w.w = pack2(o[6], o[7], bf16);
      *reinterpret_cast<uint4*>(dst) = w;
    } else {
      for (int j = 0; j < 8 && n + j < N; ++j) dst[j] = to_cd(o[j], bf16);
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

int num_sms() {
  static std::atomic<int> cached{0};
  int v = cached.load();
  if (v == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (v <= 0) v = 148;
    cached.store(v);
  }
  return v;
}

// The shared-memory opt-in is set once per device (and so never during a
// stream capture that replays the launches later).
template <bool SPARSE, int CL, bool PAIR>
cudaError_t set_smem_attr() {
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done_mask.load() & bit) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(spmm_tc_kernel<SPARSE, CL, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<SPARSE, PAIR>::kSmemBytes);
  if (e == cudaSuccess) done_mask.fetch_or(bit);
  return e;
}

long long default_budget() { return 1ll << 32; }  // about two seconds at 2 GHz

cudaError_t launch_k0(const SpmmLaunch& a, cudaStream_t s) {
  const nm_spmm_desc_t& d = a.d;
  const int64_t rows = d.order_cd == NM_ROW ? d.M : d.N, cols = d.order_cd == NM_ROW ? d.N : d.M;
  scale_c_kernel<<<grid_for(rows * cols, 256), 256, 0, s>>>(static_cast<const uint16_t*>(a.C),
                                                            static_cast<uint16_t*>(a.D), rows, cols, d.ldc, d.ldd,
                                                            a.beta_f, d.ab_type == NM_BF16);
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
  p.alpha = a.alpha_f;
  p.beta = a.beta_f;
  p.C = a.C;
  p.D = a.D;
  p.ldc = d.ldc;
  p.ldd = d.ldd;
  p.cd_col = d.order_cd == NM_COL;
  p.tma_store = a.C == nullptr;
  p.status = a.d_status;
  p.wait_budget = default_budget();
  return p;
}

// Store map over D in 32 x 32 blocks: column-major D (m contiguous) is
// staged [n][m] unswizzled; row-major D (n contiguous) is staged [m][n] with
// the 64-byte swizzle so that each lane's 64-byte row write is bank-conflict free.
bool make_store_map(CUtensorMap* map, const nm_spmm_desc_t& d, void* D) {
  if (d.order_cd == NM_COL)
    return make_map(map, D, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)d.M, (uint64_t)d.N, (uint64_t)(d.ldd * 2), 32, 32,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  return make_map(map, D, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)d.N, (uint64_t)d.M, (uint64_t)(d.ldd * 2), 32, 32,
                  CU_TENSOR_MAP_SWIZZLE_64B);
}

template <bool SPARSE, int CL, bool PAIR>
cudaError_t launch_kernel(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mD, Params p,
                          cudaStream_t s) {
  if (cudaError_t e = set_smem_attr<SPARSE, CL, PAIR>()) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<SPARSE, PAIR>::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 1 : 0;
  // persistent grid: as many clusters as can be resident at once (queried once per device)
  static std::atomic<int> resident{0};
  int max_clusters = resident.load();
  if (max_clusters == 0) {
    cfg.gridDim = dim3((unsigned)(num_sms() / CL * CL));
    int n = 0;
    if (CL > 1) {
      if (cudaOccupancyMaxActiveClusters(&n, spmm_tc_kernel<SPARSE, CL, PAIR>, &cfg) != cudaSuccess) n = 0;
      cudaGetLastError();
    }
    max_clusters = n > 0 ? n : num_sms() / CL;
    resident.store(max_clusters);
  }
  const int clusters = p.num_units < max_clusters ? p.num_units : max_clusters;
  cfg.gridDim = dim3((unsigned)(clusters * CL));
  // programmatic dependent launch (the kernel waits for the previous grid after its set-up)
  cudaLaunchAttribute attr2[2];
  attr2[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr2[0].val.programmaticStreamSerializationAllowed = 1;
  attr2[1] = attr[0];
  cfg.attrs = attr2;
  cfg.numAttrs = CL > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, spmm_tc_kernel<SPARSE, CL, PAIR>, mA, mB, mD, p);
}

// Pairs of CTAs share the B tile when the row blocks come in pairs (for the
// sparse product with algo 1 as one paired M256 product per cluster).
int cluster_for(int num_m_blk) { return (num_m_blk % 2 == 0) ? 2 : 1; }

}  // namespace tc

cudaError_t spmm_tc_sparse_impl(const SpmmLaunch& a, cudaStream_t s, int fault_test, long long budget) {
  using namespace tc;
  const nm_spmm_desc_t& d = a.d;
  if (d.K == 0) return launch_k0(a, s);
  Params p = base_params(a);
  p.fault_test = fault_test;
  if (budget > 0) p.wait_budget = budget;
  const int cl = cluster_for(p.num_m_blk);
  p.num_units = (p.num_m_blk / cl) * p.num_n_blk;
  p.num_k_steps = (int)(d.K / 32);
  // Paired CTAs on request: they halve the shared-memory traffic per SM, but their single
  // issuer's per-stage work is then exposed; on GB300 the single-CTA kernel with two
  // issuers was measured faster for the benchmark shapes, so it is the default.
  p.meta = static_cast<const uint32_t*>(a.A_meta);
  p.meta_slots = tc_slots(d.M);
  const CUtensorMapDataType u16 = CU_TENSOR_MAP_DATA_TYPE_UINT16;
  CUtensorMap mA, mB, mD;
  const int64_t kc = d.K / 2;  // compressed values per row, packed
  // paired: 128 dense K per stage, so 64 compressed values (128 B, 128B swizzle) per row of A
  const bool pair = cl == 2 && d.algo == 1;
  if (pair) {
    p.k_stages = (int)((d.K + Cfg<true, true>::kKStage - 1) / Cfg<true, true>::kKStage);
    p.stages_per_split = p.k_stages;
  }
  if (!make_map(&mA, a.A, u16, (uint64_t)kc, (uint64_t)d.M, (uint64_t)(kc * 2), pair ? 64 : 32, BM,
                pair ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&mB, a.B, u16, (uint64_t)d.K, (uint64_t)d.N, (uint64_t)(d.ldb * 2), 64, (uint32_t)(BN / cl),
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_store_map(&mD, d, a.D))
    return cudaErrorInvalidValue;
  if (pair) return launch_kernel<true, 2, true>(mA, mB, mD, p, s);
  return cl == 2 ? launch_kernel<true, 2, false>(mA, mB, mD, p, s) : launch_kernel<true, 1, false>(mA, mB, mD, p, s);
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
size_t spmm_tc_dense_masked_workspace(const nm_spmm_desc_t& d, int split_k) {
  // whole 128 x 256 tiles per split (the tiled partial order of the product's epilogue)
  const size_t tiles = (size_t)((d.M + tc::BM - 1) / tc::BM) * (size_t)((d.N + tc::BN - 1) / tc::BN);
  return split_k > 1 ? (size_t)split_k * tiles * tc::BM * tc::BN * sizeof(float) : 0;
}

cudaError_t launch_spmm_tc_dense_masked(const SpmmLaunch& a, int split_k, cudaStream_t s) {
  using namespace tc;
  const nm_spmm_desc_t& d = a.d;
  if (d.K == 0) return launch_k0(a, s);
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
  const int cl = cluster_for(p.num_m_blk);
  p.num_units = (p.num_m_blk / cl) * p.num_n_blk * p.split_k;
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
      ok = make_map(&mB, a.B, u16, (uint64_t)d.K, (uint64_t)d.N, (uint64_t)(d.ldb * 2), 64, (uint32_t)(BN / cl),
                    CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (ok) ok = make_store_map(&mD, d, a.D);
  if (!ok) return cudaErrorInvalidValue;
  cudaError_t e =
      cl == 2 ? launch_kernel<false, 2, false>(mA, mB, mD, p, s) : launch_kernel<false, 1, false>(mA, mB, mD, p, s);
  if (e != cudaSuccess || p.split_k == 1) return e;
  if (d.order_cd == NM_ROW) {
    return launch_pdl(finalize_split_rows_kernel, dim3((unsigned)((int64_t)p.num_m_blk * p.num_n_blk * (BN / 32))),
                      dim3(256), 0, s, reinterpret_cast<const float4*>(p.partial), p.split_k, p.num_m_blk,
                      p.num_n_blk, d.M, d.N, static_cast<const uint16_t*>(a.C), static_cast<uint16_t*>(a.D), d.ldc,
                      d.ldd, a.beta_f, (int)(d.ab_type == NM_BF16));
  }
  // column-major D: the stored order already runs along D's columns
  const int64_t groups = (int64_t)p.num_m_blk * p.num_n_blk * (BM * BN / 4);
  finalize_split_kernel<<<grid_for(groups, 256), 256, 0, s>>>(
      reinterpret_cast<const float4*>(p.partial), p.split_k, p.num_m_blk, p.num_n_blk, d.M, d.N,
      static_cast<const uint16_t*>(a.C), static_cast<uint16_t*>(a.D), d.ldc, d.ldd, d.order_cd == NM_COL, a.beta_f,
      d.ab_type == NM_BF16);
  return cudaGetLastError();
}

}  // namespace nmk

// Test hook (not in include/nm.h): runs the sparse kernel with the MMA lane
// waiting on a barrier nothing arrives at and a short wait budget, so the
// bounded-wait path can be exercised without hanging or faulting the GPU.
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
