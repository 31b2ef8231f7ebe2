// Tensor-core products on Blackwell (sm_103a): D = alpha * A * B + beta * C.
//
//  * SPARSE:        A is 2:4 sparse (cuSPARSELt blog, Figure 2 text: half-size
//                   values plus metadata; the sparse tensor core skips the
//                   zeros), F16/BF16 with F32 accumulation.  Issued as
//                   tcgen05.mma.sp with the metadata in tensor memory.
//  * DENSE_MASKED:  A and B dense, D = alpha * (mask .* (A B)) + beta * C, the
//                   weight gradient of a layer whose weight keeps a fixed
//                   sparsity pattern.  Issued as dense tcgen05.mma.
//
// One persistent CTA per SM walks output tiles of 128 x 128.  Warp roles:
//   warp 0      TMA producer: fills a ring of shared-memory stages of 64
//               dense K (A, B and, for SPARSE, the metadata of two k-steps)
//   warp 1      owns tensor memory; one lane issues tcgen05.cp (metadata
//               into TMEM) and tcgen05.mma, committing to mbarriers
//   warps 2..5  epilogue: tcgen05.ld the FP32 accumulator, alpha, mask,
//               convert, stage 32 x 32 blocks in shared memory and write them
//               with TMA bulk stores; the accumulator is double buffered so
//               the epilogue of one tile overlaps the main loop of the next.
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
constexpr int BN = 128;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 2 * BN;  // two accumulator buffers
// The metadata of one MMA k-step (32 dense K) occupies one TMEM column; the
// sparse MMA accepts it only at a 64-aligned column, so k-steps rotate
// through the four columns 256, 320, 384 and 448, each filled by its own
// tcgen05.cp of 128 lanes x 128 bits (the other three columns of a copy are
// filler).
constexpr int kMetaCol = kAccCols;
constexpr int kMetaColStride = 64;
constexpr int kMetaSlots = 4;
constexpr int kMetaStepBytes = BM * 16;  // one k-step: 128 slot rows x 16 B
constexpr int kKPerStage = 64;           // dense-equivalent K per stage
constexpr int kBTileBytes = BN * 128;    // BN rows x 64 elements (128B swizzle)
constexpr int kEpiBufBytes = 32 * 32 * 2;  // one 32 x 32 output block

template <bool SPARSE>
struct Cfg {
  // SPARSE: A = 128 rows x 32 compressed values (64B swizzle); DENSE: 128 x 64 (128B swizzle).
  static constexpr int kATileBytes = SPARSE ? BM * 64 : BM * 128;
  static constexpr int kMetaBytes = SPARSE ? 2 * kMetaStepBytes : 0;
  static constexpr int kStageBytes = kATileBytes + kBTileBytes + kMetaBytes;
  static constexpr int kStages = SPARSE ? 7 : 6;
  static constexpr int kEpiOffset = kStages * kStageBytes;
  static constexpr int kBarOffset = kEpiOffset + kEpiWarps * 2 * kEpiBufBytes;
  static constexpr int kSmemBytes = 1024 + kBarOffset + 256;
};

struct Params {
  int M, N, K;
  int num_m_blk, num_n_blk, num_k_stages;
  int num_k_steps;  // SPARSE: K / 32 MMA k-steps
  const uint8_t* meta;  // SPARSE: tensor-core metadata, [k-step][meta_slots][16 B]
  int64_t meta_slots;
  int a_mn, b_mn;   // DENSE_MASKED operand majors (1 = M/N contiguous)
  int bf16;         // element type: 0 f16, 1 bf16
  float alpha, beta;
  const void* C;
  void* D;
  int64_t ldc, ldd;
  int cd_col;       // 1: D[n * ldd + m]; 0: D[m * ldd + n]
  int tma_store;    // 1: D written by TMA bulk stores (C not read)
  const uint32_t* mask;
  int64_t mask_words;
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
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint (ns): the thread may sleep until the phase completes.
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\nselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Bounded wait: false if the budget ran out (then the status word and the
// CTA's abort flag are set) or another role already aborted.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, long long budget,
                                       int32_t* status) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_sleep(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      if (status != nullptr) atomicExch(status, (int)NM_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Plain bulk copy of `bytes` contiguous bytes (16-byte aligned, multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
               "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start, leading/stride byte
// offsets (16-byte units), fixed version bit 46, swizzle mode in bits 61..63.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}
constexpr uint32_t kSwizzle128 = 2, kSwizzle64 = 4, kSwizzleNone = 0;

// Instruction descriptor for kind::f16: D = F32, A/B = F16 or BF16.
__device__ __forceinline__ uint32_t idesc_f16(int bf16, int a_mn, int b_mn, bool sparse) {
  uint32_t d = (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) | ((uint32_t)a_mn << 15) |
               ((uint32_t)b_mn << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
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
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float load_cd(const void* base, int64_t off, int bf16) {
  const uint16_t b = reinterpret_cast<const uint16_t*>(base)[off];
  return bf16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
}
__device__ __forceinline__ uint16_t to_cd(float x, int bf16) {
  return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
  return (uint32_t)to_cd(lo, bf16) | ((uint32_t)to_cd(hi, bf16) << 16);
}

// ----------------------------------------------------------------- kernel
template <bool SPARSE>
__global__ void __launch_bounds__(kThreads, 1)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmD, const Params p) {
  using C = Cfg<SPARSE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain
  const uint32_t bar_full = smem_u32(bars), bar_empty = smem_u32(bars + C::kStages);
  const uint32_t bar_tfull = smem_u32(bars + 2 * C::kStages), bar_tempty = smem_u32(bars + 2 * C::kStages + 2);
  const uint32_t bar_drain = smem_u32(bars + 2 * C::kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.num_m_blk * p.num_n_blk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_tfull, 1);
    mbar_init(bar_tfull + 8, 1);
    mbar_init(bar_tempty, kEpiWarps);
    mbar_init(bar_tempty + 8, kEpiWarps);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_parity = 0;  // per-stage bits for the drain at the end
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m0 = (tile % p.num_m_blk) * BM, n0 = (tile / p.num_m_blk) * BN;
        for (int ks = 0; ks < p.num_k_stages; ++ks) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.wait_budget, p.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t sA = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sB = sA + C::kATileBytes;
          if constexpr (SPARSE) {
            // the 128 slot rows of one k-step are 2 KB of contiguous memory: one bulk copy each
            const int steps = min(2, p.num_k_steps - 2 * ks);
            mbar_expect_tx(fb, C::kATileBytes + kBTileBytes + steps * kMetaStepBytes);
            tma_load_2d(sA, &tmA, fb, ks * 32, m0);
            tma_load_2d(sB, &tmB, fb, ks * 64, n0);
            for (int j = 0; j < steps; ++j)
              bulk_load(sB + kBTileBytes + j * kMetaStepBytes,
                        p.meta + ((int64_t)(2 * ks + j) * p.meta_slots + m0) * 16, kMetaStepBytes, fb);
          } else {
            mbar_expect_tx(fb, C::kStageBytes);
            if (p.a_mn) {
              tma_load_2d(sA, &tmA, fb, m0, ks * 64);
              tma_load_2d(sA + C::kATileBytes / 2, &tmA, fb, m0 + 64, ks * 64);
            } else {
              tma_load_2d(sA, &tmA, fb, ks * 64, m0);
            }
            if (p.b_mn) {
              tma_load_2d(sB, &tmB, fb, n0, ks * 64);
              tma_load_2d(sB + kBTileBytes / 2, &tmB, fb, n0 + 64, ks * 64);
            } else {
              tma_load_2d(sB, &tmB, fb, ks * 64, n0);
            }
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: every issued copy must have landed before the CTA may exit.
      for (int s = 0; s < C::kStages; ++s)
        if ((issued >> s) & 1u) {
          const uint32_t par = (last_parity >> s) & 1u;
          const long long t0 = clock64();
          while (!mbar_try(bar_full + 8 * s, par) && clock64() - t0 < p.wait_budget) {
          }
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(p.bf16, SPARSE ? 0 : p.a_mn, SPARSE ? 0 : p.b_mn, SPARSE);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      uint32_t meta_slot = 0;  // running k-step count modulo the slot ring
      bool ok = true;
      if (p.fault_test) ok = mbar_wait(bar_drain, 0, abort_flag, p.wait_budget, p.status);  // nothing arrives: runs out
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1, abort_flag, p.wait_budget, p.status)) break;
        tc_fence_after();
        const uint32_t tacc = tmem + acc * BN;
        for (int ks = 0; ks < p.num_k_stages; ++ks) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.wait_budget, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sB = sA + C::kATileBytes;
          if constexpr (SPARSE) {
            const int steps = min(2, p.num_k_steps - 2 * ks);  // no MMA past K
            for (int j = 0; j < steps; ++j) {
              const uint32_t tmeta = tmem + kMetaCol + kMetaColStride * meta_slot;
              meta_slot = (meta_slot + 1) & (kMetaSlots - 1);
              // k-step j: 128 slot rows x 16 B, rows contiguous (8-row core matrices 128 B apart)
              const uint64_t md = sdesc(sB + kBTileBytes + j * kMetaStepBytes, 16, 128, kSwizzleNone);
              asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(tmeta), "l"(md));
              // A: 128 rows x 64 B (64B swizzle, 8-row groups 512 B apart), 16 values = 32 B per k-step
              const uint64_t ad = sdesc(sA + 32 * j, 16, 512, kSwizzle64);
              // B: BN rows x 128 B (128B swizzle), 32 values = 64 B per k-step
              const uint64_t bd = sdesc(sB + 64 * j, 16, 1024, kSwizzle128);
              mma_sparse(tacc, ad, bd, tmeta, idesc, (ks > 0 || j > 0) ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t ad = p.a_mn ? sdesc(sA + 2048 * j, C::kATileBytes / 2, 1024, kSwizzle128)
                                         : sdesc(sA + 32 * j, 16, 1024, kSwizzle128);
              const uint64_t bd = p.b_mn ? sdesc(sB + 2048 * j, kBTileBytes / 2, 1024, kSwizzle128)
                                         : sdesc(sB + 32 * j, 16, 1024, kSwizzle128);
              mma_dense(tacc, ad, bd, idesc, (ks > 0 || j > 0) ? 1u : 0u);
            }
          }
          tc_commit(bar_empty + 8 * stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(bar_tfull + 8 * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // Drain: all issued tensor-core work completes before TMEM is freed.
      tc_commit(bar_drain);
      const long long t0 = clock64();
      while (!mbar_try(bar_drain, 0u) && clock64() - t0 < p.wait_budget) {
      }
    }
  } else {
    // ------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - 2;
    uint8_t* ebuf = smem + C::kEpiOffset + ew * 2 * kEpiBufBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    int nbuf = 0;  // stores issued by this warp (selects the staging buffer)
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      if (!mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag, p.wait_budget, p.status)) break;
      tc_fence_after();
      const int m0 = (tile % p.num_m_blk) * BM, n0 = (tile / p.num_m_blk) * BN;
      const int mq = m0 + 32 * q;
      const int row = mq + lane;
      const bool row_ok = row < p.M;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        __syncwarp();  // tcgen05.ld is warp-collective: reconverge after any per-lane skip
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + acc * BN + ch * 32, v);
        if (ch == BN / 32 - 1) {
          // the accumulator buffer is drained: the next tile's MMAs may reuse it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
        }
        const int nb = n0 + ch * 32;
        if (mq >= p.M || nb >= p.N) continue;
        uint32_t mword = 0xFFFFFFFFu;
        if (!SPARSE && p.mask != nullptr && row_ok) mword = p.mask[(int64_t)row * p.mask_words + nb / 32];
        if (p.tma_store) {
          uint8_t* buf = ebuf + (nbuf & 1) * kEpiBufBytes;
          if (nbuf >= 2) {
            if (lane == 0) bulk_wait_read<1>();  // the store that used this buffer has read it
            __syncwarp();
          }
          if (p.cd_col) {
            // block [32 n][32 m], 64-byte rows: element (n, m) at (n * 32 + m) * 2
            uint16_t* b16 = reinterpret_cast<uint16_t*>(buf);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float x = ((mword >> j) & 1u) ? __uint_as_float(v[j]) * p.alpha : 0.0f;
              b16[j * 32 + lane] = to_cd(x, p.bf16);
            }
          } else {
            // block [32 m][32 n], 64-byte rows in the 64B-swizzled order the store map expects:
            // 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3)
            uint4* b4 = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int j = 8 * c + 2 * t;
                const float x0 = ((mword >> j) & 1u) ? __uint_as_float(v[j]) * p.alpha : 0.0f;
                const float x1 = ((mword >> (j + 1)) & 1u) ? __uint_as_float(v[j + 1]) * p.alpha : 0.0f;
                w[t] = pack2(x0, x1, p.bf16);
              }
              b4[c ^ ((lane >> 1) & 3)] = make_uint4(w[0], w[1], w[2], w[3]);
            }
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
          ++nbuf;
        } else {
          if (!row_ok) continue;
          const int cnt = min(32, p.N - nb);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j >= cnt) break;
            float x = ((mword >> j) & 1u) ? __uint_as_float(v[j]) : 0.0f;
            x *= p.alpha;
            const int64_t doff = p.cd_col ? (int64_t)(nb + j) * p.ldd + row : (int64_t)row * p.ldd + nb + j;
            const int64_t coff = p.cd_col ? (int64_t)(nb + j) * p.ldc + row : (int64_t)row * p.ldc + nb + j;
            if (p.C != nullptr) x = fmaf(p.beta, load_cd(p.C, coff, p.bf16), x);
            reinterpret_cast<uint16_t*>(p.D)[doff] = to_cd(x, p.bf16);
          }
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_all();  // staging buffers stay valid until the stores are done
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
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

bool make_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, const uint64_t dims[3],
                 const uint64_t pitches[2], const uint32_t box[3]) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {pitches[0], pitches[1]};
  cuuint32_t b[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dt, 3, const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
template <bool SPARSE>
cudaError_t set_smem_attr() {
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done_mask.load() & bit) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(spmm_tc_kernel<SPARSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<SPARSE>::kSmemBytes);
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
  p.num_k_stages = (int)((d.K + kKPerStage - 1) / kKPerStage);
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

}  // namespace tc

cudaError_t spmm_tc_sparse_impl(const SpmmLaunch& a, cudaStream_t s, int fault_test, long long budget) {
  using namespace tc;
  const nm_spmm_desc_t& d = a.d;
  if (d.K == 0) return launch_k0(a, s);
  Params p = base_params(a);
  p.fault_test = fault_test;
  if (budget > 0) p.wait_budget = budget;
  const CUtensorMapDataType u16 = CU_TENSOR_MAP_DATA_TYPE_UINT16;
  CUtensorMap mA, mB, mD;
  const int64_t kc = d.K / 2;  // compressed values per row, packed
  p.num_k_steps = (int)(d.K / 32);
  p.meta = static_cast<const uint8_t*>(a.A_meta);
  p.meta_slots = tc_slots(d.M);
  if (!make_map(&mA, a.A, u16, (uint64_t)kc, (uint64_t)d.M, (uint64_t)(kc * 2), 32, BM, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&mB, a.B, u16, (uint64_t)d.K, (uint64_t)d.N, (uint64_t)(d.ldb * 2), 64, BN,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_store_map(&mD, d, a.D))
    return cudaErrorInvalidValue;
  if (cudaError_t e = set_smem_attr<true>()) return e;
  const int tiles = p.num_m_blk * p.num_n_blk;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  spmm_tc_kernel<true><<<grid, kThreads, Cfg<true>::kSmemBytes, s>>>(mA, mB, mA, mD, p);
  return cudaGetLastError();
}

cudaError_t launch_spmm_tc_sparse(const SpmmLaunch& a, cudaStream_t s) { return spmm_tc_sparse_impl(a, s, 0, 0); }

int spmm_tc_dense_masked_split(const nm_spmm_desc_t&) { return 1; }
size_t spmm_tc_dense_masked_workspace(const nm_spmm_desc_t&, int) { return 0; }

cudaError_t launch_spmm_tc_dense_masked(const SpmmLaunch& a, int /*split_k*/, cudaStream_t s) {
  using namespace tc;
  const nm_spmm_desc_t& d = a.d;
  if (d.K == 0) return launch_k0(a, s);
  Params p = base_params(a);
  p.a_mn = d.order_a == NM_COL;
  p.b_mn = d.order_b == NM_ROW;
  p.mask = static_cast<const uint32_t*>(a.A_meta);
  p.mask_words = (d.N + 31) / 32;
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
      ok = make_map(&mB, a.B, u16, (uint64_t)d.K, (uint64_t)d.N, (uint64_t)(d.ldb * 2), 64, BN,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (ok) ok = make_store_map(&mD, d, a.D);
  if (!ok) return cudaErrorInvalidValue;
  if (cudaError_t e = set_smem_attr<false>()) return e;
  const int tiles = p.num_m_blk * p.num_n_blk;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  spmm_tc_kernel<false><<<grid, kThreads, Cfg<false>::kSmemBytes, s>>>(mA, mB, mA, mD, p);
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
