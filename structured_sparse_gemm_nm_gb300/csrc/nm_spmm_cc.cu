// CUDA-core product for general N:M sparse A (apex PR #1631 "[sparse] update
// support for arbitrary N:M settings sparse": m = 32 windows, the shape the
// page names for sparse GEMV, where the contraction is too thin for tensor
// cores).
//
//   D[r][b] = alpha * sum_g sum_t vals[r][g*n+t] * B[b][g*m + idx[r][g*n+t]] + beta * C
//
// B is read as N x K (K contiguous, ld = ldb).  A warp owns one row r of A at
// a time and streams that row's values and indices with 128-bit loads; the
// B columns of up to 8 batch entries sit in shared memory interleaved as
// [k][8] so one 16-byte shared load feeds the 8 products of a kept value.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "nm_device.cuh"
#include "nm_internal.h"
#include "../../include/nm_testing.h"

namespace nmk {
namespace {

constexpr int kBatch = 8;  // batch columns per pass

__device__ __forceinline__ float to_f(uint16_t b, int bf16) {
  return bf16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
}
__device__ __forceinline__ uint16_t from_f(float x, int bf16) {
  return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}

// NB = batch columns per pass (1 or 8).  x is staged in shared memory as
// [k][NB]; the staging reads B with 16-byte loads when rows of B allow it.
// NN = n when it is 4, 8 or 16 (the group of a kept value by a shift), 0 for
// any other n (a 32-bit division per kept value).
template <int NB, int NN>
__global__ void __launch_bounds__(NB == 1 ? 256 : 1024) gather_kernel(const uint16_t* __restrict__ vals, const uint8_t* __restrict__ idx,
                                                     const uint16_t* __restrict__ B, const uint16_t* __restrict__ C,
                                                     uint16_t* __restrict__ D, int64_t M, int64_t N, int64_t K, int n,
                                                     int m, int64_t ldb, int64_t ldc, int64_t ldd, int cd_col,
                                                     float alpha, float beta, int bf16) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint4 xs4[];  // K x NB halves, [k][b]
  uint16_t* xs = reinterpret_cast<uint16_t*>(xs4);
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t kc = (K / m) * n;  // kept values per row (below 2^31: K < 2^31)
  // group of the j-th kept value of a row
  auto group_of = [&](uint32_t j) -> uint32_t { return NN > 0 ? j / (uint32_t)NN : j / (uint32_t)n; };
  const bool vec = (kc % 8 == 0);
  const bool vstage = (K % 8 == 0);
  for (int64_t b0 = 0; b0 < N; b0 += NB) {
    const int nb = (int)(N - b0 < NB ? N - b0 : NB);
    const uint16_t* xg = B + b0 * ldb;  // NB == 1: x is read through the L1 cache, not staged
    __syncthreads();
    if (NB == 1) {
    } else if (vstage) {
      // a thread takes eight k of all NB (= 8) columns: eight 16-byte loads along B's rows,
      // a transpose in registers, eight 16-byte stores of one k's NB values each; k's slot
      // is k ^ ((k >> 3) & 7), so the eight lanes of a store phase hit different banks
      static_assert(NB == 1 || NB == 8, "x is staged as [k][8]");
      const int64_t k8 = K / 8;
      for (int64_t c = threadIdx.x; c < k8; c += blockDim.x) {
        const int64_t kk = c * 8;
        uint32_t q[NB][4];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (b < nb) v = __ldg(reinterpret_cast<const uint4*>(B + (b0 + b) * ldb + kk));
          q[b][0] = v.x, q[b][1] = v.y, q[b][2] = v.z, q[b][3] = v.w;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          uint32_t w[4];
#pragma unroll
          for (int pr = 0; pr < 4; ++pr)
            w[pr] = ((q[2 * pr][t / 2] >> (16 * (t % 2))) & 0xFFFFu) | ((q[2 * pr + 1][t / 2] >> (16 * (t % 2))) << 16);
          xs4[kk + (t ^ (int)(c & 7))] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    } else {
      for (int64_t i = threadIdx.x; i < K * NB; i += blockDim.x) {
        const int64_t k = i / NB;
        const int b = (int)(i - k * NB);
        xs[i] = (b < nb) ? B[(b0 + b) * ldb + k] : (uint16_t)0;
      }
    }
    __syncthreads();
    // rows interleaved over the CTAs (row r to CTA r mod grid), so that with a grid of
    // whole waves every SM gets within one row per CTA of the same count
    for (int64_t r = (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x; r < M; r += (int64_t)gridDim.x * warps) {
      float acc[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
      const uint16_t* vr = vals + r * kc;
      const uint8_t* ir = idx + r * kc;
      if (vec) {
        // up to CH chunks of 256 kept values per warp with all their loads in flight first
        constexpr int CH = NB == 1 ? 4 : 2;
        for (int64_t jb = 0; jb < kc; jb += 256 * CH) {
          uint4 v4s[CH];
          uint2 i2s[CH];
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            const int64_t j0 = jb + 256 * c + (int64_t)lane * 8;
            if (j0 < kc) {
              v4s[c] = __ldcs(reinterpret_cast<const uint4*>(vr + j0));
              i2s[c] = __ldcs(reinterpret_cast<const uint2*>(ir + j0));
            }
          }
#pragma unroll
          for (int c = 0; c < CH; ++c) {
          const int64_t j0 = jb + 256 * c + (int64_t)lane * 8;
          if (j0 >= kc) break;
          const uint4 v4 = v4s[c];
          const uint2 i2 = i2s[c];
          const uint32_t vw[4] = {v4.x, v4.y, v4.z, v4.w};
          const uint32_t iw[2] = {i2.x, i2.y};
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const uint32_t j = (uint32_t)j0 + (uint32_t)t;
            const int64_t k =
                (int64_t)group_of(j) * m + min((iw[t / 4] >> (8 * (t % 4))) & 0xFFu, (uint32_t)(m - 1));
            const float a = to_f((uint16_t)(vw[t / 2] >> (16 * (t % 2))), bf16);
            if constexpr (NB == 1) {
              acc[0] = fmaf(a, to_f(__ldg(xg + k), bf16), acc[0]);
            } else {
              const uint4 x4 = xs4[vstage ? (k ^ ((k >> 3) & 7)) : k];
              const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
              for (int b = 0; b < NB; ++b) acc[b] = fmaf(a, to_f((uint16_t)(xw[b / 2] >> (16 * (b % 2))), bf16), acc[b]);
            }
          }
          }
        }
      } else {
        for (int64_t j = lane; j < kc; j += 32) {
          const int64_t k = (int64_t)group_of((uint32_t)j) * m + min((int)ir[j], m - 1);
          const float a = to_f(vr[j], bf16);
          if constexpr (NB == 1) {
            acc[0] = fmaf(a, to_f(__ldg(xg + k), bf16), acc[0]);
          } else {
#pragma unroll
            for (int b = 0; b < NB; ++b)
              acc[b] = fmaf(a, to_f(xs[(vstage ? (k ^ ((k >> 3) & 7)) : k) * NB + b], bf16), acc[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[b] += __shfl_xor_sync(0xFFFFFFFFu, acc[b], off);
      if (lane < nb) {
        float x = 0.0f;
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (b == lane) x = acc[b];
        x *= alpha;
        const int64_t bb = b0 + lane;
        const int64_t dof = cd_col ? bb * ldd + r : r * ldd + bb;
        if (C != nullptr) x = fmaf(beta, to_f(C[cd_col ? bb * ldc + r : r * ldc + bb], bf16), x);
        D[dof] = from_f(x, bf16);
      }
    }
  }
}

template <int NB, int NN>
cudaError_t gather_launch(const SpmmLaunch& a, cudaStream_t s) {
  const nm_spmm_desc_t& d = a.d;
  const size_t smem = NB == 1 ? 0 : (size_t)d.K * NB * 2;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    // set once per device to the largest size this kernel may take
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev)) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done_mask.load() & bit)) {
      cudaError_t e = cudaFuncSetAttribute(gather_kernel<NB, NN>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      if (e != cudaSuccess) return e;
      done_mask.fetch_or(bit);
    }
  }
  // A warp per row.  NB == 1: as many CTAs as fit on every SM at once; NB > 1: x is
  // staged once per CTA, so one CTA of 32 warps per SM keeps that staging to one copy
  // per SM.  The grid is whole waves over the SMs (rows are interleaved over CTAs): a
  // grid of ceil(M / 32) CTAs left 24 of 152 SMs idle at M = 4096.
  const int threads = NB == 1 ? 256 : 1024;
  static const int per_sm = NB == 1 ? resident_ctas(gather_kernel<NB, NN>, threads, 0) : 1;
  int64_t blocks = (int64_t)num_sms_cached() * per_sm;
  if (blocks > d.M) blocks = d.M;
  if (blocks < 1) blocks = 1;
  const cudaError_t e_ = launch_pdl(gather_kernel<NB, NN>, dim3((unsigned)blocks), dim3(threads), smem, s,
                                    static_cast<const uint16_t*>(a.A), static_cast<const uint8_t*>(a.A_meta),
                                    static_cast<const uint16_t*>(a.B), static_cast<const uint16_t*>(a.C),
                                    static_cast<uint16_t*>(a.D), d.M, d.N, d.K, d.n, d.m, d.ldb, d.ldc, d.ldd,
                                    d.order_cd == NM_COL, a.alpha_f, a.beta_f, d.ab_type == NM_BF16);
  return e_;
}

}  // namespace

template <int NB>
cudaError_t gather_launch_n(const SpmmLaunch& a, cudaStream_t s) {
  switch (a.d.n) {
    case 4: return gather_launch<NB, 4>(a, s);
    case 8: return gather_launch<NB, 8>(a, s);
    case 16: return gather_launch<NB, 16>(a, s);
    default: return gather_launch<NB, 0>(a, s);
  }
}

cudaError_t launch_spmm_nm_gather(const SpmmLaunch& a, cudaStream_t s) {
  return a.d.N == 1 ? gather_launch_n<1>(a, s) : gather_launch_n<kBatch>(a, s);
}

// ---------------------------------------------------------------------------
// 2:4 sparse INT8 product with INT32 accumulation (cuSPARSELt blog, "key
// features": INT8 inputs, INT32 Tensor Core accumulation).  The tcgen05 MMA
// has no int8 kind on sm_103a, so this uses the warp-level sparse MMA
// m16n8k64 (s8 x s8 -> s32) with the canonical metadata: lane 4g+t supplies
// the 32-bit word of row g + 8*(t&1) covering columns 32*(t>>1) .. +31 of the
// 64-column k-step, which is exactly two consecutive uint16 words of the
// canonical layout.
//
// CTA tile 128 x 128, 8 warps (4 along M x 2 along N, 32 x 64 each), four stages of 128
// dense K.  A (128 rows x 64 compressed bytes) and B (128 rows x 128 bytes) arrive by TMA
// in the 64-byte and 128-byte swizzles, which keep the fragment loads free of bank
// conflicts; the metadata (128 rows x 16 bytes) by cp.async, so that rows past M and a K
// tail can hold the valid code 0x4 instead of TMA's zero fill.
namespace {

constexpr int I8_BM = 128, I8_BN = 128, I8_BK = 128, I8_STAGES = 4;
constexpr int I8_BBYTES = I8_BN * 128;  // stage offset 0 (1024-byte aligned for the 128-byte swizzle)
constexpr int I8_ABYTES = I8_BM * 64;   // at 16384 (512-byte aligned for the 64-byte swizzle)
constexpr int I8_MPITCH = 16;           // 8 uint16 metadata words per row per stage
constexpr int I8_MBYTES = I8_BM * I8_MPITCH;
constexpr int I8_STAGE_BYTES = I8_BBYTES + I8_ABYTES + I8_MBYTES;  // 26 KB, a multiple of 1024
constexpr int I8_TX_BYTES = I8_BBYTES + I8_ABYTES;
static_assert(I8_STAGE_BYTES % 1024 == 0, "stage alignment");

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void i8_tma_load(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Four 8 x 16-byte matrices: lanes 8i .. 8i + 7 give the row addresses of matrix i, and lane
// (g, t) receives bytes 4t .. 4t + 3 of row g of matrix i in register i.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ bool i8_mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// OUT8: int8 D (and C) with float scales: D = saturate(rne(alpha * acc + beta * C)), each
// product and the sum rounded to float32; otherwise int32 D = alpha * acc + beta * C modulo 2^32.
// A stage barrier that has not completed within `budget` cycles writes NM_ERR_TIMEOUT to
// *status (nullable) and the CTA stops issuing MMAs (D is then not defined).
template <bool OUT8>
__global__ void __launch_bounds__(256, 1) spmm_i8_kernel(const __grid_constant__ CUtensorMap tmA,
                                                      const __grid_constant__ CUtensorMap tmB,
                                                      const uint16_t* __restrict__ meta, const void* __restrict__ Cv,
                                                      void* __restrict__ Dv, int M, int N, int K, int64_t ldc,
                                                      int64_t ldd, int cd_col, int32_t alpha, int32_t beta,
                                                      float alpha_f, float beta_f, int32_t* status, long long budget) {
  extern __shared__ uint4 smem4[];
  __shared__ __align__(8) uint64_t full[I8_STAGES];
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem4) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int wm = warp & 3, wn = warp >> 2;
  const int m0 = blockIdx.y * I8_BM, n0 = blockIdx.x * I8_BN;
  const int64_t mrow = K / 16;      // uint16 metadata words per row
  const int kstages = (K + I8_BK - 1) / I8_BK;
  const int ksteps = K / 64;        // MMA k-steps in K
  const uint32_t smem_base = (uint32_t)__cvta_generic_to_shared(smem);
  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < I8_STAGES; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(&full[i])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  int issued = 0;  // stages whose copies have been issued (the same count in every thread)
  auto load_stage = [&](int ks, int buf) {
    ++issued;
    const uint32_t base = smem_base + buf * I8_STAGE_BYTES;
    if (tid == 0) {
      const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&full[buf]);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(I8_TX_BYTES) : "memory");
      i8_tma_load(base, &tmB, bar, ks * 128, n0);
      i8_tma_load(base + I8_BBYTES, &tmA, bar, ks * 64, m0);
    }
    // metadata: 128 rows x 16 bytes; rows past M (or a K tail) get the valid code 0x4
    if (tid < I8_BM * 2) {
      const int r = tid >> 1, h = tid & 1;
      const int64_t w = (int64_t)ks * 8 + h * 4;
      const uint32_t dst = base + I8_BBYTES + I8_ABYTES + r * I8_MPITCH + h * 8;
      if (m0 + r < M && w < mrow) {
        cp_async8(dst, meta + (int64_t)(m0 + r) * mrow + w);
      } else {
        asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(dst), "r"(0x44444444u) : "memory");
      }
    }
  };

  int32_t acc[2][8][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0;

  for (int s = 0; s < I8_STAGES - 1; ++s) {
    if (s < kstages) load_stage(s, s);
    cp_commit();
  }
  bool ok = true;
  for (int ks = 0; ks < kstages; ++ks) {
    const int buf = ks % I8_STAGES;
    cp_wait<I8_STAGES - 2>();  // this thread's metadata copies of stage ks
    if (ok) {                  // the stage's A and B boxes (bounded wait)
      const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&full[buf]);
      const uint32_t parity = (uint32_t)(ks / I8_STAGES) & 1u;
      if (!i8_mbar_try(bar, parity)) {
        const long long t0 = clock64();
        while (!i8_mbar_try(bar, parity)) {
          if (abort_flag || clock64() - t0 > budget) {
            if (!abort_flag && status != nullptr) atomicExch(status, (int)NM_ERR_TIMEOUT);
            abort_flag = 1;
            ok = false;
            break;
          }
        }
      }
    }
    __syncthreads();  // every thread's metadata copies, and the buffer of stage ks - 1 is free
    if (abort_flag) ok = false;
    const int nxt = ks + I8_STAGES - 1;
    if (ok && nxt < kstages) load_stage(nxt, nxt % I8_STAGES);
    cp_commit();
    if (!ok) continue;
    const uint8_t* sb = smem + buf * I8_STAGE_BYTES;
    const uint8_t* sa = sb + I8_BBYTES;
    const uint8_t* sm = sa + I8_ABYTES;
    const uint32_t sb_u = smem_base + buf * I8_STAGE_BYTES, sa_u = sb_u + I8_BBYTES;
    const int li = lane & 7, lm = lane >> 3;  // ldmatrix: this lane's row within matrix lm
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      if (ks * 2 + kk >= ksteps) break;  // no MMA past K
      uint32_t bf[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        // matrix r: the eight B rows (columns of D) of this n-tile, 16-byte chunk 4 kk + r; 128-byte
        // rows in the 128-byte swizzle: chunk c of row n at chunk c ^ (n & 7)
        const int rn = wn * 64 + nt * 8 + li;
        ldsm_x4(sb_u + rn * 128 + (((4 * kk + lm) ^ (rn & 7)) << 4), bf[nt]);
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int rb = wm * 32 + mt * 16;
        uint32_t af[4];
        {
          // matrix r: A rows rb + 8 (r & 1) .. + 7, 16-byte chunk 2 kk + (r >> 1); 64-byte rows in the
          // 64-byte swizzle: chunk c of row m at chunk c ^ ((m >> 1) & 3)
          const int ra = rb + 8 * (lm & 1) + li;
          ldsm_x4(sa_u + ra * 64 + (((2 * kk + (lm >> 1)) ^ ((ra >> 1) & 3)) << 4), af);
        }
        const uint32_t e =
            *reinterpret_cast<const uint32_t*>(sm + (rb + g + 8 * (t & 1)) * I8_MPITCH + kk * 8 + (t >> 1) * 4);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          asm volatile(
              "mma.sp::ordered_metadata.sync.aligned.m16n8k64.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
              "{%8,%9,%10,%11}, {%0,%1,%2,%3}, %12, 0x0;"
              : "+r"(acc[mt][nt][0]), "+r"(acc[mt][nt][1]), "+r"(acc[mt][nt][2]), "+r"(acc[mt][nt][3])
              : "r"(af[0]), "r"(af[1]), "r"(af[2]), "r"(af[3]), "r"(bf[nt][0]), "r"(bf[nt][1]), "r"(bf[nt][2]),
                "r"(bf[nt][3]), "r"(e));
        }
      }
    }
  }
  cp_wait<0>();
  if (!ok && tid == 0) {
    // copies still in flight land before the CTA's shared memory is released (bounded): the
    // last I8_STAGES stages issued use distinct barriers, each with one pending phase at most
    for (int k = issued > I8_STAGES ? issued - I8_STAGES : 0; k < issued; ++k) {
      const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&full[k % I8_STAGES]);
      const long long t0 = clock64();
      while (!i8_mbar_try(bar, (uint32_t)(k / I8_STAGES) & 1u) && clock64() - t0 < budget) {
      }
    }
  }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = m0 + wm * 32 + mt * 16 + g + 8 * (r >> 1);
        const int col = n0 + wn * 64 + nt * 8 + 2 * t + (r & 1);
        if (row >= M || col >= N) continue;
        const int64_t coff = cd_col ? (int64_t)col * ldc + row : (int64_t)row * ldc + col;
        const int64_t doff = cd_col ? (int64_t)col * ldd + row : (int64_t)row * ldd + col;
        if constexpr (OUT8) {
          float x = __fmul_rn(alpha_f, __int2float_rn(acc[mt][nt][r]));
          if (Cv != nullptr) x = __fadd_rn(x, __fmul_rn(beta_f, (float)static_cast<const int8_t*>(Cv)[coff]));
          const int q = __float2int_rn(x);
          static_cast<int8_t*>(Dv)[doff] = (int8_t)max(-128, min(127, q));
        } else {
          // D = alpha * acc + beta * C in int32 arithmetic modulo 2^32
          uint32_t x = (uint32_t)alpha * (uint32_t)acc[mt][nt][r];
          if (Cv != nullptr) x += (uint32_t)beta * (uint32_t)static_cast<const int32_t*>(Cv)[coff];
          static_cast<int32_t*>(Dv)[doff] = (int32_t)x;
        }
      }
}

}  // namespace

cudaError_t launch_spmm_i8(const SpmmLaunch& a, cudaStream_t s) {
  const nm_spmm_desc_t& d = a.d;
  if (d.K == 0) return cudaErrorInvalidValue;  // rejected by the plan
  if (cudaError_t e = tc::bind_context()) return e;
  const int smem = I8_STAGES * I8_STAGE_BYTES + 1024;  // + alignment of the stages to 1024 bytes
  const bool out8 = d.cd_type == NM_I8;
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done_mask.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(spmm_i8_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(spmm_i8_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    done_mask.fetch_or(bit);
  }
  // A: M rows of K / 2 compressed bytes; B: N rows (columns of D) of K bytes, ldb apart
  CUtensorMap mA, mB;
  if (!tc::make_map(&mA, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)(d.K / 2), (uint64_t)d.M, (uint64_t)(d.K / 2),
                    64, I8_BM, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !tc::make_map(&mB, a.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)d.K, (uint64_t)d.N, (uint64_t)d.ldb, 128, I8_BN,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const long long budget = 1ll << 32;  // cycles, about two seconds
  dim3 grid((unsigned)((d.N + I8_BN - 1) / I8_BN), (unsigned)((d.M + I8_BM - 1) / I8_BM));
  if (out8)
    spmm_i8_kernel<true><<<grid, 256, smem, s>>>(mA, mB, static_cast<const uint16_t*>(a.A_meta), a.C, a.D, (int)d.M,
                                                 (int)d.N, (int)d.K, d.ldc, d.ldd, d.order_cd == NM_COL, 0, 0,
                                                 a.alpha_f, a.beta_f, a.d_status, budget);
  else
    spmm_i8_kernel<false><<<grid, 256, smem, s>>>(mA, mB, static_cast<const uint16_t*>(a.A_meta), a.C, a.D, (int)d.M,
                                                  (int)d.N, (int)d.K, d.ldc, d.ldd, d.order_cd == NM_COL, a.alpha_i,
                                                  a.beta_i, 0.0f, 0.0f, a.d_status, budget);
  return cudaGetLastError();
}

}  // namespace nmk

namespace {
// Rate probe: four independent accumulator chains per warp on register operands (metadata
// code 0x4 = positions 0 and 1 of every group, selector 0), no memory traffic in the loop.
__global__ void __launch_bounds__(256) i8_sparse_mma_rate_kernel(int iters, int32_t* out, uint32_t seed) {
  int32_t acc[4][4] = {};
  const uint32_t a0 = seed * 0x9E3779B9u + threadIdx.x, a1 = a0 ^ 0x55u, a2 = a0 + 7u, a3 = a0 * 3u;
  const uint32_t b0 = seed + threadIdx.x * 13u, b1 = b0 ^ 0xAAu, b2 = b0 + 5u, b3 = b0 * 5u;
  const uint32_t e = 0x44444444u;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      asm volatile(
          "mma.sp::ordered_metadata.sync.aligned.m16n8k64.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9,%10,%11}, {%0,%1,%2,%3}, %12, 0x0;"
          : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(b2), "r"(b3), "r"(e));
  }
  int32_t sum = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) sum += acc[c][0] + acc[c][1] + acc[c][2] + acc[c][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = sum;  // keeps the chains live
}
}  // namespace

extern "C" nm_status_t nm_test_i8_sparse_mma_rate(int iters, float* ms, double* ops) {
  if (iters < 1 || iters > 1000000 || ms == nullptr || ops == nullptr) return NM_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return NM_ERR_CUDA;
  constexpr int kThreads = 256;
  int32_t* out = nullptr;
  if (cudaMalloc(&out, sizeof(int32_t) * (size_t)sms * kThreads) != cudaSuccess) return NM_ERR_CUDA;
  cudaEvent_t t0 = nullptr, t1 = nullptr;
  bool ok = cudaEventCreate(&t0) == cudaSuccess && cudaEventCreate(&t1) == cudaSuccess;
  if (ok) {
    i8_sparse_mma_rate_kernel<<<sms, kThreads>>>(iters, out, 1u);  // warm-up
    ok = cudaEventRecord(t0) == cudaSuccess;
    i8_sparse_mma_rate_kernel<<<sms, kThreads>>>(iters, out, 2u);
    ok = ok && cudaGetLastError() == cudaSuccess && cudaEventRecord(t1) == cudaSuccess &&
         cudaEventSynchronize(t1) == cudaSuccess && cudaEventElapsedTime(ms, t0, t1) == cudaSuccess;
  }
  *ops = 2.0 * 16 * 8 * 64 * 4.0 * (double)iters * (kThreads / 32) * sms;
  if (t0) cudaEventDestroy(t0);
  if (t1) cudaEventDestroy(t1);
  const bool freed = cudaFree(out) == cudaSuccess;
  return ok && freed ? NM_OK : NM_ERR_CUDA;
}

