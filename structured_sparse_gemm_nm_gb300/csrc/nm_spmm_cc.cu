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

namespace nmk {
namespace {

constexpr int kBatch = 8;  // batch columns per pass

__device__ __forceinline__ float to_f(uint16_t b, int bf16) {
  return bf16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
}
__device__ __forceinline__ uint16_t from_f(float x, int bf16) {
  return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}

__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ vals, const uint8_t* __restrict__ idx,
                                                     const uint16_t* __restrict__ B, const uint16_t* __restrict__ C,
                                                     uint16_t* __restrict__ D, int64_t M, int64_t N, int64_t K, int n,
                                                     int m, int64_t ldb, int64_t ldc, int64_t ldd, int cd_col,
                                                     float alpha, float beta, int bf16) {
  extern __shared__ uint4 xs4[];  // K x kBatch halves, [k][b]
  uint16_t* xs = reinterpret_cast<uint16_t*>(xs4);
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t kc = (K / m) * n;  // kept values per row
  const bool vec = (kc % 8 == 0);
  for (int64_t b0 = 0; b0 < N; b0 += kBatch) {
    const int nb = (int)(N - b0 < kBatch ? N - b0 : kBatch);
    __syncthreads();
    for (int64_t i = threadIdx.x; i < K * kBatch; i += blockDim.x) {
      const int64_t k = i / kBatch;
      const int b = (int)(i - k * kBatch);
      xs[i] = (b < nb) ? B[(b0 + b) * ldb + k] : (uint16_t)0;
    }
    __syncthreads();
    for (int64_t r = blockIdx.x * (int64_t)warps + (threadIdx.x >> 5); r < M; r += (int64_t)gridDim.x * warps) {
      float acc[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) acc[b] = 0.0f;
      const uint16_t* vr = vals + r * kc;
      const uint8_t* ir = idx + r * kc;
      if (vec) {
        for (int64_t j0 = (int64_t)lane * 8; j0 < kc; j0 += 256) {
          const uint4 v4 = *reinterpret_cast<const uint4*>(vr + j0);
          const uint2 i2 = *reinterpret_cast<const uint2*>(ir + j0);
          const uint32_t vw[4] = {v4.x, v4.y, v4.z, v4.w};
          const uint32_t iw[2] = {i2.x, i2.y};
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int64_t j = j0 + t;
            const int64_t k = (j / n) * m + min((iw[t / 4] >> (8 * (t % 4))) & 0xFFu, (uint32_t)(m - 1));
            const float a = to_f((uint16_t)(vw[t / 2] >> (16 * (t % 2))), bf16);
            const uint4 x4 = *reinterpret_cast<const uint4*>(xs + k * kBatch);
            const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int b = 0; b < kBatch; ++b) acc[b] = fmaf(a, to_f((uint16_t)(xw[b / 2] >> (16 * (b % 2))), bf16), acc[b]);
          }
        }
      } else {
        for (int64_t j = lane; j < kc; j += 32) {
          const int64_t k = (j / n) * m + min((int)ir[j], m - 1);
          const float a = to_f(vr[j], bf16);
#pragma unroll
          for (int b = 0; b < kBatch; ++b) acc[b] = fmaf(a, to_f(xs[k * kBatch + b], bf16), acc[b]);
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[b] += __shfl_xor_sync(0xFFFFFFFFu, acc[b], off);
      if (lane < nb) {
        float x = 0.0f;
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
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

}  // namespace

cudaError_t launch_spmm_nm_gather(const SpmmLaunch& a, cudaStream_t s) {
  const nm_spmm_desc_t& d = a.d;
  const size_t smem = (size_t)d.K * kBatch * 2;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    // set once per device to the largest size this kernel may take
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev)) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done_mask.load() & bit)) {
      cudaError_t e = cudaFuncSetAttribute(gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      if (e != cudaSuccess) return e;
      done_mask.fetch_or(bit);
    }
  }
  const int threads = 256;
  int64_t blocks = (d.M + 7) / 8;
  if (blocks > 152 * 2) blocks = 152 * 2;
  if (blocks < 1) blocks = 1;
  gather_kernel<<<(unsigned)blocks, threads, smem, s>>>(
      static_cast<const uint16_t*>(a.A), static_cast<const uint8_t*>(a.A_meta), static_cast<const uint16_t*>(a.B),
      static_cast<const uint16_t*>(a.C), static_cast<uint16_t*>(a.D), d.M, d.N, d.K, d.n, d.m, d.ldb, d.ldc, d.ldd,
      d.order_cd == NM_COL, a.alpha_f, a.beta_f, d.ab_type == NM_BF16);
  return cudaGetLastError();
}

cudaError_t launch_spmm_i8(const SpmmLaunch&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace nmk
