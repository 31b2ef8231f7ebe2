// Transposable 2:4 pruning on 4x4 tiles (PyTorch issue #126420, maintainer
// reply: the forward product W x and the backward product W^T dL/dy both run
// on 2:4 sparse hardware only if every 4x4 tile keeps two entries per row and
// two per column).
//
// Per tile the kernel scores the 90 patterns with two kept entries in every
// row and column, score = ((p0 + p1) + p2) + p3 in float32 where p_r is the
// sum of row r's two kept magnitudes, and keeps the first pattern (row 0's
// pair outermost, pairs in the order (0,1),(0,2),(0,3),(1,2),(1,3),(2,3))
// with the largest score.
//
// Work layout: one warp per 16 x 32 block of W, lane l owns the tile in tile
// row l/8 and tile column l%8 of the block.  Every packed output word (a
// 32-bit mask word of one row, a 16-bit metadata word of four groups) then
// comes from lanes of the same warp and is assembled with shuffles.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "nm_device.cuh"
#include "nm_internal.h"

namespace nmk {
namespace {

// Column bits of pair q in (0,1),(0,2),(0,3),(1,2),(1,3),(2,3).
__host__ __device__ constexpr uint32_t pair_bits(int q) {
  return q == 0 ? 0x3u : q == 1 ? 0x5u : q == 2 ? 0x9u : q == 3 ? 0x6u : q == 4 ? 0xAu : 0xCu;
}
__host__ __device__ constexpr int pair_of_bits(uint32_t b) {
  return b == 0x3u ? 0 : b == 0x5u ? 1 : b == 0x9u ? 2 : b == 0x6u ? 3 : b == 0xAu ? 4 : b == 0xCu ? 5 : -1;
}
__host__ __device__ constexpr int col_count(int a, int b, int c, int j) {
  return (int)((pair_bits(a) >> j) & 1u) + (int)((pair_bits(b) >> j) & 1u) + (int)((pair_bits(c) >> j) & 1u);
}
// Pair that row 3 must keep after rows 0..2 chose a, b, c, or -1 if none completes a valid tile.
__host__ __device__ constexpr int completion(int a, int b, int c) {
  uint32_t need = 0;
  for (int j = 0; j < 4; ++j) {
    const int k = col_count(a, b, c, j);
    if (k < 1 || k > 2) return -1;
    if (k == 1) need |= 1u << j;
  }
  return pair_of_bits(need);
}
__host__ __device__ constexpr uint32_t tile_mask(int a, int b, int c, int d) {
  return pair_bits(a) | (pair_bits(b) << 4) | (pair_bits(c) << 8) | (pair_bits(d) << 12);
}

template <int DT>
__device__ __forceinline__ float tile_mag(typename Elem<DT>::T v) {
  if constexpr (DT == kI8) {
    return fabsf((float)v);
  } else {
    return mag_f32((uint16_t)v, DT);
  }
}

// Four consecutive elements of a tile row in one access (VEC: 8 bytes for
// 16-bit types, 4 for int8), or element by element.
template <bool VEC>
__device__ __forceinline__ void load4(const uint16_t* p, uint16_t (&o)[4]) {
  if constexpr (VEC) {
    const uint2 q = *reinterpret_cast<const uint2*>(p);
    o[0] = (uint16_t)q.x, o[1] = (uint16_t)(q.x >> 16), o[2] = (uint16_t)q.y, o[3] = (uint16_t)(q.y >> 16);
  } else {
    for (int c = 0; c < 4; ++c) o[c] = p[c];
  }
}
template <bool VEC>
__device__ __forceinline__ void load4(const int8_t* p, int8_t (&o)[4]) {
  if constexpr (VEC) {
    const uint32_t q = *reinterpret_cast<const uint32_t*>(p);
    for (int c = 0; c < 4; ++c) o[c] = (int8_t)(q >> (8 * c));
  } else {
    for (int c = 0; c < 4; ++c) o[c] = p[c];
  }
}
template <bool VEC>
__device__ __forceinline__ void store4(uint16_t* p, const uint16_t (&o)[4]) {
  if constexpr (VEC) {
    *reinterpret_cast<uint2*>(p) = make_uint2(o[0] | ((uint32_t)o[1] << 16), o[2] | ((uint32_t)o[3] << 16));
  } else {
    for (int c = 0; c < 4; ++c) p[c] = o[c];
  }
}
template <bool VEC>
__device__ __forceinline__ void store4(int8_t* p, const int8_t (&o)[4]) {
  if constexpr (VEC) {
    uint32_t q = 0;
    for (int c = 0; c < 4; ++c) q |= (uint32_t)(uint8_t)o[c] << (8 * c);
    *reinterpret_cast<uint32_t*>(p) = q;
  } else {
    for (int c = 0; c < 4; ++c) p[c] = o[c];
  }
}
template <bool VEC>
__device__ __forceinline__ void store2(uint16_t* p, uint16_t a, uint16_t b) {
  if constexpr (VEC) {
    *reinterpret_cast<uint32_t*>(p) = a | ((uint32_t)b << 16);
  } else {
    p[0] = a, p[1] = b;
  }
}
template <bool VEC>
__device__ __forceinline__ void store2(int8_t* p, int8_t a, int8_t b) {
  if constexpr (VEC) {
    *reinterpret_cast<uint16_t*>(p) = (uint16_t)((uint8_t)a | ((uint32_t)(uint8_t)b << 8));
  } else {
    p[0] = a, p[1] = b;
  }
}

// One SGD step on a 16-bit element: w + round(-lr * g), both operations rounded to float32
// separately (no contraction into a fused multiply-add), then rounded to the element type.
template <int DT>
__device__ __forceinline__ uint16_t sgd_elem(uint16_t w, uint16_t g, float nlr) {
  float wf, gf;
  if constexpr (DT == kBF16) {
    wf = __uint_as_float((uint32_t)w << 16);
    gf = __uint_as_float((uint32_t)g << 16);
  } else {
    wf = __half2float(__ushort_as_half(w));
    gf = __half2float(__ushort_as_half(g));
  }
  const float x = __fadd_rn(wf, __fmul_rn(nlr, gf));
  if constexpr (DT == kBF16)
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else
    return __half_as_ushort(__float2half_rn(x));
}

// UPD: the tile is first updated with one SGD step (W <- W - lr * G, written back to W_upd)
// and the updated values are pruned and compressed.
template <int DT, bool VEC, bool UPD>
__global__ void __launch_bounds__(128, 7) transposable_kernel(const typename Elem<DT>::T* W, int64_t rows,
                                                           int64_t cols, int64_t ld, typename Elem<DT>::T* W_out,
                                                           int64_t ld_out, uint32_t* __restrict__ mask_bits,
                                                           typename Elem<DT>::T* __restrict__ vals,
                                                           void* __restrict__ meta,
                                                           typename Elem<DT>::T* __restrict__ valsT,
                                                           void* __restrict__ metaT, int meta_tc,
                                                           const typename Elem<DT>::T* __restrict__ G, int64_t ld_g,
                                                           float nlr, typename Elem<DT>::T* W_upd) {
  using T = typename Elem<DT>::T;
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int tr = lane >> 3, tcol = lane & 7;
  const int64_t nbr = (rows + 15) / 16, nbc = (cols + 31) / 32;
  const int64_t nblocks = nbr * nbc;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t mw = (cols + 15) / 16, mwT = (rows + 15) / 16;
  const int64_t nslots = ((rows + 127) / 128) * 128, nslotsT = ((cols + 127) / 128) * 128;
  const int64_t mask_words = (cols + 31) / 32;
  for (int64_t blk = blockIdx.x * (int64_t)(blockDim.x / 32) + (threadIdx.x >> 5); blk < nblocks; blk += warps) {
    const int64_t br = blk / nbc, bc = blk - br * nbc;
    const int64_t R0 = br * 16 + tr * 4, C0 = bc * 32 + tcol * 4;
    const bool valid = R0 < rows && C0 < cols;
    T v[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (valid) {
        load4<VEC>(W + (R0 + r) * ld + C0, v[r]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) v[r][c] = (T)0;
      }
    }
    if constexpr (UPD) {
      if constexpr (DT != kI8) {
        if (valid) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            T g[4];
            load4<VEC>(G + (R0 + r) * ld_g + C0, g);
#pragma unroll
            for (int c = 0; c < 4; ++c) v[r][c] = sgd_elem<DT>(v[r][c], g[c], nlr);
            store4<VEC>(W_upd + (R0 + r) * ld + C0, v[r]);
          }
        }
      }
    }
    // the tile packed into 32-bit words (two 16-bit or four 8-bit elements each) while the
    // patterns are scored
    constexpr int kEB = 8 * (int)sizeof(T), kWords = (4 * kEB) / 32;
    uint32_t vw[4][kWords];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
#pragma unroll
      for (int w = 0; w < kWords; ++w) vw[r][w] = 0u;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        vw[r][(c * kEB) >> 5] |= (uint32_t)(sizeof(T) == 2 ? (uint32_t)(uint16_t)v[r][c] : (uint32_t)(uint8_t)v[r][c])
                                 << ((c * kEB) & 31);
    }
    auto elem = [&](int r, int c) -> T { return (T)(vw[r][(c * kEB) >> 5] >> ((c * kEB) & 31)); };
    float p[4][6];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float mg[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) mg[c] = tile_mag<DT>(v[r][c]);
      p[r][0] = mg[0] + mg[1];
      p[r][1] = mg[0] + mg[2];
      p[r][2] = mg[0] + mg[3];
      p[r][3] = mg[1] + mg[2];
      p[r][4] = mg[1] + mg[3];
      p[r][5] = mg[2] + mg[3];
    }
    // The first pattern in (a, b, c) order with the largest score: one chain per row-0 pair a
    // over its 15 patterns, then the chains in a order, each comparison keeping the earlier
    // pattern on equal scores.  Scores are never NaN (magnitudes are >= 0 or +Inf) and a valid
    // pattern scores >= 0.
    auto keep_first = [](float& s, uint32_t& m, float s2, uint32_t m2) {
      if (s2 > s) {
        s = s2;
        m = m2;
      }
    };
    float s_best = -1.0f;
    uint32_t m_best = 0u;
#pragma unroll
    for (int a = 0; a < 6; ++a) {
      float sa = -1.0f;
      uint32_t ma = 0u;
#pragma unroll
      for (int b = 0; b < 6; ++b) {
        const float s01 = p[0][a] + p[1][b];
#pragma unroll
        for (int c = 0; c < 6; ++c) {
          const int d = completion(a, b, c);
          if (d >= 0) keep_first(sa, ma, (s01 + p[2][c]) + p[3][d], tile_mask(a, b, c, d));
        }
      }
      keep_first(s_best, m_best, sa, ma);
    }
    uint32_t bmask = valid ? m_best : 0u;

    // ---- pruned copy
    if (W_out != nullptr && valid) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        T o[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) o[c] = ((bmask >> (4 * r + c)) & 1u) ? elem(r, c) : (T)0;
        store4<VEC>(W_out + (R0 + r) * ld_out + C0, o);
      }
    }
    // ---- mask bits: 8 lanes of a tile row form one 32-bit word per row
    if (mask_bits != nullptr) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        uint32_t w = ((bmask >> (4 * r)) & 0xFu) << (4 * tcol);
        w |= __shfl_xor_sync(0xFFFFFFFFu, w, 1);
        w |= __shfl_xor_sync(0xFFFFFFFFu, w, 2);
        w |= __shfl_xor_sync(0xFFFFFFFFu, w, 4);
        if (tcol == 0 && R0 < rows) mask_bits[(R0 + r) * mask_words + bc] = w;
      }
    }
    // ---- row-compressed W: per row two values and one 4-bit code
    if (vals != nullptr || meta != nullptr) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t km = (bmask >> (4 * r)) & 0xFu;
        const uint32_t i0 = (km & 1u) ? 0u : ((km & 2u) ? 1u : 2u);
        const uint32_t i1 = (km & 8u) ? 3u : ((km & 4u) ? 2u : 1u);
        if (vals != nullptr && valid) {
          store2<VEC>(vals + (R0 + r) * (cols / 2) + C0 / 2, (km & 1u) ? elem(r, 0) : ((km & 2u) ? elem(r, 1) : elem(r, 2)),
                      (km & 8u) ? elem(r, 3) : ((km & 4u) ? elem(r, 2) : elem(r, 1)));
        }
        if (meta != nullptr) {
          uint32_t code = valid ? (i0 | (i1 << 2)) << (4 * (tcol & 3)) : 0u;
          code |= __shfl_xor_sync(0xFFFFFFFFu, code, 1);
          code |= __shfl_xor_sync(0xFFFFFFFFu, code, 2);
          if ((tcol & 3) == 0 && valid) {
            const int64_t row = R0 + r, k = C0 / 16;
            if (meta_tc)
              tc_store(meta, row, k, nslots, code);
            else
              reinterpret_cast<uint16_t*>(meta)[row * mw + k] = (uint16_t)code;
          }
        }
      }
    }
    // ---- column-compressed (W^T): per tile column two values and one code
    if (valsT != nullptr || metaT != nullptr) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t km = ((bmask >> c) & 1u) | (((bmask >> (4 + c)) & 1u) << 1) | (((bmask >> (8 + c)) & 1u) << 2) |
                            (((bmask >> (12 + c)) & 1u) << 3);
        const uint32_t i0 = (km & 1u) ? 0u : ((km & 2u) ? 1u : 2u);
        const uint32_t i1 = (km & 8u) ? 3u : ((km & 4u) ? 2u : 1u);
        if (valsT != nullptr && valid) {
          store2<VEC>(valsT + (C0 + c) * (rows / 2) + R0 / 2, (km & 1u) ? elem(0, c) : ((km & 2u) ? elem(1, c) : elem(2, c)),
                      (km & 8u) ? elem(3, c) : ((km & 4u) ? elem(2, c) : elem(1, c)));
        }
        if (metaT != nullptr) {
          // four tile rows of the block share one 16-bit word: lanes tcol, tcol+8, tcol+16, tcol+24
          uint32_t code = valid ? (i0 | (i1 << 2)) << (4 * tr) : 0u;
          code |= __shfl_xor_sync(0xFFFFFFFFu, code, 8);
          code |= __shfl_xor_sync(0xFFFFFFFFu, code, 16);
          if (tr == 0 && C0 < cols) {
            const int64_t row = C0 + c, k = br;
            if (meta_tc)
              tc_store(metaT, row, k, nslotsT, code);
            else
              reinterpret_cast<uint16_t*>(metaT)[row * mwT + k] = (uint16_t)code;
          }
        }
      }
    }
  }
}

template <int DT>
cudaError_t transposable_dt(const TransposableLaunch& a, cudaStream_t s) {
  using T = typename Elem<DT>::T;
  if (a.meta_tc) {
    if (a.meta != nullptr) {
      const int64_t slots = tc_slots(a.rows);
      if (slots != a.rows) {
        cudaError_t e = cudaMemsetAsync(a.meta, 0x44, (size_t)((a.cols / 32) * slots * 4), s);
        if (e != cudaSuccess) return e;
      }
    }
    if (a.metaT != nullptr) {
      const int64_t slots = tc_slots(a.cols);
      if (slots != a.cols) {
        cudaError_t e = cudaMemsetAsync(a.metaT, 0x44, (size_t)((a.rows / 32) * slots * 4), s);
        if (e != cudaSuccess) return e;
      }
    }
  }
  const int64_t nblocks = ((a.rows + 15) / 16) * ((a.cols + 31) / 32);
  // 128-thread CTAs (four 16 x 32 blocks each) spread small matrices over every SM
  const unsigned grid = grid_for(nblocks * 32, 128);
  // Vector accesses need 4-element rows aligned (W, W_out) and 2-element pairs aligned (vals, valsT).
  const uintptr_t a4 = 4 * sizeof(T), a2 = 2 * sizeof(T);
  const bool vec = (reinterpret_cast<uintptr_t>(a.W) % a4) == 0 && a.ld % 4 == 0 &&
                   (a.W_out == nullptr || ((reinterpret_cast<uintptr_t>(a.W_out) % a4) == 0 && a.ld_out % 4 == 0)) &&
                   (reinterpret_cast<uintptr_t>(a.vals) % a2) == 0 && (reinterpret_cast<uintptr_t>(a.valsT) % a2) == 0;
  const T* W = static_cast<const T*>(a.W);
  T* W_out = static_cast<T*>(a.W_out);
  T* vals = static_cast<T*>(a.vals);
  T* valsT = static_cast<T*>(a.valsT);
  const T* G = static_cast<const T*>(a.grad);
  T* W_upd = static_cast<T*>(a.W_upd);
  const float nlr = -a.lr;
  if (G != nullptr) {
    const bool vecg = vec && (reinterpret_cast<uintptr_t>(G) % a4) == 0 && a.ld_grad % 4 == 0;
    if (vecg)
      return launch_pdl(transposable_kernel<DT, true, true>, dim3(grid), dim3(128), 0, s, W, a.rows, a.cols, a.ld,
                        W_out, a.ld_out, a.mask_bits, vals, a.meta, valsT, a.metaT, a.meta_tc, G, a.ld_grad, nlr,
                        W_upd);
    return launch_pdl(transposable_kernel<DT, false, true>, dim3(grid), dim3(128), 0, s, W, a.rows, a.cols, a.ld,
                      W_out, a.ld_out, a.mask_bits, vals, a.meta, valsT, a.metaT, a.meta_tc, G, a.ld_grad, nlr,
                      W_upd);
  }
  if (vec)
    return launch_pdl(transposable_kernel<DT, true, false>, dim3(grid), dim3(128), 0, s, W, a.rows, a.cols, a.ld,
                      W_out, a.ld_out, a.mask_bits, vals, a.meta, valsT, a.metaT, a.meta_tc, (const T*)nullptr,
                      (int64_t)0, 0.0f, (T*)nullptr);
  return launch_pdl(transposable_kernel<DT, false, false>, dim3(grid), dim3(128), 0, s, W, a.rows, a.cols, a.ld,
                    W_out, a.ld_out, a.mask_bits, vals, a.meta, valsT, a.metaT, a.meta_tc, (const T*)nullptr,
                    (int64_t)0, 0.0f, (T*)nullptr);
}

}  // namespace

cudaError_t launch_transposable(const TransposableLaunch& a, cudaStream_t s) {
  if (a.rows == 0 || a.cols == 0) return cudaSuccess;
  switch (a.dt) {
    case kF16: return transposable_dt<kF16>(a, s);
    case kBF16: return transposable_dt<kBF16>(a, s);
    default: return a.grad != nullptr ? cudaErrorInvalidValue : transposable_dt<kI8>(a, s);
  }
}

}  // namespace nmk
