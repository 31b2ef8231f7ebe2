// N:M greedy magnitude pruning, compression, decompression and pattern check.
//
// Selection rule (apex PR #1631 "[sparse] update support for arbitrary N:M
// settings sparse", extension 1, mn_1d_greedy): in every group of m
// consecutive elements of a row keep the n largest |w|; equal magnitudes go
// to the lower position; NaN ranks above every number.  Compression
// (cuSPARSELt blog, Figure 2 text) stores the kept values at n/m of the size
// plus position metadata.
//
// 2:4 kernels give each thread one 16-column segment of a row: four groups,
// one uint16 of canonical metadata (or one 16-bit half of a tensor-core
// metadata word), one 16-bit half of a mask word.  For aligned 16-bit data
// the segment is two 128-bit loads and the eight kept values one 128-bit
// store.  Other N:M shapes give each thread one group.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "nm_device.cuh"
#include "nm_internal.h"

namespace nmk {
namespace {

// Position of logical element (r, c) in the stored matrix.
template <bool TRANS>
__device__ __forceinline__ int64_t at(int64_t r, int64_t c, int64_t ld) {
  return TRANS ? c * ld + r : r * ld + c;
}

// Selects the two kept positions of a group of four keys (lower position wins
// ties) and returns the 4-bit keep mask.
__device__ __forceinline__ uint32_t keep2of4(uint32_t k0, uint32_t k1, uint32_t k2, uint32_t k3) {
  // cij (i < j): element i beats element j  <=>  k_i >= k_j
  const uint32_t c01 = k0 >= k1, c02 = k0 >= k2, c03 = k0 >= k3;
  const uint32_t c12 = k1 >= k2, c13 = k1 >= k3, c23 = k2 >= k3;
  const uint32_t r0 = (c01 ^ 1) + (c02 ^ 1) + (c03 ^ 1);
  const uint32_t r1 = c01 + (c12 ^ 1) + (c13 ^ 1);
  const uint32_t r2 = c02 + c12 + (c23 ^ 1);
  const uint32_t r3 = c03 + c13 + c23;
  return (uint32_t)(r0 < 2) | ((uint32_t)(r1 < 2) << 1) | ((uint32_t)(r2 < 2) << 2) | ((uint32_t)(r3 < 2) << 3);
}

template <int DT, bool VEC, bool TRANS>
__global__ void __launch_bounds__(256) prune24_kernel(const typename Elem<DT>::T* __restrict__ W, int64_t rowsL,
                                                      int64_t colsL, int64_t ld, typename Elem<DT>::T* W_out,
                                                      int64_t ld_out, uint32_t* __restrict__ mask_bits,
                                                      typename Elem<DT>::T* __restrict__ vals, void* __restrict__ meta,
                                                      int meta_tc) {
  using T = typename Elem<DT>::T;
  const int64_t segs = (colsL + 15) / 16;
  const int64_t total = rowsL * segs;
  const int64_t half_cols = colsL / 2;
  const int64_t mask_halves = ((colsL + 31) / 32) * 2;
  const int64_t nslots = ((rowsL + 127) / 128) * 128;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / segs;
    const int64_t k = idx - r * segs;
    const int64_t c0 = k * 16;
    const int ncol = (int)(colsL - c0 < 16 ? colsL - c0 : 16);
    T v[16];
    if constexpr (VEC) {
      const uint4* p = reinterpret_cast<const uint4*>(W + r * ld + c0);
      if constexpr (sizeof(T) == 2) {
        const uint4 a = __ldg(p), b = __ldg(p + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[2 * j] = (T)(w[j] & 0xFFFFu);
          v[2 * j + 1] = (T)(w[j] >> 16);
        }
      } else {
        const uint4 a = __ldg(p);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = (T)(int8_t)((w[j / 4] >> (8 * (j % 4))) & 0xFFu);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = (j < ncol) ? W[at<TRANS>(r, c0 + j, ld)] : (T)0;
    }
    uint32_t keep = 0, code = 0;
    T kv[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const T* e = v + 4 * g;
      const uint32_t km = keep2of4(Elem<DT>::key(e[0]), Elem<DT>::key(e[1]), Elem<DT>::key(e[2]), Elem<DT>::key(e[3]));
      const uint32_t kmask = (4 * g < ncol) ? km : 0u;
      const uint32_t i0 = (km & 1u) ? 0u : ((km & 2u) ? 1u : 2u);
      const uint32_t i1 = (km & 8u) ? 3u : ((km & 4u) ? 2u : 1u);
      kv[2 * g] = (4 * g < ncol) ? ((km & 1u) ? e[0] : ((km & 2u) ? e[1] : e[2])) : (T)0;
      kv[2 * g + 1] = (4 * g < ncol) ? ((km & 8u) ? e[3] : ((km & 4u) ? e[2] : e[1])) : (T)0;
      keep |= kmask << (4 * g);
      code |= ((4 * g < ncol) ? (i0 | (i1 << 2)) : 0u) << (4 * g);
    }
    if (vals != nullptr) {
      T* out = vals + r * half_cols + c0 / 2;
      if constexpr (VEC) {
        if constexpr (sizeof(T) == 2) {
          uint4 o;
          o.x = (uint32_t)kv[0] | ((uint32_t)kv[1] << 16);
          o.y = (uint32_t)kv[2] | ((uint32_t)kv[3] << 16);
          o.z = (uint32_t)kv[4] | ((uint32_t)kv[5] << 16);
          o.w = (uint32_t)kv[6] | ((uint32_t)kv[7] << 16);
          *reinterpret_cast<uint4*>(out) = o;
        } else {
          uint2 o;
          o.x = 0;
          o.y = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            o.x |= ((uint32_t)(uint8_t)kv[j]) << (8 * j);
            o.y |= ((uint32_t)(uint8_t)kv[4 + j]) << (8 * j);
          }
          *reinterpret_cast<uint2*>(out) = o;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (2 * j < ncol) out[j] = kv[j];
      }
    }
    if (meta != nullptr) {
      if (meta_tc) {
        tc_store(meta, r, k, nslots, code);
      } else {
        reinterpret_cast<uint16_t*>(meta)[r * segs + k] = (uint16_t)code;
      }
    }
    if constexpr (!TRANS) {
      if (mask_bits != nullptr) {
        uint16_t* mh = reinterpret_cast<uint16_t*>(mask_bits) + r * mask_halves;
        mh[k] = (uint16_t)keep;
        if (k == segs - 1 && (segs & 1)) mh[k + 1] = 0;  // unused upper half of the row's last word
      }
      if (W_out != nullptr) {
        T o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = ((keep >> j) & 1u) ? v[j] : (T)0;
        T* q = W_out + r * ld_out + c0;
        if constexpr (VEC) {
          if constexpr (sizeof(T) == 2) {
            uint4 a, b;
            a.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
            a.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
            a.z = (uint32_t)o[4] | ((uint32_t)o[5] << 16);
            a.w = (uint32_t)o[6] | ((uint32_t)o[7] << 16);
            b.x = (uint32_t)o[8] | ((uint32_t)o[9] << 16);
            b.y = (uint32_t)o[10] | ((uint32_t)o[11] << 16);
            b.z = (uint32_t)o[12] | ((uint32_t)o[13] << 16);
            b.w = (uint32_t)o[14] | ((uint32_t)o[15] << 16);
            reinterpret_cast<uint4*>(q)[0] = a;
            reinterpret_cast<uint4*>(q)[1] = b;
          } else {
            uint4 a;
            uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j / 4] |= ((uint32_t)(uint8_t)o[j]) << (8 * (j % 4));
            a.x = w[0];
            a.y = w[1];
            a.z = w[2];
            a.w = w[3];
            *reinterpret_cast<uint4*>(q) = a;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < ncol) q[j] = o[j];
        }
      }
    }
  }
}

// Positions of the two largest of four keys, lower position first on ties,
// as the 4-bit code i0 | i1 << 2.  Composite keys (key << 2 | (3 - position))
// are distinct and order exactly like the rule; the second largest of four is
// max(min of the two pair maxima, max of the two pair minima).
__device__ __forceinline__ uint32_t top2of4(uint32_t k0, uint32_t k1, uint32_t k2, uint32_t k3) {
  const uint32_t c0 = (k0 << 2) | 3u, c1 = (k1 << 2) | 2u, c2 = (k2 << 2) | 1u, c3 = k3 << 2;
  const uint32_t a = max(c0, c1), b = min(c0, c1), c = max(c2, c3), d = min(c2, c3);
  const uint32_t first = max(a, c), second = max(min(a, c), max(b, d));
  const uint32_t t = first & 3u, u = second & 3u;  // 3 - position
  return (max(t, u) | (min(t, u) << 2)) ^ 15u;
}
__device__ __forceinline__ uint32_t keep_of_code(uint32_t code) { return (1u << (code & 3u)) | (1u << (code >> 2)); }

template <int DT>
__device__ __forceinline__ uint32_t key_lo(uint32_t w) {
  return min(w & 0x7FFFu, DT == kF16 ? 0x7C01u : 0x7F81u);
}
template <int DT>
__device__ __forceinline__ uint32_t key_hi(uint32_t w) {
  return min((w >> 16) & 0x7FFFu, DT == kF16 ? 0x7C01u : 0x7F81u);
}
__device__ __forceinline__ uint32_t key_i8(uint32_t w, int b) {
  const int x = (int)(int8_t)(w >> (8 * b));
  return (uint32_t)(x < 0 ? -x : x);
}

// 2:4 for aligned rows whose length is a multiple of 32: one thread per 32
// columns (two segments), all loads of the pair issued before any selection,
// selection on packed words (one byte permute gathers a group's kept pair),
// one mask word and one 32-bit canonical metadata word per thread; the grid
// covers the matrix in a single pass.
template <int DT>
__global__ void __launch_bounds__(256) prune24_pair_kernel(const typename Elem<DT>::T* __restrict__ W, int64_t rows,
                                                           int64_t cols, int64_t ld, typename Elem<DT>::T* W_out,
                                                           int64_t ld_out, uint32_t* __restrict__ mask_bits,
                                                           typename Elem<DT>::T* __restrict__ vals,
                                                           void* __restrict__ meta, int meta_tc) {
  using T = typename Elem<DT>::T;
  constexpr bool k16 = sizeof(T) == 2;
  constexpr int kWords = k16 ? 16 : 8;  // 32-bit words of the thread's 32 elements
  const int64_t ppr = cols / 32;        // pairs of segments per row
  const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (idx >= rows * ppr) return;
  const int64_t r = idx / ppr, p = idx - r * ppr;
  const uint4* src = reinterpret_cast<const uint4*>(W + r * ld + p * 32);
  uint32_t w[kWords];
#pragma unroll
  for (int q = 0; q < kWords / 4; ++q) {
    const uint4 a = __ldcs(src + q);
    w[4 * q] = a.x, w[4 * q + 1] = a.y, w[4 * q + 2] = a.z, w[4 * q + 3] = a.w;
  }
  // eight groups of four
  uint32_t code = 0, keep = 0;
  uint32_t vw[k16 ? 8 : 4];  // kept values, packed
  uint32_t ow[kWords];       // pruned copy
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    uint32_t c, km;
    if constexpr (k16) {
      const uint32_t w0 = w[2 * g], w1 = w[2 * g + 1];
      c = top2of4(key_lo<DT>(w0), key_hi<DT>(w0), key_lo<DT>(w1), key_hi<DT>(w1));
      const uint32_t i0 = c & 3u, i1 = c >> 2;
      vw[g] = __byte_perm(w0, w1, (i0 * 0x22u + 0x10u) | ((i1 * 0x22u + 0x10u) << 8));
      km = keep_of_code(c);
      ow[2 * g] = w0 & ((km & 1u) * 0xFFFFu | (km & 2u) * 0x7FFF8000u);
      ow[2 * g + 1] = w1 & (((km >> 2) & 1u) * 0xFFFFu | ((km >> 2) & 2u) * 0x7FFF8000u);
    } else {
      const uint32_t w0 = w[g];
      c = top2of4(key_i8(w0, 0), key_i8(w0, 1), key_i8(w0, 2), key_i8(w0, 3));
      const uint32_t kv = __byte_perm(w0, 0u, (c & 3u) | ((c >> 2) << 4)) & 0xFFFFu;
      if (g % 2 == 0) vw[g / 2] = kv; else vw[g / 2] |= kv << 16;
      km = keep_of_code(c);
      ow[g] = w0 & ((km & 1u) * 0xFFu | (km & 2u) * 0x7F80u | (km & 4u) * 0x3FC000u | (km & 8u) * 0x1FE00000u);
    }
    code |= c << (4 * g);
    keep |= km << (4 * g);
  }
  if (W_out != nullptr) {
    uint4* dst = reinterpret_cast<uint4*>(W_out + r * ld_out + p * 32);
#pragma unroll
    for (int q = 0; q < kWords / 4; ++q) dst[q] = make_uint4(ow[4 * q], ow[4 * q + 1], ow[4 * q + 2], ow[4 * q + 3]);
  }
  if (vals != nullptr) {
    uint4* vo = reinterpret_cast<uint4*>(vals + r * (cols / 2) + p * 16);
#pragma unroll
    for (int q = 0; q < (k16 ? 2 : 1); ++q) vo[q] = make_uint4(vw[4 * q], vw[4 * q + 1], vw[4 * q + 2], vw[4 * q + 3]);
  }
  if (meta != nullptr) {
    if (meta_tc) {
      const int64_t nslots = ((rows + 127) / 128) * 128;
      tc_store(meta, r, 2 * p, nslots, code & 0xFFFFu);
      tc_store(meta, r, 2 * p + 1, nslots, code >> 16);
    } else {
      reinterpret_cast<uint32_t*>(meta)[r * ppr + p] = code;
    }
  }
  if (mask_bits != nullptr) mask_bits[r * ppr + p] = keep;
}

// 2:4 for 16-bit rows stored back to back (ld == cols, cols % 32 == 0): the
// matrix is read as one array of 16-byte words, lane-contiguous, so every warp
// access covers 512 consecutive bytes; a word holds two groups and yields 8
// bytes of kept values, one byte of canonical metadata (the two 16-bit halves
// of a tensor-core metadata word come from a lane and its neighbour) and one
// byte of the mask.  Every warp of a resident grid takes an equal share of
// the words (a multiple of 32), four words per lane in flight.
constexpr int kLaneWords = 4;
struct LaneSplit {
  unsigned grid;
  int64_t per;  // words per warp
};
inline LaneSplit lane_split(int64_t words, int ctas_per_sm = 5) {
  LaneSplit s;
  int64_t g = (int64_t)num_sms_cached() * ctas_per_sm;  // up to five 256-thread CTAs per SM are resident
  const int64_t need = (words + 255) / 256;
  if (need < g) g = need;
  if (g < 1) g = 1;
  s.grid = (unsigned)g;
  const int64_t warps = g * 8;
  s.per = ((words + warps - 1) / warps + 31) / 32 * 32;
  return s;
}

template <int DT>
__global__ void __launch_bounds__(256, 5) prune24_lanes_kernel(const uint4* __restrict__ W, int64_t rows, int64_t cols,
                                                               int64_t per, uint4* W_out, uint8_t* __restrict__ mask_bytes,
                                                               uint2* __restrict__ vals, void* __restrict__ meta,
                                                               int meta_tc) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t n16 = rows * cols / 8;
  const int64_t lo = ((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5) * per;
  const int64_t hi = lo + per < n16 ? lo + per : n16;
  const int64_t nslots = ((rows + 127) / 128) * 128;
  for (int64_t base = lo; base < hi; base += 32 * kLaneWords) {
    uint4 x[kLaneWords];
#pragma unroll
    for (int u = 0; u < kLaneWords; ++u) {
      const int64_t i = base + u * 32 + lane;
      x[u] = i < hi ? __ldcs(W + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kLaneWords; ++u) {
      const int64_t i = base + u * 32 + lane;
      const uint32_t w0 = x[u].x, w1 = x[u].y, w2 = x[u].z, w3 = x[u].w;
      const uint32_t c0 = top2of4(key_lo<DT>(w0), key_hi<DT>(w0), key_lo<DT>(w1), key_hi<DT>(w1));
      const uint32_t c1 = top2of4(key_lo<DT>(w2), key_hi<DT>(w2), key_lo<DT>(w3), key_hi<DT>(w3));
      const uint32_t code = c0 | (c1 << 4);
      if (meta != nullptr && meta_tc) {  // uniform: the even lane of each pair stores 16 columns' code
        const uint32_t code_hi = __shfl_down_sync(0xFFFFFFFFu, code, 1);
        if (i < hi && (lane & 1) == 0) {
          const int64_t e = i * 8, r = e / cols;
          tc_store(meta, r, (e - r * cols) / 16, nslots, code | (code_hi << 8));
        }
      }
      if (i < hi) {
        if (vals != nullptr)
          vals[i] = make_uint2(__byte_perm(w0, w1, ((c0 & 3u) * 0x22u + 0x10u) | (((c0 >> 2) * 0x22u + 0x10u) << 8)),
                               __byte_perm(w2, w3, ((c1 & 3u) * 0x22u + 0x10u) | (((c1 >> 2) * 0x22u + 0x10u) << 8)));
        if (meta != nullptr && !meta_tc) static_cast<uint8_t*>(meta)[i] = (uint8_t)code;
        if (W_out != nullptr || mask_bytes != nullptr) {
          const uint32_t k0 = keep_of_code(c0), k1 = keep_of_code(c1);
          if (W_out != nullptr)
            W_out[i] = make_uint4(w0 & ((k0 & 1u) * 0xFFFFu | (k0 & 2u) * 0x7FFF8000u),
                                  w1 & (((k0 >> 2) & 1u) * 0xFFFFu | ((k0 >> 2) & 2u) * 0x7FFF8000u),
                                  w2 & ((k1 & 1u) * 0xFFFFu | (k1 & 2u) * 0x7FFF8000u),
                                  w3 & (((k1 >> 2) & 1u) * 0xFFFFu | ((k1 >> 2) & 2u) * 0x7FFF8000u));
          if (mask_bytes != nullptr) mask_bytes[i] = (uint8_t)(k0 | (k1 << 4));
        }
      }
    }
  }
}

// General n:m (m <= 32), one thread per group.  Composite keys (key << 5 |
// (31 - position)) are all distinct; an element is kept when fewer than n
// composite keys of its group exceed its own.
template <int DT, bool TRANS>
__global__ void __launch_bounds__(256) prune_nm_kernel(const typename Elem<DT>::T* __restrict__ W, int64_t rowsL,
                                                       int64_t colsL, int64_t ld, int n, int m,
                                                       typename Elem<DT>::T* W_out, int64_t ld_out,
                                                       uint32_t* __restrict__ mask_bits,
                                                       typename Elem<DT>::T* __restrict__ vals,
                                                       uint8_t* __restrict__ meta) {
  using T = typename Elem<DT>::T;
  const int64_t gpr = colsL / m;
  const int64_t total = rowsL * gpr;
  const int64_t words = (colsL + 31) / 32;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / gpr;
    const int64_t g = idx - r * gpr;
    const int64_t c0 = g * m;
    T v[32];
    uint32_t ck[32];
    for (int j = 0; j < m; ++j) {
      v[j] = W[at<TRANS>(r, c0 + j, ld)];
      ck[j] = (Elem<DT>::key(v[j]) << 5) | (uint32_t)(31 - j);
    }
    uint32_t keep = 0;
    for (int j = 0; j < m; ++j) {
      int rank = 0;
      for (int i = 0; i < m; ++i) rank += ck[i] > ck[j];
      if (rank < n) keep |= 1u << j;
    }
    if (vals != nullptr || meta != nullptr) {
      int o = 0;
      const int64_t base = r * gpr * n + g * n;
      for (int j = 0; j < m; ++j) {
        if ((keep >> j) & 1u) {
          if (vals != nullptr) vals[base + o] = v[j];
          if (meta != nullptr) meta[base + o] = (uint8_t)j;
          ++o;
        }
      }
    }
    if constexpr (!TRANS) {
      if (W_out != nullptr) {
        for (int j = 0; j < m; ++j) W_out[r * ld_out + c0 + j] = ((keep >> j) & 1u) ? v[j] : (T)0;
      }
      if (mask_bits != nullptr && keep != 0u) {  // buffer was zeroed by the launcher
        const int64_t w0 = c0 / 32;
        const int sh = (int)(c0 % 32);
        atomicOr(mask_bits + r * words + w0, keep << sh);
        if (sh + m > 32) atomicOr(mask_bits + r * words + w0 + 1, keep >> (32 - sh));
      }
    }
  }
}

// n:32 for 16-bit types (apex PR #1631: "Normally we set M = 32"), one thread
// per group, aligned rows.  The sign-cleared bit patterns of f16/bf16 order
// exactly like the magnitudes when compared as half/bfloat16 values (for groups
// without NaN), so the n-th largest key T is found with packed (two elements
// per instruction) min/max: a sorting network orders the 16 keys of each
// half-stream (even and odd positions) at once (for n = 4 a selection network
// that keeps only the 4 largest), and T is the n-th largest of the two sorted
// lists' union (about 4x fewer instructions than a 15-step
// bisection over packed compare counts).  The kept set is every key > T plus
// the lowest-position keys == T.  Kept values are
// gathered through a padded shared-memory copy of the group.  Groups holding a
// NaN take an exact scalar path (composite keys), so NaN still ranks first.
template <int DT> struct Pair;
template <> struct Pair<kF16> {
  using T2 = __half2;
  static constexpr uint32_t kInf = 0x7C00u;
  __device__ __forceinline__ static T2 as(uint32_t w) { return *reinterpret_cast<const __half2*>(&w); }
  __device__ __forceinline__ static uint32_t bits(T2 v) { return *reinterpret_cast<const uint32_t*>(&v); }
};
template <> struct Pair<kBF16> {
  using T2 = __nv_bfloat162;
  static constexpr uint32_t kInf = 0x7F80u;
  __device__ __forceinline__ static T2 as(uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); }
  __device__ __forceinline__ static uint32_t bits(T2 v) { return *reinterpret_cast<const uint32_t*>(&v); }
};

// Batcher's odd-even merge sort of 16 elements: 63 compare-exchanges, built at compile time.
struct CmpX {
  int a, b;
};
struct Batcher16 {
  CmpX c[63];
};
__host__ __device__ constexpr Batcher16 make_batcher16() {
  Batcher16 r{};
  int n = 0;
  for (int p = 1; p < 16; p <<= 1)
    for (int k = p; k >= 1; k >>= 1)
      for (int j = k % p; j + k < 16; j += 2 * k)
        for (int i = 0; i < k && i < 16 - j - k; ++i)
          if ((i + j) / (2 * p) == (i + j + k) / (2 * p)) r.c[n++] = CmpX{i + j, i + j + k};
  return r;
}
// Sorts 16 packed pairs descending in each half (two elements per compare-exchange).
template <typename T2>
__device__ __forceinline__ void sort16_desc(T2 (&t)[16]) {
  constexpr Batcher16 kNet = make_batcher16();
#pragma unroll
  for (int q = 0; q < 63; ++q) {
    const T2 a = t[kNet.c[q].a], b = t[kNet.c[q].b];
    t[kNet.c[q].a] = __hmax2(a, b);
    t[kNet.c[q].b] = __hmin2(a, b);
  }
}

// The 4 largest of 16 packed pairs, sorted descending in each half, into t[0..3]: each group of
// four sorted (5 compare-exchanges), then pairs of sorted fours merged by taking
// max(a[i], b[3 - i]) (the top four, in bitonic order) and a 4-element bitonic sort.
template <typename T2>
__device__ __forceinline__ void cmpx_desc(T2& a, T2& b) {
  const T2 hi = __hmax2(a, b), lo = __hmin2(a, b);
  a = hi;
  b = lo;
}
template <typename T2>
__device__ __forceinline__ void top4_desc(T2 (&t)[16]) {
#pragma unroll
  for (int o = 0; o < 16; o += 4) {
    cmpx_desc(t[o], t[o + 1]);
    cmpx_desc(t[o + 2], t[o + 3]);
    cmpx_desc(t[o], t[o + 2]);
    cmpx_desc(t[o + 1], t[o + 3]);
    cmpx_desc(t[o + 1], t[o + 2]);
  }
  auto merge = [&](int oa, int ob) {
    T2 m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = __hmax2(t[oa + i], t[ob + 3 - i]);
    cmpx_desc(m[0], m[2]);
    cmpx_desc(m[1], m[3]);
    cmpx_desc(m[0], m[1]);
    cmpx_desc(m[2], m[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) t[oa + i] = m[i];
  };
  merge(0, 4);
  merge(8, 12);
  merge(0, 8);
}

template <int DT, int N>
__global__ void __launch_bounds__(128) prune32_kernel(const uint16_t* __restrict__ W, int64_t rows, int64_t cols,
                                                      int64_t ld, uint16_t* W_out, int64_t ld_out,
                                                      uint32_t* __restrict__ mask_bits, uint16_t* __restrict__ vals,
                                                      uint8_t* __restrict__ meta) {
  pdl_trigger();
  pdl_wait();
  using P = Pair<DT>;
  __shared__ uint4 srow4[128][5];  // the thread's group (64 B) at an 80-byte pitch: conflict-free
  const int64_t gpr = cols / 32;
  const int64_t total = rows * gpr;
  uint4* mine = srow4[threadIdx.x];
  const uint16_t* mine16 = reinterpret_cast<const uint16_t*>(mine);
  if (total == 0) return;
  // row and group of gidx, stepped with the grid stride (one 64-bit division per thread)
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t g_first = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t dr = stride / gpr, dg = stride - dr * gpr;
  int64_t r = g_first / gpr, gi = g_first - r * gpr;
  for (int64_t gidx = g_first; gidx < total; gidx += stride, r += dr, gi += dg) {
    if (gi >= gpr) {
      gi -= gpr;
      ++r;
    }
    const uint4* src = reinterpret_cast<const uint4*>(W + r * ld + gi * 32);
    uint32_t w[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 q = __ldg(src + c);
      mine[c] = q;
      w[4 * c] = q.x;
      w[4 * c + 1] = q.y;
      w[4 * c + 2] = q.z;
      w[4 * c + 3] = q.w;
    }
    // sign-cleared keys; a half holds a NaN iff key > kInf, i.e. iff key + (0x7FFF - kInf) sets
    // its bit 15 (the sum stays below 0x10000, so no carry reaches the other half)
    uint32_t k[16];
    uint32_t nan_bits = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      k[i] = w[i] & 0x7FFF7FFFu;
      nan_bits |= k[i] + (0x7FFFu - P::kInf) * 0x00010001u;
    }
    const bool nan = (nan_bits & 0x80008000u) != 0u;
    uint32_t kept = 0;
    if (!nan) {
      // t[0] >= t[1] >= ... in each half: the keys of the half-stream of even positions (low
      // halves) and of odd positions (high halves), sorted
      typename P::T2 t[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) t[i] = P::as(k[i]);
      if constexpr (N == 4)
        top4_desc(t);  // only the 4 largest are needed
      else
        sort16_desc(t);
      static_assert(N >= 1 && N <= 16, "n of 32");
      // the N-th largest of the union of the two sorted lists A (low halves) and B (high
      // halves): the largest of B[N-1], A[N-1] and min(A[i-1], B[N-1-i]) for 0 < i < N
      auto lo = [&](int j) { return P::bits(t[j]) & 0xFFFFu; };
      auto hi = [&](int j) { return P::bits(t[j]) >> 16; };
      uint32_t T = max(lo(N - 1), hi(N - 1));
#pragma unroll
      for (int i = 1; i < N; ++i) T = max(T, min(lo(i - 1), hi(N - 1 - i)));
      uint32_t gtm = 0, eqm = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t lo = k[i] & 0xFFFFu, hi = k[i] >> 16;
        gtm |= ((uint32_t)(lo > T) | ((uint32_t)(hi > T) << 1)) << (2 * i);
        eqm |= ((uint32_t)(lo == T) | ((uint32_t)(hi == T) << 1)) << (2 * i);
      }
      kept = gtm;
      const int need = N - __popc(gtm);
      for (int j = 0; j < need; ++j) {  // lowest positions among the ties
        kept |= eqm & (0u - eqm);
        eqm &= eqm - 1u;
      }
    } else {
      // exact path: composite keys (key << 5 | (31 - position)), NaN above everything
#pragma unroll 1
      for (int e = 0; e < 32; ++e) {
        const uint32_t ke = (min((uint32_t)mine16[e] & 0x7FFFu, P::kInf + 1u) << 5) | (uint32_t)(31 - e);
        int rank = 0;
#pragma unroll 1
        for (int f = 0; f < 32; ++f)
          rank += ((min((uint32_t)mine16[f] & 0x7FFFu, P::kInf + 1u) << 5) | (uint32_t)(31 - f)) > ke;
        if (rank < N) kept |= 1u << e;
      }
    }
    // compressed values and positions, ascending position order
    uint32_t ov[N / 2], oi[N / 4];
    uint32_t rem = kept;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const uint32_t pos = (uint32_t)(__ffs(rem) - 1);
      rem &= rem - 1u;
      const uint32_t val = mine16[pos];
      if (j % 2 == 0) ov[j / 2] = val; else ov[j / 2] |= val << 16;
      if (j % 4 == 0) oi[j / 4] = pos; else oi[j / 4] |= pos << (8 * (j % 4));
    }
    if (vals != nullptr) {
      uint16_t* vo = vals + gidx * N;
      if constexpr (N == 4) {
        *reinterpret_cast<uint2*>(vo) = make_uint2(ov[0], ov[1]);
      } else {
#pragma unroll
        for (int c = 0; c < N / 8; ++c)
          reinterpret_cast<uint4*>(vo)[c] = make_uint4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
      }
    }
    if (meta != nullptr) {
      uint8_t* mo = meta + gidx * N;
      if constexpr (N == 4) {
        *reinterpret_cast<uint32_t*>(mo) = oi[0];
      } else if constexpr (N == 8) {
        *reinterpret_cast<uint2*>(mo) = make_uint2(oi[0], oi[1]);
      } else {
        *reinterpret_cast<uint4*>(mo) = make_uint4(oi[0], oi[1], oi[2], oi[3]);
      }
    }
    if (mask_bits != nullptr) mask_bits[r * gpr + gi] = kept;
    if (W_out != nullptr) {
      uint4* dst = reinterpret_cast<uint4*>(W_out + r * ld_out + gi * 32);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int e = 8 * c + 2 * t;
          const uint32_t m2 = ((kept >> e) & 1u ? 0x0000FFFFu : 0u) | ((kept >> (e + 1)) & 1u ? 0xFFFF0000u : 0u);
          o[t] = w[4 * c + t] & m2;
        }
        dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// ---- decompression -------------------------------------------------------
template <int DT, bool VEC>
__global__ void __launch_bounds__(256) decompress24_kernel(const typename Elem<DT>::T* __restrict__ vals,
                                                           const void* __restrict__ meta, int64_t rows, int64_t cols,
                                                           int meta_tc, typename Elem<DT>::T* __restrict__ W_out,
                                                           int64_t ld_out) {
  using T = typename Elem<DT>::T;
  const int64_t segs = (cols + 15) / 16;
  const int64_t total = rows * segs;
  const int64_t nslots = ((rows + 127) / 128) * 128;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / segs;
    const int64_t k = idx - r * segs;
    const int64_t c0 = k * 16;
    const int ncol = (int)(cols - c0 < 16 ? cols - c0 : 16);
    const uint32_t code = meta_tc ? *reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(meta) +
                                                                      tc_half_offset(r, k, nslots))
                                  : reinterpret_cast<const uint16_t*>(meta)[r * segs + k];
    T kv[8];
    const T* in = vals + r * (cols / 2) + c0 / 2;
#pragma unroll
    for (int j = 0; j < 8; ++j) kv[j] = (2 * j < ncol) ? in[j] : (T)0;
    T o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = (T)0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t c = (code >> (4 * g)) & 0xFu;
      const uint32_t i0 = c & 3u, i1 = c >> 2;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (t == (int)i0) o[4 * g + t] = kv[2 * g];
        if (t == (int)i1) o[4 * g + t] = kv[2 * g + 1];
      }
    }
    T* q = W_out + r * ld_out + c0;
    if constexpr (VEC && sizeof(T) == 2) {
      uint4 a, b;
      a.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
      a.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
      a.z = (uint32_t)o[4] | ((uint32_t)o[5] << 16);
      a.w = (uint32_t)o[6] | ((uint32_t)o[7] << 16);
      b.x = (uint32_t)o[8] | ((uint32_t)o[9] << 16);
      b.y = (uint32_t)o[10] | ((uint32_t)o[11] << 16);
      b.z = (uint32_t)o[12] | ((uint32_t)o[13] << 16);
      b.w = (uint32_t)o[14] | ((uint32_t)o[15] << 16);
      reinterpret_cast<uint4*>(q)[0] = a;
      reinterpret_cast<uint4*>(q)[1] = b;
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < ncol) q[j] = o[j];
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(256) decompress_nm_kernel(const typename Elem<DT>::T* __restrict__ vals,
                                                            const uint8_t* __restrict__ meta, int64_t rows,
                                                            int64_t cols, int n, int m,
                                                            typename Elem<DT>::T* __restrict__ W_out, int64_t ld_out) {
  using T = typename Elem<DT>::T;
  const int64_t gpr = cols / m;
  const int64_t total = rows * gpr;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / gpr;
    const int64_t g = idx - r * gpr;
    T* q = W_out + r * ld_out + g * m;
    for (int j = 0; j < m; ++j) q[j] = (T)0;
    const int64_t base = r * gpr * n + g * n;
    for (int t = 0; t < n; ++t) {
      const int p = meta[base + t];
      if (p < m) q[p] = vals[base + t];
    }
  }
}

// ---- pattern check ---------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(256) check_kernel(const typename Elem<DT>::T* __restrict__ W, int64_t rows,
                                                    int64_t cols, int64_t ld, int n, int m, int transposable,
                                                    int32_t* __restrict__ d_violations) {
  const int64_t gpr = cols / m;
  const int64_t row_groups = rows * gpr;
  const int64_t col_groups = transposable ? (rows / 4) * cols : 0;
  int count = 0;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < row_groups + col_groups;
       idx += (int64_t)gridDim.x * blockDim.x) {
    int nz = 0;
    if (idx < row_groups) {
      const int64_t r = idx / gpr;
      const int64_t c0 = (idx - r * gpr) * m;
      for (int j = 0; j < m; ++j) nz += Elem<DT>::nonzero(W[r * ld + c0 + j]);
      count += nz > n;
    } else {
      const int64_t t = idx - row_groups;
      const int64_t rg = t / cols;
      const int64_t c = t - rg * cols;
      for (int j = 0; j < 4; ++j) nz += Elem<DT>::nonzero(W[(4 * rg + j) * ld + c]);
      count += nz > 2;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) count += __shfl_xor_sync(0xFFFFFFFFu, count, off);
  if ((threadIdx.x & 31) == 0 && count) atomicAdd(d_violations, count);
}

// 2:4 check of 16-bit rows in one pass over strips of four rows: a thread reads the
// same 16-byte word (eight columns) of the strip's four rows, counts the two row
// groups of each and, for the transposable check, every column of the strip.
// Nonzero bits: (w & 0x7FFF7FFF) + 0x7FFF7FFF carries into bit 15 / 31 exactly for
// a half that is not +-0 (no carry crosses the halves).
__device__ __forceinline__ uint32_t nz8(const uint4 x) {
  auto h = [](uint32_t w) { return ((w & 0x7FFF7FFFu) + 0x7FFF7FFFu) & 0x80008000u; };
  const uint32_t a = h(x.x), b = h(x.y), c = h(x.z), d = h(x.w);
  return ((a >> 15) & 1u) | ((a >> 30) & 2u) | ((b >> 13) & 4u) | ((b >> 28) & 8u) | ((c >> 11) & 16u) |
         ((c >> 26) & 32u) | ((d >> 9) & 64u) | ((d >> 24) & 128u);
}
// The check's counter set to zero in the launch chain (a memset node would end the chain of
// dependent launches before the check).
__global__ void zero_count_kernel(int32_t* __restrict__ d_violations) {
  pdl_trigger();
  pdl_wait();
  *d_violations = 0;
}

// U items per lane and pass: a warp's `per` items go out in one pass when per <= 32 U.
template <int U>
__global__ void __launch_bounds__(256) check24_strips_kernel(const uint4* __restrict__ W, int64_t rows, int64_t wpr,
                                                             int64_t ldw, int transposable, int64_t per,
                                                             int32_t* __restrict__ d_violations) {
  pdl_trigger();
  pdl_wait();
  // every warp takes `per` consecutive items (strip, word), U per lane in flight
  const int lane = threadIdx.x & 31;
  const int64_t total = ((rows + 3) / 4) * wpr;
  const int64_t lo = ((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5) * per;
  const int64_t hi = lo + per < total ? lo + per : total;
  int count = 0;  // a warp with no items (lo >= hi) skips the loop and adds 0
  // strip and word of the lane's U items, stepped by 32 U items per pass (a 64-bit
  // division per item had cost more issue slots than the check itself)
  int64_t st[U], wd[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t idx = lo + 32 * u + lane;
    st[u] = idx / wpr;
    wd[u] = idx - st[u] * wpr;
  }
  for (int64_t base = lo; base < hi; base += 32 * U) {
    uint32_t m[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t idx = base + 32 * u + lane;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t r = 4 * st[u] + j;
        m[u][j] = (idx < hi && r < rows) ? nz8(__ldcs(W + r * ldw + wd[u])) : 0u;
      }
      wd[u] += 32 * U;
      if (wd[u] >= wpr) {
        if (wpr >= 32 * U) {
          wd[u] -= wpr;
          ++st[u];
        } else {
          st[u] += wd[u] / wpr;
          wd[u] %= wpr;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int j = 0; j < 4; ++j) count += (__popc(m[u][j] & 0xFu) > 2) + (__popc(m[u][j] >> 4) > 2);
      if (transposable)  // columns with at least three of the strip's four entries nonzero
        count += __popc((m[u][0] & m[u][1] & (m[u][2] | m[u][3])) | ((m[u][0] | m[u][1]) & m[u][2] & m[u][3]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) count += __shfl_xor_sync(0xFFFFFFFFu, count, off);
  // one atomic per CTA: thousands of same-address atomics, one per warp, had serialised at
  // the counter when most groups violate
  __shared__ int warp_count[8];
  if (lane == 0) warp_count[threadIdx.x >> 5] = count;
  __syncthreads();
  if (threadIdx.x == 0) {
    int total_count = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) total_count += warp_count[w];
    if (total_count) atomicAdd(d_violations, total_count);
  }
}

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte-permute selectors that scatter a group's kept pair back to its four
// positions: for code i0 | i1 << 2, output element t takes the first kept
// value if t == i0, the second if t == i1, zero otherwise.  16-bit elements:
// two selectors (elements 0-1, 2-3) in one word; int8: one selector.
__host__ __device__ constexpr uint32_t scatter_nibble16(uint32_t code, int t) {
  return (uint32_t)t == (code & 3u) ? 0x10u : ((uint32_t)t == (code >> 2) ? 0x32u : 0x44u);
}
__host__ __device__ constexpr uint32_t scatter_sel16(uint32_t code) {
  return scatter_nibble16(code, 0) | (scatter_nibble16(code, 1) << 8) | (scatter_nibble16(code, 2) << 16) |
         (scatter_nibble16(code, 3) << 24);
}
__host__ __device__ constexpr uint32_t scatter_sel8(uint32_t code) {
  uint32_t sel = 0;
  for (int t = 0; t < 4; ++t)
    sel |= ((uint32_t)t == (code & 3u) ? 0u : ((uint32_t)t == (code >> 2) ? 1u : 4u)) << (4 * t);
  return sel;
}

// 2:4 for 16-bit rows with tensor-core metadata: one CTA per 16-row x 512-column
// tile.  The selection runs as in the lane kernel (thread (r, g) takes words
// g, g + 16, g + 32, g + 48 of tile row r, so each row is read in 256-byte runs)
// and leaves each word's code byte in shared memory; then each thread writes one
// whole metadata word, the two rows 8 apart that share it, so a k-step's 16 slot
// words are one 64-byte run.  Slots of rows past the matrix get the valid code 0x4.
template <int DT>
__global__ void __launch_bounds__(256) prune24_tc_tile_kernel(const uint4* __restrict__ W, int64_t rows, int64_t cols,
                                                              int64_t ldw, uint4* W_out, int64_t ldw_out,
                                                              uint8_t* __restrict__ mask_bytes,
                                                              uint2* __restrict__ vals, uint32_t* __restrict__ meta) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint8_t codes[16][64];
  const int64_t wpr = cols / 8;  // 16-byte words per row
  const int64_t tiles_c = (wpr + 63) / 64, tiles = ((rows + 15) / 16) * tiles_c;
  const int64_t nslots = ((rows + 127) / 128) * 128;
  const int tr = threadIdx.x >> 4, g = threadIdx.x & 15;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t row0 = (tile / tiles_c) * 16, w0 = (tile % tiles_c) * 64;
    const int64_t r = row0 + tr;
    uint4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t w = w0 + g + 16 * u;
      x[u] = (r < rows && w < wpr) ? __ldcs(W + r * ldw + w) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t w = w0 + g + 16 * u;
      const uint32_t w0_ = x[u].x, w1 = x[u].y, w2 = x[u].z, w3 = x[u].w;
      const uint32_t c0 = top2of4(key_lo<DT>(w0_), key_hi<DT>(w0_), key_lo<DT>(w1), key_hi<DT>(w1));
      const uint32_t c1 = top2of4(key_lo<DT>(w2), key_hi<DT>(w2), key_lo<DT>(w3), key_hi<DT>(w3));
      codes[tr][g + 16 * u] = (uint8_t)(r < rows ? (c0 | (c1 << 4)) : 0x44u);
      if (r < rows && w < wpr) {
        const int64_t i = r * wpr + w;  // index in the packed values and mask
        if (vals != nullptr)
          vals[i] = make_uint2(
              __byte_perm(w0_, w1, ((c0 & 3u) * 0x22u + 0x10u) | (((c0 >> 2) * 0x22u + 0x10u) << 8)),
              __byte_perm(w2, w3, ((c1 & 3u) * 0x22u + 0x10u) | (((c1 >> 2) * 0x22u + 0x10u) << 8)));
        if (W_out != nullptr || mask_bytes != nullptr) {
          const uint32_t k0 = keep_of_code(c0), k1 = keep_of_code(c1);
          if (W_out != nullptr)
            W_out[r * ldw_out + w] = make_uint4(w0_ & ((k0 & 1u) * 0xFFFFu | (k0 & 2u) * 0x7FFF8000u),
                                                w1 & (((k0 >> 2) & 1u) * 0xFFFFu | ((k0 >> 2) & 2u) * 0x7FFF8000u),
                                                w2 & ((k1 & 1u) * 0xFFFFu | (k1 & 2u) * 0x7FFF8000u),
                                                w3 & (((k1 >> 2) & 1u) * 0xFFFFu | ((k1 >> 2) & 2u) * 0x7FFF8000u));
          if (mask_bytes != nullptr) mask_bytes[i] = (uint8_t)(k0 | (k1 << 4));
        }
      }
    }
    __syncthreads();
    if (meta != nullptr) {
      // word (k-step j, slot si): rows si & 7 (low half) and (si & 7) + 8 (high half) of the
      // tile, 16-column segment 2 j + (si >> 3), i.e. code bytes of words 2 seg and 2 seg + 1
      const int j = threadIdx.x >> 4, si = threadIdx.x & 15;
      const int64_t kstep = w0 / 4 + j;
      if (kstep < wpr / 4) {
        const int lo_r = si & 7, seg = 2 * j + (si >> 3);
        const uint32_t word = codes[lo_r][2 * seg] | ((uint32_t)codes[lo_r][2 * seg + 1] << 8) |
                              ((uint32_t)codes[lo_r + 8][2 * seg] << 16) |
                              ((uint32_t)codes[lo_r + 8][2 * seg + 1] << 24);
        meta[kstep * nslots + row0 + si] = word;
      }
    }
    __syncthreads();
  }
}

// Decompression in the same lane-contiguous order and split: 8 bytes of kept
// values and a canonical metadata byte per 16-byte output word.
template <int DT>
__global__ void __launch_bounds__(256, 5) decompress24_lanes_kernel(const uint2* __restrict__ vals,
                                                                    const uint8_t* __restrict__ meta, int64_t n16,
                                                                    int64_t per, uint4* __restrict__ W_out) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t lo = ((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5) * per;
  const int64_t hi = lo + per < n16 ? lo + per : n16;
  for (int64_t base = lo; base < hi; base += 32 * kLaneWords) {
    uint2 v[kLaneWords];
    uint32_t code[kLaneWords];
#pragma unroll
    for (int u = 0; u < kLaneWords; ++u) {
      const int64_t i = base + u * 32 + lane;
      v[u] = i < hi ? __ldcs(vals + i) : make_uint2(0u, 0u);
      code[u] = i < hi ? (uint32_t)__ldcs(meta + i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kLaneWords; ++u) {
      const int64_t i = base + u * 32 + lane;
      if (i >= hi) continue;
      const uint32_t s0 = scatter_sel16(code[u] & 0xFu), s1 = scatter_sel16((code[u] >> 4) & 0xFu);
      W_out[i] = make_uint4(__byte_perm(v[u].x, 0u, s0 & 0xFFFFu), __byte_perm(v[u].x, 0u, s0 >> 16),
                            __byte_perm(v[u].y, 0u, s1 & 0xFFFFu), __byte_perm(v[u].y, 0u, s1 >> 16));
    }
  }
}

// Decompression with tensor-core metadata in the prune kernel's 16 x 512 tiles: each
// thread reads one whole metadata word (a k-step's 16 slot words are one 64-byte
// run) and leaves its four code bytes in shared memory, then thread (r, g) expands
// words g, g + 16, g + 32, g + 48 of tile row r.
template <int DT>
__global__ void __launch_bounds__(256) decompress24_tc_tile_kernel(const uint2* __restrict__ vals,
                                                                   const uint32_t* __restrict__ meta, int64_t rows,
                                                                   int64_t cols, uint4* __restrict__ W_out,
                                                                   int64_t ldw_out) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint8_t codes[16][64];
  const int64_t wpr = cols / 8;
  const int64_t tiles_c = (wpr + 63) / 64, tiles = ((rows + 15) / 16) * tiles_c;
  const int64_t nslots = ((rows + 127) / 128) * 128;
  const int tr = threadIdx.x >> 4, g = threadIdx.x & 15;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t row0 = (tile / tiles_c) * 16, w0 = (tile % tiles_c) * 64;
    {
      const int j = threadIdx.x >> 4, si = threadIdx.x & 15;
      const int64_t kstep = w0 / 4 + j;
      if (kstep < wpr / 4) {
        const uint32_t word = __ldcs(meta + kstep * nslots + row0 + si);
        const int lo_r = si & 7, seg = 2 * j + (si >> 3);
        codes[lo_r][2 * seg] = (uint8_t)word;
        codes[lo_r][2 * seg + 1] = (uint8_t)(word >> 8);
        codes[lo_r + 8][2 * seg] = (uint8_t)(word >> 16);
        codes[lo_r + 8][2 * seg + 1] = (uint8_t)(word >> 24);
      }
    }
    __syncthreads();
    const int64_t r = row0 + tr;
    uint2 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t w = w0 + g + 16 * u;
      v[u] = (r < rows && w < wpr) ? __ldcs(vals + r * wpr + w) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t w = w0 + g + 16 * u;
      if (r >= rows || w >= wpr) continue;
      const uint32_t c = codes[tr][g + 16 * u];
      const uint32_t s0 = scatter_sel16(c & 0xFu), s1 = scatter_sel16((c >> 4) & 0xFu);
      W_out[r * ldw_out + w] = make_uint4(__byte_perm(v[u].x, 0u, s0 & 0xFFFFu), __byte_perm(v[u].x, 0u, s0 >> 16),
                                          __byte_perm(v[u].y, 0u, s1 & 0xFFFFu), __byte_perm(v[u].y, 0u, s1 >> 16));
    }
    __syncthreads();
  }
}

// Decompression for aligned rows whose length is a multiple of 32: one thread
// per 32 columns; the kept values and codes are loaded as words, each group's
// four outputs come from byte permutes with a selector looked up by its code.
template <int DT>
__global__ void __launch_bounds__(256) decompress24_pair_kernel(const typename Elem<DT>::T* __restrict__ vals,
                                                                const void* __restrict__ meta, int64_t rows,
                                                                int64_t cols, int meta_tc,
                                                                typename Elem<DT>::T* __restrict__ W_out,
                                                                int64_t ld_out) {
  using T = typename Elem<DT>::T;
  constexpr bool k16 = sizeof(T) == 2;
  __shared__ uint32_t sel[16];
  if (threadIdx.x < 16) sel[threadIdx.x] = k16 ? scatter_sel16(threadIdx.x) : scatter_sel8(threadIdx.x);
  __syncthreads();
  const int64_t ppr = cols / 32;
  const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (idx >= rows * ppr) return;
  const int64_t r = idx / ppr, p = idx - r * ppr;
  uint32_t code;
  if (meta_tc) {
    const int64_t nslots = ((rows + 127) / 128) * 128;
    const char* mb = reinterpret_cast<const char*>(meta);
    code = *reinterpret_cast<const uint16_t*>(mb + tc_half_offset(r, 2 * p, nslots)) |
           ((uint32_t)*reinterpret_cast<const uint16_t*>(mb + tc_half_offset(r, 2 * p + 1, nslots)) << 16);
  } else {
    code = __ldcs(reinterpret_cast<const uint32_t*>(meta) + r * ppr + p);
  }
  const uint4* vin = reinterpret_cast<const uint4*>(vals + r * (cols / 2) + p * 16);
  uint32_t kw[k16 ? 8 : 4];
#pragma unroll
  for (int q = 0; q < (k16 ? 2 : 1); ++q) {
    const uint4 a = __ldcs(vin + q);
    kw[4 * q] = a.x, kw[4 * q + 1] = a.y, kw[4 * q + 2] = a.z, kw[4 * q + 3] = a.w;
  }
  uint32_t ow[k16 ? 16 : 8];
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint32_t sg = sel[(code >> (4 * g)) & 0xFu];
    if constexpr (k16) {
      ow[2 * g] = __byte_perm(kw[g], 0u, sg & 0xFFFFu);
      ow[2 * g + 1] = __byte_perm(kw[g], 0u, sg >> 16);
    } else {
      ow[g] = __byte_perm(kw[g / 2] >> (16 * (g % 2)), 0u, sg);
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(W_out + r * ld_out + p * 32);
#pragma unroll
  for (int q = 0; q < (k16 ? 4 : 2); ++q) dst[q] = make_uint4(ow[4 * q], ow[4 * q + 1], ow[4 * q + 2], ow[4 * q + 3]);
}

template <int DT>
cudaError_t prune_dt(const PruneLaunch& a, cudaStream_t s) {
  using T = typename Elem<DT>::T;
  const int threads = 256;
  const T* W = static_cast<const T*>(a.W);
  T* W_out = static_cast<T*>(a.W_out);
  T* vals = static_cast<T*>(a.vals);
  if (a.n == 2 && a.m == 4) {
    const int64_t segs = (a.colsL + 15) / 16;
    const unsigned grid = grid_for(a.rowsL * segs, threads);
    if (a.meta != nullptr && a.meta_tc) {
      // slot rows of rows past the matrix hold the valid code 0x4 (positions 0 and 1)
      const int64_t slots = tc_slots(a.rowsL);
      if (slots != a.rowsL) {
        cudaError_t e = cudaMemsetAsync(a.meta, 0x44, (size_t)((a.colsL / 32) * slots * 4), s);
        if (e != cudaSuccess) return e;
      }
    }
    const int64_t es = (int64_t)sizeof(T);
    const bool vec = !a.trans && (a.colsL % 16 == 0) && (a.ld * es) % 16 == 0 && aligned16(W) &&
                     (W_out == nullptr || ((a.ld_out * es) % 16 == 0 && aligned16(W_out))) && aligned16(vals);
    const bool lanes = sizeof(T) == 2 && vec && a.colsL % 32 == 0 && a.ld == a.colsL &&
                       (W_out == nullptr || a.ld_out == a.colsL);
    if (lanes && a.meta != nullptr && a.meta_tc) {
      if constexpr (sizeof(T) == 2) {
        const int64_t tiles = ((a.rowsL + 15) / 16) * ((a.colsL / 8 + 63) / 64);
        const unsigned g = (unsigned)std::min<int64_t>(tiles, (int64_t)num_sms_cached() * 8);
        if (cudaError_t e = launch_pdl(prune24_tc_tile_kernel<DT>, dim3(g), dim3(256), 0, s,
                                       reinterpret_cast<const uint4*>(W), a.rowsL, a.colsL, a.ld / 8,
                                       reinterpret_cast<uint4*>(W_out), a.ld_out / 8,
                                       reinterpret_cast<uint8_t*>(a.mask_bits), reinterpret_cast<uint2*>(vals),
                                       static_cast<uint32_t*>(a.meta)))
          return e;
      }
    } else if (lanes) {
      if constexpr (sizeof(T) == 2) {
        const LaneSplit ls = lane_split(a.rowsL * a.colsL / 8);
        if (cudaError_t e = launch_pdl(prune24_lanes_kernel<DT>, dim3(ls.grid), dim3(256), 0, s,
                                       reinterpret_cast<const uint4*>(W), a.rowsL, a.colsL, ls.per,
                                       reinterpret_cast<uint4*>(W_out), reinterpret_cast<uint8_t*>(a.mask_bits),
                                       reinterpret_cast<uint2*>(vals), a.meta, a.meta_tc))
          return e;
      }
    } else if (vec && a.colsL % 32 == 0) {
      const int64_t pairs = a.rowsL * (a.colsL / 32);
      prune24_pair_kernel<DT><<<(unsigned)((pairs + threads - 1) / threads), threads, 0, s>>>(
          W, a.rowsL, a.colsL, a.ld, W_out, a.ld_out, a.mask_bits, vals, a.meta, a.meta_tc);
    } else if (vec)
      prune24_kernel<DT, true, false><<<grid, threads, 0, s>>>(W, a.rowsL, a.colsL, a.ld, W_out, a.ld_out,
                                                                a.mask_bits, vals, a.meta, a.meta_tc);
    else if (!a.trans)
      prune24_kernel<DT, false, false><<<grid, threads, 0, s>>>(W, a.rowsL, a.colsL, a.ld, W_out, a.ld_out,
                                                                 a.mask_bits, vals, a.meta, a.meta_tc);
    else
      prune24_kernel<DT, false, true><<<grid, threads, 0, s>>>(W, a.rowsL, a.colsL, a.ld, nullptr, 0, nullptr,
                                                                vals, a.meta, a.meta_tc);
    return cudaGetLastError();
  }
  if constexpr (sizeof(T) == 2) {
    const bool fast = !a.trans && a.m == 32 && (a.n == 4 || a.n == 8 || a.n == 16) && (a.ld % 8) == 0 &&
                      aligned16(W) && (W_out == nullptr || ((a.ld_out % 8) == 0 && aligned16(W_out))) &&
                      aligned16(vals) && aligned16(a.meta);
    if (fast) {
      const unsigned grid = grid_for(a.rowsL * (a.colsL / 32), 128, 16);
      const uint16_t* W16 = reinterpret_cast<const uint16_t*>(W);
      uint16_t* Wo16 = reinterpret_cast<uint16_t*>(W_out);
      uint16_t* v16 = reinterpret_cast<uint16_t*>(vals);
      uint8_t* m8 = static_cast<uint8_t*>(a.meta);
      cudaError_t e_;
      if (a.n == 4)
        e_ = launch_pdl(prune32_kernel<DT, 4>, dim3(grid), dim3(128), 0, s, W16, a.rowsL, a.colsL, a.ld, Wo16, a.ld_out,
                        a.mask_bits, v16, m8);
      else if (a.n == 8)
        e_ = launch_pdl(prune32_kernel<DT, 8>, dim3(grid), dim3(128), 0, s, W16, a.rowsL, a.colsL, a.ld, Wo16, a.ld_out,
                        a.mask_bits, v16, m8);
      else
        e_ = launch_pdl(prune32_kernel<DT, 16>, dim3(grid), dim3(128), 0, s, W16, a.rowsL, a.colsL, a.ld, Wo16,
                        a.ld_out, a.mask_bits, v16, m8);
      return e_;
    }
  }
  if (a.mask_bits != nullptr && !a.trans) {
    const size_t bytes = (size_t)a.rowsL * (size_t)((a.colsL + 31) / 32) * 4;
    cudaError_t e = cudaMemsetAsync(a.mask_bits, 0, bytes, s);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = grid_for(a.rowsL * (a.colsL / a.m), threads);
  uint8_t* meta = static_cast<uint8_t*>(a.meta);
  if (!a.trans)
    prune_nm_kernel<DT, false><<<grid, threads, 0, s>>>(W, a.rowsL, a.colsL, a.ld, a.n, a.m, W_out, a.ld_out,
                                                         a.mask_bits, vals, meta);
  else
    prune_nm_kernel<DT, true><<<grid, threads, 0, s>>>(W, a.rowsL, a.colsL, a.ld, a.n, a.m, nullptr, 0, nullptr,
                                                        vals, meta);
  return cudaGetLastError();
}

template <int DT>
cudaError_t decompress_dt(const DecompressLaunch& a, cudaStream_t s) {
  using T = typename Elem<DT>::T;
  const int threads = 256;
  const T* vals = static_cast<const T*>(a.vals);
  T* W_out = static_cast<T*>(a.W_out);
  if (a.n == 2 && a.m == 4) {
    const int64_t segs = (a.cols + 15) / 16;
    const unsigned grid = grid_for(a.rows * segs, threads);
    const bool vec = sizeof(T) == 2 && a.cols % 16 == 0 && (a.ld_out * 2) % 16 == 0 && aligned16(W_out);
    const bool pair = a.cols % 32 == 0 && (a.ld_out * (int64_t)sizeof(T)) % 16 == 0 && aligned16(W_out) &&
                      aligned16(vals) && (a.meta_tc || (reinterpret_cast<uintptr_t>(a.meta) & 3u) == 0);
    // lane order for canonical metadata; tensor-core metadata is stored by row slots, which
    // the one-thread-per-32-columns kernel reads with fewer scattered accesses
    if (pair && sizeof(T) == 2 && a.ld_out == a.cols && !a.meta_tc) {
      if constexpr (sizeof(T) == 2) {
        const LaneSplit ls = lane_split(a.rows * a.cols / 8);
        if (cudaError_t e = launch_pdl(decompress24_lanes_kernel<DT>, dim3(ls.grid), dim3(256), 0, s,
                                       reinterpret_cast<const uint2*>(vals), static_cast<const uint8_t*>(a.meta),
                                       a.rows * a.cols / 8, ls.per, reinterpret_cast<uint4*>(W_out)))
          return e;
      }
    } else if (pair && sizeof(T) == 2 && a.meta_tc && (reinterpret_cast<uintptr_t>(a.meta) & 3u) == 0) {
      if constexpr (sizeof(T) == 2) {
        const int64_t tiles = ((a.rows + 15) / 16) * ((a.cols / 8 + 63) / 64);
        const unsigned g = (unsigned)std::min<int64_t>(tiles, (int64_t)num_sms_cached() * 8);
        if (cudaError_t e = launch_pdl(decompress24_tc_tile_kernel<DT>, dim3(g), dim3(256), 0, s,
                                       reinterpret_cast<const uint2*>(vals), static_cast<const uint32_t*>(a.meta),
                                       a.rows, a.cols, reinterpret_cast<uint4*>(W_out), a.ld_out / 8))
          return e;
      }
    } else if (pair) {
      const int64_t pairs = a.rows * (a.cols / 32);
      decompress24_pair_kernel<DT><<<(unsigned)((pairs + threads - 1) / threads), threads, 0, s>>>(
          vals, a.meta, a.rows, a.cols, a.meta_tc, W_out, a.ld_out);
    } else if (vec)
      decompress24_kernel<DT, true><<<grid, threads, 0, s>>>(vals, a.meta, a.rows, a.cols, a.meta_tc, W_out, a.ld_out);
    else
      decompress24_kernel<DT, false><<<grid, threads, 0, s>>>(vals, a.meta, a.rows, a.cols, a.meta_tc, W_out,
                                                              a.ld_out);
  } else {
    const unsigned grid = grid_for(a.rows * (a.cols / a.m), threads);
    decompress_nm_kernel<DT><<<grid, threads, 0, s>>>(vals, static_cast<const uint8_t*>(a.meta), a.rows, a.cols, a.n,
                                                      a.m, W_out, a.ld_out);
  }
  return cudaGetLastError();
}

template <int DT>
cudaError_t check_dt(const void* W, int64_t rows, int64_t cols, int64_t ld, int n, int m, int transposable,
                     int32_t* d_violations, cudaStream_t s) {
  using T = typename Elem<DT>::T;
  cudaError_t e = launch_pdl(zero_count_kernel, dim3(1), dim3(32), 0, s, d_violations);
  if (e != cudaSuccess) return e;
  const int64_t work = rows * (cols / m) + (transposable ? (rows / 4) * cols : 0);
  if (work == 0) return cudaSuccess;
  if (sizeof(T) == 2 && n == 2 && m == 4 && cols % 8 == 0 && ld % 8 == 0 && aligned16(W) &&
      (!transposable || rows % 4 == 0)) {
    const int64_t wpr = cols / 8;
    const LaneSplit ls = lane_split(((rows + 3) / 4) * wpr);
    // one pass per warp when its share is at most 96 items (12 loads of 16 bytes per lane in
    // flight), else passes of 64
    const uint4* W4 = static_cast<const uint4*>(W);
    cudaError_t e_;
    if (ls.per <= 32)
      e_ = launch_pdl(check24_strips_kernel<1>, dim3(ls.grid), dim3(256), 0, s, W4, rows, wpr, ld / 8, transposable,
                      ls.per, d_violations);
    else if (ls.per <= 96)
      e_ = launch_pdl(check24_strips_kernel<3>, dim3(ls.grid), dim3(256), 0, s, W4, rows, wpr, ld / 8, transposable,
                      ls.per, d_violations);
    else
      e_ = launch_pdl(check24_strips_kernel<2>, dim3(ls.grid), dim3(256), 0, s, W4, rows, wpr, ld / 8, transposable,
                      ls.per, d_violations);
    return e_;
  }
  check_kernel<DT><<<grid_for(work, 256), 256, 0, s>>>(static_cast<const T*>(W), rows, cols, ld, n, m, transposable,
                                                       d_violations);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prune(const PruneLaunch& a, cudaStream_t s) {
  if (a.rowsL == 0 || a.colsL == 0) return cudaSuccess;
  switch (a.dt) {
    case kF16: return prune_dt<kF16>(a, s);
    case kBF16: return prune_dt<kBF16>(a, s);
    default: return prune_dt<kI8>(a, s);
  }
}

cudaError_t launch_decompress(const DecompressLaunch& a, cudaStream_t s) {
  if (a.rows == 0 || a.cols == 0) return cudaSuccess;
  switch (a.dt) {
    case kF16: return decompress_dt<kF16>(a, s);
    case kBF16: return decompress_dt<kBF16>(a, s);
    default: return decompress_dt<kI8>(a, s);
  }
}

cudaError_t launch_check(int dt, const void* W, int64_t rows, int64_t cols, int64_t ld, int n, int m,
                         int transposable, int32_t* d_violations, cudaStream_t s) {
  switch (dt) {
    case kF16: return check_dt<kF16>(W, rows, cols, ld, n, m, transposable, d_violations, s);
    case kBF16: return check_dt<kBF16>(W, rows, cols, ld, n, m, transposable, d_violations, s);
    default: return check_dt<kI8>(W, rows, cols, ld, n, m, transposable, d_violations, s);
  }
}

}  // namespace nmk
