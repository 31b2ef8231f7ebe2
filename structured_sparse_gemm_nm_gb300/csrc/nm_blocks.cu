// Vector-wise (1 x 32) and block-wise (32 x 32) pruning and the product over
// the kept units (apex PR #1631 "[sparse] update support for arbitrary N:M
// settings sparse", extension 2: unstructured vector-wise and block-wise
// masks).
//
// Selection keeps the `keep` units (1 x 32 vectors or 32 x 32 blocks) with the
// largest score; equal scores go to the lower unit index (row-major order).
// Scores are exact integers: an f16 value is a whole number of 2^-24 units
// below 2^40, so the score of a unit of at most 1024 elements is an integer
// below 2^51 (int8: below 2^18).  A unit's 64-bit key orders it: 0 for a NaN
// score, score + 1 for a finite score, 2^62 for an infinite one.
//
// Four launches, none of which waits on another CTA:
//   1. score      key of every unit and a histogram of a log-scale bucket of
//                 the key (64 buckets per octave); the last CTA to finish
//                 finds the bucket holding the keep-th largest key.
//   2. candidates the keys of that bucket are gathered; the last CTA finds the
//                 exact threshold key T by a radix search over them.
//   3. count      per chunk of 256 units: keys above T and keys equal to T,
//                 as prefixes within groups of 8 chunks plus group totals;
//                 the last CTA turns the group totals into exclusive prefixes.
//   4. write      kept flag and output position of every unit, then the CSR
//                 arrays, the packed values, the bit mask and the pruned copy.
// A unit is kept if its key is above T, or equal to T and among the first
// `need_eq` such units in index order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstring>

#include "nm_device.cuh"
#include "nm_internal.h"

namespace nmk {
namespace {

constexpr int kUnitW = 32;         // unit width (columns) of both kinds
constexpr int kBins = 4096;        // log-scale buckets
constexpr int kChunk = 256;        // units per CTA in the count and write kernels
constexpr int kCountChunks = 8;    // chunks per CTA of the count kernel (one group)
constexpr uint64_t kKeyInf = 1ull << 62;

struct Ctl {
  uint32_t ticket[3];
  uint32_t cand_count;
  int32_t bucket;  // bucket to refine, or -1 when T is already final
  uint32_t pad;
  uint64_t k_rem;    // keys still to take inside `bucket`
  uint64_t T;        // threshold key
  uint64_t need_eq;  // keys equal to T that are kept
};

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t hist, ctl, keys, cand, cnt_gt, cnt_eq, total;
};
// cnt_gt / cnt_eq: one entry per chunk (the prefix within its group) followed by one
// per group of kCountChunks chunks (the group's prefix).
constexpr WsLayout ws_layout(int64_t units) {
  const int64_t chunks = (units + kChunk - 1) / kChunk;
  const int64_t groups = (chunks + kCountChunks - 1) / kCountChunks;
  WsLayout w{};
  w.hist = 0;
  w.ctl = align256(kBins * 4);
  w.keys = w.ctl + align256(sizeof(Ctl));
  w.cand = w.keys + align256((size_t)units * 8);
  w.cnt_gt = w.cand + align256((size_t)units * 8);
  w.cnt_eq = w.cnt_gt + align256((size_t)(chunks + groups) * 4);
  w.total = w.cnt_eq + align256((size_t)(chunks + groups) * 4);
  return w;
}

// ---------------------------------------------------------------- scoring
// Exact scores: the sum of a unit's elements (SIGNED) or of their magnitudes, in units
// of 2^-24 for f16.
//
// f16, in fp32 on the FMA pipe: an f16 x converts exactly; adding and then subtracting
// C = 1.5 * 2^20 rounds it to hi, the nearest multiple of 2^-3 (x + C stays inside
// [2^20, 2^21), whose spacing is 2^-3), and lo = x - hi is exact, a multiple of 2^-24
// of magnitude at most 2^-4.  The hi parts of up to 32 elements sum exactly in fp32
// (below 32 * 65504 * 8 < 2^24 units of 2^-3); the lo parts of one 8-element segment
// sum exactly (within 2^23 units of 2^-24) and go to a 32-bit integer sum.  The score
// is hi_sum * 2^21 + lo_int.  (The integer form of the same split, shift-and-add per
// element, spent twice the issue slots on the half-rate integer pipe.)  An Inf or NaN
// makes hi_sum non-finite; seg_flags then classifies the unit.
//
// int8: a dp4a with ones sums four elements; for magnitudes each byte is multiplied by
// its sign (+1 or -1 per byte, no carry between bytes).
struct ScoreAcc {
  float hs = 0.f;   // f16: exact sum of the hi parts (at most 32 elements)
  int32_t li = 0;   // f16: sum of the lo parts in units of 2^-24; int8: the sum itself
};

template <int DT, bool SIGNED>
__device__ __forceinline__ void acc_seg(const uint4 v, ScoreAcc& a) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (DT == kF16) {
    constexpr float C = 1572864.0f;  // 1.5 * 2^20
    float ls = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 hh;
      memcpy(&hh, &w[i], 4);
      const float2 f2 = __half22float2(hh);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float x = SIGNED ? (j ? f2.y : f2.x) : fabsf(j ? f2.y : f2.x);
        const float hi = __fsub_rn(__fadd_rn(x, C), C);
        a.hs = __fadd_rn(a.hs, hi);
        ls = __fadd_rn(ls, __fsub_rn(x, hi));
      }
    }
    a.li += __float2int_rn(ls * 16777216.0f);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (SIGNED) {
        a.li = __dp4a((int)w[i], 0x01010101, a.li);
      } else {
        const uint32_t neg = (w[i] >> 7) & 0x01010101u;  // 1 in each negative byte
        a.li = __dp4a((int)w[i], (int)(0x01010101u + neg * 0xFEu), a.li);
      }
    }
  }
}

// The accumulated score; `special` is set when an f16 Inf or NaN took part.
template <int DT>
__device__ __forceinline__ int64_t acc_value(const ScoreAcc& a, bool& special) {
  if constexpr (DT == kF16) {
    special = !(fabsf(a.hs) <= 3.0e38f);
    return (int64_t)__float2int_rn(a.hs * 8.0f) * (1 << 21) + a.li;
  } else {
    special = false;
    return a.li;
  }
}

// Flags of the f16 specials in a segment: 1 NaN, 2 +Inf, 4 -Inf.
__device__ __forceinline__ uint32_t seg_flags(const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t fl = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t h = (i & 1) ? w[i >> 1] >> 16 : w[i >> 1] & 0xFFFFu;
    if ((h & 0x7C00u) == 0x7C00u) fl |= (h & 0x3FFu) ? 1u : ((h & 0x8000u) ? 4u : 2u);
  }
  return fl;
}

template <bool SIGNED>
__device__ __forceinline__ uint64_t make_key(int64_t x, uint32_t fl) {
  if (SIGNED) {
    if ((fl & 1u) || (fl & 6u) == 6u) return 0;
    if (fl) return kKeyInf;
    return (uint64_t)(x < 0 ? -x : x) + 1;
  }
  if (fl & 1u) return 0;
  if (fl) return kKeyInf;
  return (uint64_t)x + 1;
}

// Monotone log-scale bucket: keys below 128 are their own bucket; above, the
// leading bit position and the next 6 bits.
__device__ __forceinline__ int key_bucket(uint64_t k) {
  if (k < 64) return (int)k;
  const int lead = 63 - __clzll((long long)k);  // >= 6
  return (lead - 5) * 64 + (int)((k >> (lead - 6)) & 63);
}

__device__ __forceinline__ int64_t shfl_xor64(int64_t v, int m) {
  const int lo = __shfl_xor_sync(0xFFFFFFFFu, (int)(uint32_t)(uint64_t)v, m);
  const int hi = __shfl_xor_sync(0xFFFFFFFFu, (int)(uint32_t)((uint64_t)v >> 32), m);
  return (int64_t)(((uint64_t)(uint32_t)hi << 32) | (uint32_t)lo);
}

// True in every thread of the CTA that finished last; its writes and those of
// all other CTAs are visible to it afterwards (threadfence + ticket pattern).
__device__ __forceinline__ bool last_cta(uint32_t* ticket) {
  __shared__ bool is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (is_last) __threadfence();
  return is_last;
}

// Inclusive prefix sum over the 256 threads of a CTA (one value each, thread order);
// `total` receives the sum over the CTA.  Every thread must call it.
template <typename T>
__device__ __forceinline__ T cta_inclusive_scan256(T v, T& total) {
  __shared__ T wsum[8];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T u = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) wsum[w] = v;
  __syncthreads();
  T add = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    add += i < w ? wsum[i] : T(0);
    tot += wsum[i];
  }
  __syncthreads();  // wsum is free again on return
  total = tot;
  return v + add;
}

// Run by the last score CTA: the bucket that holds the keep-th largest key.  Thread t
// holds 16 bins, highest bins first over t; a prefix sum over the threads finds the one
// whose bins hold the keep-th key, and that thread walks its bins.
__device__ void select_bucket(const uint32_t* hist, Ctl* ctl, uint64_t keep) {
  constexpr int per = kBins / 256;
  const int top = kBins - per * (int)threadIdx.x;  // bins [top - per, top)
  uint32_t c[per];
  unsigned long long sum = 0, total;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    c[j] = __ldcg(hist + top - 1 - j);
    sum += c[j];
  }
  const unsigned long long incl = cta_inclusive_scan256<unsigned long long>(sum, total);
  const unsigned long long excl = incl - sum;
  if (keep == 0) {
    if (threadIdx.x == 0) {
      ctl->bucket = -1;
      ctl->T = ~0ull;
      ctl->need_eq = 0;
    }
    return;
  }
  if (!(excl < keep && keep <= incl)) return;  // exactly one thread goes on (keep <= units)
  uint64_t above = excl, k_rem = 0;
  int b = -1;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    if (b < 0) {
      if (above + c[j] >= keep) {
        b = top - 1 - j;
        k_rem = keep - above;
      } else {
        above += c[j];
      }
    }
  }
  if (b < 128) {  // a single key value
    ctl->bucket = -1;
    ctl->T = (uint64_t)b;
    ctl->need_eq = k_rem;
  } else {
    ctl->bucket = b;
    ctl->k_rem = k_rem;
  }
}

// Vector-wise keys: a thread scores whole vectors (64 or 32 bytes, loaded as 16-byte
// segments), two at a time; no cross-lane reduction.
template <int DT, bool SIGNED>
__global__ void __launch_bounds__(256) vw_score_kernel(const uint8_t* __restrict__ W, int64_t rows, int64_t cols,
                                                       int64_t ld_bytes, uint64_t* __restrict__ keys,
                                                       uint32_t* __restrict__ hist, Ctl* ctl, uint64_t keep) {
  pdl_trigger();
  pdl_wait();
  constexpr int kSegElems = DT == kF16 ? 8 : 16;
  constexpr int kSpv = kUnitW / kSegElems;  // segments per vector: 4 (f16) or 2 (int8)
  constexpr int kVecBytes = kSpv * 16;
  constexpr int kVecs = 2;  // vectors in flight per thread
  __shared__ uint32_t sh[kBins];
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const int64_t vpr = cols / kUnitW;  // vectors per row
  const int64_t units = rows * vpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // Row and column of the thread's next vector, stepped by `stride` (one division per
  // thread, not one per vector).
  const int64_t u_first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t r = u_first / vpr, c = u_first - r * vpr;
  const int64_t dr = stride / vpr, dc = stride - dr * vpr;
  for (int64_t u0 = (int64_t)blockIdx.x * blockDim.x; u0 < units; u0 += kVecs * stride) {
    uint4 v[kVecs][kSpv];
    bool ok[kVecs];
#pragma unroll
    for (int j = 0; j < kVecs; ++j) {
      ok[j] = u0 + j * stride + threadIdx.x < units;
      const uint4* p = reinterpret_cast<const uint4*>(W + r * ld_bytes + c * kVecBytes);
#pragma unroll
      for (int q = 0; q < kSpv; ++q) v[j][q] = ok[j] ? __ldcs(p + q) : make_uint4(0, 0, 0, 0);
      c += dc;
      r += dr;
      if (c >= vpr) {
        c -= vpr;
        ++r;
      }
    }
#pragma unroll
    for (int j = 0; j < kVecs; ++j) {
      ScoreAcc a;
#pragma unroll
      for (int q = 0; q < kSpv; ++q) acc_seg<DT, SIGNED>(v[j][q], a);
      bool sp;
      const int64_t x = acc_value<DT>(a, sp);
      uint32_t fl = 0;
      if (sp) {  // an Inf or NaN in the vector (rare)
#pragma unroll
        for (int q = 0; q < kSpv; ++q) fl |= seg_flags(v[j][q]);
      }
      if (ok[j]) {
        const uint64_t key = make_key<SIGNED>(x, fl);
        keys[u0 + j * stride + threadIdx.x] = key;
        atomicAdd(&sh[key_bucket(key)], 1u);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (sh[i]) atomicAdd(hist + i, sh[i]);
  if (last_cta(&ctl->ticket[0])) select_bucket(hist, ctl, keep);
}

// Block-wise keys: a warp scores one 32 x 32 block (sum of |w|).
template <int DT>
__global__ void __launch_bounds__(256) bw_score_kernel(const uint8_t* __restrict__ W, int64_t rows, int64_t cols,
                                                       int64_t ld_bytes, uint64_t* __restrict__ keys,
                                                       uint32_t* __restrict__ hist, Ctl* ctl, uint64_t keep) {
  pdl_trigger();
  pdl_wait();
  constexpr int kSegElems = DT == kF16 ? 8 : 16;
  constexpr int kSpr = kUnitW / kSegElems;  // segments per block row: 4 or 2
  constexpr int kRowsPer = 32 / kSpr;       // block rows per warp load: 8 or 16
  constexpr int es = DT == kF16 ? 2 : 1;
  __shared__ uint32_t sh[kBins];
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const int64_t bn = cols / kUnitW, units = (rows / 32) * bn;
  const int lane = threadIdx.x & 31;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += wstride) {
    const int64_t bi = u / bn, bj = u - bi * bn;
    const uint8_t* base = W + (bi * 32 + lane / kSpr) * ld_bytes + (bj * kUnitW + (lane % kSpr) * kSegElems) * es;
    uint4 v[32 / kRowsPer];
#pragma unroll
    for (int p = 0; p < 32 / kRowsPer; ++p) v[p] = __ldcs(reinterpret_cast<const uint4*>(base + p * kRowsPer * ld_bytes));
    ScoreAcc acc;  // a lane's 32 elements (f16) or 32 int8 elements
#pragma unroll
    for (int p = 0; p < 32 / kRowsPer; ++p) acc_seg<DT, false>(v[p], acc);
    bool sp;
    int64_t a = acc_value<DT>(acc, sp);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) a += shfl_xor64(a, m);
    uint32_t fl = 0;
    if (__any_sync(0xFFFFFFFFu, sp)) {  // an Inf or NaN in the block (rare)
#pragma unroll
      for (int p = 0; p < 32 / kRowsPer; ++p) fl |= seg_flags(v[p]);
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, m);
    }
    if (lane == 0) {
      const uint64_t key = make_key<false>(a, fl);
      keys[u] = key;
      atomicAdd(&sh[key_bucket(key)], 1u);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (sh[i]) atomicAdd(hist + i, sh[i]);
  if (last_cta(&ctl->ticket[0])) select_bucket(hist, ctl, keep);
}

// ---------------------------------------------------------------- threshold
__global__ void __launch_bounds__(256) candidates_kernel(const uint64_t* __restrict__ keys, int64_t units, Ctl* ctl,
                                                         uint64_t* __restrict__ cand) {
  pdl_trigger();
  pdl_wait();
  const int B = ctl->bucket;
  if (B < 0) return;  // T already final (uniform across the grid)
  // A CTA gathers its candidates in shared memory and claims room for them in the global
  // array with one atomic (a global atomic per warp serialised thousands of same-address
  // updates); past the shared buffer's capacity each candidate claims its own slot.
  constexpr int kCap = 4096;  // also holds all candidates for the radix search when they fit
  __shared__ uint64_t sc[kCap];
  __shared__ uint32_t scount, sbase;
  if (threadIdx.x == 0) scount = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  constexpr int kLoads = 4;  // keys in flight per thread
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); i0 < units; i0 += kLoads * stride) {
    uint64_t k4[kLoads];
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      const int64_t i = i0 + q * stride + lane;
      k4[q] = i < units ? keys[i] : 0;
    }
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      const int64_t i = i0 + q * stride + lane;
      const uint64_t key = k4[q];
      const bool c = i < units && key_bucket(key) == B;
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, c);
      if (bal) {
        const int leader = __ffs(bal) - 1;
        uint32_t base = 0;
        if (lane == leader) base = atomicAdd(&scount, (uint32_t)__popc(bal));
        base = __shfl_sync(0xFFFFFFFFu, base, leader);
        const uint32_t at = base + __popc(bal & ((1u << lane) - 1u));
        if (c) {
          if (at < kCap)
            sc[at] = key;
          else
            cand[atomicAdd(&ctl->cand_count, 1u)] = key;
        }
      }
    }
  }
  __syncthreads();
  const uint32_t mine = scount < kCap ? scount : kCap;
  if (threadIdx.x == 0) sbase = mine ? atomicAdd(&ctl->cand_count, mine) : 0u;
  __syncthreads();
  for (uint32_t t = threadIdx.x; t < mine; t += blockDim.x) cand[sbase + t] = sc[t];
  if (!last_cta(&ctl->ticket[1])) return;
  // Radix search, 8 bits at a time, over the bits the bucket leaves open.
  __shared__ uint32_t h[256];
  __shared__ uint64_t s_prefix, s_k;
  const uint32_t n = __ldcg(&ctl->cand_count);
  const int lead = B / 64 + 5;
  const int hi_bit = lead - 7;  // highest bit not fixed by the bucket (B >= 128 so lead >= 7)
  if (threadIdx.x == 0) {
    s_prefix = (uint64_t)(64 + (B & 63)) << (lead - 6);
    s_k = __ldcg(&ctl->k_rem);
  }
  // The passes read the candidates from shared memory when they fit (one global read).
  const bool staged = n <= (uint32_t)kCap;
  if (staged) {
    uint32_t i = threadIdx.x;
    for (; i + 3 * 256 < n; i += 4 * 256) {
      uint64_t k4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) k4[q] = __ldcg(cand + i + q * 256);
#pragma unroll
      for (int q = 0; q < 4; ++q) sc[i + q * 256] = k4[q];
    }
    for (; i < n; i += 256) sc[i] = __ldcg(cand + i);
  }
  for (int shift = (hi_bit / 8) * 8; shift >= 0; shift -= 8) {
    h[threadIdx.x] = 0;
    __syncthreads();
    const uint64_t want = s_prefix >> (shift + 8);
    uint32_t i = threadIdx.x;
    if (staged) {
      for (; i < n; i += 256) {
        const uint64_t key = sc[i];
        if ((key >> (shift + 8)) == want) atomicAdd(&h[(key >> shift) & 255], 1u);
      }
    }
    for (; i + 3 * 256 < n; i += 4 * 256) {  // four loads in flight per thread
      uint64_t k4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) k4[q] = __ldcg(cand + i + q * 256);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if ((k4[q] >> (shift + 8)) == want) atomicAdd(&h[(k4[q] >> shift) & 255], 1u);
    }
    for (; i < n; i += 256) {
      const uint64_t key = __ldcg(cand + i);
      if ((key >> (shift + 8)) == want) atomicAdd(&h[(key >> shift) & 255], 1u);
    }
    __syncthreads();
    // Digit of the k-th largest: thread t holds digit 255 - t, prefix over threads.
    const uint32_t cnt = h[255 - threadIdx.x];
    uint32_t tot;
    const uint32_t incl = cta_inclusive_scan256<uint32_t>(cnt, tot);
    const uint64_t k = s_k;
    __syncthreads();
    if ((uint64_t)(incl - cnt) < k && k <= (uint64_t)incl) {
      s_k = k - (incl - cnt);
      s_prefix = (s_prefix & ~(255ull << shift)) | ((uint64_t)(255 - threadIdx.x) << shift);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    ctl->T = s_prefix;
    ctl->need_eq = s_k;
  }
}

// ---------------------------------------------------------------- ordering
// In-place exclusive prefix of a[0..n) by one CTA of 256 threads.
__device__ void cta_exclusive_scan(uint32_t* a, int64_t n) {
  constexpr int kPer = 8;  // a thread takes kPer consecutive entries of a 2048-entry tile
  uint32_t carry = 0;
  for (int64_t base = 0; base < n; base += 256 * kPer) {
    const int64_t first = base + (int64_t)threadIdx.x * kPer;
    uint32_t v[kPer], s = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      v[j] = first + j < n ? __ldcg(a + first + j) : 0u;
      s += v[j];
    }
    uint32_t tile;
    uint32_t run = carry + cta_inclusive_scan256<uint32_t>(s, tile) - s;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (first + j < n) a[first + j] = run;
      run += v[j];
    }
    carry += tile;
  }
}

// Counts of keys above and at the threshold per chunk of kChunk keys.  A CTA takes one
// group of kCountChunks chunks and writes each chunk's prefix within the group and the
// group's totals; the last CTA turns the group totals into prefixes, so its scan covers
// groups, not chunks.
__global__ void __launch_bounds__(kChunk) count_kernel(const uint64_t* __restrict__ keys, int64_t units, Ctl* ctl,
                                                       uint32_t* __restrict__ cnt_gt, uint32_t* __restrict__ cnt_eq) {
  pdl_trigger();
  pdl_wait();
  const uint64_t T = ctl->T;
  const int64_t chunks = (units + kChunk - 1) / kChunk;
  const int64_t groups = (chunks + kCountChunks - 1) / kCountChunks;
  uint64_t key[kCountChunks];
#pragma unroll
  for (int q = 0; q < kCountChunks; ++q) {  // every load in flight before the counts
    const int64_t i = ((int64_t)blockIdx.x * kCountChunks + q) * kChunk + threadIdx.x;
    key[q] = i < units ? keys[i] : 0;
  }
  uint32_t run_gt = 0, run_eq = 0;
#pragma unroll
  for (int q = 0; q < kCountChunks; ++q) {
    const int64_t chunk = (int64_t)blockIdx.x * kCountChunks + q;
    if (chunk >= chunks) break;  // uniform across the CTA
    const bool in = chunk * kChunk + threadIdx.x < units;
    const int gt = __syncthreads_count(in && key[q] > T);
    const int eq = __syncthreads_count(in && key[q] == T);
    if (threadIdx.x == 0) {
      cnt_gt[chunk] = run_gt;
      cnt_eq[chunk] = run_eq;
    }
    run_gt += (uint32_t)gt;
    run_eq += (uint32_t)eq;
  }
  if (threadIdx.x == 0) {
    cnt_gt[chunks + blockIdx.x] = run_gt;
    cnt_eq[chunks + blockIdx.x] = run_eq;
  }
  if (!last_cta(&ctl->ticket[2])) return;
  cta_exclusive_scan(cnt_gt + chunks, groups);
  __syncthreads();
  cta_exclusive_scan(cnt_eq + chunks, groups);
}

// Exclusive prefix of a per-thread flag over the CTA (kChunk threads).
__device__ __forceinline__ uint32_t cta_rank(bool f, uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, f);
  __syncthreads();
  if (lane == 0) warp_tot[w] = __popc(bal);
  __syncthreads();
  uint32_t before = 0;
  for (int j = 0; j < w; ++j) before += warp_tot[j];
  return before + __popc(bal & ((1u << lane) - 1u));
}

template <int DT, bool BLOCK>
__global__ void __launch_bounds__(kChunk) write_kernel(const uint8_t* __restrict__ W, int64_t rows, int64_t cols,
                                                       int64_t ld_bytes, const uint64_t* __restrict__ keys,
                                                       int64_t units, const Ctl* ctl, const uint32_t* __restrict__ pre_gt,
                                                       const uint32_t* __restrict__ pre_eq, uint8_t* W_out,
                                                       int64_t ldo_bytes, uint32_t* __restrict__ mask,
                                                       int32_t* __restrict__ csr, uint8_t* __restrict__ vals) {
  pdl_trigger();
  pdl_wait();
  constexpr int es = DT == kF16 ? 2 : 1;
  constexpr int kSegElems = 16 / es;
  constexpr int kSpr = kUnitW / kSegElems;         // segments per unit row
  constexpr int kUnitRows = BLOCK ? 32 : 1;
  constexpr int kSpu = kSpr * kUnitRows;           // segments per unit
  constexpr int kUnitBytes = kUnitW * kUnitRows * es;
  __shared__ uint32_t warp_tot[kChunk / 32];
  const uint64_t T = ctl->T, need_eq = ctl->need_eq;
  const int64_t upr = cols / kUnitW;  // units per unit row
  const int64_t urows = units / upr;
  const int64_t i = (int64_t)blockIdx.x * kChunk + threadIdx.x;
  const bool valid = i < units;
  const uint64_t key = valid ? keys[i] : 0;
  const bool gt = valid && key > T, eq = valid && key == T;
  const int64_t chunks = gridDim.x, grp = chunks + blockIdx.x / kCountChunks;
  const uint64_t eq0 = pre_eq[blockIdx.x] + pre_eq[grp], gt0 = pre_gt[blockIdx.x] + pre_gt[grp];
  const uint64_t eq_rank = eq0 + cta_rank(eq, warp_tot);
  const bool kept = gt || (eq && eq_rank < need_eq);
  const uint64_t before = gt0 + (eq0 < need_eq ? eq0 : need_eq);
  const int64_t pos = (int64_t)(before + cta_rank(kept, warp_tot));
  // Unit row and column of unit (warp's first unit) + k, 0 <= k < 32, from one
  // division per thread (a 64-bit division per segment dominated the issue slots).
  const int lane = threadIdx.x & 31;
  const int64_t r0 = (i - lane) / upr, c0 = (i - lane) - r0 * upr;
  auto unit_at = [&](int k, int64_t& r, int64_t& c) {
    r = r0;
    c = c0 + k;
    if (c >= upr) {
      const uint32_t q = (uint32_t)c / (uint32_t)upr;  // c < upr + 32
      r += q;
      c -= (int64_t)q * upr;
    }
  };
  if (csr != nullptr && valid) {
    int64_t ur, uc;
    unit_at(lane, ur, uc);
    if (uc == 0) csr[ur] = (int32_t)pos;
    if (i == units - 1) csr[urows] = (int32_t)(pos + (kept ? 1 : 0));
    if (kept) csr[urows + 1 + pos] = (int32_t)uc;
  }
  // Data movement: each warp handles its 32 units, 16-byte segments spread
  // over the lanes.
  if (mask != nullptr) {
    const int64_t mw = cols / 32;  // mask words per row
    if (!BLOCK) {
      if (valid) mask[i] = kept ? 0xFFFFFFFFu : 0u;  // a 32-column vector is one mask word
    } else {
      for (int k = 0; k < 32; ++k) {
        const int64_t u = i - lane + k;
        const bool kv = __shfl_sync(0xFFFFFFFFu, kept, k);
        if (u < units) {
          int64_t bi, bj;
          unit_at(k, bi, bj);
          mask[(bi * 32 + lane) * mw + bj] = kv ? 0xFFFFFFFFu : 0u;
        }
      }
    }
  }
  if (W_out == nullptr && vals == nullptr) return;
  if constexpr (!BLOCK) {
    // Every load is issued before the first store (W_out may alias W, which would
    // otherwise order each load after the previous store).  A thread reads and writes
    // the same addresses, so an in-place call stays correct.
    uint4 v[kSpu];
    bool kv[kSpu], in[kSpu];
    int64_t kp[kSpu], off_w[kSpu], off_o[kSpu];
#pragma unroll
    for (int it = 0; it < kSpu; ++it) {
      const int g = it * 32 + lane;
      const int k = g / kSpu, part = g % kSpu;
      kv[it] = __shfl_sync(0xFFFFFFFFu, kept, k);
      kp[it] = (int64_t)__shfl_sync(0xFFFFFFFFu, (long long)pos, k) * kUnitBytes + part * 16;
      const int64_t u = i - lane + k;
      in[it] = u < units;
      int64_t r, c;
      unit_at(k, r, c);
      const int64_t col_b = (c * kUnitW + part * kSegElems) * es;
      off_w[it] = r * ld_bytes + col_b;
      off_o[it] = r * ldo_bytes + col_b;
      v[it] = make_uint4(0, 0, 0, 0);
      if (in[it] && kv[it]) v[it] = *reinterpret_cast<const uint4*>(W + off_w[it]);
    }
#pragma unroll
    for (int it = 0; it < kSpu; ++it) {
      if (!in[it]) continue;
      if (W_out != nullptr) *reinterpret_cast<uint4*>(W_out + off_o[it]) = v[it];
      if (kv[it] && vals != nullptr) *reinterpret_cast<uint4*>(vals + kp[it]) = v[it];
    }
  } else {
    for (int k = 0; k < 32; ++k) {
      const bool kv = __shfl_sync(0xFFFFFFFFu, kept, k);
      const int64_t kp = (int64_t)__shfl_sync(0xFFFFFFFFu, (long long)pos, k);
      const int64_t u = i - lane + k;
      if (u >= units) break;  // uniform across the warp
      if (!kv && W_out == nullptr) continue;
      int64_t bi, bj;
      unit_at(k, bi, bj);
      constexpr int kIt = kSpu / 32;
      uint4 v[kIt];
#pragma unroll
      for (int it = 0; it < kIt; ++it) {  // loads first, as in the vector case
        const int g = it * 32 + lane;
        const int64_t row = bi * 32 + g / kSpr;
        v[it] = make_uint4(0, 0, 0, 0);
        if (kv) v[it] = *reinterpret_cast<const uint4*>(W + row * ld_bytes + (bj * kUnitW + (g % kSpr) * kSegElems) * es);
      }
#pragma unroll
      for (int it = 0; it < kIt; ++it) {
        const int g = it * 32 + lane;
        const int64_t row = bi * 32 + g / kSpr;
        const int64_t col_b = (bj * kUnitW + (g % kSpr) * kSegElems) * es;
        if (W_out != nullptr) *reinterpret_cast<uint4*>(W_out + row * ldo_bytes + col_b) = v[it];
        if (kv && vals != nullptr) *reinterpret_cast<uint4*>(vals + kp * kUnitBytes + g * 16) = v[it];
      }
    }
  }
}

// ---------------------------------------------------------------- product
__device__ __forceinline__ float h2f(uint32_t b, int bf16) {
  return bf16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((uint16_t)b));
}
__device__ __forceinline__ uint16_t f2h(float x, int bf16) {
  return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}
template <int NB>
__device__ __forceinline__ void dot8(const uint4 a, const uint16_t* x, int64_t ldb, int nb, int bf16, float* acc) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  float af[8];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    af[2 * t] = h2f(aw[t] & 0xFFFFu, bf16);
    af[2 * t + 1] = h2f(aw[t] >> 16, bf16);
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (b < nb) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + b * ldb));
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        acc[b] = fmaf(af[2 * t], h2f(xw[t] & 0xFFFFu, bf16), acc[b]);
        acc[b] = fmaf(af[2 * t + 1], h2f(xw[t] >> 16, bf16), acc[b]);
      }
    }
  }
}

__device__ __forceinline__ void store_d(const SpmmLaunch& a, int64_t r, int64_t b, float x, int bf16) {
  const nm_spmm_desc_t& d = a.d;
  const bool col = d.order_cd == NM_COL;
  x *= a.alpha_f;
  if (a.C != nullptr) {
    const uint16_t* C = static_cast<const uint16_t*>(a.C);
    x = fmaf(a.beta_f, h2f(C[col ? b * d.ldc + r : r * d.ldc + b], bf16), x);
  }
  static_cast<uint16_t*>(a.D)[col ? b * d.ldd + r : r * d.ldd + b] = f2h(x, bf16);
}

// Vector-wise: a warp per row; 8 kept vectors per step, 4 lanes per vector.
template <int NB>
__global__ void __launch_bounds__(256) vw_spmv_kernel(const SpmmLaunch a) {
  const nm_spmm_desc_t& d = a.d;
  const int bf16 = d.ab_type == NM_BF16;
  const int lane = threadIdx.x & 31;
  const int32_t* csr = static_cast<const int32_t*>(a.A_meta);
  const int32_t* colidx = csr + d.M + 1;
  const uint16_t* vals = static_cast<const uint16_t*>(a.A);
  const uint16_t* B = static_cast<const uint16_t*>(a.B);
  const int q = lane >> 2, part = lane & 3;
  // rows interleaved over the CTAs of a whole-wave grid (row r to CTA r mod grid)
  for (int64_t r = (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x; r < d.M; r += 8 * (int64_t)gridDim.x) {
    const int p0 = csr[r], p1 = csr[r + 1];
    for (int64_t b0 = 0; b0 < d.N; b0 += NB) {
      const int nb = (int)(d.N - b0 < NB ? d.N - b0 : NB);
      float acc[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
      // batch 1: four steps of eight vectors at a time, their column indices and values all
      // loaded before the first product needs them (7.1 -> 5.1 us at 4096^2, density 0.25);
      // batch 8 keeps one step at a time (four at once measured 12.6 -> 17.4 us there)
      constexpr int kSteps = NB == 1 ? 4 : 1;
      for (int p = p0 + q; p < p1; p += 8 * kSteps) {
        int64_t cs[kSteps];
        uint4 avs[kSteps];
#pragma unroll
        for (int k = 0; k < kSteps; ++k) {
          const int pk = p + 8 * k;
          if (pk < p1) {
            cs[k] = colidx[pk];
            avs[k] = __ldcs(reinterpret_cast<const uint4*>(vals + (int64_t)pk * kUnitW + part * 8));
          }
        }
#pragma unroll
        for (int k = 0; k < kSteps; ++k)
          if (p + 8 * k < p1) dot8<NB>(avs[k], B + b0 * d.ldb + cs[k] * kUnitW + part * 8, d.ldb, nb, bf16, acc);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) acc[b] += __shfl_xor_sync(0xFFFFFFFFu, acc[b], m);
#pragma unroll
      for (int b = 0; b < NB; ++b)
        if (lane == b && b < nb) store_d(a, r, b0 + b, acc[b], bf16);
    }
  }
}

// Block-wise: a CTA per block row; its warps split the kept blocks.  Lane l
// covers columns 8*(l%4)..+7 of block rows l/4 + 8j, j = 0..3, so that every
// warp load reads 512 contiguous bytes of a block.
// One CTA of bw_warps(NB) warps per 32-row block row: each warp takes every
// bw_warps-th kept block, so a block row's kept blocks (a quarter of them at the
// benchmark's density) are all in flight at once.  Batch 1: 32 warps.  Batch 8:
// 16 warps, so that a lane has the registers to convert its 32 values of a block
// and each batch column's 8 values of x once and reuse them across its 4 rows.
__host__ __device__ constexpr int bw_warps(int nb) { return nb == 1 ? 32 : 16; }
template <int NB>
__global__ void __launch_bounds__(bw_warps(NB) * 32) bw_spmv_kernel(const SpmmLaunch a) {
  constexpr int kBwWarps = bw_warps(NB);
  const nm_spmm_desc_t& d = a.d;
  const int bf16 = d.ab_type == NM_BF16;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t bi = blockIdx.x;
  const int64_t brows = d.M / 32;
  const int32_t* csr = static_cast<const int32_t*>(a.A_meta);
  const int32_t* colidx = csr + brows + 1;
  const uint16_t* vals = static_cast<const uint16_t*>(a.A);
  const uint16_t* B = static_cast<const uint16_t*>(a.B);
  const int p0 = csr[bi], p1 = csr[bi + 1];
  const int part = lane & 3, rq = lane >> 2;
  __shared__ float red[kBwWarps][32][NB];
  for (int64_t b0 = 0; b0 < d.N; b0 += NB) {
    const int nb = (int)(d.N - b0 < NB ? d.N - b0 : NB);
    float acc[4][NB];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[j][b] = 0.0f;
    for (int p = p0 + w; p < p1; p += kBwWarps) {
      const int64_t c = colidx[p];
      const uint16_t* blk = vals + (int64_t)p * 1024;
      uint4 av[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) av[j] = __ldcs(reinterpret_cast<const uint4*>(blk + (rq + 8 * j) * 32 + part * 8));
      if constexpr (NB == 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) dot8<NB>(av[j], B + b0 * d.ldb + c * kUnitW + part * 8, d.ldb, nb, bf16, acc[j]);
      } else {
        float af[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t aw[4] = {av[j].x, av[j].y, av[j].z, av[j].w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            af[j][2 * t] = h2f(aw[t] & 0xFFFFu, bf16);
            af[j][2 * t + 1] = h2f(aw[t] >> 16, bf16);
          }
        }
        const uint16_t* x = B + b0 * d.ldb + c * kUnitW + part * 8;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b < nb) {
            const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + b * d.ldb));
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
            float xf[8];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              xf[2 * t] = h2f(xw[t] & 0xFFFFu, bf16);
              xf[2 * t + 1] = h2f(xw[t] >> 16, bf16);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[j][b] = fmaf(af[j][e], xf[e], acc[j][b]);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float v = acc[j][b];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
        if (part == 0) red[w][rq + 8 * j][b] = v;
      }
    __syncthreads();
    for (int t = threadIdx.x; t < 32 * NB; t += blockDim.x) {
      const int row = t / NB, b = t - row * NB;
      if (b < nb) {
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < kBwWarps; ++k) s += red[k][row][b];
        store_d(a, bi * 32 + row, b0 + b, s, bf16);
      }
    }
    __syncthreads();
  }
}

// The histogram and control block set to zero in the launch chain (a memset node would end
// the chain of dependent launches before the scoring kernel).
__global__ void __launch_bounds__(256) zero_words_kernel(uint4* __restrict__ p, int64_t n16) {
  pdl_trigger();
  pdl_wait();
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) p[i] = make_uint4(0u, 0u, 0u, 0u);
}

template <int DT>
cudaError_t launch_blocks_dt(const BlocksLaunch& a, const WsLayout& L, cudaStream_t s) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  Ctl* ctl = reinterpret_cast<Ctl*>(ws + L.ctl);
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + L.keys);
  uint64_t* cand = reinterpret_cast<uint64_t*>(ws + L.cand);
  uint32_t* cgt = reinterpret_cast<uint32_t*>(ws + L.cnt_gt);
  uint32_t* ceq = reinterpret_cast<uint32_t*>(ws + L.cnt_eq);
  constexpr int es = DT == kF16 ? 2 : 1;
  const int64_t units = a.units;
  const int64_t chunks = (units + kChunk - 1) / kChunk;
  const uint8_t* W = static_cast<const uint8_t*>(a.W);
  // histogram + control block (L.keys bytes, a multiple of 256)
  if (cudaError_t e = launch_pdl(zero_words_kernel, dim3(1), dim3(256), 0, s, reinterpret_cast<uint4*>(ws),
                                 (int64_t)(L.keys / 16)))
    return e;
  cudaError_t e_;
  if (a.bh == 1) {
    const int64_t segs = a.rows * (a.cols * es / 16);
    if (a.abs_of_sum)
      e_ = launch_pdl(vw_score_kernel<DT, true>, dim3(grid_for(segs, 256, 4)), dim3(256), 0, s, W, a.rows, a.cols,
                      a.ld * es, keys, hist, ctl, (uint64_t)a.keep);
    else
      e_ = launch_pdl(vw_score_kernel<DT, false>, dim3(grid_for(segs, 256, 4)), dim3(256), 0, s, W, a.rows, a.cols,
                      a.ld * es, keys, hist, ctl, (uint64_t)a.keep);
  } else {
    e_ = launch_pdl(bw_score_kernel<DT>, dim3(grid_for(units * 32, 256, 4)), dim3(256), 0, s, W, a.rows, a.cols,
                    a.ld * es, keys, hist, ctl, (uint64_t)a.keep);
  }
  if (e_ != cudaSuccess) return e_;
  e_ = launch_pdl(candidates_kernel, dim3(grid_for(units, 256, 4)), dim3(256), 0, s, keys, units, ctl, cand);
  if (e_ != cudaSuccess) return e_;
  e_ = launch_pdl(count_kernel, dim3((unsigned)((chunks + kCountChunks - 1) / kCountChunks)), dim3(kChunk), 0, s, keys,
                  units, ctl, cgt, ceq);
  if (e_ != cudaSuccess) return e_;
  if (a.bh == 1) {
    e_ = launch_pdl(write_kernel<DT, false>, dim3((unsigned)chunks), dim3(kChunk), 0, s, W, a.rows, a.cols, a.ld * es,
                    keys, units, ctl, cgt, ceq, static_cast<uint8_t*>(a.W_out), a.ld_out * es, a.mask_bits, a.csr,
                    static_cast<uint8_t*>(a.vals));
  } else {
    e_ = launch_pdl(write_kernel<DT, true>, dim3((unsigned)chunks), dim3(kChunk), 0, s, W, a.rows, a.cols, a.ld * es,
                    keys, units, ctl, cgt, ceq, static_cast<uint8_t*>(a.W_out), a.ld_out * es, a.mask_bits, a.csr,
                    static_cast<uint8_t*>(a.vals));
  }
  return e_;
}

}  // namespace

size_t blocks_workspace(int64_t units) { return ws_layout(units).total; }

// ---------------------------------------------------------------- fixed scratch
// Scratch for the selection of at most kFixedScratchUnits units, held by every
// device that loads the library for as long as the process runs (about 8 MiB).
// Host code must not pass `g_units_scratch` itself to a kernel: on the host it
// names a host-side shadow, not device memory.  Its device address is looked
// up once per device below.
constexpr int64_t kFixedScratchUnits = int64_t(1) << 19;
static_assert(kFixedScratchUnits == NM_NOALLOC_MAX_UNITS, "the header advertises the fixed scratch's limit");
constexpr size_t kFixedScratchBytes = ws_layout(kFixedScratchUnits).total;
static __device__ __align__(256) uint8_t g_units_scratch[kFixedScratchBytes];

int64_t fixed_scratch_units() { return kFixedScratchUnits; }

cudaError_t fixed_scratch(void** ptr, size_t* bytes) {
  static std::atomic<void*> addr[64];
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* p = addr[dev].load();
  if (p == nullptr) {
    // the current device is `dev`: this resolves the array's address on it
    if (cudaError_t e = cudaGetSymbolAddress(&p, g_units_scratch)) return e;
    addr[dev].store(p);
  }
  *ptr = p;
  *bytes = kFixedScratchBytes;
  return cudaSuccess;
}

cudaError_t launch_blocks(const BlocksLaunch& a, cudaStream_t s) {
  const WsLayout L = ws_layout(a.units);
  if (a.units == 0) {
    if (a.csr != nullptr) return cudaMemsetAsync(a.csr, 0, (size_t)(a.unit_rows + 1) * 4, s);
    return cudaSuccess;
  }
  return a.dt == kF16 ? launch_blocks_dt<kF16>(a, L, s) : launch_blocks_dt<kI8>(a, L, s);
}

cudaError_t launch_spmm_blocks(const SpmmLaunch& a, cudaStream_t s) {
  const nm_spmm_desc_t& d = a.d;
  if (d.n == 1) {
    // whole waves over the SMs; a grid of ceil(M / 8) CTAs left some SMs a CTA short
    static const int per_sm1 = resident_ctas(vw_spmv_kernel<1>, 256, 0);
    static const int per_sm8 = resident_ctas(vw_spmv_kernel<8>, 256, 0);
    int64_t grid = (int64_t)num_sms_cached() * (d.N == 1 ? per_sm1 : per_sm8);
    if (grid > d.M) grid = d.M;  // a CTA's spare warps exit at once
    if (d.N == 1)
      vw_spmv_kernel<1><<<(unsigned)grid, 256, 0, s>>>(a);
    else
      vw_spmv_kernel<8><<<(unsigned)grid, 256, 0, s>>>(a);
  } else {
    const unsigned grid = (unsigned)(d.M / 32);
    if (d.N == 1)
      bw_spmv_kernel<1><<<grid, bw_warps(1) * 32, 0, s>>>(a);
    else
      bw_spmv_kernel<8><<<grid, bw_warps(8) * 32, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace nmk
