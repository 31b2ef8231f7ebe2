// Device-side helpers shared by the library's kernels: element traits and the
// magnitude key that orders elements for N:M selection.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nmk {

// Element type tags, equal to nm_dtype_t values.
constexpr int kF16 = 0, kBF16 = 1, kI8 = 2;

template <int DT> struct Elem;
template <> struct Elem<kF16> {
  using T = uint16_t;
  // |w| order on bit patterns: clear the sign; every NaN maps to one key above +Inf (0x7C00).
  __device__ __forceinline__ static uint32_t key(T v) { return min((uint32_t)v & 0x7FFFu, 0x7C01u); }
  __device__ __forceinline__ static bool nonzero(T v) { return (v & 0x7FFFu) != 0; }
};
template <> struct Elem<kBF16> {
  using T = uint16_t;
  __device__ __forceinline__ static uint32_t key(T v) { return min((uint32_t)v & 0x7FFFu, 0x7F81u); }
  __device__ __forceinline__ static bool nonzero(T v) { return (v & 0x7FFFu) != 0; }
};
template <> struct Elem<kI8> {
  using T = int8_t;
  __device__ __forceinline__ static uint32_t key(T v) { return (uint32_t)abs((int)v); }  // |-128| = 128
  __device__ __forceinline__ static bool nonzero(T v) { return v != 0; }
};

// Float32 magnitude used by the transposable tile score: exact for every
// input type; NaN scores as +Inf.
__device__ __forceinline__ float mag_f32(uint16_t v, int dt) {
  float f;
  if (dt == kF16) {
    f = __half2float(__ushort_as_half(v));
  } else {
    f = __uint_as_float((uint32_t)v << 16);
  }
  f = fabsf(f);
  return (f != f) ? __int_as_float(0x7F800000) : f;
}

// Tensor-core order of 2:4 metadata: for each k-step s (32 columns) `nslots`
// uint32 words; word s * nslots + (16b + 8h + i) holds the codes of row 16b+i
// (low half) and row 16b+8+i (high half) for columns 32s+16h .. 32s+16h+15.
// Byte offset of the 16-bit half that holds 16-column segment k of row r:
__host__ __device__ __forceinline__ int64_t tc_half_offset(int64_t r, int64_t k, int64_t nslots) {
  const int64_t slot = (r & ~int64_t(15)) + 8 * (k & 1) + (r & 7);
  return ((k >> 1) * nslots + slot) * 4 + ((r >> 3) & 1) * 2;
}
inline int64_t tc_slots(int64_t rows) { return ((rows + 127) / 128) * 128; }

__device__ __forceinline__ void tc_store(void* meta, int64_t r, int64_t k, int64_t nslots, uint32_t code16) {
  *reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(meta) + tc_half_offset(r, k, nslots)) = (uint16_t)code16;
}

// Programmatic dependent launch.  A grid launched with launch_pdl may be scheduled
// while the previous grid of its stream is still finishing: pdl_wait() returns once
// that grid has completed and its memory operations are visible (at once for a grid
// launched without the attribute), so every kernel calls it before its first global
// memory access; pdl_trigger() lets the next grid be scheduled as this one's CTAs
// exit (called once every CTA of this grid runs, so the next grid never takes the
// resources a CTA of this one still waits for).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// CTAs of `kernel` that fit on one SM at `threads` threads and `smem` dynamic shared bytes
// (1 if the query fails).
template <typename Kernel>
inline int resident_ctas(Kernel kernel, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 1;
  }
  return n;
}

// Streaming multiprocessors of the current device (queried once).
inline int num_sms_cached() {
  static const int v = [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    return n;
  }();
  return v;
}

// Grid size for grid-stride loops: enough CTAs to fill 152 SMs several times.
inline unsigned grid_for(int64_t work_items, int threads, int max_ctas_per_sm = 8) {
  int64_t g = (work_items + threads - 1) / threads;
  int64_t cap = 152LL * max_ctas_per_sm;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (unsigned)g;
}

}  // namespace nmk
