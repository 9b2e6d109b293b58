// Shared device helpers of the Medusa step kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cfloat>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/medusa.h"

#define MEDUSA_API extern "C" __attribute__((visibility("default")))

namespace medusa {

constexpr int kWarp = 32;

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// --------------------------------------------------------------------------
// Element access for the two storage types
// --------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPer16B = 4;
  __device__ static inline float to_f(float x) { return x; }
  __device__ static inline float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kPer16B = 8;
  __device__ static inline float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static inline __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// 16-byte streaming load that does not allocate in L1 (weights are read once).
__device__ inline uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Unpack 16 bytes into fp32 values.
__device__ inline void unpack16(const uint4& v, float (&f)[8], __nv_bfloat16*) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ inline void unpack16(const uint4& v, float (&f)[4], float*) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}

// --------------------------------------------------------------------------
// Warp reductions
// --------------------------------------------------------------------------
__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (value, id) ordering used by every top-k / argmax: larger value first, equal
// values by lower id; NaN is never "better" than anything.
__device__ inline bool better(float va, int ia, float vb, int ib) {
  return (va > vb) || (va == vb && ia < ib);
}

__device__ inline void warp_argmax(float& v, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, id, o);
    if (better(ov, oi, v, id)) { v = ov; id = oi; }
  }
}

__device__ inline uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: wait until the grids this one depends on have
// completed and their writes are visible (a no-op when launched without the
// attribute), and let the next grid in the stream start launching.
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 2^x on the special-function unit (flush-to-zero; 2^-inf = 0).
__device__ inline float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded-wait limit for every device-side spin (about one second).
constexpr uint64_t kSpinLimitNs = 1000000000ull;

// Process-wide count of kernels this library has launched (or captured).
void note_launch();

// Streaming multiprocessors of the current device (148 when the query fails).
int device_sm_count();

// Opt `kernel` in to `bytes` of dynamic shared memory.  The attribute stays
// set, so the driver call is made only when a kernel needs more than it was
// last given on the current device (per-step calls stay cheap on the host).
template <typename... KArgs>
bool ensure_dyn_smem(void (*kernel)(KArgs...), size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> granted;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = granted.find(key);
  if (it != granted.end() && it->second >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  granted[key] = bytes;
  return true;
}

// Launch `kernel` with programmatic dependent launch allowed: the grid may
// start while the previous kernel in the stream is still finishing, and the
// kernel itself waits (pdl_wait) before it touches what that work produced.
// Every kernel launched this way calls pdl_wait in all of its CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace medusa

// Host-side check after every kernel launch of an entry point.
#define MEDUSA_LAUNCH_CHECK()                                  \
  do {                                                         \
    if (cudaPeekAtLastError() != cudaSuccess) {                \
      (void)cudaGetLastError();                                \
      return MEDUSA_ERR_CUDA;                                  \
    }                                                          \
    medusa::note_launch();                                     \
  } while (0)
