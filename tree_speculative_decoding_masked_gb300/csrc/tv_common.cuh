// Shared device helpers for the tree-verification kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "treeverify.h"

#ifndef TV_WAIT_NS
// Upper bound for any spin wait inside a kernel (mbarrier, flag): 1 second.
#define TV_WAIT_NS 1000000000ull
#endif

namespace tv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint32_t u = __float_as_uint(f);
  uint32_t bias = ((u >> 16) & 1u) + 0x7FFFu;
  return (uint16_t)((u + bias) >> 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)f32_to_bf16_rn(lo) | ((uint32_t)f32_to_bf16_rn(hi) << 16);
}

__device__ __forceinline__ void set_dev_status(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

template <typename T>
__device__ __forceinline__ T warp_max(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (max, sum-exp) pair in base-2 units: represents sum_i 2^(z_i) = s * 2^m.
struct MaxSum {
  float m;
  float s;
};

__device__ __forceinline__ MaxSum maxsum_merge(MaxSum a, MaxSum b) {
  float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.f};
  float s = a.s * exp2f(a.m - m) + b.s * exp2f(b.m - m);
  return {m, s};
}

// argmax candidate: larger value wins, equal values -> smaller index.
struct ArgMax {
  float v;
  int i;
};

__device__ __forceinline__ ArgMax argmax_merge(ArgMax a, ArgMax b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}

// Block-wide exclusive scan of 64-bit values; returns this thread's exclusive prefix and
// sets *total.  red holds at least 33 entries.
static __device__ unsigned long long block_scan_u64(unsigned long long v, unsigned long long* red,
                                                    unsigned long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) red[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const unsigned long long x = lane < (int)(blockDim.x >> 5) ? red[lane] : 0ull;
    unsigned long long xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += y;
    }
    red[lane] = xi - x;
    if (lane == 31) red[32] = xi;
  }
  __syncthreads();
  const unsigned long long excl = red[wid] + (incl - v);
  *total = red[32];
  __syncthreads();
  return excl;
}

// Launch with programmatic stream serialization: the kernel's CTAs may start while the
// previous kernel of the stream is finishing (after it calls griddep_launch_dependents)
// and wait in griddep_wait() for its completion, which hides the launch latency between
// dependent kernels.  Optional extra attributes (e.g. a cluster shape) come first.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              const cudaLaunchAttribute* extra, int n_extra, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[4];
  int n = 0;
  for (int i = 0; i < n_extra && n < 3; ++i) attr[n++] = extra[i];
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace tv
