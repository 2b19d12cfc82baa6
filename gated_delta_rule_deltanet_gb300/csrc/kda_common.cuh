// kda_common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// ---------------------------------------------------------------- element access

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Load element i of a q/k/v row stored as fp32 (IS_BF16 = false) or bf16.
template <bool IS_BF16>
__device__ __forceinline__ float load_elem(const void* base, int64_t i) {
  if constexpr (IS_BF16) {
    return bf16_bits_to_f32(static_cast<const uint16_t*>(base)[i]);
  } else {
    return static_cast<const float*>(base)[i];
  }
}

// Four consecutive elements (16-byte aligned for fp32, 8-byte for bf16).
template <bool IS_BF16>
__device__ __forceinline__ float4 load4(const void* base, int64_t i) {
  if constexpr (IS_BF16) {
    uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + i);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  } else {
    return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
  }
}

template <bool IS_BF16>
__device__ __forceinline__ void store4(void* base, int64_t i, float4 v) {
  if constexpr (IS_BF16) {
    uint32_t lo = static_cast<uint32_t>(f32_to_bf16_bits(v.x)) |
                  (static_cast<uint32_t>(f32_to_bf16_bits(v.y)) << 16);
    uint32_t hi = static_cast<uint32_t>(f32_to_bf16_bits(v.z)) |
                  (static_cast<uint32_t>(f32_to_bf16_bits(v.w)) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + i) = make_uint2(lo, hi);
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(base) + i) = v;
  }
}

// Two-wide fp32 arithmetic (one instruction for two lanes of a float2, sm_100 and later):
// a * b + c, a * b and a + b, each component rounded to nearest as the scalar operations.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(*reinterpret_cast<unsigned long long*>(&d))
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
        "l"(*reinterpret_cast<unsigned long long*>(&c)));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(*reinterpret_cast<unsigned long long*>(&d))
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(*reinterpret_cast<unsigned long long*>(&d))
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
  return d;
}

// 2^x by the hardware approximation (PTX ex2.approx, flushing subnormal results to zero);
// callers keep their exponents in log2 units, so a decay factor costs one instruction
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp32 rounded to the nearest tf32 (10-bit mantissa, ties away from zero; the low 13 bits
// zero): what a kind::tf32 MMA operand should hold, since the MMA reads only the top bits
__device__ __forceinline__ float tf32_nearest(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// sum over the 16 lanes of each half-warp
__device__ __forceinline__ float halfwarp_sum(float v) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Record the first device-side problem; later ones keep the first code.
__device__ __forceinline__ void raise_device_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- host-side launch records

// Optional per-kernel timing events (kda_set_stage_events): mark(0) before the
// first launch of a call, mark(i) after its i-th kernel.
struct Stages {
  cudaEvent_t ev[8];
  int n;
  void mark(int i, cudaStream_t s) const {
    if (i < n) cudaEventRecord(ev[i], s);
  }
};

// Per-call problem description handed to the kernels (plain values, device pointers).
struct Problem {
  int32_t num_seqs, HK, HV, D, num_slots, chunk;
  int64_t T;
  float scale;
  int32_t l2norm;
  uint32_t flags;
  int64_t q_stride, k_stride, v_stride;  // elements between tokens
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* g;
  const uint32_t* offsets;
  const uint32_t* slot_idx;
  void* pool;
  float* o;
  int32_t* err;
};

// streaming multiprocessors of the current device (cached per device)
inline int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace kda
