// Device helpers shared by the kernels of libsv.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace sv {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Programmatic dependent launch. pdl_trigger: this CTA lets the next kernel in
// the stream start its independent prologue (the first call in a CTA counts).
// pdl_wait: block until the kernels before this one have completed and their
// writes are visible. Both are no-ops for a kernel launched without the
// programmatic attribute.
//
// Every kernel of the library triggers only after its own wait. Then at most
// two kernels of a stream overlap, the running one (past its wait, so its
// predecessor has completed) and the next one's prologue, and a prologue may
// read anything written two or more kernels back (the row maps of the row
// preparation, the committed lengths, the cached keys and values).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Store one activation element as float32 or bf16 (round to nearest even).
__device__ __forceinline__ void store_act(void* base, long long idx, float v, int act_bf16) {
  if (act_bf16)
    reinterpret_cast<uint16_t*>(base)[idx] = f32_to_bf16_bits(v);
  else
    reinterpret_cast<float*>(base)[idx] = v;
}

__device__ __forceinline__ float load_act(const void* base, long long idx, int act_bf16) {
  if (act_bf16) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

// x tensors: float32, or hi/lo bf16 planes (hi at i, lo at plane + i).
__device__ __forceinline__ void store_x(void* base, long long plane, long long idx, float v, int pair) {
  if (pair) {
    const uint16_t hi = f32_to_bf16_bits(v);
    const uint16_t lo = f32_to_bf16_bits(v - bf16_bits_to_f32(hi));
    reinterpret_cast<uint16_t*>(base)[idx] = hi;
    reinterpret_cast<uint16_t*>(base)[plane + idx] = lo;
  } else {
    reinterpret_cast<float*>(base)[idx] = v;
  }
}

// kind 0: float32; 1: one bf16 plane; 2: hi/lo bf16 planes (see XKind).
__device__ __forceinline__ float load_x(const void* base, long long plane, long long idx, int kind) {
  if (kind == 0) return reinterpret_cast<const float*>(base)[idx];
  const uint16_t* p = reinterpret_cast<const uint16_t*>(base);
  const float hi = bf16_bits_to_f32(p[idx]);
  return kind == 2 ? hi + bf16_bits_to_f32(p[plane + idx]) : hi;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value, index) argmax; ties go to the lower index.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_merge(v, i, v2, i2);
  }
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024). `red` holds 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : -INFINITY;
  t = warp_max(t);
  return t;
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11, section 3.3): two
// 32x32->64 products per round on words 0 and 2, a Weyl key schedule, ten rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// u in [0, 1), a multiple of 2^-24: counter (position, stream, request lo, request hi),
// key (seed lo, seed hi), word 0 >> 8.
__device__ __forceinline__ float philox_uniform(unsigned long long seed, long long req, long long pos,
                                                unsigned stream) {
  const unsigned long long r = static_cast<unsigned long long>(req);
  const uint4 c = make_uint4(static_cast<uint32_t>(pos), stream, static_cast<uint32_t>(r),
                             static_cast<uint32_t>(r >> 32));
  const uint2 k = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  return static_cast<float>(philox4x32_10(c, k).x >> 8) * (1.0f / 16777216.0f);
}

}  // namespace sv
