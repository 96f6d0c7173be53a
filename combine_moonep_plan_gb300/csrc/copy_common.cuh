// 16-byte global-memory helpers shared by the copy kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace moonep {

// Streaming read: every byte is read once, keep it out of L1.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Read once through L2 from memory this kernel also writes (no .nc path).
__device__ __forceinline__ float4 ld_once_f4(const float4 *p) {
  float4 v;
  asm volatile("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_global(uint4 *p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_global_f4(float4 *p, float4 v) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// |dst| of the signed route encoding.
__device__ __forceinline__ int64_t decode_row(int32_t d) {
  return d >= 0 ? (int64_t)d : -(int64_t)d - 1;
}

}  // namespace moonep
