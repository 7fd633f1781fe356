// Device helpers and internal launcher declarations for the xq library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace xq {

constexpr int kQ4kBytes = 144;  // GGUF Q4_K super-block: 256 weights
constexpr int kQ6kBytes = 210;  // GGUF Q6_K super-block: 256 weights
constexpr int kNumSMs = 152;    // GB300: 2 dies x 76 SMs

// ---------------------------------------------------------------- loads

// Streaming 16-byte load for weight bytes: read once per launch, so it skips
// L1 allocation (the read-only path still goes through L2).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned ld_stream4(const void* p) {
  unsigned v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Activation loads: small, re-read by every row of the CTA, so they stay
// cacheable in L1.
__device__ __forceinline__ uint4 ld_act16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ----------------------------------------------------------- integer ops

// Four-way byte dot product: unsigned bytes of a times signed bytes of b,
// accumulated into c.
__device__ __forceinline__ int dp4a_us(unsigned a, unsigned b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Byte permute of the 8-byte pair (hi:lo).
__device__ __forceinline__ unsigned prmt(unsigned lo, unsigned hi, unsigned sel) {
  unsigned d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(lo), "r"(hi), "r"(sel));
  return d;
}

__device__ __forceinline__ float half_bits_to_float(unsigned bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// --------------------------------------------------------- launchers

struct GemvArgs {
  const uint8_t* W;     // weight super-blocks
  const int8_t* qs;     // Q8 quants [M][K]
  const float* d8;      // Q8 scales [M][K/32]
  const float* s8;      // Q8 scale*sum [M][K/32]
  int M, N, K;          // M in 1..8 for one launch
  float* y;             // [M][N], row stride ldy (floats)
  long long ldy;
  int32_t* isum;        // optional sub-block sums (test hook)
};

cudaError_t launch_quantize_q8(const float* x, int M, int K, int8_t* qs, float* d8, float* s8,
                               cudaStream_t s);
cudaError_t launch_gemv_q4k(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_gemv_q6k(const GemvArgs& a, cudaStream_t s);

}  // namespace xq
