// One 32-block of Q8 activation quantization per warp, one element per lane
// (the q8_1 kind; xLLM v0.7 article, sections B1.3 and C.1), and the SwiGLU
// feed of the down projection. Shared by the quantize kernel and the fused
// SwiGLU epilogue of the grouped GEMV, so both write the same bytes:
//   amax = max |x|          (warp max over the IEEE bit patterns of |x|)
//   d8   = amax / 127       (IEEE round-to-nearest divide)
//   id   = 1 / d8, 0 if d8 == 0 (IEEE round-to-nearest reciprocal)
//   q    = clamp(roundf(x * id), -127, 127), roundf = half away from zero,
//          clamped in float (NaN -> 0) before the int conversion
//   s8   = d8 * (float)sum(q)
// Each step is one correctly rounded fp32 operation, written with explicit
// _rn intrinsics so that no contraction or fast-math substitution can change
// a bit.
#pragma once

#include <cuda_fp16.h>

#include <cstddef>
#include <cstdint>

namespace xq {

struct Q8Lane {
  int q;    // this lane's quant
  float d;  // the block's d8 (every lane)
  float s;  // the block's s8 (every lane)
};

// h = silu(g) * u = g / (1 + e^-g) * u, each step one fp32 operation (CUDA's
// expf, IEEE add, divide and multiply); g -> -inf gives e^-g = inf and h = +-0.
__device__ __forceinline__ float swiglu(float g, float u) {
  const float e = expf(-g);
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, e)), u);
}

// Quantize the warp's block; every lane passes its element and all 32 call.
__device__ __forceinline__ Q8Lane q8_quantize_lane(float v) {
  // |x| >= 0, so its IEEE bit pattern orders like the value itself.
  const unsigned amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
  const float amax = __uint_as_float(amax_bits);
  Q8Lane r;
  r.d = __fdiv_rn(amax, 127.0f);
  const float id = (r.d != 0.0f) ? __frcp_rn(r.d) : 0.0f;
  float x = roundf(__fmul_rn(v, id));
  // Saturate in float: if 1/d8 overflowed (amax below ~1.5e-36), x*id is
  // +-inf (-> +-127) or 0*inf = NaN (-> 0).
  x = (x != x) ? 0.0f : x;
  x = x > 127.0f ? 127.0f : (x < -127.0f ? -127.0f : x);
  r.q = static_cast<int>(x);
  const int isum = __reduce_add_sync(0xffffffffu, r.q);
  r.s = __fmul_rn(r.d, static_cast<float>(isum));
  return r;
}

// Position of lane's element among its 8 operand slots of the GEMV image:
// slot order 0,2,1,3,4,6,5,7 (an involution), so slot = perm[lane & 7].
__device__ __forceinline__ int gemv_image_slot(int lane) {
  const int i = lane & 7;
  return (i == 1 || i == 2 || i == 5 || i == 6) ? (i ^ 3) : i;
}

// Token m's entries of 32-block j in the GEMV operand image (layout in
// xq_common.cuh): the fp16 quant of this lane, and (lane 0) the scale quad
// halves d8 and s8. Padding tokens of a chunk are written with q = d = s = 0.
__device__ __forceinline__ void write_gemv_image(uint8_t* frag_base, uint8_t* fsc_base, int nsub, int m, int j,
                                                 int lane, int q, float d, float s) {
  const int c = m >> 3, n = m & 7, t = lane >> 3;
  __half* frag = reinterpret_cast<__half*>(frag_base);
  frag[((static_cast<size_t>(c) * nsub + j) * 32 + 4 * n + t) * 8 + gemv_image_slot(lane)] = __int2half_rn(q);
  if (lane == 0) {
    float* fsc = reinterpret_cast<float*>(fsc_base);
    const size_t base = ((static_cast<size_t>(c) * nsub + j) * 4 + (n >> 1)) * 4;
    fsc[base + (n & 1)] = d;
    fsc[base + 2 + (n & 1)] = s;
  }
}

}  // namespace xq
