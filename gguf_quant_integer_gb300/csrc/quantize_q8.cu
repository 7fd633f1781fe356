// Q8 activation quantization: fp32 [M][K] -> int8 quants + fp32 scale + fp32
// scale*sum per block of 32 (the q8_1 kind; xLLM v0.7 article, sections B1.3
// and C.1; Agent Telemetry log, "批次化 MMVQ").
//
// One warp per 32-block, one element per lane:
//   amax = max |x|          (warp max over the IEEE bit patterns of |x|)
//   d8   = amax / 127       (IEEE round-to-nearest divide)
//   id   = 1 / d8, 0 if d8 == 0 (IEEE round-to-nearest reciprocal)
//   q    = clamp(roundf(x * id), -127, 127), roundf = half away from zero,
//          clamped in float (NaN -> 0) before the int conversion
//   s8   = d8 * (float)sum(q)
// Each step is one correctly rounded fp32 operation, written with explicit
// _rn intrinsics so that no contraction or fast-math substitution can change
// a bit. The result is therefore the same on any IEEE implementation that
// performs the same steps.
#include "xq_common.cuh"

namespace xq {

__global__ void __launch_bounds__(256)
quantize_q8_kernel(const float* __restrict__ x, long long nblocks,
                   int8_t* __restrict__ qs, float* __restrict__ d8, float* __restrict__ s8) {
  const int lane = threadIdx.x & 31;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long blk = warp; blk < nblocks; blk += nwarps) {
    const float v = __ldg(x + blk * 32 + lane);
    // |x| >= 0, so its IEEE bit pattern orders like the value itself.
    const unsigned amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
    const float amax = __uint_as_float(amax_bits);
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    float r = roundf(__fmul_rn(v, id));
    // Saturate in float: if 1/d8 overflowed (amax below ~1.5e-36), x*id is
    // +-inf (-> +-127) or 0*inf = NaN (-> 0).
    r = (r != r) ? 0.0f : r;
    r = r > 127.0f ? 127.0f : (r < -127.0f ? -127.0f : r);
    const int q = static_cast<int>(r);
    qs[blk * 32 + lane] = static_cast<int8_t>(q);
    const int isum = __reduce_add_sync(0xffffffffu, q);
    if (lane == 0) {
      d8[blk] = d;
      s8[blk] = __fmul_rn(d, static_cast<float>(isum));
    }
  }
}

cudaError_t launch_quantize_q8(const float* x, int M, int K, int8_t* qs, float* d8, float* s8,
                               cudaStream_t s) {
  const long long nblocks = static_cast<long long>(M) * (K / 32);
  if (nblocks == 0) return cudaSuccess;
  const int threads = 256;
  long long want = (nblocks + 7) / 8;  // 8 warps per CTA, one block per warp
  const long long cap = static_cast<long long>(kNumSMs) * 16;
  const int grid = static_cast<int>(want < cap ? want : cap);
  quantize_q8_kernel<<<grid, threads, 0, s>>>(x, nblocks, qs, d8, s8);
  return cudaGetLastError();
}

}  // namespace xq
