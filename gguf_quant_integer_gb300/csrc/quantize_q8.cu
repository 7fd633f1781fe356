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
//
// The same pass writes the tensor-core operand image of the quants (fp16
// copies in m16n8k16 B-fragment order, 8 token columns per chunk) and the
// per-32-block scale quads the MMA epilogue reads, so that the matmuls never
// convert activations themselves. One launch serves all inputs of a layer.
#include "xq_common.cuh"

namespace xq {

struct QuantGroup {
  QuantJob job[kMaxProj];
  long long blk0[kMaxProj + 1];  // prefix of padded 32-blocks per job
  unsigned int* zero_words;      // optional: words set to 0 (the next matmul's scheduling state)
  int zero_count;
  int n;
};

__global__ void __launch_bounds__(256)
quantize_q8_kernel(const __grid_constant__ QuantGroup G) {
  // Inputs may be written by the previous kernel on the stream.
  cudaGridDependencySynchronize();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < G.zero_count; i += blockDim.x) G.zero_words[i] = 0u;
  const int lane = threadIdx.x & 31;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long total = G.blk0[G.n];
  // Position of this lane's element inside its lane's 8 operand slots:
  // slot order is perm = 0,2,1,3,4,6,5,7 (an involution), so slot = perm[l & 7].
  const int t = lane >> 3;
  const int i = lane & 7;
  const int slot = (i == 1 || i == 2 || i == 5 || i == 6) ? (i ^ 3) : i;

  int jb = 0;
  for (long long blk = warp; blk < total; blk += nwarps) {
    while (blk >= G.blk0[jb + 1]) ++jb;
    const QuantJob& J = G.job[jb];
    const long long local = blk - G.blk0[jb];
    const int nsub = J.K >> 5;
    const int m = static_cast<int>(local / nsub);
    const int j = static_cast<int>(local - static_cast<long long>(m) * nsub);
    const Q8Layout L = q8_layout(J.M, J.K);
    const int c = m >> 3, n = m & 7;

    float d = 0.0f, s = 0.0f;
    int q = 0;
    if (m < J.M) {
      const float v = __ldg(J.x + static_cast<size_t>(m) * J.K + 32 * j + lane);
      // |x| >= 0, so its IEEE bit pattern orders like the value itself.
      const unsigned amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
      const float amax = __uint_as_float(amax_bits);
      d = __fdiv_rn(amax, 127.0f);
      const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
      float r = roundf(__fmul_rn(v, id));
      // Saturate in float: if 1/d8 overflowed (amax below ~1.5e-36), x*id is
      // +-inf (-> +-127) or 0*inf = NaN (-> 0).
      r = (r != r) ? 0.0f : r;
      r = r > 127.0f ? 127.0f : (r < -127.0f ? -127.0f : r);
      q = static_cast<int>(r);
      const int isum = __reduce_add_sync(0xffffffffu, q);
      s = __fmul_rn(d, static_cast<float>(isum));
      J.xq[L.qs + static_cast<size_t>(m) * J.K + 32 * j + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
      if (lane == 0) {
        reinterpret_cast<float*>(J.xq + L.d8)[static_cast<size_t>(m) * nsub + j] = d;
        reinterpret_cast<float*>(J.xq + L.s8)[static_cast<size_t>(m) * nsub + j] = s;
      }
    }
    // operand image (zeros for padding tokens)
    __half* frag = reinterpret_cast<__half*>(J.xq + L.frag);
    frag[((static_cast<size_t>(c) * nsub + j) * 32 + 4 * n + t) * 8 + slot] = __int2half_rn(q);
    if (lane == 0) {
      float* fsc = reinterpret_cast<float*>(J.xq + L.fsc);
      const size_t base = ((static_cast<size_t>(c) * nsub + j) * 4 + (n >> 1)) * 4;
      fsc[base + (n & 1)] = d;
      fsc[base + 2 + (n & 1)] = s;
    }
  }
  cudaTriggerProgrammaticLaunchCompletion();
}

cudaError_t launch_quantize_q8(const QuantJob* jobs, int n, cudaStream_t s, bool pdl, unsigned int* zero_words,
                               int zero_count) {
  if (n <= 0 || n > kMaxProj) return cudaErrorInvalidValue;
  QuantGroup G;
  G.n = n;
  G.zero_words = zero_words;
  G.zero_count = zero_words ? zero_count : 0;
  G.blk0[0] = 0;
  for (int k = 0; k < n; ++k) {
    G.job[k] = jobs[k];
    const long long mp = 8LL * ((jobs[k].M + 7) / 8);
    G.blk0[k + 1] = G.blk0[k] + mp * (jobs[k].K / 32);
  }
  const long long nblocks = G.blk0[n];
  if (nblocks == 0) return cudaSuccess;
  long long want = (nblocks + 7) / 8;  // 8 warps per CTA, one block per warp
  const long long cap = static_cast<long long>(kNumSMs) * 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quantize_q8_kernel, G);
}

}  // namespace xq
