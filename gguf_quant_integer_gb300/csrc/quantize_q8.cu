// Q8 activation quantization: fp32 [M][K] -> int8 quants + fp32 scale + fp32
// scale*sum per block of 32 (the q8_1 kind; xLLM v0.7 article, sections B1.3
// and C.1; Agent Telemetry log, "批次化 MMVQ").
//
// One warp per 32-block, one element per lane, by the steps of
// q8_quantize_lane (q8_block.cuh): each one correctly rounded fp32
// operation, so the result is the same on any IEEE implementation that
// performs the same steps.
//
// The same pass writes the tensor-core operand image of the quants, so that
// the matmuls never convert activations themselves: for M <= 64 fp16 copies
// in m16n8k16 B-fragment order plus per-32-block scale quads; for M > 64 the
// 128-token tiles of the tcgen05 B operand, their d8 rows and the three-piece
// bf16 split of s8 (layouts in xq_common.cuh). One launch serves all inputs
// of a layer.
#include "q8_block.cuh"
#include "xq_check.cuh"
#include "xq_common.cuh"

namespace xq {

// Byte offset of token r, k-slot ks in a 128-token x 32-slot operand in the
// K-major no-swizzle layout (8x8 core matrices of 128 bytes: slot groups of
// 8 strided by 128 bytes, token groups of 8 strided by 512 bytes).
__device__ __forceinline__ int tile_offset(int r, int ks) {
  return (r >> 3) * 512 + (ks >> 3) * 128 + (r & 7) * 16 + (ks & 7) * 2;
}

// One input of a grouped launch, with its buffer layout resolved on the host.
struct QuantItem {
  const float* x;
  const float* up;  // non-null: quantize h = silu(x) * up
  float* h_out;     // optional copy of h
  uint8_t* xq;
  size_t d8, s8, frag, fsc, tile;  // byte offsets in xq (layout in xq_common.cuh)
  size_t total;                    // bytes of xq (bounds checks of checked builds)
  int M, K, nsub, ttiles;
};

struct QuantGroup {
  QuantItem job[kMaxProj];
  unsigned blk0[kMaxProj + 1];  // prefix of padded 32-blocks per input
  unsigned int* zero_words;     // optional: words set to 0 (the next matmul's scheduling state)
  int zero_count;
  int n;
};

__global__ void __launch_bounds__(1024)
quantize_q8_kernel(const __grid_constant__ QuantGroup G) {
  const int lane = threadIdx.x & 31;
  const unsigned warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  const unsigned total = G.blk0[G.n];
  // Inputs may be written by the previous kernel on the stream, so they are
  // read only after the dependency wait. Before it, the lines they occupy
  // are requested into L2 (L2 is coherent for the device, so a line the
  // previous kernel writes afterwards is read with its new contents).
  {
    int jb = 0;
    for (unsigned blk = warp; blk < total; blk += nwarps) {
      while (blk >= G.blk0[jb + 1]) ++jb;
      const QuantItem& J = G.job[jb];
      const unsigned local = blk - G.blk0[jb];
      const int m = static_cast<int>(local / static_cast<unsigned>(J.nsub));
      const int j = static_cast<int>(local - static_cast<unsigned>(m) * J.nsub);
      if (m < J.M && (lane == 0 || lane == 31)) {
        const size_t idx = static_cast<size_t>(m) * J.K + 32 * j + lane;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(J.x + idx));
        if (J.up) asm volatile("prefetch.global.L2 [%0];" ::"l"(J.up + idx));
      }
    }
  }
  // The next kernel may launch at once: it waits for this grid's completion
  // before reading what it writes.
  cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < G.zero_count; i += blockDim.x) G.zero_words[i] = 0u;
  // Position of this lane's element inside its lane's 8 operand slots.
  const int slot = gemv_image_slot(lane);

  int jb = 0;
  for (unsigned blk = warp; blk < total; blk += nwarps) {
    while (blk >= G.blk0[jb + 1]) ++jb;
    const QuantItem& J = G.job[jb];
    const unsigned local = blk - G.blk0[jb];
    const int nsub = J.nsub;
    const int m = static_cast<int>(local / static_cast<unsigned>(nsub));
    const int j = static_cast<int>(local - static_cast<unsigned>(m) * nsub);
    const QuantItem& L = J;

    float d = 0.0f, s = 0.0f;
    int q = 0;
    // (checked builds: the block inside [M][K] and every region of xq this
    // block writes inside the buffer)
    const bool blk_ok = XQ_CHECKED(j >= 0 && 32 * j + 32 <= J.K, kChkQuantX) &&
                        XQ_CHECKED(L.s8 + 4 * (static_cast<size_t>(J.M) * nsub) <= J.total, kChkQuantQ8) &&
                        XQ_CHECKED(L.ttiles != 0 || L.fsc + static_cast<size_t>((m >> 3) + 1) * nsub * 64 <= J.total,
                                   kChkQuantImage) &&
                        XQ_CHECKED(L.ttiles == 0 || L.tile + (static_cast<size_t>(m >> 7) + 1) * (J.K >> 8) *
                                                                   kTileRecord <= J.total,
                                   kChkQuantImage);
    if (!blk_ok) continue;
    if (m < J.M) {
      const size_t idx = static_cast<size_t>(m) * J.K + 32 * j + lane;
      float v = __ldg(J.x + idx);
      if (J.up) {
        // SwiGLU feed of the down projection
        v = swiglu(v, __ldg(J.up + idx));
        if (J.h_out) J.h_out[idx] = v;
      }
      const Q8Lane r = q8_quantize_lane(v);
      q = r.q;
      d = r.d;
      s = r.s;
      J.xq[static_cast<size_t>(m) * J.K + 32 * j + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
      if (lane == 0) {
        reinterpret_cast<float*>(J.xq + L.d8)[static_cast<size_t>(m) * nsub + j] = d;
        reinterpret_cast<float*>(J.xq + L.s8)[static_cast<size_t>(m) * nsub + j] = s;
      }
    }
    if (L.ttiles == 0) {
      // GEMV operand image (zeros for padding tokens)
      write_gemv_image(J.xq + L.frag, J.xq + L.fsc, nsub, m, j, lane, q, d, s);
    } else {
      // tile image: token r of tile tt, 32-block j = 8b + ib
      const int tt = m >> 7, r = m & 127, b = j >> 3, ib = j & 7;
      uint8_t* rec = J.xq + L.tile + (static_cast<size_t>(tt) * (J.K >> 8) + b) * kTileRecord;
      uint8_t* item = rec + ib * kTileItem;
      const int ks = (lane & ~7) | slot;  // k-slot of this lane's feature
      *reinterpret_cast<__half*>(item + tile_offset(r, ks)) = __int2half_rn(q);
      if (lane == 0) reinterpret_cast<float*>(item + kTileItemOp)[r] = d;
      uint8_t* beta = rec + 8 * kTileItem;
      if (lane < 3) {
        // s8 = p0 + p1 + p2, each piece a bf16 (upper 16 bits of an fp32)
        const float p0 = __uint_as_float(__float_as_uint(s) & 0xFFFF0000u);
        const float r1 = __fsub_rn(s, p0);
        const float p1 = __uint_as_float(__float_as_uint(r1) & 0xFFFF0000u);
        const float p2 = __fsub_rn(r1, p1);
        const float pc = lane == 0 ? p0 : (lane == 1 ? p1 : p2);
        *reinterpret_cast<uint16_t*>(beta + tile_offset(r, 3 * ib + lane)) =
            static_cast<uint16_t>(__float_as_uint(pc) >> 16);
      } else if (ib == 7 && lane < 11) {
        *reinterpret_cast<uint16_t*>(beta + tile_offset(r, 21 + lane)) = 0;
      }
    }
  }
}

// The same quantization for inputs whose Q8 buffer holds the tile image
// (M > 64 tokens): one warp per (token, 256-feature super-block), lane l
// taking feature l of each of its eight 32-blocks, so that eight 128-byte
// loads are in flight per warp and each block's max and quant sum come from
// warp reductions. Every element goes through the steps of q8_quantize_lane
// (the max and the integer sum do not depend on their order), so the bytes
// equal quantize_q8_kernel's. Padding tokens of the last 128-token tile get
// zeros in the image, as there.
__global__ void __launch_bounds__(256)
quantize_q8_tile_kernel(const __grid_constant__ QuantGroup G) {
  const int lane = threadIdx.x & 31;
  const unsigned warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  const unsigned total = G.blk0[G.n] >> 3;  // super-block units (blk0 counts padded 32-blocks)
  {
    int jb = 0;
    for (unsigned u = warp; u < total; u += nwarps) {
      while (u >= (G.blk0[jb + 1] >> 3)) ++jb;
      const QuantItem& J = G.job[jb];
      const unsigned local = u - (G.blk0[jb] >> 3);
      const int nsb = J.K >> 8;
      const int m = static_cast<int>(local / static_cast<unsigned>(nsb));
      const int b = static_cast<int>(local - static_cast<unsigned>(m) * nsb);
      if (m < J.M && lane < 8) {
        const size_t idx = static_cast<size_t>(m) * J.K + 256 * b + 32 * lane;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(J.x + idx));
        if (J.up) asm volatile("prefetch.global.L2 [%0];" ::"l"(J.up + idx));
      }
    }
  }
  cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < G.zero_count; i += blockDim.x) G.zero_words[i] = 0u;
  const int ks = (lane & ~7) | gemv_image_slot(lane);  // k-slot of this lane's feature in a tile item

  int jb = 0;
  for (unsigned u = warp; u < total; u += nwarps) {
    while (u >= (G.blk0[jb + 1] >> 3)) ++jb;
    const QuantItem& J = G.job[jb];
    const unsigned local = u - (G.blk0[jb] >> 3);
    const int nsb = J.K >> 8, nsub = J.nsub;
    const int m = static_cast<int>(local / static_cast<unsigned>(nsb));
    const int b = static_cast<int>(local - static_cast<unsigned>(m) * nsb);
    const bool live = m < J.M;
    if (!XQ_CHECKED(J.ttiles > 0 && J.tile + (static_cast<size_t>(m >> 7) + 1) * nsb * kTileRecord <= J.total &&
                        J.s8 + 4 * (static_cast<size_t>(J.M) * nsub) <= J.total,
                    kChkQuantImage))
      continue;
    float v[8];
    const size_t base = static_cast<size_t>(m) * J.K + 256 * b + lane;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = live ? __ldg(J.x + base + 32 * i) : 0.0f;
    if (J.up && live) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = swiglu(v[i], __ldg(J.up + base + 32 * i));
        if (J.h_out) J.h_out[base + 32 * i] = v[i];
      }
    }
    float d[8], sc[8];
    int q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // the steps of q8_quantize_lane, block i
      const unsigned amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[i])));
      d[i] = __fdiv_rn(__uint_as_float(amax_bits), 127.0f);
      const float id = (d[i] != 0.0f) ? __frcp_rn(d[i]) : 0.0f;
      float x = roundf(__fmul_rn(v[i], id));
      x = (x != x) ? 0.0f : x;
      x = x > 127.0f ? 127.0f : (x < -127.0f ? -127.0f : x);
      q[i] = static_cast<int>(x);
      sc[i] = __fmul_rn(d[i], static_cast<float>(__reduce_add_sync(0xffffffffu, q[i])));
    }
    if (live) {
#pragma unroll
      for (int i = 0; i < 8; ++i) J.xq[base + 32 * i] = static_cast<uint8_t>(static_cast<int8_t>(q[i]));
      if (lane < 8) {
        float dl = d[0], sl = sc[0];
#pragma unroll
        for (int i = 1; i < 8; ++i)
          if (lane == i) {
            dl = d[i];
            sl = sc[i];
          }
        reinterpret_cast<float*>(J.xq + J.d8)[static_cast<size_t>(m) * nsub + 8 * b + lane] = dl;
        reinterpret_cast<float*>(J.xq + J.s8)[static_cast<size_t>(m) * nsub + 8 * b + lane] = sl;
      }
    }
    // tile image record (tile m / 128, super-block b), token r = m % 128
    const int r = m & 127;
    uint8_t* rec = J.xq + J.tile + (static_cast<size_t>(m >> 7) * nsb + b) * kTileRecord;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint8_t* item = rec + i * kTileItem;
      *reinterpret_cast<__half*>(item + tile_offset(r, ks)) = __int2half_rn(q[i]);
      if (lane == i) reinterpret_cast<float*>(item + kTileItemOp)[r] = d[i];
    }
    // min-term operand: slot 3i + p holds bf16 piece p of s8 of block i
    // (s8 = p0 + p1 + p2, each the upper 16 bits of an fp32), slots 24-31 zero
    uint16_t piece = 0;
    if (lane < 24) {
      const int i = lane / 3, pc = lane - 3 * i;
      float sv = sc[0];
#pragma unroll
      for (int k = 1; k < 8; ++k)
        if (i == k) sv = sc[k];
      const float p0 = __uint_as_float(__float_as_uint(sv) & 0xFFFF0000u);
      const float r1 = __fsub_rn(sv, p0);
      const float p1 = __uint_as_float(__float_as_uint(r1) & 0xFFFF0000u);
      const float p2 = __fsub_rn(r1, p1);
      const float pv = pc == 0 ? p0 : (pc == 1 ? p1 : p2);
      piece = static_cast<uint16_t>(__float_as_uint(pv) >> 16);
    }
    *reinterpret_cast<uint16_t*>(rec + 8 * kTileItem + tile_offset(r, lane)) = piece;
  }
}

cudaError_t take_quant_check(unsigned int* code) { return take_check_word(code); }

cudaError_t launch_quantize_q8(const QuantJob* jobs, int n, cudaStream_t s, bool pdl, unsigned int* zero_words,
                               int zero_count) {
  if (n <= 0 || n > kMaxProj) return cudaErrorInvalidValue;
  QuantGroup G;
  G.n = n;
  G.zero_words = zero_words;
  G.zero_count = zero_words ? zero_count : 0;
  G.blk0[0] = 0;
  long long nblocks = 0;
  for (int k = 0; k < n; ++k) {
    const QuantJob& q = jobs[k];
    const Q8Layout L = q8_layout(q.M, q.K, q.gemv_image);
    QuantItem& it = G.job[k];
    it.x = q.x;
    it.up = q.up;
    it.h_out = q.h_out;
    it.xq = q.xq;
    it.d8 = L.d8;
    it.s8 = L.s8;
    it.frag = L.frag;
    it.fsc = L.fsc;
    it.tile = L.tile;
    it.total = L.total;
    it.M = q.M;
    it.K = q.K;
    it.nsub = q.K / 32;
    it.ttiles = L.ttiles;
    // padded token count: the operand image's chunk (8) or tile (128)
    const long long mp = (q.M > kGemvMaxTokens && !q.gemv_image) ? 128LL * ((q.M + 127) / 128) : 8LL * ((q.M + 7) / 8);
    nblocks += mp * (q.K / 32);
    if (nblocks >= (1LL << 31)) return cudaErrorInvalidValue;
    G.blk0[k + 1] = static_cast<unsigned>(nblocks);
  }
  if (nblocks == 0) return cudaSuccess;
  bool tiles = true;  // every input in the tile layout: the super-block quantizer
  for (int k = 0; k < n; ++k) tiles = tiles && G.job[k].ttiles > 0;
  if (tiles) {
    const long long units = nblocks / 8;
    long long want = (units + 7) / 8;  // 8 warps per CTA, one super-block per warp and pass
    const long long cap = static_cast<long long>(kNumSMs) * 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, quantize_q8_tile_kernel, G);
  }
  long long want = (nblocks + 31) / 32;  // 32 warps per CTA, one block per warp
  const long long cap = static_cast<long long>(kNumSMs) * 2;  // all resident
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
  cfg.blockDim = dim3(1024);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quantize_q8_kernel, G);
}

}  // namespace xq
