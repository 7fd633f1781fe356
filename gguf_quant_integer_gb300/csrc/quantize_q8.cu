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
// (M > 64 tokens): one warp per 8 tokens x one 256-feature super-block.
// Lane l takes token 8u + l/4 and features 8g..8g+7 (g = l%4) of each of the
// eight 32-blocks, so each lane keeps its 16 16-byte loads in flight and
// stores whole 16-byte chunks: 8 fp16 quants of the tile operand (k-slots
// 8g..8g+7 of its token, in operand slot order), 8 int8 quants of qs, and 8
// bf16 pieces of the min-term operand. Every element goes through the steps
// of q8_quantize_lane, the block max and quant sum taken over the token's 4
// lanes (neither depends on its order), so the bytes equal
// quantize_q8_kernel's. Padding tokens of the last 128-token tile get zeros
// in the image, as there.
__global__ void __launch_bounds__(256)
quantize_q8_tile_kernel(const __grid_constant__ QuantGroup G) {
  const int lane = threadIdx.x & 31;
  const int t = lane >> 2, g = lane & 3;
  const unsigned warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
  // units: (8-token group, super-block) of every job; blk0 counts padded
  // 32-blocks, 64 of them per unit
  const unsigned total = G.blk0[G.n] >> 6;
  {
    int jb = 0;
    for (unsigned u = warp; u < total; u += nwarps) {
      while (u >= (G.blk0[jb + 1] >> 6)) ++jb;
      const QuantItem& J = G.job[jb];
      const unsigned local = u - (G.blk0[jb] >> 6);
      const int nsb = J.K >> 8;
      const int m = 8 * static_cast<int>(local / static_cast<unsigned>(nsb)) + t;
      const int b = static_cast<int>(local % static_cast<unsigned>(nsb));
      if (m < J.M && g < 2) {  // the token's 1 KB of the super-block: 8 lines over its 4 lanes
        const size_t idx = static_cast<size_t>(m) * J.K + 256 * b + 128 * g;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(J.x + idx));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(J.x + idx + 32));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(J.x + idx + 64));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(J.x + idx + 96));
        if (J.up) {
          asm volatile("prefetch.global.L2 [%0];" ::"l"(J.up + idx));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(J.up + idx + 32));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(J.up + idx + 64));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(J.up + idx + 96));
        }
      }
    }
  }
  cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < G.zero_count; i += blockDim.x) G.zero_words[i] = 0u;

  int jb = 0;
  for (unsigned u = warp; u < total; u += nwarps) {
    while (u >= (G.blk0[jb + 1] >> 6)) ++jb;
    const QuantItem& J = G.job[jb];
    const unsigned local = u - (G.blk0[jb] >> 6);
    const int nsb = J.K >> 8, nsub = J.nsub;
    const int m = 8 * static_cast<int>(local / static_cast<unsigned>(nsb)) + t;
    const int b = static_cast<int>(local % static_cast<unsigned>(nsb));
    const bool live = m < J.M;
    if (!XQ_CHECKED(J.ttiles > 0 && J.tile + (static_cast<size_t>(m >> 7) + 1) * nsb * kTileRecord <= J.total &&
                        J.s8 + 4 * (static_cast<size_t>(J.M) * nsub) <= J.total,
                    kChkQuantImage))
      continue;
    // this lane's 64 features: 8 per 32-block, all loads issued first
    const size_t base = static_cast<size_t>(m) * J.K + 256 * b + 8 * g;
    float4 v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const size_t at = base + 32 * (k >> 1) + 4 * (k & 1);
      v[k] = live ? __ldg(reinterpret_cast<const float4*>(J.x + at)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    if (J.up && live) {
      // SwiGLU feed of the down projection
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const size_t at = base + 32 * (k >> 1) + 4 * (k & 1);
        const float4 w = __ldg(reinterpret_cast<const float4*>(J.up + at));
        v[k] = make_float4(swiglu(v[k].x, w.x), swiglu(v[k].y, w.y), swiglu(v[k].z, w.z), swiglu(v[k].w, w.w));
        if (J.h_out) *reinterpret_cast<float4*>(J.h_out + at) = v[k];
      }
    }
    const int r = m & 127;  // token of its 128-token tile
    uint8_t* rec = J.xq + J.tile + (static_cast<size_t>(m >> 7) * nsb + b) * kTileRecord;
    float sblk[8];  // s8 of the token's eight 32-blocks
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float e[8] = {v[2 * i].x, v[2 * i].y, v[2 * i].z, v[2 * i].w,
                          v[2 * i + 1].x, v[2 * i + 1].y, v[2 * i + 1].z, v[2 * i + 1].w};
      // the steps of q8_quantize_lane over the token's 4 lanes
      unsigned ab = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) ab = max(ab, __float_as_uint(fabsf(e[k])));
      ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 1));
      ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 2));
      const float d = __fdiv_rn(__uint_as_float(ab), 127.0f);
      const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
      int q[8], isum = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float x = roundf(__fmul_rn(e[k], id));
        x = (x != x) ? 0.0f : x;
        x = x > 127.0f ? 127.0f : (x < -127.0f ? -127.0f : x);
        q[k] = static_cast<int>(x);
        isum += q[k];
      }
      isum += __shfl_xor_sync(0xffffffffu, isum, 1);
      isum += __shfl_xor_sync(0xffffffffu, isum, 2);
      const float sc = __fmul_rn(d, static_cast<float>(isum));
      sblk[i] = sc;
      if (live) {
        uint2 qb;
        qb.x = (q[0] & 255) | (q[1] & 255) << 8 | (q[2] & 255) << 16 | static_cast<unsigned>(q[3] & 255) << 24;
        qb.y = (q[4] & 255) | (q[5] & 255) << 8 | (q[6] & 255) << 16 | static_cast<unsigned>(q[7] & 255) << 24;
        *reinterpret_cast<uint2*>(J.xq + base + 32 * i) = qb;
        if (g == 0) {
          reinterpret_cast<float*>(J.xq + J.d8)[static_cast<size_t>(m) * nsub + 8 * b + i] = d;
          reinterpret_cast<float*>(J.xq + J.s8)[static_cast<size_t>(m) * nsub + 8 * b + i] = sc;
        }
      }
      // tile operand of 32-block i: k-slots 8g..8g+7 of token r, slot s
      // holding feature perm(s) of the lane's 8 (perm = 0,2,1,3,4,6,5,7)
      uint8_t* item = rec + i * kTileItem;
      const __half2 h01 = __halves2half2(__int2half_rn(q[0]), __int2half_rn(q[2]));
      const __half2 h23 = __halves2half2(__int2half_rn(q[1]), __int2half_rn(q[3]));
      const __half2 h45 = __halves2half2(__int2half_rn(q[4]), __int2half_rn(q[6]));
      const __half2 h67 = __halves2half2(__int2half_rn(q[5]), __int2half_rn(q[7]));
      uint4 w;
      w.x = *reinterpret_cast<const unsigned*>(&h01);
      w.y = *reinterpret_cast<const unsigned*>(&h23);
      w.z = *reinterpret_cast<const unsigned*>(&h45);
      w.w = *reinterpret_cast<const unsigned*>(&h67);
      *reinterpret_cast<uint4*>(item + tile_offset(r, 8 * g)) = w;
      if (g == 0) reinterpret_cast<float*>(item + kTileItemOp)[r] = d;
    }
    // min-term operand: slot 3i + p holds bf16 piece p of s8 of block i
    // (s8 = p0 + p1 + p2, each the upper 16 bits of an fp32), slots 24-31
    // zero; this lane writes slots 8g..8g+7
    uint32_t pk[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t pair = 0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int slot = 8 * g + 2 * h + e;
        uint32_t piece = 0;
        if (slot < 24) {
          const int i = slot / 3, pc = slot - 3 * i;
          float sv = sblk[0];
#pragma unroll
          for (int k = 1; k < 8; ++k)
            if (i == k) sv = sblk[k];
          const float p0 = __uint_as_float(__float_as_uint(sv) & 0xFFFF0000u);
          const float r1 = __fsub_rn(sv, p0);
          const float p1 = __uint_as_float(__float_as_uint(r1) & 0xFFFF0000u);
          const float p2 = __fsub_rn(r1, p1);
          const float pv = pc == 0 ? p0 : (pc == 1 ? p1 : p2);
          piece = __float_as_uint(pv) >> 16;
        }
        pair |= piece << (16 * e);
      }
      pk[h] = pair;
    }
    *reinterpret_cast<uint4*>(rec + 8 * kTileItem + tile_offset(r, 8 * g)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
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
    const long long units = nblocks / 64;
    long long want = (units + 7) / 8;  // 8 warps per CTA, 8 tokens x one super-block per warp and pass
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
