// Q4_K x Q8 -> fp32 for M <= 8 tokens on the tensor cores (mma.sync
// m16n8k16, fp16 operands holding exact integers, fp32 accumulation).
//
// What it computes (xLLM v0.7 long-context article, section 一; M template
// of section B2): for output row n and token m,
//   y[m][n] = sum over super-blocks b, sub-blocks j of
//             d*sc_j*d8[m][8b+j]*isum_j  -  dmin*m_j*s8[m][8b+j]
//   isum_j  = sum_{i<32} q[32j+i] * q8[m][256b+32j+i]        (exact)
//
// Why tensor cores at M <= 8: with one dp4a per 4 MACs, a 144-byte Q4_K
// super-block costs 512 dp4a at M = 8, which at 64 integer ops per clock per
// SM is slower than the HBM stream on GB300. One m16n8k16 MMA does the 2048
// MACs of 16 rows x 16 weights x 8 tokens. It is not a dequantization: the
// A operand is the raw 4-bit quant, the B operand the raw int8 activation.
//
// Exactness. A quant nibble masked in place, q & 0x000F000F, is the fp16 bit
// pattern of the subnormal q * 2^-24; a high nibble masked in place,
// q & 0x00F000F0, is 16q * 2^-24. The activations are fp16 integers in
// [-127, 127]. Every product and every partial sum of a 32-weight sub-block
// is an integer multiple of 2^-24 below 2^-2 in magnitude, so the fp32
// accumulation is exact and isum = D * 2^24 (low nibbles) or D * 2^20 (high
// nibbles), bit for bit. The 2^24 / 2^20 factors are folded into d.
//
// Fragment mapping. Lane (n8 = lane/4, t = lane%4) loads 8 quant bytes
// 32g + 8t .. 32g + 8t + 7 of rows n8 and n8+8 for each g = 0..3: its low
// nibbles are positions 8t..8t+7 of sub-block 2g, its high nibbles the same
// positions of sub-block 2g+1. Even bytes (mask) and odd bytes (shift 8,
// mask) give the k-slot pairs (2t, 2t+1) and (2t+8, 2t+9) of two MMAs; the
// activation image written by the quantizer uses the same position order.
//
// Schedule. Persistent CTAs of 4 warps walk a task list covering every
// projection of the launch. A task is 16 rows whose K is split in quarters
// over the 4 warps (halves or whole for K < 1024); the partials meet in
// shared memory in a fixed order. Each warp keeps the next super-block's
// weight loads in flight while it computes the current one, across task
// boundaries.
#include "xq_common.cuh"

namespace xq {

namespace {

struct Proj {
  const uint8_t* W;
  const uint4* frag;   // [K/32][32] 16-byte lane operands (chunk 0)
  const float4* fsc;   // [K/32][4]
  float* y;
  int32_t* isum;
  int N, K, M, kw, task0;
};

struct Group {
  Proj p[kMaxProj];
  int n, total;
};

struct Pos {
  int p, rg, b0, b1;
  bool valid;
};

__device__ __forceinline__ Pos locate(const Group& G, int task, int warp) {
  Pos s;
  s.valid = task < G.total;
  if (!s.valid) {
    s.p = 0; s.rg = 0; s.b0 = 0; s.b1 = 0;
    return s;
  }
  int p = 0;
#pragma unroll 1
  while (p + 1 < G.n && task >= G.p[p + 1].task0) ++p;
  const Proj& P = G.p[p];
  const int kw = P.kw;
  const int tl = task - P.task0;
  const int nsb = P.K >> 8;
  const int kp = warp % kw;
  s.p = p;
  s.rg = tl * (4 / kw) + warp / kw;
  s.b0 = nsb * kp / kw;
  s.b1 = nsb * (kp + 1) / kw;
  return s;
}

__device__ __forceinline__ void mma16816(float (&d)[4], unsigned a0, unsigned a1, unsigned a2,
                                         unsigned a3, unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kRing = 4;            // weight steps in flight per warp
constexpr int kStepBytes = 16 * kQ4kBytes;  // 16 rows x one super-block

// Shared-memory slot of weight row i (0..15) of a step. Lane (n8, t) reads
// rows n8 and n8+8; with 144-byte rows, slot 2*(n8%4) + n8/4 puts the four
// rows a half-warp reads 8 banks apart, so the 8-byte quant loads and the
// 16-byte header loads are conflict-free.
__device__ __forceinline__ int row_slot(int i) {
  return 8 * (i >> 3) + 2 * (i & 3) + ((i >> 2) & 1);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

// Packed fp32 pairs.
__device__ __forceinline__ unsigned long long pk(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float lo32(unsigned long long v) { return __uint_as_float(static_cast<unsigned>(v)); }
__device__ __forceinline__ float hi32(unsigned long long v) { return __uint_as_float(static_cast<unsigned>(v >> 32)); }

// Byte k of a packed word as 2^23 + byte, an exact fp32 (0x4B0000xx).
__device__ __forceinline__ float byte_plus_2p23(unsigned w, int k) {
  return __uint_as_float(prmt(w, 0x4B000000u, 0x7540u | static_cast<unsigned>(k)));
}

// Issue the copies of one step (16 rows x super-block b) into a ring slot.
// Chunk c (0..143) of the step is 16 bytes: row c/9, piece c%9.
__device__ __forceinline__ void issue_step(const Proj& P, int rg, int b, uint32_t slot_base, int lane) {
  const int nsb = P.K >> 8;
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int c = lane + 32 * k;
    if (c < 144) {
      const int i = c / 9, piece = c - 9 * (c / 9);
      const int row = rg * 16 + i;
      const bool ok = row < P.N;
      const uint8_t* src = ok ? P.W + (static_cast<size_t>(row) * nsb + b) * kQ4kBytes + 16 * piece : P.W;
      cp_async16(slot_base + row_slot(i) * kQ4kBytes + 16 * piece, src, ok ? 16u : 0u);
    }
  }
}

template <bool ISUM>
__device__ __forceinline__ void compute_step(const uint8_t* st, const Proj& P, int rg, int b, int n8,
                                             int t, int lane, unsigned long long (&acc)[2]) {
  // Weight operands of rows n8 and n8 + 8 from the ring slot.
  const int s0 = row_slot(n8), s1 = row_slot(n8 + 8);
  const uint4 h0 = *reinterpret_cast<const uint4*>(st + s0 * kQ4kBytes);
  const uint4 h1 = *reinterpret_cast<const uint4*>(st + s1 * kQ4kBytes);
  uint2 q0[4], q1[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    q0[g] = *reinterpret_cast<const uint2*>(st + s0 * kQ4kBytes + 16 + 32 * g + 8 * t);
    q1[g] = *reinterpret_cast<const uint2*>(st + s1 * kQ4kBytes + 16 + 32 * g + 8 * t);
  }
  // sc and m of the 8 sub-blocks as packed bytes:
  //   j < 4 : sc = s[j] & 63, m = s[j+4] & 63
  //   j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4
  unsigned scw[2][2], mnw[2][2];
  float dl[2], dh[2], dm[2];
  const uint4 hh[2] = {h0, h1};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 hd = hh[h];
    scw[h][0] = hd.y & 0x3F3F3F3Fu;
    mnw[h][0] = hd.z & 0x3F3F3F3Fu;
    scw[h][1] = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
    mnw[h][1] = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
    const float d = half_bits_to_float(hd.x);
    dl[h] = d * 16777216.0f;  // 2^24: low-nibble sums arrive as isum * 2^-24
    dh[h] = d * 1048576.0f;   // 2^20: high-nibble sums arrive as 16 * isum * 2^-24
    dm[h] = -half_bits_to_float(hd.x >> 16);
  }
  const int nsub = P.K >> 5;
  // Activation operands of the 8 sub-blocks, loaded one sub-block ahead.
  const uint4* fp = P.frag + static_cast<size_t>(8 * b) * 32 + lane;
  const float4* sp = P.fsc + static_cast<size_t>(8 * b) * 4 + t;
  uint4 Bn = __ldg(fp);
  float4 fn = __ldg(sp);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const unsigned w0a = q0[g].x, w1a = q0[g].y;  // row n8
    const unsigned w0b = q1[g].x, w1b = q1[g].y;  // row n8 + 8
    const unsigned s0a = w0a >> 8, s1a = w1a >> 8, s0b = w0b >> 8, s1b = w1b >> 8;
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      const unsigned mk = hi ? 0x00F000F0u : 0x000F000Fu;
      const int j = 2 * g + hi;
      const uint4 B = Bn;
      const float4 f = fn;
      if (j < 7) {
        Bn = __ldg(fp + (j + 1) * 32);
        fn = __ldg(sp + (j + 1) * 4);
      }
      float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      mma16816(D, w0a & mk, w0b & mk, s0a & mk, s0b & mk, B.x, B.y);
      mma16816(D, w1a & mk, w1b & mk, s1a & mk, s1b & mk, B.z, B.w);
      // alpha = d*sc*2^24 (or 2^20), beta = -dmin*m, each from the byte via
      // (2^23 + byte)*x - 2^23*x: one rounding of an exact product.
      const int k = j & 3, wsel = j >> 2;
      const float a0 = fmaf(byte_plus_2p23(scw[0][wsel], k), hi ? dh[0] : dl[0], -8388608.0f * (hi ? dh[0] : dl[0]));
      const float a1 = fmaf(byte_plus_2p23(scw[1][wsel], k), hi ? dh[1] : dl[1], -8388608.0f * (hi ? dh[1] : dl[1]));
      const float b0 = fmaf(byte_plus_2p23(mnw[0][wsel], k), dm[0], -8388608.0f * dm[0]);
      const float b1 = fmaf(byte_plus_2p23(mnw[1][wsel], k), dm[1], -8388608.0f * dm[1]);
      const unsigned long long d8p = pk(f.x, f.y), s8p = pk(f.z, f.w);
      acc[0] = fma2(mul2(pk(a0, a0), d8p), pk(D[0], D[1]), fma2(pk(b0, b0), s8p, acc[0]));
      acc[1] = fma2(mul2(pk(a1, a1), d8p), pk(D[2], D[3]), fma2(pk(b1, b1), s8p, acc[1]));
      if (ISUM) {
        const float scale = hi ? 1048576.0f : 16777216.0f;
        const int sb = 8 * b + j;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = rg * 16 + n8 + 8 * (e >> 1);
          const int col = 2 * t + (e & 1);
          if (row < P.N && col < P.M)
            P.isum[(static_cast<size_t>(col) * P.N + row) * nsub + sb] = static_cast<int32_t>(D[e] * scale);
        }
      }
    }
  }
}

__device__ __forceinline__ void store_y(const Proj& P, int rg, int n8, int t, float v00, float v01,
                                        float v10, float v11) {
  const int r0 = rg * 16 + n8, r1 = r0 + 8, c0 = 2 * t, c1 = c0 + 1;
  if (r0 < P.N) {
    if (c0 < P.M) P.y[static_cast<size_t>(c0) * P.N + r0] = v00;
    if (c1 < P.M) P.y[static_cast<size_t>(c1) * P.N + r0] = v01;
  }
  if (r1 < P.N) {
    if (c0 < P.M) P.y[static_cast<size_t>(c0) * P.N + r1] = v10;
    if (c1 < P.M) P.y[static_cast<size_t>(c1) * P.N + r1] = v11;
  }
}

// A cursor over this warp's steps: (task, super-block) pairs.
struct Cursor {
  int task;
  Pos pos;
  int b;
};

__device__ __forceinline__ void cursor_init(Cursor& c, const Group& G, int task, int warp) {
  c.task = task;
  c.pos = locate(G, task, warp);
  c.b = c.pos.b0;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const Group& G, int warp) {
  if (++c.b >= c.pos.b1) cursor_init(c, G, c.task + gridDim.x, warp);
}

template <bool ISUM>
__global__ void __launch_bounds__(128, 4)
gemv_q4k_mma_kernel(const __grid_constant__ Group G) {
  cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int n8 = lane >> 2, t = lane & 3;
  __shared__ __align__(16) uint8_t ring[4][kRing][kStepBytes];
  __shared__ float4 red[2][4][32];
  int nbar = 0;
  const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(&ring[warp][0][0]));

  // Producer cursor runs kRing - 1 steps ahead of the consumer cursor.
  Cursor pc, cc;
  cursor_init(pc, G, blockIdx.x, warp);
  cc = pc;
  int issued = 0;
#pragma unroll
  for (int k = 0; k < kRing - 1; ++k) {
    if (pc.pos.valid) {
      issue_step(G.p[pc.pos.p], pc.pos.rg, pc.b, ring_base + (issued % kRing) * kStepBytes, lane);
      cursor_next(pc, G, warp);
    }
    cp_async_commit();
    ++issued;
  }
  int consumed = 0;
  while (cc.pos.valid) {
    const Proj& P = G.p[cc.pos.p];
    unsigned long long acc[2] = {0ull, 0ull};
    const int rg = cc.pos.rg;
    const int b1 = cc.pos.b1;
    for (int b = cc.pos.b0; b < b1; ++b) {
      if (pc.pos.valid) {
        issue_step(G.p[pc.pos.p], pc.pos.rg, pc.b, ring_base + (issued % kRing) * kStepBytes, lane);
        cursor_next(pc, G, warp);
      }
      cp_async_commit();
      ++issued;
      cp_async_wait<kRing - 1>();
      __syncwarp();
      compute_step<ISUM>(&ring[warp][consumed % kRing][0], P, rg, b, n8, t, lane, acc);
      __syncwarp();
      ++consumed;
    }
    if (P.kw == 1) {
      store_y(P, rg, n8, t, lo32(acc[0]), hi32(acc[0]), lo32(acc[1]), hi32(acc[1]));
    } else {
      const int buf = nbar & 1;
      ++nbar;
      red[buf][warp][lane] = make_float4(lo32(acc[0]), hi32(acc[0]), lo32(acc[1]), hi32(acc[1]));
      __syncthreads();
      if (warp % P.kw == 0) {
        float4 v = red[buf][warp][lane];
        for (int w = 1; w < P.kw; ++w) {
          const float4 u = red[buf][warp + w][lane];
          v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
        }
        store_y(P, rg, n8, t, v.x, v.y, v.z, v.w);
      }
    }
    cursor_init(cc, G, cc.task + gridDim.x, warp);
  }
  cp_async_wait<0>();
}

// Split-K factor: 4 warps share each 16-row group whenever K allows, so a
// layer has thousands of short tasks and the persistent grid ends evenly.
int choose_kw(int nsb) {
  if (nsb >= 4) return 4;
  if (nsb >= 2) return 2;
  return 1;
}

template <bool ISUM>
int max_ctas() {
  static int per_sm = -1;
  if (per_sm < 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_q4k_mma_kernel<ISUM>, 128, 0) != cudaSuccess || n < 1)
      n = 1;
    per_sm = n;
  }
  return per_sm * kNumSMs;
}

}  // namespace

cudaError_t launch_gemv_q4k_mma(const MmaProj* projs, int n, cudaStream_t s, bool pdl) {
  if (n <= 0 || n > kMaxProj) return cudaErrorInvalidValue;
  Group G;
  G.n = n;
  int total = 0;
  bool isum = false;
  for (int k = 0; k < n; ++k) {
    const MmaProj& q = projs[k];
    const int nsb = q.K >> 8;
    int kw = choose_kw(nsb);
    if (kw > nsb) kw = 1;
    const Q8Layout L = q8_layout(q.M_total, q.K);
    const int m0 = 8 * q.chunk;
    Proj& P = G.p[k];
    P.W = q.W;
    P.frag = reinterpret_cast<const uint4*>(q.xq + L.frag + static_cast<size_t>(q.chunk) * 16 * q.K);
    P.fsc = reinterpret_cast<const float4*>(q.xq + L.fsc + static_cast<size_t>(q.chunk) * 2 * q.K);
    P.y = q.y + static_cast<size_t>(m0) * q.N;
    P.isum = q.isum;
    P.N = q.N;
    P.K = q.K;
    P.M = (q.M_total - m0) < 8 ? (q.M_total - m0) : 8;
    P.kw = kw;
    P.task0 = total;
    const int rows_per_task = 16 * (4 / kw);
    total += (q.N + rows_per_task - 1) / rows_per_task;
    isum = isum || (q.isum != nullptr);
  }
  G.total = total;
  if (total == 0) return cudaSuccess;
  const int cap = isum ? max_ctas<true>() : max_ctas<false>();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(total < cap ? total : cap));
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return isum ? cudaLaunchKernelEx(&cfg, gemv_q4k_mma_kernel<true>, G)
              : cudaLaunchKernelEx(&cfg, gemv_q4k_mma_kernel<false>, G);
}

}  // namespace xq
