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
// projection of the launch. A task is 64 rows (4 warps x 16 rows, full K),
// 32 rows (2 warps split K in halves) or 16 rows (4 warps split K in
// quarters), chosen per projection so every warp streams 12..24 super-blocks;
// split-K partials meet in shared memory in a fixed order. Each warp keeps
// the next super-block's weight loads in flight while it computes the
// current one, across task boundaries.
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

struct Raw {
  uint2 q[2][4];  // [row n8 / n8+8][g]
  uint4 h[2];     // super-block headers of the two rows
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

__device__ __forceinline__ void load_raw(Raw& r, const Proj& P, int rg, int b, int n8, int t) {
  const int nsb = P.K >> 8;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = rg * 16 + n8 + 8 * h;
    if (row < P.N) {
      const uint8_t* blk = P.W + (static_cast<size_t>(row) * nsb + b) * kQ4kBytes;
      r.h[h] = ld_stream16(blk);
#pragma unroll
      for (int g = 0; g < 4; ++g) r.q[h][g] = ld_stream8(blk + 16 + 32 * g + 8 * t);
    } else {
      r.h[h] = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int g = 0; g < 4; ++g) r.q[h][g] = make_uint2(0, 0);
    }
  }
}

__device__ __forceinline__ void mma16816(float (&d)[4], unsigned a0, unsigned a1, unsigned a2,
                                         unsigned a3, unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool ISUM>
__device__ __forceinline__ void compute_step(const Raw& r, const Proj& P, int rg, int b, int n8,
                                             int t, int lane, float (&acc)[4]) {
  // Scales: sc and m of the 8 sub-blocks as packed bytes, for both rows.
  unsigned scw[2][2], mnw[2][2];
  float dl[2], dh[2], dm[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 hd = r.h[h];
    scw[h][0] = hd.y & 0x3F3F3F3Fu;
    mnw[h][0] = hd.z & 0x3F3F3F3Fu;
    scw[h][1] = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
    mnw[h][1] = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
    const float d = half_bits_to_float(hd.x);
    dl[h] = d * 16777216.0f;  // 2^24: low-nibble sums arrive as isum * 2^-24
    dh[h] = d * 1048576.0f;   // 2^20: high-nibble sums arrive as 16 * isum * 2^-24
    dm[h] = half_bits_to_float(hd.x >> 16);
  }
  const int nsub = P.K >> 5;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const unsigned w0a = r.q[0][g].x, w1a = r.q[0][g].y;  // row n8
    const unsigned w0b = r.q[1][g].x, w1b = r.q[1][g].y;  // row n8 + 8
    const unsigned s0a = w0a >> 8, s1a = w1a >> 8, s0b = w0b >> 8, s1b = w1b >> 8;
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      const unsigned mk = hi ? 0x00F000F0u : 0x000F000Fu;
      const int j = 2 * g + hi;
      const int sb = 8 * b + j;
      const uint4 B = __ldg(P.frag + static_cast<size_t>(sb) * 32 + lane);
      float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      mma16816(D, w0a & mk, w0b & mk, s0a & mk, s0b & mk, B.x, B.y);
      mma16816(D, w1a & mk, w1b & mk, s1a & mk, s1b & mk, B.z, B.w);
      const float4 f = __ldg(P.fsc + static_cast<size_t>(sb) * 4 + t);
      const int sh = 8 * (j & 3);
      const float sc0 = static_cast<float>((scw[0][j >> 2] >> sh) & 0xFFu);
      const float sc1 = static_cast<float>((scw[1][j >> 2] >> sh) & 0xFFu);
      const float mn0 = static_cast<float>((mnw[0][j >> 2] >> sh) & 0xFFu);
      const float mn1 = static_cast<float>((mnw[1][j >> 2] >> sh) & 0xFFu);
      const float a0 = (hi ? dh[0] : dl[0]) * sc0, a1 = (hi ? dh[1] : dl[1]) * sc1;
      const float b0 = dm[0] * mn0, b1 = dm[1] * mn1;
      acc[0] = fmaf(a0 * f.x, D[0], fmaf(-b0, f.z, acc[0]));
      acc[1] = fmaf(a0 * f.y, D[1], fmaf(-b0, f.w, acc[1]));
      acc[2] = fmaf(a1 * f.x, D[2], fmaf(-b1, f.z, acc[2]));
      acc[3] = fmaf(a1 * f.y, D[3], fmaf(-b1, f.w, acc[3]));
      if (ISUM) {
        const float scale = hi ? 1048576.0f : 16777216.0f;
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

template <bool ISUM>
__global__ void __launch_bounds__(128)
gemv_q4k_mma_kernel(const __grid_constant__ Group G) {
  cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int n8 = lane >> 2, t = lane & 3;
  __shared__ float4 red[2][4][32];
  int nbar = 0;

  int task = blockIdx.x;
  Pos cur = locate(G, task, warp);
  Raw rc;
  if (cur.valid) load_raw(rc, G.p[cur.p], cur.rg, cur.b0, n8, t);
  while (cur.valid) {
    const Proj& P = G.p[cur.p];
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    Pos nxt = cur;
#pragma unroll 1
    for (int b = cur.b0; b < cur.b1; ++b) {
      int nb = b + 1;
      if (nb >= cur.b1) {
        nxt = locate(G, task + gridDim.x, warp);
        nb = nxt.b0;
      }
      Raw rn;
      if (nxt.valid) load_raw(rn, G.p[nxt.p], nxt.rg, nb, n8, t);
      compute_step<ISUM>(rc, P, cur.rg, b, n8, t, lane, acc);
      rc = rn;
    }
    if (P.kw == 1) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = cur.rg * 16 + n8 + 8 * (e >> 1);
        const int col = 2 * t + (e & 1);
        if (row < P.N && col < P.M) P.y[static_cast<size_t>(col) * P.N + row] = acc[e];
      }
    } else {
      const int buf = nbar & 1;
      ++nbar;
      red[buf][warp][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      __syncthreads();
      if (warp % P.kw == 0) {
        float4 v = red[buf][warp][lane];
        for (int w = 1; w < P.kw; ++w) {
          const float4 u = red[buf][warp + w][lane];
          v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
        }
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = cur.rg * 16 + n8 + 8 * (e >> 1);
          const int col = 2 * t + (e & 1);
          if (row < P.N && col < P.M) P.y[static_cast<size_t>(col) * P.N + row] = vv[e];
        }
      }
    }
    task += gridDim.x;
    cur = nxt;
  }
}

// Split-K factor: keep every warp at 12..24 super-blocks of one row group.
int choose_kw(int nsb) {
  if (nsb > 40) return 4;
  if (nsb > 24) return 2;
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
