// Q4_K x Q8 -> fp32 for a small token batch M (1..8), integer dot products.
//
// What it computes (xLLM v0.7 long-context article, section 一; M template
// of section B2; batched MMVQ of the Agent Telemetry log): for each output
// row n and token m,
//   y[m][n] = sum over super-blocks b, sub-blocks j of
//             d*sc_j*d8[m][8b+j]*isum_j  -  dmin*m_j*s8[m][8b+j]
//   isum_j  = sum_{i<32} q[32j+i] * q8[m][256b+32j+i]   (exact int32)
// Each weight byte is read once for all M tokens.
//
// Work split. A warp covers 8 super-blocks per step: lane = 4*slot + g, slot
// picks the super-block, g the 32 quant bytes 32g..32g+31, i.e. the low
// nibbles (sub-block 2g) and high nibbles (sub-block 2g+1). So every lane
// owns two whole sub-blocks and produces their exact integer sums by itself.
// A warp handles R rows at once, so each activation load serves R rows. kw
// warps of a CTA split the super-blocks of the same rows (for short rows or
// few rows); their partial sums meet in shared memory in a fixed order.
//
// Unpacking: low nibbles are q & 0x0F0F0F0F; high nibbles are taken as
// q & 0xF0F0F0F0 (16x the quant, as unsigned bytes) and the 1/16 is applied
// to the exact integer sum, so no shift is needed per word.
#include "xq_common.cuh"

namespace xq {

// (sc, m) for sub-blocks 2g and 2g+1, packed as two bytes each.
// s0, s1, s2 are the 12 scale bytes 0..3, 4..7, 8..11 of the super-block:
//   j < 4 : sc = s[j] & 63,                          m = s[j+4] & 63
//   j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4
__device__ __forceinline__ void q4k_scale_pair(unsigned s0, unsigned s1, unsigned s2, int g,
                                               unsigned& sc2, unsigned& mn2) {
  const int sh = (g & 1) * 16;
  const unsigned a = s0 >> sh, b = s1 >> sh, c = s2 >> sh;
  if (g < 2) {
    sc2 = a & 0x3F3Fu;
    mn2 = b & 0x3F3Fu;
  } else {
    sc2 = (c & 0x0F0Fu) | ((a >> 2) & 0x3030u);
    mn2 = ((c >> 4) & 0x0F0Fu) | ((b >> 2) & 0x3030u);
  }
}

template <int M, int R, bool ISUM>
__global__ void __launch_bounds__(256)
gemv_q4k_dp4a_kernel(GemvArgs a, int kw) {
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int slot = lane >> 2;
  const int g = lane & 3;
  const int kk = wib % kw;
  const int rg = wib / kw;
  const int groups = 8 / kw;
  const int K = a.K, N = a.N;
  const int nsb = K >> 8;
  const int nsub = K >> 5;
  const long long row0 = (static_cast<long long>(blockIdx.x) * groups + rg) * R;

  float acc[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;

  for (int b = slot + 8 * kk; b < nsb; b += 8 * kw) {
    uint4 hdr[R], qa[R], qb[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const long long row = row0 + r;
      if (row < N) {
        const uint8_t* blk = a.W + (static_cast<size_t>(row) * nsb + b) * kQ4kBytes;
        hdr[r] = ld_stream16(blk);
        qa[r] = ld_stream16(blk + 16 + 32 * g);
        qb[r] = ld_stream16(blk + 32 + 32 * g);
      } else {
        hdr[r] = make_uint4(0, 0, 0, 0);
        qa[r] = hdr[r];
        qb[r] = hdr[r];
      }
    }
    // Per-row scale factors for the two sub-blocks this lane owns.
    float al[R], ah[R], bl[R], bh[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      unsigned sc2, mn2;
      q4k_scale_pair(hdr[r].y, hdr[r].z, hdr[r].w, g, sc2, mn2);
      const float d = half_bits_to_float(hdr[r].x);
      const float dmin = half_bits_to_float(hdr[r].x >> 16);
      al[r] = d * static_cast<float>(sc2 & 0xFFu);
      ah[r] = d * static_cast<float>(sc2 >> 8);
      bl[r] = dmin * static_cast<float>(mn2 & 0xFFu);
      bh[r] = dmin * static_cast<float>(mn2 >> 8);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int8_t* xa = a.qs + static_cast<size_t>(m) * K + static_cast<size_t>(b) * 256 + 64 * g;
      const uint4 x0 = ld_act16(xa);
      const uint4 x1 = ld_act16(xa + 16);
      const uint4 x2 = ld_act16(xa + 32);
      const uint4 x3 = ld_act16(xa + 48);
      const size_t si = static_cast<size_t>(m) * nsub + 8 * b + 2 * g;
      const float2 dd = __ldg(reinterpret_cast<const float2*>(a.d8 + si));
      const float2 ss = __ldg(reinterpret_cast<const float2*>(a.s8 + si));
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const unsigned L = 0x0F0F0F0Fu, H = 0xF0F0F0F0u;
        int lo = 0, hi = 0;
        lo = dp4a_us(qa[r].x & L, x0.x, lo);
        lo = dp4a_us(qa[r].y & L, x0.y, lo);
        lo = dp4a_us(qa[r].z & L, x0.z, lo);
        lo = dp4a_us(qa[r].w & L, x0.w, lo);
        lo = dp4a_us(qb[r].x & L, x1.x, lo);
        lo = dp4a_us(qb[r].y & L, x1.y, lo);
        lo = dp4a_us(qb[r].z & L, x1.z, lo);
        lo = dp4a_us(qb[r].w & L, x1.w, lo);
        hi = dp4a_us(qa[r].x & H, x2.x, hi);
        hi = dp4a_us(qa[r].y & H, x2.y, hi);
        hi = dp4a_us(qa[r].z & H, x2.z, hi);
        hi = dp4a_us(qa[r].w & H, x2.w, hi);
        hi = dp4a_us(qb[r].x & H, x3.x, hi);
        hi = dp4a_us(qb[r].y & H, x3.y, hi);
        hi = dp4a_us(qb[r].z & H, x3.z, hi);
        hi = dp4a_us(qb[r].w & H, x3.w, hi);
        hi >>= 4;  // exact: hi is 16 * (sum of high-nibble products)
        float t = acc[r][m];
        t = fmaf(al[r] * dd.x, static_cast<float>(lo), t);
        t = fmaf(ah[r] * dd.y, static_cast<float>(hi), t);
        t = fmaf(-bl[r], ss.x, t);
        t = fmaf(-bh[r], ss.y, t);
        acc[r][m] = t;
        if (ISUM) {
          const long long row = row0 + r;
          if (row < N) {
            int32_t* o = a.isum + (static_cast<size_t>(m) * N + row) * nsub + 8 * b + 2 * g;
            *reinterpret_cast<int2*>(o) = make_int2(lo, hi);
          }
        }
      }
    }
  }

  // Warp tree reduction of every (row, token) partial.
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = acc[r][m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[r][m] = v;
    }

  if (kw == 1) {
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const long long row = row0 + r;
        if (row < N)
#pragma unroll
          for (int m = 0; m < M; ++m) a.y[m * a.ldy + row] = acc[r][m];
      }
    }
    return;
  }
  // kw warps share these rows: combine in shared memory in warp order.
  __shared__ float red[8][R * M];
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) red[wib][r * M + m] = acc[r][m];
  }
  __syncthreads();
  if (kk == 0 && lane < R * M) {
    const int r = lane / M, m = lane % M;
    float v = red[wib][lane];
    for (int w = 1; w < kw; ++w) v += red[wib + w][lane];
    const long long row = row0 + r;
    if (row < N) a.y[m * a.ldy + row] = v;
  }
}

// Warps of a CTA that split one row's super-blocks: as many 8-block steps as
// the row has, up to 8. It depends on K only, so a row's summation order,
// and with it every output bit, is the same whatever N (or slice of N) is
// launched.
static int choose_kw(int nsb) {
  int kw = 1;
  while (kw < 8 && 8 * (2 * kw) <= nsb) kw *= 2;
  return kw;
}

template <int M, bool ISUM>
static cudaError_t launch_m(const GemvArgs& a, cudaStream_t s) {
  constexpr int R = (M <= 4) ? 4 : 2;
  const int nsb = a.K >> 8;
  const int kw = choose_kw(nsb);
  const long long rows_per_cta = static_cast<long long>(8 / kw) * R;
  const long long grid = (a.N + rows_per_cta - 1) / rows_per_cta;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  gemv_q4k_dp4a_kernel<M, R, ISUM><<<static_cast<unsigned>(grid), 256, 0, s>>>(a, kw);
  return cudaGetLastError();
}

template <bool ISUM>
static cudaError_t dispatch(const GemvArgs& a, cudaStream_t s) {
  switch (a.M) {
    case 1: return launch_m<1, ISUM>(a, s);
    case 2: return launch_m<2, ISUM>(a, s);
    case 3: return launch_m<3, ISUM>(a, s);
    case 4: return launch_m<4, ISUM>(a, s);
    case 5: return launch_m<5, ISUM>(a, s);
    case 6: return launch_m<6, ISUM>(a, s);
    case 7: return launch_m<7, ISUM>(a, s);
    case 8: return launch_m<8, ISUM>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemv_q4k(const GemvArgs& a, cudaStream_t s) {
  return a.isum ? dispatch<true>(a, s) : dispatch<false>(a, s);
}

}  // namespace xq
