// Q6_K x Q8 -> fp32 for a small token batch M (1..8), integer dot products.
//
// What it computes (xLLM v0.7 long-context article, sections 一 and A2):
//   y[m][n] = sum over super-blocks b, 16-weight groups g of
//             d * s_g * d8[m][(256b+16g)/32] * isum_g
//   isum_g  = sum_{i<16} (q[16g+i] - 32) * q8[m][256b+16g+i]   (exact int32)
// with the 6-bit quant q = low 4 bits from ql | 2 bits from qh << 4 (public
// GGUF Q6_K layout: ql[128] @0, qh[64] @128, int8 scales[16] @192, d @208).
//
// Work split as for Q4_K: a warp covers 8 super-blocks per step, 4 lanes per
// super-block. Lane u = 2h + p takes half h (weights 128h..128h+127) and the
// 16-wide column p of its four 32-weight quarters, i.e. exactly the four
// scale groups g = 8h + 2qq + p (qq = 0..3). It needs 16 bytes of ql for
// quarters 0/2, 16 for quarters 1/3 and 16 of qh.
//
// Alignment: 210-byte blocks start on 2-byte boundaries only, so a 16-byte
// run is assembled from five aligned 32-bit words with a byte permute; the
// extra word read stays inside the same super-block.
//
// The -32 offset: sum (q-32)*a = dot(q, a) - 32*sum(a). The activation sums
// are computed once per token and reused for all R rows of the warp.
#include "xq_check.cuh"
#include "xq_common.cuh"

namespace xq {

// 16 bytes starting at a 2-byte aligned address, from aligned words.
__device__ __forceinline__ uint4 load16_a2(const uint8_t* p) {
  const uintptr_t ad = reinterpret_cast<uintptr_t>(p);
  const uint8_t* w = reinterpret_cast<const uint8_t*>(ad & ~static_cast<uintptr_t>(3));
  const unsigned sel = (ad & 2) ? 0x5432u : 0x3210u;
  const unsigned w0 = ld_stream4(w), w1 = ld_stream4(w + 4), w2 = ld_stream4(w + 8),
                 w3 = ld_stream4(w + 12), w4 = ld_stream4(w + 16);
  return make_uint4(prmt(w0, w1, sel), prmt(w1, w2, sel), prmt(w2, w3, sel), prmt(w3, w4, sel));
}

// 6-bit quants of one quarter: low nibbles (qq 0/1) or high nibbles (qq 2/3)
// of the ql word, plus bits 2qq..2qq+1 of each qh byte as bits 4..5.
__device__ __forceinline__ unsigned q6_word(unsigned ql, unsigned qh, int qq) {
  const unsigned lo = (qq >= 2 ? (ql >> 4) : ql) & 0x0F0F0F0Fu;
  const unsigned hi = ((qh >> (2 * qq)) & 0x03030303u) << 4;
  return lo | hi;
}

template <int M, int R, bool ISUM>
__global__ void __launch_bounds__(256)
gemv_q6k_dp4a_kernel(GemvArgs a, int kw) {
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int slot = lane >> 2;
  const int u = lane & 3;
  const int h = u >> 1, p = u & 1;
  const int kk = wib % kw;
  const int rg = wib / kw;
  const int groups = 8 / kw;
  const int K = a.K, N = a.N;
  const int nsb = K >> 8;
  const int nsub = K >> 5;
  const int ngrp = K >> 4;
  const long long row0 = (static_cast<long long>(blockIdx.x) * groups + rg) * R;

  float acc[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;

  for (int b = slot + 8 * kk; b < nsb; b += 8 * kw) {
    uint4 l0[R], l1[R], hh[R];
    float sd[R][4];  // d * s_g for the lane's four groups
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const long long row = row0 + r;
      if (row < N && XQ_CHECKED(row >= 0 && b >= 0 && (static_cast<size_t>(row) * nsb + b + 1) * kQ6kBytes <=
                                                          static_cast<size_t>(N) * nsb * kQ6kBytes,
                                kChkQ6W)) {
        const uint8_t* blk = a.W + (static_cast<size_t>(row) * nsb + b) * kQ6kBytes;
        l0[r] = load16_a2(blk + 64 * h + 16 * p);
        l1[r] = load16_a2(blk + 64 * h + 32 + 16 * p);
        hh[r] = load16_a2(blk + 128 + 32 * h + 16 * p);
        // scales s[8h + 2qq + p] live at bytes 192 + 8h + p + 2qq
        const uint8_t* sp = blk + 192 + 8 * h;
        const uintptr_t ad = reinterpret_cast<uintptr_t>(sp);
        const uint8_t* w = reinterpret_cast<const uint8_t*>(ad & ~static_cast<uintptr_t>(3));
        const unsigned sel = (ad & 2) ? 0x5432u : 0x3210u;
        // Aligned: bytes are w0, w1. Shifted by 2: w0..w2, ending exactly at
        // the end of the 8 scale bytes, so no read leaves the super-block.
        const unsigned w0 = ld_stream4(w), w1 = ld_stream4(w + 4);
        const unsigned w2 = (ad & 2) ? ld_stream4(w + 8) : 0u;
        const unsigned s03 = prmt(w0, w1, sel), s47 = prmt(w1, w2, sel);
        const unsigned short dbits = __ldg(reinterpret_cast<const unsigned short*>(blk + 208));
        const float d = half_bits_to_float(dbits);
        const unsigned sw[2] = {s03, s47};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int byte = p + 2 * qq;  // 0..7 within the 8 bytes at 192+8h
          const int sv = static_cast<int>(static_cast<int8_t>((sw[byte >> 2] >> (8 * (byte & 3))) & 0xFFu));
          sd[r][qq] = d * static_cast<float>(sv);
        }
      } else {
        l0[r] = make_uint4(0, 0, 0, 0);
        l1[r] = l0[r];
        hh[r] = l0[r];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) sd[r][qq] = 0.0f;
      }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int8_t* xa = a.qs + static_cast<size_t>(m) * K + static_cast<size_t>(b) * 256 + 128 * h + 16 * p;
      // (checked builds: the token's quants and scales of this super-block inside [M][K] and [M][K/32])
      if (!XQ_CHECKED(static_cast<size_t>(m) * K + static_cast<size_t>(b) * 256 + 256 <= static_cast<size_t>(a.M) * K &&
                          static_cast<size_t>(m) * nsub + 8 * b + 8 <= static_cast<size_t>(a.M) * nsub,
                      kChkQ6Act))
        continue;
      const float4 dd = __ldg(reinterpret_cast<const float4*>(a.d8 + static_cast<size_t>(m) * nsub + 8 * b + 4 * h));
      const float dq[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const uint4 x = ld_act16(xa + 32 * qq);
        int sa = 0;
        sa = dp4a_us(0x01010101u, x.x, sa);
        sa = dp4a_us(0x01010101u, x.y, sa);
        sa = dp4a_us(0x01010101u, x.z, sa);
        sa = dp4a_us(0x01010101u, x.w, sa);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint4 L = (qq & 1) ? l1[r] : l0[r];
          int s = 0;
          s = dp4a_us(q6_word(L.x, hh[r].x, qq), x.x, s);
          s = dp4a_us(q6_word(L.y, hh[r].y, qq), x.y, s);
          s = dp4a_us(q6_word(L.z, hh[r].z, qq), x.z, s);
          s = dp4a_us(q6_word(L.w, hh[r].w, qq), x.w, s);
          const int isum = s - 32 * sa;
          acc[r][m] = fmaf(sd[r][qq] * dq[qq], static_cast<float>(isum), acc[r][m]);
          if (ISUM) {
            const long long row = row0 + r;
            const size_t ii = (static_cast<size_t>(m) * N + row) * ngrp + 16 * b + 8 * h + 2 * qq + p;
            if (row < N && XQ_IN(ii, static_cast<size_t>(a.M) * N * ngrp, kChkQ6Isum)) a.isum[ii] = isum;
          }
        }
      }
    }
  }

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
          for (int m = 0; m < M; ++m)
            if (XQ_IN(m * a.ldy + row, (a.M - 1) * a.ldy + N, kChkQ6Y)) a.y[m * a.ldy + row] = acc[r][m];
      }
    }
    return;
  }
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
    if (row < N && XQ_IN(m * a.ldy + row, (a.M - 1) * a.ldy + N, kChkQ6Y)) a.y[m * a.ldy + row] = v;
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
  gemv_q6k_dp4a_kernel<M, R, ISUM><<<static_cast<unsigned>(grid), 256, 0, s>>>(a, kw);
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

cudaError_t take_q6k_check(unsigned int* code) { return take_check_word(code); }

cudaError_t launch_gemv_q6k(const GemvArgs& a, cudaStream_t s) {
  return a.isum ? dispatch<true>(a, s) : dispatch<false>(a, s);
}

}  // namespace xq
