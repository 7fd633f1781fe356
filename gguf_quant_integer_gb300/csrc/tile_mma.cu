// Q4_K / Q6_K x Q8 -> fp32 for M > 8 tokens on the fifth-generation tensor
// cores: tcgen05.mma kind::f16 with exact small-integer operands and fp32
// accumulators in tensor memory (TMEM).
//
// What it computes is the sum of the GEMV kernels (xLLM v0.7 long-context
// article, section 一, for the super-block; section B2 for the tile MMQ that
// reuses one unpacked weight tile for many tokens):
//   Q4_K: y[m][n] = sum_b d[n,b] * sum_j d8[m][8b+j] * sc_j isum_j
//                 - sum_b dmin[n,b] * sum_j mn_j * s8[m][8b+j]
//   Q6_K: y[m][n] = sum_b d[n,b] * sum_p d8[m][8b+p] * sum_{k<32} s_g(k) (q_k - 32) q8_k
// The tile is 128 weight rows (MMA M, the TMEM lanes) x 128 tokens (MMA N).
//
// A operand (weights), written into TMEM by the unpack warps (tcgen05.st):
//   Q4_K: sc_j * q * 2^-14 in fp16 (sc*q <= 945, exact): the nibble masked in
//         place is the fp16 subnormal q * 2^-24 (16q * 2^-24 for a high
//         nibble), and one fp16 multiply by sc * 2^10 (sc * 2^6) is exact.
//   Q6_K: s * (q - 32) in fp16 when |s| <= 64 (magnitude <= 2048, exact).
//         Rows with a larger scale use two operands, 2*(s>>1)*(q - 32) (even,
//         <= 4096, exact) and (s&1)*(q - 32), multiplied by the same token
//         operand into the same accumulator; the second pair of MMAs is issued
//         only when some row of the tile needs it.
// B operand (tokens) in shared memory: the q8 values as fp16 integers, read
// from the tile image the quantizer writes (one bulk copy per 32-block).
// Exactness: every product is an integer (times 2^-14 for Q4_K) and every
// partial sum of a 32-block accumulator stays below 2^24 in magnitude
// (Q4_K: 945*127*32; Q6_K, worst split: 129*32*127*32 = 16,776,192), so
// each accumulator is exact whatever the order of accumulation.
// Q4_K min term: one bf16 MMA per super-block, A = mn_j (exact) against the
// three-piece bf16 split of s8 (exact), i.e. exact products summed in fp32.
//
// Epilogue: per 32-block acc[m] += d8[m][j] * D[m] (one fp32 FMA per output);
// per super-block run[m] += d' * acc[m] (- dmin * Dmin[m]), d' = d*2^14 for
// Q4_K and d for Q6_K, with run kept
// in TMEM and written to y after the last super-block.
//
// Warp roles (448 threads): warps 0-3 unpack (thread = weight row = TMEM
// lane), warps 4-11 epilogue (warp w reads lane quarter w%4, token half
// (w-4)/4), warp 12 producer (raw weights by TMA or row copies, token items
// by bulk copy), warp 13 MMA issuer and TMEM owner. TMEM columns: [0,128)
// running sums, [128,384) two accumulators, [384,512) four A buffers of 32
// columns (16 for a 32-block of fp16 pairs, 16 more for the Q6_K second
// operand). Every mbarrier wait is bounded (about 2^32 clocks); on expiry
// the kernel records an error code, leaves its loops, waits for its own
// tensor-core work and frees TMEM.
#include <cuda.h>

#include "xq_common.cuh"
#include "xq_ptx.cuh"

namespace xq {

__device__ unsigned int g_tile_error;  // set by a timed-out wait (never expected)

namespace {

using namespace ptx;

constexpr int kRows = 128;        // weight rows per tile
constexpr int kNumA = 4;          // A buffers in TMEM
constexpr int kTokStages = 8;     // token item ring
constexpr int kRawStages = 3;     // raw weight ring (one super-block of 128 rows per stage)
constexpr uint32_t kColRun = 0, kColD = 128, kColA = 384;
constexpr int kThreads = 448;
constexpr int kWarpEpi0 = 4, kWarpProd = 12, kWarpMma = 13;
constexpr long long kWaitClocks = 1LL << 32;
constexpr int kQ6Window = 224;    // bytes copied per Q6_K row and super-block
constexpr int kQ6Pitch = 240;     // their pitch in shared memory (conflict-free 16-byte reads)

template <int TYPE>
struct Fmt;
template <>
struct Fmt<12> {
  static constexpr int kRawRow = kQ4kBytes, kItems = 9;  // 8 sub-blocks + the min-term item
};
template <>
struct Fmt<14> {
  static constexpr int kRawRow = kQ6Pitch, kItems = 8;
};

constexpr int kBarRawFull = 0;
constexpr int kBarRawEmpty = kBarRawFull + kRawStages;
constexpr int kBarTokFull = kBarRawEmpty + kRawStages;
constexpr int kBarTokEmpty = kBarTokFull + kTokStages;
constexpr int kBarAFull = kBarTokEmpty + kTokStages;
constexpr int kBarAEmpty = kBarAFull + kNumA;
constexpr int kBarDFull = kBarAEmpty + kNumA;
constexpr int kBarDEmpty = kBarDFull + 2;
constexpr int kBarDone = kBarDEmpty + 2;
constexpr int kNumBars = kBarDone + 1;

template <int TYPE>
constexpr int raw_stage_bytes() {
  return kRows * Fmt<TYPE>::kRawRow;
}
template <int TYPE>
constexpr int smem_bytes() {
  return kRawStages * raw_stage_bytes<TYPE>() + kTokStages * kTileItem + kNumBars * 8 + 16 + kNumA * 4 * 4;
}

struct TileArgs {
  CUtensorMap map;             // Q4_K: {row_bytes/8, N} of u64, box {18, 128}
  const uint8_t* W;
  const uint8_t* img;          // tile image of the Q8 buffer
  float* y;                    // [M][N]
  unsigned long long w_bytes;  // N * row_bytes
  int N, K, M, nsb, row_bytes, ttiles;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, unsigned parity, unsigned code) {
  return mbar_wait(bar, parity, &g_tile_error, code, kWaitClocks);
}
// Every lane waits; the warp goes on only if all of them saw the phase.
__device__ __forceinline__ bool warp_wait(uint32_t bar, unsigned parity, unsigned code) {
  const bool ok = wait_bar(bar, parity, code);
  return __all_sync(0xffffffffu, ok);
}

// Bytes of the Q6_K row window copied for row n, super-block b: 224 from
// the 16-byte boundary at or below the super-block start (which lies 0..14
// bytes in), cut to a multiple of 16 at the end of the weight buffer.
__device__ __forceinline__ unsigned q6_window(const TileArgs& A, int n, int b) {
  const unsigned long long start = static_cast<unsigned long long>(n) * A.row_bytes + 210ull * b;
  const unsigned long long src = start & ~15ull;
  return src + kQ6Window <= A.w_bytes ? kQ6Window : static_cast<unsigned>((A.w_bytes - src) & ~15ull);
}

// nw 32-bit words starting at a 2-byte aligned shared-memory address.
template <int NW>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&out)[NW]) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~static_cast<uintptr_t>(3));
  const unsigned sh = static_cast<unsigned>(a & 3) * 8;
  uint32_t prev = w[0];
#pragma unroll
  for (int k = 0; k < NW; ++k) {
    const uint32_t next = w[k + 1];
    out[k] = __funnelshift_r(prev, next, sh);
    prev = next;
  }
}

__device__ __forceinline__ uint32_t half2_of(float v) {
  const uint32_t h = __half_as_ushort(__float2half_rn(v));
  return h | (h << 16);
}

template <int TYPE>
__device__ __forceinline__ unsigned load_coef(const TileArgs& A, int n, int b) {
  const uint8_t* p = A.W + static_cast<size_t>(n) * A.row_bytes;
  if (TYPE == 12) return __ldg(reinterpret_cast<const unsigned*>(p + static_cast<size_t>(b) * kQ4kBytes));
  return __ldg(reinterpret_cast<const unsigned short*>(p + static_cast<size_t>(b) * kQ6kBytes + 208));
}

template <int TYPE>
__global__ void __launch_bounds__(kThreads, 1) tile_mma_kernel(const __grid_constant__ TileArgs A) {
  using F = Fmt<TYPE>;
  constexpr int kRawBytes = raw_stage_bytes<TYPE>();
  constexpr int kItems = F::kItems;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* raw_ring = smem;
  uint8_t* tok_ring = smem + kRawStages * kRawBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tok_ring + kTokStages * kTileItem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  int* split_flag = reinterpret_cast<int*>(tmem_slot + 4);  // [kNumA][4 unpack warps]
  const uint32_t bar0 = smem_addr(bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tt = blockIdx.x % A.ttiles, wt = blockIdx.x / A.ttiles;
  const int nitems = A.nsb * kItems;
#define BAR(i) (bar0 + 8u * static_cast<uint32_t>(i))

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(BAR(kBarRawFull + s), 1);
      mbar_init(BAR(kBarRawEmpty + s), 4);
    }
    for (int s = 0; s < kTokStages; ++s) {
      mbar_init(BAR(kBarTokFull + s), 1);
      mbar_init(BAR(kBarTokEmpty + s), 8);
    }
    for (int s = 0; s < kNumA; ++s) {
      mbar_init(BAR(kBarAFull + s), 4);
      mbar_init(BAR(kBarAEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(kBarDFull + s), 1);
      mbar_init(BAR(kBarDEmpty + s), 8);
    }
    mbar_init(BAR(kBarDone), 1);
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The tile image is written by the previous kernel on the stream.
  cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();

  if (warp == kWarpProd) {
    // ------------------------------------------------------- producer
    const uint8_t* rec = A.img + static_cast<size_t>(tt) * A.nsb * kTileRecord;
    const int row0 = wt * kRows;
    const int rows = min(kRows, A.N - row0);
    unsigned tf = 0;  // token items issued
    bool ok = true;
    for (int b = 0; b < A.nsb && ok; ++b) {
      const int rs = b % kRawStages;
      if (b >= kRawStages && !warp_wait(BAR(kBarRawEmpty + rs), ((b / kRawStages) - 1) & 1, 1)) break;
      const uint32_t dst = smem_addr(raw_ring + rs * kRawBytes);
      if (TYPE == 12) {
        if (lane == 0) {
          mbar_expect_tx(BAR(kBarRawFull + rs), kRawBytes);  // rows past N arrive zero-filled
          tma_load_2d(dst, &A.map, b * (kQ4kBytes / 8), row0, BAR(kBarRawFull + rs));
        }
      } else {
        unsigned mine = 0;
        for (int r = lane; r < rows; r += 32) mine += q6_window(A, row0 + r, b);
        const unsigned total = __reduce_add_sync(0xffffffffu, mine);
        if (lane == 0) mbar_expect_tx(BAR(kBarRawFull + rs), total);
        __syncwarp();
        for (int r = lane; r < rows; r += 32) {
          const unsigned long long start = static_cast<unsigned long long>(row0 + r) * A.row_bytes + 210ull * b;
          bulk_load(dst + r * kQ6Pitch, A.W + (start & ~15ull), q6_window(A, row0 + r, b), BAR(kBarRawFull + rs));
        }
      }
      for (int it = 0; it < kItems; ++it, ++tf) {
        const int ts = tf % kTokStages;
        if (tf >= kTokStages && !warp_wait(BAR(kBarTokEmpty + ts), ((tf / kTokStages) - 1) & 1, 2)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const unsigned bytes = it < 8 ? kTileItem : kTileItemOp;
          mbar_expect_tx(BAR(kBarTokFull + ts), bytes);
          bulk_load(smem_addr(tok_ring + ts * kTileItem), rec + static_cast<size_t>(b) * kTileRecord + it * kTileItem,
                    bytes, BAR(kBarTokFull + ts));
        }
      }
    }
    // No copy may still be landing when the CTA exits: wait for the last
    // fill of every stage (already complete on the normal path).
    if (lane == 0) {
      const int nb = A.nsb;
      for (int b = nb > kRawStages ? nb - kRawStages : 0; b < nb; ++b)
        wait_bar(BAR(kBarRawFull + b % kRawStages), (b / kRawStages) & 1, 11);
      for (unsigned f = tf > kTokStages ? tf - kTokStages : 0; f < tf; ++f)
        wait_bar(BAR(kBarTokFull + f % kTokStages), (f / kTokStages) & 1, 12);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------------------------------- unpack
    const int r = threadIdx.x;  // tile row = TMEM lane
    const int n = wt * kRows + r;
    const bool row_ok = n < A.N;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    unsigned af = 0;  // A buffers filled
    bool ok = true;
    for (int b = 0; b < A.nsb && ok; ++b) {
      const int rs = b % kRawStages;
      if (!warp_wait(BAR(kBarRawFull + rs), (b / kRawStages) & 1, 3)) break;
      const uint8_t* raw = raw_ring + rs * kRawBytes + r * F::kRawRow;
      if (TYPE == 12) {
        // Scales and mins (public Q4_K packing): j < 4: sc = s[j] & 63,
        // m = s[j+4] & 63; j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
        // m = (s[j+4] >> 4) | (s[j] >> 6) << 4. Rows past N are zero-filled.
        const uint4 h = *reinterpret_cast<const uint4*>(raw);
        const uint32_t sc_lo = h.y & 0x3F3F3F3Fu, mn_lo = h.z & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
        const uint32_t mn_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
#pragma unroll
        for (int it = 0; it < 9; ++it, ++af) {
          const int a = af % kNumA;
          if (af >= kNumA && !warp_wait(BAR(kBarAEmpty + a), ((af / kNumA) - 1) & 1, 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t v[16];
          if (it < 8) {
            const int g = it >> 1;
            const bool hi = (it & 1) != 0;
            const uint32_t sc = ((it < 4 ? sc_lo : sc_hi) >> (8 * (it & 3))) & 0xFFu;
            const uint32_t S = half2_of(static_cast<float>(sc) * (hi ? 64.0f : 1024.0f));
            const uint4* qp = reinterpret_cast<const uint4*>(raw + 16 + 32 * g);
            const uint4 q0 = qp[0], q1 = qp[1];
            const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            const uint32_t mk = hi ? 0x00F000F0u : 0x000F000Fu;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              // columns 2i, 2i+1 = k-slots 4i..4i+3 = weights 4i, 4i+2, 4i+1, 4i+3
              v[2 * i] = hmul2(w[i] & mk, S);
              v[2 * i + 1] = hmul2((w[i] >> 8) & mk, S);
            }
          } else {
            // min-term operand: slot k < 24 holds mn_{k/3} as bf16, the rest 0
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              uint32_t pair = 0;
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int k = 2 * c + e;
                if (k < 24) {
                  const int j = k / 3;
                  const uint32_t mn = ((j < 4 ? mn_lo : mn_hi) >> (8 * (j & 3))) & 0xFFu;
                  pair |= (__float_as_uint(static_cast<float>(mn)) >> 16) << (16 * e);
                }
              }
              v[c] = pair;
            }
          }
          tmem_st16(tl + kColA + 32 * a, v);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(kBarAFull + a));
        }
      } else {
        // Q6_K: ql[128] at 0, qh[64] at 128, scales int8[16] at 192, d at
        // 208. The row's window starts `off` (even, 0..14) bytes before the
        // super-block.
        const unsigned long long start = static_cast<unsigned long long>(n) * A.row_bytes + 210ull * b;
        const uint8_t* sb = raw + (start & 15);
        uint32_t sw[4] = {0u, 0u, 0u, 0u};
        if (row_ok) {
          if ((start & ~15ull) + kQ6Window <= A.w_bytes) {
            load_words<4>(sb + 192, sw);
          } else {
            // the window was cut at the end of the buffer: scales from memory
            const unsigned short* gs = reinterpret_cast<const unsigned short*>(A.W + start + 192);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              sw[k] = static_cast<uint32_t>(__ldg(gs + 2 * k)) | (static_cast<uint32_t>(__ldg(gs + 2 * k + 1)) << 16);
          }
        }
        // |s| > 64 anywhere in the row needs the two-operand form
        bool big = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) big = big || (__vcmpgtu4(__vabsss4(sw[k]), 0x40404040u) != 0u);
        const bool split = __any_sync(0xffffffffu, big);
        uint32_t ql[16], qh[8];
#pragma unroll
        for (int it = 0; it < 8; ++it, ++af) {
          const int hh = it >> 2, rr = it & 3;
          if (rr == 0 && row_ok) {
            load_words<16>(sb + 64 * hh, ql);
            load_words<8>(sb + 128 + 32 * hh, qh);
          }
          const int a = af % kNumA;
          if (af >= kNumA && !warp_wait(BAR(kBarAEmpty + a), ((af / kNumA) - 1) & 1, 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // scales of the two 16-groups of this 32-block
          uint32_t Shi[2], Slo[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int g = 2 * it + e;
            const int s = static_cast<int>(static_cast<int8_t>((sw[g >> 2] >> (8 * (g & 3))) & 0xFFu));
            const bool wide = s > 64 || s < -64;
            Shi[e] = half2_of(static_cast<float>(wide ? 2 * (s >> 1) : s));
            Slo[e] = half2_of(static_cast<float>(wide ? (s & 1) : 0));
          }
          uint32_t v[16], u[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t L = (rr >> 1) ? (ql[8 * (rr & 1) + i] >> 4) : ql[8 * (rr & 1) + i];
            const uint32_t H = rr == 0 ? (qh[i] << 4) : (rr == 1 ? (qh[i] << 2) : (rr == 2 ? qh[i] : (qh[i] >> 2)));
            const uint32_t q = (L & 0x0F0F0F0Fu) | (H & 0x30303030u);  // 6-bit quants of weights 4i..4i+3
            // fp16 1024 + q, then q - 32 (both exact)
            const uint32_t x0 = hsub2(prmt(q, 0x64646464u, 0x4240u), 0x64206420u);  // weights 4i, 4i+2
            const uint32_t x1 = hsub2(prmt(q, 0x64646464u, 0x4341u), 0x64206420u);  // weights 4i+1, 4i+3
            const int e = i >> 2;
            v[2 * i] = row_ok ? hmul2(x0, Shi[e]) : 0u;
            v[2 * i + 1] = row_ok ? hmul2(x1, Shi[e]) : 0u;
            u[2 * i] = row_ok ? hmul2(x0, Slo[e]) : 0u;
            u[2 * i + 1] = row_ok ? hmul2(x1, Slo[e]) : 0u;
          }
          tmem_st16(tl + kColA + 32 * a, v);
          if (split) tmem_st16(tl + kColA + 32 * a + 16, u);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            split_flag[4 * a + warp] = split ? 1 : 0;
            mbar_arrive(BAR(kBarAFull + a));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(kBarRawEmpty + rs));
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t kIdH = idesc_f16(kRows, kTileTokens, false);
      constexpr uint32_t kIdB = idesc_f16(kRows, kTileTokens, true);
      for (int f = 0; f < nitems; ++f) {
        const int it = f % kItems, ts = f % kTokStages, a = f % kNumA, d = f & 1;
        if (!wait_bar(BAR(kBarTokFull + ts), (f / kTokStages) & 1, 5)) break;
        if (!wait_bar(BAR(kBarAFull + a), (f / kNumA) & 1, 6)) break;
        if (f >= 2 && !wait_bar(BAR(kBarDEmpty + d), ((f >> 1) - 1) & 1, 7)) break;
        tc_fence_after();
        const uint32_t dt = tmem + kColD + 128u * d, at = tmem + kColA + 32u * a;
        const uint32_t bs = smem_addr(tok_ring + ts * kTileItem);
        const uint64_t b0 = smem_desc(bs, 128, 512), b1 = smem_desc(bs + 256, 128, 512);
        const uint32_t id = (TYPE == 12 && it == 8) ? kIdB : kIdH;
        mma_f16_ts(dt, at, b0, id, false);
        mma_f16_ts(dt, at + 8, b1, id, true);
        if (TYPE == 14) {
          const int* fl = split_flag + 4 * a;
          if (fl[0] | fl[1] | fl[2] | fl[3]) {
            mma_f16_ts(dt, at + 16, b0, id, true);
            mma_f16_ts(dt, at + 24, b1, id, true);
          }
        }
        tc_commit(BAR(kBarAEmpty + a));
        tc_commit(BAR(kBarDFull + d));
      }
      // all issued MMAs complete before TMEM is freed
      tc_commit(BAR(kBarDone));
      wait_bar(BAR(kBarDone), 0, 8);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue
    const int quarter = warp & 3, half = (warp - kWarpEpi0) >> 2;
    const int r = quarter * 32 + lane, n = wt * kRows + r;
    const bool row_ok = n < A.N;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int m0 = tt * kTileTokens + 64 * half;  // token of column 0 of this thread
    f2 acc[32];                                   // token pairs (2i, 2i+1) of the current super-block
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0ull;
    unsigned coef = row_ok ? load_coef<TYPE>(A, n, 0) : 0u;
    bool ok = true;
    int f = 0;
    for (int b = 0; b < A.nsb && ok; ++b) {
      const unsigned cur = coef;
      if (row_ok && b + 1 < A.nsb) coef = load_coef<TYPE>(A, n, b + 1);
      // d, times 2^14 for Q4_K (its operand carries sc*q*2^-14)
      const float da = half_bits_to_float(cur) * (TYPE == 12 ? 16384.0f : 1.0f);
      const float dm = TYPE == 12 ? -half_bits_to_float(cur >> 16) : 0.0f;
      const f2 da2 = pk(da, da), dm2 = pk(dm, dm);
      for (int it = 0; it < kItems; ++it, ++f) {
        const int d = f & 1, ts = f % kTokStages;
        if (!warp_wait(BAR(kBarDFull + d), (f >> 1) & 1, 9) ||
            !warp_wait(BAR(kBarTokFull + ts), (f / kTokStages) & 1, 10)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dcol = tl + kColD + 128u * d + 64u * half;
        if (it < 8) {
          const float4* d8 = reinterpret_cast<const float4*>(tok_ring + ts * kTileItem + kTileItemOp) + 16 * half;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[16];
            tmem_ld16(dcol + 16 * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float4 s = d8[4 * c + k];
              acc[8 * c + 2 * k] = fma2(pk(s.x, s.y), pk(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1])),
                                        acc[8 * c + 2 * k]);
              acc[8 * c + 2 * k + 1] =
                  fma2(pk(s.z, s.w), pk(__uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3])),
                       acc[8 * c + 2 * k + 1]);
            }
          }
        }
        if (it == kItems - 1) {
          // super-block end: run += d' * acc (- dmin * Dmin)
          const bool last = b == A.nsb - 1;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t run[16], dmin[16];
            if (b > 0) tmem_ld16(tl + kColRun + 64u * half + 16u * c, run);
            if (TYPE == 12) tmem_ld16(dcol + 16 * c, dmin);
            tmem_wait_ld();
            uint32_t out[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              f2 rv = b > 0 ? pk(__uint_as_float(run[2 * k]), __uint_as_float(run[2 * k + 1])) : 0ull;
              rv = fma2(da2, acc[8 * c + k], rv);
              if (TYPE == 12) rv = fma2(dm2, pk(__uint_as_float(dmin[2 * k]), __uint_as_float(dmin[2 * k + 1])), rv);
              out[2 * k] = static_cast<uint32_t>(rv);
              out[2 * k + 1] = static_cast<uint32_t>(rv >> 32);
              acc[8 * c + k] = 0ull;
            }
            if (last) {
              if (row_ok) {
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                  const int m = m0 + 16 * c + k;
                  if (m < A.M) A.y[static_cast<size_t>(m) * A.N + n] = __uint_as_float(out[k]);
                }
              }
            } else {
              tmem_st16(tl + kColRun + 64u * half + 16u * c, out);
            }
          }
          if (!last) tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(BAR(kBarDEmpty + d));
          mbar_arrive(BAR(kBarTokEmpty + ts));
        }
      }
    }
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int TYPE>
cudaError_t launch_tile(const TileArgs& A, int grid, cudaStream_t s, bool pdl) {
  static bool smem_set = false;
  if (!smem_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(tile_mma_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<TYPE>());
    if (e != cudaSuccess) return e;
    smem_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes<TYPE>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tile_mma_kernel<TYPE>, A);
}

}  // namespace

cudaError_t launch_tile_mma(int type, const uint8_t* W, const uint8_t* xq, int M, int N, int K, float* y,
                            cudaStream_t s, bool pdl) {
  if (M <= 8 || N <= 0 || K <= 0 || (K & 255) != 0 || (type != 12 && type != 14)) return cudaErrorInvalidValue;
  const Q8Layout L = q8_layout(M, K);
  TileArgs A = {};
  A.W = W;
  A.img = xq + L.tile;
  A.y = y;
  A.N = N;
  A.K = K;
  A.M = M;
  A.nsb = K >> 8;
  A.row_bytes = A.nsb * (type == 12 ? kQ4kBytes : kQ6kBytes);
  A.w_bytes = static_cast<unsigned long long>(N) * A.row_bytes;
  A.ttiles = L.ttiles;
  const int grid = ((N + kRows - 1) / kRows) * L.ttiles;
  if (type == 12) {
    if (!encode_tma_2d(&A.map, CU_TENSOR_MAP_DATA_TYPE_UINT64, W, A.row_bytes / 8, static_cast<unsigned long long>(N),
                       A.row_bytes, kQ4kBytes / 8, kRows))
      return cudaErrorInvalidValue;
    return launch_tile<12>(A, grid, s, pdl);
  }
  return launch_tile<14>(A, grid, s, pdl);
}

}  // namespace xq
