// Q4_K / Q6_K x Q8 -> fp32 for M <= 8 tokens on the tensor cores (mma.sync
// m16n8k16, fp16 operands holding exact integers, fp32 accumulation), with
// the weights streamed by TMA through a shared-memory ring. The Q4_K
// description follows; Q6_K differences are described at decode_scales_q6
// and compute_block_q6.
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
// Fragment mapping. Lane (n8 = lane/4, t = lane%4) takes 8 quant bytes
// 32g + 8t .. 32g + 8t + 7 of two rows for each g = 0..3: its low nibbles
// are positions 8t..8t+7 of sub-block 2g, its high nibbles the same
// positions of sub-block 2g+1. Even bytes (mask) and odd bytes (shift 8,
// mask) give the k-slot pairs (2t, 2t+1) and (2t+8, 2t+9) of two MMAs; the
// activation image written by the quantizer uses the same position order.
// MMA row i holds weight row pi(i) = 8*(i/8) + 2*(i%4) + (i%8)/4 of the
// 16-row group, which makes the 8-byte shared-memory loads bank-conflict
// free on 144-byte rows.
//
// Pipeline. Each CTA has one producer lane and 4 consumer warps. A task is
// 64 rows (16 per consumer warp) x a range of super-blocks; every ring stage
// holds one super-block of those 64 rows (four 2D TMA boxes of 16 rows x
// 144 bytes, rows past N zero-filled by the tensor map) and the activation
// operands of that super-block (two 1D bulk copies, 4.6 KB), which all four
// warps share. The producer writes each stage's task id and runs ahead
// across tasks through a 4-stage ring guarded by mbarriers, with no
// CTA-wide barrier. Each CTA's first task is its own index; later tasks come
// from a static stride, or, when a work counter is given, from an atomic
// counter over a list ordered by cost. The weight boxes of the first task's
// first stages are requested before the kernel waits for the previous grid
// on the stream (which writes the activation image and zeroes the counter).
// Long rows (more than 24 super-blocks) can be split into K-chunks of about
// 16 super-blocks (8 when a launch has few tasks) handled by different CTAs:
// each consumer warp writes its 16 rows' partial sums to a workspace and
// bumps that 16-row group's arrival count, and the last warp to arrive adds
// the chunks in chunk order and writes y, so the result does not depend on
// which CTA finishes last. (The geometry constants kGemvWarps, kGemvRows and
// kGemvCtasPerSM are in xq_common.cuh; the figures above are their values.)
//
// Every mbarrier wait is bounded (about 2^32 clocks); on expiry the kernel
// records an error code and returns.
#include <cuda.h>

#include "q8_block.cuh"
#include "xq_check.cuh"
#include "xq_common.cuh"
#include "xq_ptx.cuh"

namespace xq {

__device__ unsigned int g_gemv_error;  // set by a timed-out wait (never expected)

namespace {

struct Proj {
  CUtensorMap map;     // Q4_K: {row_bytes/8 u64, N}, box {18, 16}; Q6_K: {row_bytes u8, N}, box {240, 16}
  const uint8_t* frag; // [K/32][32][16 B] lane operands of the 8-token chunk
  const uint8_t* fsc;  // [K/32][4][16 B]
  float* y;
  int32_t* isum;
  float* partial;      // split: [nch][8][kGemvRows * row blocks]
  unsigned int* arrive;  // split: one arrival count per 16-row group
  uint32_t cb[4];        // IQ4_XS: codebook bytes with their sign bits flipped
  const uint8_t* aq;     // small-M form: int8 quants [M][K] of the Q8 buffer
  const float* ad8;      // small-M form: d8 [M][K/32]
  const float* as8;      // small-M form: s8 [M][K/32]
  int N, K, M, task0, nch;
  int gs;                // Q6_K grouped view: 2^gs consecutive rows form one tensor-map row (else 0)
  const uint8_t* xq0;    // the Q8 buffer and its size (bounds checks of checked builds)
  unsigned long long xq_bytes;
  unsigned long long y_elems;  // elements of y from P.y on that the launch may write (checked builds)
};

// The SwiGLU feed of a down projection computed inside the launch that runs
// gate and up: h = silu(y_gate) * y_up, quantized to Q8 (qs, d8, s8 and the
// GEMV operand image) by the warp that completes a 32-row block of gate and
// up, then counted ready per super-block. A down projection in the same
// launch waits, per super-block, for those counts before copying its
// activations; one in a later launch reads h after this grid completes.
struct Ffn {
  unsigned int* arrive;  // per 32-block of h: gate and up warps done with its rows (4 = all); null: no feed
  unsigned int* ready;   // per super-block of h: 32-blocks written (8 = all)
  uint8_t* hq;           // h's Q8 buffer
  float* h_out;          // optional fp32 copy of h [M][F]
  unsigned long long qs, d8, s8, frag, fsc;  // region offsets in hq
  unsigned long long hq_bytes;               // size of h's Q8 buffer
  int gate, up, down;    // slots in Group::p (down -1: not in this launch)
  int F, M;              // h features (N of gate and up, K of down), tokens (<= 8)
  int stall;             // test hook: h is written but never counted ready, so down's waits run out
  long long ready_limit; // clocks down's producer waits for a super-block of h
};

struct Group {
  Proj p[kMaxProj];
  Ffn ffn;
  unsigned int* counter;  // dynamic task counter (zeroed before launch) or null
  long long wait_limit;   // clocks a wait may take before it records an error and gives up
  int stall;              // test hook: the producer issues no stage, so the consumers' first waits run out
  int n, total;
  // 0: the launch needs nothing the previous grid on the stream writes (it
  // follows another grouped launch of the same layer, whose CTAs trigger only
  // after their own wait for the quantizer): skip the dependency wait.
  int wait_prev;
};

constexpr int kDecBytes = 8 * 16 * 16;  // per warp: one float4 per (32-block, row)

// Stage layout per weight type: four 16-row TMA boxes of one super-block,
// then the activation operands (8 x 512 B) and scale quads (8 x 64 B).
// Q4_K boxes are the 144-byte super-blocks; Q6_K boxes are 240-byte windows
// starting at the 16-byte boundary at or below the 210-byte super-block.
template <int TYPE>
struct GLay {
  static constexpr int kBoxRow = TYPE == 12 ? kQ4kBytes : (TYPE == 8 ? kQ80Group : (TYPE == 23 ? 144 : 240));
  static constexpr int kStages = kGemvWarps == 4 ? ((TYPE == 12 || TYPE == 23) ? 4 : 3) : ((TYPE == 12 || TYPE == 23) ? 4 : 2);
  static constexpr int kBlockBytes = 16 * kBoxRow;  // 16 rows x one super-block
  static constexpr int kFragOff = kGemvWarps * kBlockBytes;
  static constexpr int kFscOff = kFragOff + 8 * 512;
  static constexpr int kStageBytes = kFscOff + 8 * 64;
  static constexpr int kSmemBytes = kStages * kStageBytes + kGemvWarps * kDecBytes + kStages * 16 + 2 * kStages * 8;
};
static_assert(kGemvWarps != 4 || GLay<12>::kStageBytes == 13824, "Q4_K stage layout");
static_assert(kGemvCtasPerSM * (GLay<12>::kSmemBytes + 1024) <= 228 * 1024, "Q4_K: resident CTAs per SM");
static_assert(kGemvCtasPerSM * (GLay<14>::kSmemBytes + 1024) <= 228 * 1024, "Q6_K: resident CTAs per SM");
static_assert(kGemvCtasPerSM * (GLay<8>::kSmemBytes + 1024) <= 228 * 1024, "Q8_0: resident CTAs per SM");
static_assert(kGemvCtasPerSM * (GLay<23>::kSmemBytes + 1024) <= 228 * 1024, "IQ4_XS: resident CTAs per SM");
constexpr long long kWaitClocks = 1LL << 32;
constexpr long long kStallWaitClocks = 100000;  // the test hook's short limit (about 50 us)

__device__ __forceinline__ int mma_row(int i) { return 8 * (i >> 3) + 2 * (i & 3) + ((i >> 2) & 1); }

// TMA x coordinate of super-block (or 8-block group) b in the weight map.
template <int TYPE>
__device__ __forceinline__ int weight_box_x(int b) {
  if constexpr (TYPE == 12) return b * (kQ4kBytes / 8);
  else if constexpr (TYPE == 8) return b * (kQ80Group / 8);
  else if constexpr (TYPE == 23) return (kIq4xsBytes * b) & ~15;
  else return (kQ6kBytes * b) & ~15;
}

// Weight row of row k (0..15) of the 16-row group rg. Without the grouped
// view (gs = 0) the group holds rows 16rg .. 16rg+15. Q6_K rows that are not
// 16-byte multiples are mapped 2^gs rows to a tensor-map row (the smallest
// count whose bytes are a multiple of 16); group rg then holds rows
// i, i + g, ..., i + 15g of the block of 16g rows starting at 16g(rg >> gs),
// with g = 2^gs and i = rg mod g, so all its rows share one position i in
// their tensor-map rows and one in-window offset.
__device__ __forceinline__ int group_row(const Proj& P, int rg, int k) {
  return ((16 * (rg >> P.gs) + k) << P.gs) + (rg & ((1 << P.gs) - 1));
}

// TMA coordinates of the 16-row box of group rg at super-block b.
template <int TYPE>
__device__ __forceinline__ void weight_box(const Proj& P, int rg, int b, int& x, int& y) {
  if constexpr (TYPE == 14) {
    const int i = rg & ((1 << P.gs) - 1);
    x = (kQ6kBytes * ((P.K >> 8) * i + b)) & ~15;
    y = 16 * (rg >> P.gs);
  } else {
    x = weight_box_x<TYPE>(b);
    y = 16 * rg;
  }
  // x in map elements (8 bytes for Q4_K and Q8_0, 1 byte otherwise)
  const int xb = (TYPE == 12 || TYPE == 8) ? 8 * x : x;
  (void)XQ_CHECKED((xb & 15) == 0 && x >= 0 && y >= 0 && y < (P.N >> P.gs), kChkGemvBox);
}

// ---------------------------------------------------------------- PTX
using namespace ptx;

// Bounded wait: false (and an error code recorded) if the phase does not
// complete within `limit` clocks.
__device__ __forceinline__ bool mbar_wait(uint32_t a, unsigned parity, unsigned code, long long limit) {
  return ptx::mbar_wait(a, parity, &g_gemv_error, code, limit);
}

__device__ __forceinline__ void mma16816(float (&d)[4], unsigned a0, unsigned a1, unsigned a2,
                                         unsigned a3, unsigned b0, unsigned b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte k of a packed word as 2^23 + byte, an exact fp32 (0x4B0000xx).
__device__ __forceinline__ float byte_plus_2p23(unsigned w, int k) {
  return __uint_as_float(prmt(w, 0x4B000000u, 0x7540u | static_cast<unsigned>(k)));
}

// Arrival count increment of a split hand-off: an acquire-release atomic,
// executed by lane 0 after a warp barrier. As a release it publishes the
// stores every lane made before the barrier; as an acquire it makes the
// stores published by earlier arrivals visible to this warp, so the warp
// that arrives last can read every chunk's partial sums with no other fence.
__device__ __forceinline__ unsigned arrive_acq_rel(unsigned int* count) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(count) : "memory");
  return old;
}

// ---------------------------------------------------------------- tasks
struct TaskPos {
  int p, rb, b0, b1, c;
};

__device__ __forceinline__ TaskPos task_pos(const Group& G, int task) {
  int p = 0;
#pragma unroll 1
  while (p + 1 < G.n && task >= G.p[p + 1].task0) ++p;
  const Proj& P = G.p[p];
  const int local = task - P.task0;
  const int nsb = P.K >> 8;
  TaskPos s;
  s.p = p;
  s.rb = local / P.nch;
  s.c = local - s.rb * P.nch;
  s.b0 = nsb * s.c / P.nch;
  s.b1 = nsb * (s.c + 1) / P.nch;
  return s;
}

// Decode the 16 rows' scales of one super-block into the warp's table:
// lane l takes weight row l%16 and sub-blocks 4*(l/16) .. +3, writing
// (alpha, alpha, beta, beta) with alpha = d*sc*2^24 (low nibbles) or
// d*sc*2^20 (high), beta = -dmin*m, each as (2^23 + byte)*x - 2^23*x: one
// rounding of an exact product. Packed bytes (public Q4_K layout):
//   j < 4 : sc = s[j] & 63, m = s[j+4] & 63
//   j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4
// Each half-warp's stores cover 256 consecutive bytes (no bank conflicts).
__device__ __forceinline__ void decode_scales_q4(const uint8_t* blk, float4* dec, int lane) {
  const int r = lane & 15, half = lane >> 4;
  const uint4 hd = *reinterpret_cast<const uint4*>(blk + r * kQ4kBytes);
  const unsigned scw = half ? ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u)) : (hd.y & 0x3F3F3F3Fu);
  const unsigned mnw = half ? (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u)) : (hd.z & 0x3F3F3F3Fu);
  const float d = half_bits_to_float(hd.x);
  const float dl = d * 16777216.0f, dh = d * 1048576.0f;
  const float dm = -half_bits_to_float(hd.x >> 16);
  const float cl = -8388608.0f * dl, ch = -8388608.0f * dh, cm = -8388608.0f * dm;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 4 * half + k;
    const float a = (k & 1) ? fmaf(byte_plus_2p23(scw, k), dh, ch) : fmaf(byte_plus_2p23(scw, k), dl, cl);
    const float bm = fmaf(byte_plus_2p23(mnw, k), dm, cm);
    dec[j * 16 + r] = make_float4(a, a, bm, bm);
  }
}


// NW 32-bit words starting at a 2-byte aligned shared-memory address.
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

// Q6_K (public layout: ql[128] @0, qh[64] @128, int8 scales[16] @192, d @208;
// the super-block starts `off` bytes into the row's window). Lane l takes
// weight row l%16 and 32-blocks 4*(l/16) .. +3, writing for each 32-block p
// (alpha_2p, alpha_2p, delta_p, delta_p) with alpha_2p = d * s_2p and
// delta_p = d * (s_2p+1 - s_2p): exact products (11 x 9 significant bits),
// so each is exact in fp32. Each half-warp's stores cover 256 consecutive
// bytes.
__device__ __forceinline__ void decode_scales_q6(const uint8_t* blk, int off, float4* dec, int lane) {
  const int r = lane & 15, half = lane >> 4;
  const uint8_t* sb = blk + r * GLay<14>::kBoxRow + off;
  uint32_t sw[2];
  load_words<2>(sb + 192 + 8 * half, sw);
  const float d = half_bits_to_float(*reinterpret_cast<const unsigned short*>(sb + 208));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w = sw[k >> 1];
    const int b0 = 2 * (k & 1);
    const int s0 = static_cast<int8_t>((w >> (8 * b0)) & 0xFFu);
    const int s1 = static_cast<int8_t>((w >> (8 * b0 + 8)) & 0xFFu);
    const float a0 = d * static_cast<float>(s0);
    const float dl = d * static_cast<float>(s1 - s0);
    dec[(4 * half + k) * 16 + r] = make_float4(a0, a0, dl, dl);
  }
}

template <bool ISUM>
__device__ __forceinline__ void compute_block_q4(const uint8_t* blk, const uint8_t* act, const float4* dec,
                                              const Proj& P, int rg, int b, int n8, int t, int lane, f2 (&acc)[2]) {
  const int r0 = mma_row(n8), r1 = r0 + 8;
  uint2 q0[4], q1[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    q0[g] = *reinterpret_cast<const uint2*>(blk + r0 * kQ4kBytes + 16 + 32 * g + 8 * t);
    q1[g] = *reinterpret_cast<const uint2*>(blk + r1 * kQ4kBytes + 16 + 32 * g + 8 * t);
  }
  // Activation operands and scale quads of the super-block, from the stage.
  const uint4* fp = reinterpret_cast<const uint4*>(act) + lane;
  const ulonglong2* sp = reinterpret_cast<const ulonglong2*>(act + (GLay<12>::kFscOff - GLay<12>::kFragOff)) + t;
  const ulonglong2* dp = reinterpret_cast<const ulonglong2*>(dec);
  // The four shared-memory operands of a sub-block are loaded one sub-block
  // ahead of their use.
  uint4 Bn = fp[0];
  ulonglong2 fn = sp[0], e0n = dp[r0], e1n = dp[r1];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const unsigned w0a = q0[g].x, w1a = q0[g].y;  // row r0
    const unsigned w0b = q1[g].x, w1b = q1[g].y;  // row r1
    const unsigned s0a = w0a >> 8, s1a = w1a >> 8, s0b = w0b >> 8, s1b = w1b >> 8;
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      const unsigned mk = hi ? 0x00F000F0u : 0x000F000Fu;
      const int j = 2 * g + hi;
      const uint4 B = Bn;
      const ulonglong2 f = fn;  // (d8 c0, d8 c1), (s8 c0, s8 c1)
      const ulonglong2 e0 = e0n, e1 = e1n;  // (a, a), (b, b) of rows r0, r1
      if (j < 7) {
        Bn = fp[(j + 1) * 32];
        fn = sp[(j + 1) * 4];
        e0n = dp[(j + 1) * 16 + r0];
        e1n = dp[(j + 1) * 16 + r1];
      }
      float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      mma16816(D, w0a & mk, w0b & mk, s0a & mk, s0b & mk, B.x, B.y);
      mma16816(D, w1a & mk, w1b & mk, s1a & mk, s1b & mk, B.z, B.w);
      acc[0] = fma2(mul2(e0.x, f.x), pk(D[0], D[1]), fma2(e0.y, f.y, acc[0]));
      acc[1] = fma2(mul2(e1.x, f.x), pk(D[2], D[3]), fma2(e1.y, f.y, acc[1]));
      if (ISUM) {
        const float scale = hi ? 1048576.0f : 16777216.0f;
        const int nsub = P.K >> 5;
        const int sb = 8 * b + j;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = group_row(P, rg, (e >> 1) ? r1 : r0);
          const int col = 2 * t + (e & 1);
          const size_t ii = (static_cast<size_t>(col) * P.N + row) * nsub + sb;
          if (row < P.N && col < P.M && XQ_IN(ii, static_cast<size_t>(P.M) * P.N * nsub, kChkGemvIsum))
            P.isum[ii] = static_cast<int32_t>(D[e] * scale);
        }
      }
    }
  }
}


// Q6_K 32-block p of rows r0, r1: lane (n8, t) holds the quants of weights
// 8t..8t+7 of p, i.e. of group 2p for t < 2 and group 2p+1 for t >= 2
// (the activation image's slot order, as for Q4_K). Each quant is
// q = (ql nibble) | (qh 2 bits) << 4; the operand is q - 32 in fp16
// (1024 + q from a byte permute, then an exact subtraction). Four MMAs per
// 32-block: two give Da = isum_2p + isum_2p+1, and two more, with the
// activation operands of group 2p's lanes zeroed, give D1 = isum_2p+1 (all
// exact: |isum_g| <= 32*127*16). Since
//   alpha_2p isum_2p + alpha_2p+1 isum_2p+1 = alpha_2p Da + delta_p D1,
// the combine is acc += (alpha_2p d8) Da + (delta_p d8) D1.
template <bool ISUM>
__device__ __forceinline__ void compute_block_q6(const uint8_t* blk, int off, const uint8_t* act, const float4* dec,
                                                 const Proj& P, int rg, int b, int n8, int t, int lane,
                                                 f2 (&acc)[2]) {
  const int r0 = mma_row(n8), r1 = r0 + 8;
  const uint8_t* s0 = blk + r0 * GLay<14>::kBoxRow + off;
  const uint8_t* s1 = blk + r1 * GLay<14>::kBoxRow + off;
  const uint4* fp = reinterpret_cast<const uint4*>(act) + lane;
  const ulonglong2* sp = reinterpret_cast<const ulonglong2*>(act + (GLay<14>::kFscOff - GLay<14>::kFragOff)) + t;
  const ulonglong2* dp = reinterpret_cast<const ulonglong2*>(dec);
  const bool first = t < 2;  // this lane's weights belong to group 2p
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    // ql bytes 64hh + 8t (32-blocks 0, 2 of the half) and 64hh + 32 + 8t (1, 3);
    // qh bytes 128 + 32hh + 8t (all four)
    uint32_t la0[2], lb0[2], hq0[2], la1[2], lb1[2], hq1[2];
    load_words<2>(s0 + 64 * hh + 8 * t, la0);
    load_words<2>(s0 + 64 * hh + 32 + 8 * t, lb0);
    load_words<2>(s0 + 128 + 32 * hh + 8 * t, hq0);
    load_words<2>(s1 + 64 * hh + 8 * t, la1);
    load_words<2>(s1 + 64 * hh + 32 + 8 * t, lb1);
    load_words<2>(s1 + 128 + 32 * hh + 8 * t, hq1);
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int p = 4 * hh + rr;
      uint32_t a[2][4];  // [k-half][a0..a3]
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint32_t L0 = (rr & 1) ? lb0[w] : la0[w], L1 = (rr & 1) ? lb1[w] : la1[w];
        const uint32_t H0 = rr == 0 ? (hq0[w] << 4) : (rr == 1 ? (hq0[w] << 2) : (rr == 2 ? hq0[w] : (hq0[w] >> 2)));
        const uint32_t H1 = rr == 0 ? (hq1[w] << 4) : (rr == 1 ? (hq1[w] << 2) : (rr == 2 ? hq1[w] : (hq1[w] >> 2)));
        const uint32_t q0 = (((rr >> 1) ? (L0 >> 4) : L0) & 0x0F0F0F0Fu) | (H0 & 0x30303030u);
        const uint32_t q1 = (((rr >> 1) ? (L1 >> 4) : L1) & 0x0F0F0F0Fu) | (H1 & 0x30303030u);
        // (1024 + q) pairs, minus 1056: weights (4w, 4w+2) -> a0/a1, (4w+1, 4w+3) -> a2/a3
        a[w][0] = hsub2(prmt(q0, 0x64646464u, 0x4240u), 0x64206420u);
        a[w][1] = hsub2(prmt(q1, 0x64646464u, 0x4240u), 0x64206420u);
        a[w][2] = hsub2(prmt(q0, 0x64646464u, 0x4341u), 0x64206420u);
        a[w][3] = hsub2(prmt(q1, 0x64646464u, 0x4341u), 0x64206420u);
      }
      const uint4 B = fp[p * 32];
      float Da[4] = {0.0f, 0.0f, 0.0f, 0.0f}, D1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const uint32_t g1 = first ? 0u : 0xFFFFFFFFu;  // keeps group 2p+1's activations
      mma16816(Da, a[0][0], a[0][1], a[0][2], a[0][3], B.x, B.y);
      mma16816(Da, a[1][0], a[1][1], a[1][2], a[1][3], B.z, B.w);
      mma16816(D1, a[0][0], a[0][1], a[0][2], a[0][3], B.x & g1, B.y & g1);
      mma16816(D1, a[1][0], a[1][1], a[1][2], a[1][3], B.z & g1, B.w & g1);
      const ulonglong2 f = sp[p * 4];  // (d8 c0, d8 c1), (s8 c0, s8 c1)
      const ulonglong2 e0 = dp[p * 16 + r0], e1 = dp[p * 16 + r1];
      acc[0] = fma2(mul2(e0.x, f.x), pk(Da[0], Da[1]), fma2(mul2(e0.y, f.x), pk(D1[0], D1[1]), acc[0]));
      acc[1] = fma2(mul2(e1.x, f.x), pk(Da[2], Da[3]), fma2(mul2(e1.y, f.x), pk(D1[2], D1[3]), acc[1]));
      if (ISUM) {
        const int ngrp = P.K >> 4;
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = group_row(P, rg, (e >> 1) ? r1 : r0);
            const int col = 2 * t + (e & 1);
            const size_t ii = (static_cast<size_t>(col) * P.N + row) * ngrp + 16 * b + 2 * p + g;
            if (row < P.N && col < P.M && XQ_IN(ii, static_cast<size_t>(P.M) * P.N * ngrp, kChkGemvIsum))
              P.isum[ii] = static_cast<int32_t>(g ? D1[e] : Da[e] - D1[e]);
          }
      }
    }
  }
}

// Q8_0 (xLLM v0.7 long-context article, section B3 + B4; public GGUF block:
// fp16 d at byte 0, 32 int8 quants at bytes 2..33). A stage row holds 8
// blocks (272 bytes, 16-byte aligned). Lane l takes row l%16 and blocks
// 4*(l/16) .. +3, writing (d, d, 0, 0) into the warp's table (no min term).
__device__ __forceinline__ void decode_scales_q8_0(const uint8_t* blk, float4* dec, int lane) {
  const int r = lane & 15, half = lane >> 4;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 4 * half + k;
    const float d = half_bits_to_float(*reinterpret_cast<const unsigned short*>(blk + r * kQ80Group + 34 * j));
    dec[j * 16 + r] = make_float4(d, d, 0.0f, 0.0f);
  }
}

// Q8_0 block j of rows r0, r1: lane (n8, t) takes the quants of weights
// 8t..8t+7 (the activation image's slot order, as for Q4_K). Each int8 q
// becomes the exact fp16 integer q: the byte with its sign bit flipped is
// q + 128, placed under the exponent of 1024 by a byte permute (1024 + q +
// 128), then 1152 is subtracted. Products are at most 128*127 and a block
// sum at most 520,192 in magnitude, so D = isum exactly. Combine:
// acc += (d * d8) * D.
template <bool ISUM>
__device__ __forceinline__ void compute_block_q8_0(const uint8_t* blk, const uint8_t* act, const float4* dec,
                                                   const Proj& P, int rg, int b, int n8, int t, int lane,
                                                   f2 (&acc)[2]) {
  const int r0 = mma_row(n8), r1 = r0 + 8;
  const uint4* fp = reinterpret_cast<const uint4*>(act) + lane;
  const ulonglong2* sp = reinterpret_cast<const ulonglong2*>(act + (GLay<8>::kFscOff - GLay<8>::kFragOff)) + t;
  const ulonglong2* dp = reinterpret_cast<const ulonglong2*>(dec);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t w0[2], w1[2];
    load_words<2>(blk + r0 * kQ80Group + 34 * j + 2 + 8 * t, w0);
    load_words<2>(blk + r1 * kQ80Group + 34 * j + 2 + 8 * t, w1);
    uint32_t a[2][4];  // [k-half][a0..a3]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t x0 = w0[h] ^ 0x80808080u, x1 = w1[h] ^ 0x80808080u;
      a[h][0] = hsub2(prmt(x0, 0x64646464u, 0x4240u), 0x64806480u);  // row r0, weights 4h', 4h'+2
      a[h][1] = hsub2(prmt(x1, 0x64646464u, 0x4240u), 0x64806480u);  // row r1
      a[h][2] = hsub2(prmt(x0, 0x64646464u, 0x4341u), 0x64806480u);  // row r0, weights 4h'+1, 4h'+3
      a[h][3] = hsub2(prmt(x1, 0x64646464u, 0x4341u), 0x64806480u);  // row r1
    }
    const uint4 B = fp[j * 32];
    float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    mma16816(D, a[0][0], a[0][1], a[0][2], a[0][3], B.x, B.y);
    mma16816(D, a[1][0], a[1][1], a[1][2], a[1][3], B.z, B.w);
    const ulonglong2 f = sp[j * 4];  // (d8 c0, d8 c1), (s8 c0, s8 c1)
    const ulonglong2 e0 = dp[j * 16 + r0], e1 = dp[j * 16 + r1];
    acc[0] = fma2(mul2(e0.x, f.x), pk(D[0], D[1]), acc[0]);
    acc[1] = fma2(mul2(e1.x, f.x), pk(D[2], D[3]), acc[1]);
    if (ISUM) {
      const int nsub = P.K >> 5;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = group_row(P, rg, (e >> 1) ? r1 : r0);
        const int col = 2 * t + (e & 1);
        const size_t ii = (static_cast<size_t>(col) * P.N + row) * nsub + 8 * b + j;
        if (row < P.N && col < P.M && XQ_IN(ii, static_cast<size_t>(P.M) * P.N * nsub, kChkGemvIsum))
          P.isum[ii] = static_cast<int32_t>(D[e]);
      }
    }
  }
}

// IQ4_XS (Agent Telemetry log, entries on the IQ4_XS batch kernels: 4-bit
// indices into a 16-entry int8 codebook; public GGUF block, 136 bytes: fp16 d
// at 0, scales_h at 2, scales_l[4] at 4, 128 index bytes at 8). A stage row
// is the 144-byte window from the 16-byte boundary at or below the
// super-block, which begins `off` = 0 or 8 bytes in (136 b mod 16). Lane l
// takes weight row l%16 and sub-blocks 4*(l/16) .. +3, writing (alpha, alpha,
// 0, 0) with alpha = d * (ls_j - 32), an exact product: ls_j is 4 bits of
// scales_l at bit 4j and 2 bits of scales_h at bit 2j.
__device__ __forceinline__ void decode_scales_iq4xs(const uint8_t* blk, int off, float4* dec, int lane) {
  const int r = lane & 15, half = lane >> 4;
  const uint2 h = *reinterpret_cast<const uint2*>(blk + r * GLay<23>::kBoxRow + off);  // d | scales_h, scales_l
  const float d = half_bits_to_float(h.x);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 4 * half + k;
    const int ls = static_cast<int>(((h.y >> (4 * j)) & 15u) | (((h.x >> (16 + 2 * j)) & 3u) << 4));
    const float a = d * static_cast<float>(ls - 32);
    dec[j * 16 + r] = make_float4(a, a, 0.0f, 0.0f);
  }
}

// Codebook bytes (sign bits flipped) of four 4-bit indices, one index per
// byte of x: two byte permutes over the codebook halves, chosen per byte by
// index bit 3 (a sign-replicating permute of x << 4 makes the byte mask).
__device__ __forceinline__ uint32_t iq4_lookup(uint32_t x, const uint32_t (&cb)[4]) {
  const uint32_t sel = prmt(x | (x >> 4), 0u, 0x4420u) & 0x7777u;  // the four indices' low 3 bits, as selectors
  const uint32_t lo = prmt(cb[0], cb[1], sel), hi = prmt(cb[2], cb[3], sel);
  const uint32_t m = prmt(x << 4, 0u, 0xBA98u);
  return (hi & m) | (lo & ~m);
}

// IQ4_XS sub-block j of rows r0, r1: lane (n8, t) takes weights 8t..8t+7
// (the activation image's slot order): low nibbles of index bytes
// 16j + 8t .. +7 for t < 2, high nibbles of bytes 16j + 8(t-2) .. +7 for
// t >= 2. Each index becomes its codebook value, then the exact fp16 integer
// as for Q8_0 (sign bit flipped, placed under the exponent of 1024, 1152
// subtracted). |value| <= 128, so a sub-block sum is at most 128*127*32 in
// magnitude and D = isum exactly. Combine: acc += (alpha * d8) * D.
template <bool ISUM>
__device__ __forceinline__ void compute_block_iq4xs(const uint8_t* blk, int off, const uint8_t* act, const float4* dec,
                                                    const Proj& P, int rg, int b, int n8, int t, int lane,
                                                    f2 (&acc)[2]) {
  const int r0 = mma_row(n8), r1 = r0 + 8;
  const uint8_t* q0 = blk + r0 * GLay<23>::kBoxRow + off + 8 + 8 * (t & 1);
  const uint8_t* q1 = blk + r1 * GLay<23>::kBoxRow + off + 8 + 8 * (t & 1);
  const unsigned sh = 4u * static_cast<unsigned>(t >> 1);
  const uint32_t cb[4] = {P.cb[0], P.cb[1], P.cb[2], P.cb[3]};
  const uint4* fp = reinterpret_cast<const uint4*>(act) + lane;
  const ulonglong2* sp = reinterpret_cast<const ulonglong2*>(act + (GLay<23>::kFscOff - GLay<23>::kFragOff)) + t;
  const ulonglong2* dp = reinterpret_cast<const ulonglong2*>(dec);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint2 w0 = *reinterpret_cast<const uint2*>(q0 + 16 * j);
    const uint2 w1 = *reinterpret_cast<const uint2*>(q1 + 16 * j);
    uint32_t a[2][4];  // [k-half][a0..a3]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t x0 = iq4_lookup(((h ? w0.y : w0.x) >> sh) & 0x0F0F0F0Fu, cb);
      const uint32_t x1 = iq4_lookup(((h ? w1.y : w1.x) >> sh) & 0x0F0F0F0Fu, cb);
      a[h][0] = hsub2(prmt(x0, 0x64646464u, 0x4240u), 0x64806480u);  // row r0, weights 4h', 4h'+2
      a[h][1] = hsub2(prmt(x1, 0x64646464u, 0x4240u), 0x64806480u);  // row r1
      a[h][2] = hsub2(prmt(x0, 0x64646464u, 0x4341u), 0x64806480u);  // row r0, weights 4h'+1, 4h'+3
      a[h][3] = hsub2(prmt(x1, 0x64646464u, 0x4341u), 0x64806480u);  // row r1
    }
    const uint4 B = fp[j * 32];
    float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    mma16816(D, a[0][0], a[0][1], a[0][2], a[0][3], B.x, B.y);
    mma16816(D, a[1][0], a[1][1], a[1][2], a[1][3], B.z, B.w);
    const ulonglong2 f = sp[j * 4];  // (d8 c0, d8 c1), (s8 c0, s8 c1)
    const ulonglong2 e0 = dp[j * 16 + r0], e1 = dp[j * 16 + r1];
    acc[0] = fma2(mul2(e0.x, f.x), pk(D[0], D[1]), acc[0]);
    acc[1] = fma2(mul2(e1.x, f.x), pk(D[2], D[3]), acc[1]);
    if (ISUM) {
      const int nsub = P.K >> 5;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = group_row(P, rg, (e >> 1) ? r1 : r0);
        const int col = 2 * t + (e & 1);
        const size_t ii = (static_cast<size_t>(col) * P.N + row) * nsub + 8 * b + j;
        if (row < P.N && col < P.M && XQ_IN(ii, static_cast<size_t>(P.M) * P.N * nsub, kChkGemvIsum))
          P.isum[ii] = static_cast<int32_t>(D[e]);
      }
    }
  }
}

__device__ __forceinline__ void store_y(const Proj& P, int rg, int n8, int t, float v00, float v01, float v10,
                                        float v11) {
  const int r0 = group_row(P, rg, mma_row(n8)), r1 = group_row(P, rg, mma_row(n8) + 8), c0 = 2 * t, c1 = c0 + 1;
  auto put = [&](int c, int r, float v) {
    const size_t i = static_cast<size_t>(c) * P.N + r;
    if (c < P.M && r < P.N && XQ_IN(i, P.y_elems, kChkGemvY)) P.y[i] = v;
  };
  put(c0, r0, v00);
  put(c1, r0, v01);
  put(c0, r1, v10);
  put(c1, r1, v11);
}

// The last warp to finish a split 16-row group: y = the group's K-chunk
// partials added in chunk order (the loads of 4 chunks issued together).
__device__ __forceinline__ void reduce_chunks(const Proj& P, int rg, int n8, int t) {
  const int rows_pad = gemv_row_blocks(P.N) * kGemvRows;
  const int r0 = rg * 16 + mma_row(n8), r1 = r0 + 8, c0 = 2 * t, c1 = c0 + 1;
  float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int c0k = 0; c0k < P.nch; c0k += 4) {
    float pv[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (c0k + u < P.nch) {
        const float* pc = P.partial + static_cast<size_t>(c0k + u) * 8 * rows_pad;
        pv[u][0] = __ldcg(pc + static_cast<size_t>(c0) * rows_pad + r0);
        pv[u][1] = __ldcg(pc + static_cast<size_t>(c1) * rows_pad + r0);
        pv[u][2] = __ldcg(pc + static_cast<size_t>(c0) * rows_pad + r1);
        pv[u][3] = __ldcg(pc + static_cast<size_t>(c1) * rows_pad + r1);
        // (checked builds: the highest of the four reads inside the partial sums)
        (void)XQ_IN((static_cast<size_t>(c0k + u) * 8 + c1) * rows_pad + (r0 > r1 ? r0 : r1),
                    static_cast<size_t>(P.nch) * 8 * rows_pad, kChkGemvPartial);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c0k + u < P.nch)
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] += pv[u][e];
  }
  store_y(P, rg, n8, t, v[0], v[1], v[2], v[3]);
}

// A consumer warp has written the final y of 16-row group rg of gate or up.
// The warp that completes a 32-row block (the fourth of the two gate and two
// up warps to arrive) computes that block of h for every token and writes
// its Q8 bytes and operand image, then counts the block ready. The arrival
// is an acquire-release increment (arrive_acq_rel, as in the split hand-off),
// so the fourth warp reads the others' y with no further fence. The proxy
// fence makes the generic-proxy writes of h visible to the bulk copies
// (async proxy) that read them.
__device__ __noinline__ void ffn_arrive(const Group& G, int rg, int lane) {
  const Ffn& F = G.ffn;
  __syncwarp();
  unsigned old = 0;
  if (lane == 0) old = arrive_acq_rel(F.arrive + (rg >> 1));
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != 3u) return;
  // All tokens at once: lane l takes token n = l/4 and elements 8g..8g+7,
  // g = l%4, of the block. The steps are those of q8_quantize_lane and
  // swiglu (the same fp32 operations, the block max and quant sum taken over
  // the token's 4 lanes instead of 32), so the bytes equal the quantize
  // kernel's.
  const int j = rg >> 1, nsub = F.F >> 5;
  const int n = lane >> 2, g = lane & 3;
  const bool live = n < F.M;
  float v[8];
  // (checked builds: the block inside h, and h's Q8 regions inside its buffer)
  const bool ffn_ok = XQ_CHECKED(j >= 0 && 32 * j + 32 <= F.F && F.fsc + static_cast<size_t>(F.F / 32) * 64 <= F.hq_bytes &&
                                     F.s8 + 4ull * F.M * (F.F / 32) <= F.hq_bytes && F.qs + 1ull * F.M * F.F <= F.hq_bytes,
                                 kChkGemvFfn);
  if (!ffn_ok) return;
  if (live) {
    const size_t idx = static_cast<size_t>(n) * F.F + 32 * j + 8 * g;
    const float4* gp = reinterpret_cast<const float4*>(G.p[F.gate].y + idx);
    const float4* up = reinterpret_cast<const float4*>(G.p[F.up].y + idx);
    const float4 g0 = __ldcg(gp), g1 = __ldcg(gp + 1), u0 = __ldcg(up), u1 = __ldcg(up + 1);
    v[0] = swiglu(g0.x, u0.x);
    v[1] = swiglu(g0.y, u0.y);
    v[2] = swiglu(g0.z, u0.z);
    v[3] = swiglu(g0.w, u0.w);
    v[4] = swiglu(g1.x, u1.x);
    v[5] = swiglu(g1.y, u1.y);
    v[6] = swiglu(g1.z, u1.z);
    v[7] = swiglu(g1.w, u1.w);
    if (F.h_out) {
      float4* hp = reinterpret_cast<float4*>(F.h_out + idx);
      hp[0] = make_float4(v[0], v[1], v[2], v[3]);
      hp[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.0f;
  }
  // amax over the token's 32 values: IEEE bit patterns of |x| order like the values
  unsigned ab = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) ab = max(ab, __float_as_uint(fabsf(v[e])));
  ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 1));
  ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 2));
  const float d = __fdiv_rn(__uint_as_float(ab), 127.0f);
  const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
  int q[8], isum = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float x = roundf(__fmul_rn(v[e], id));
    x = (x != x) ? 0.0f : x;
    x = x > 127.0f ? 127.0f : (x < -127.0f ? -127.0f : x);
    q[e] = static_cast<int>(x);
    isum += q[e];
  }
  isum += __shfl_xor_sync(0xffffffffu, isum, 1);
  isum += __shfl_xor_sync(0xffffffffu, isum, 2);
  const float sc = __fmul_rn(d, static_cast<float>(isum));
  if (live) {
    uint2 qb;
    qb.x = (q[0] & 255) | (q[1] & 255) << 8 | (q[2] & 255) << 16 | static_cast<unsigned>(q[3] & 255) << 24;
    qb.y = (q[4] & 255) | (q[5] & 255) << 8 | (q[6] & 255) << 16 | static_cast<unsigned>(q[7] & 255) << 24;
    *reinterpret_cast<uint2*>(F.hq + F.qs + static_cast<size_t>(n) * F.F + 32 * j + 8 * g) = qb;
    if (g == 0) {
      reinterpret_cast<float*>(F.hq + F.d8)[static_cast<size_t>(n) * nsub + j] = d;
      reinterpret_cast<float*>(F.hq + F.s8)[static_cast<size_t>(n) * nsub + j] = sc;
    }
  }
  // GEMV image (chunk 0): the lane's 8 fp16 quants fill operand slots
  // 0..7 of (token n, quad g), slot s holding element perm(s), perm =
  // 0,2,1,3,4,6,5,7 (write_gemv_image's order); padding tokens write zeros.
  {
    const __half2 h01 = __halves2half2(__int2half_rn(q[0]), __int2half_rn(q[2]));
    const __half2 h23 = __halves2half2(__int2half_rn(q[1]), __int2half_rn(q[3]));
    const __half2 h45 = __halves2half2(__int2half_rn(q[4]), __int2half_rn(q[6]));
    const __half2 h67 = __halves2half2(__int2half_rn(q[5]), __int2half_rn(q[7]));
    uint4 w;
    w.x = *reinterpret_cast<const unsigned*>(&h01);
    w.y = *reinterpret_cast<const unsigned*>(&h23);
    w.z = *reinterpret_cast<const unsigned*>(&h45);
    w.w = *reinterpret_cast<const unsigned*>(&h67);
    reinterpret_cast<uint4*>(F.hq + F.frag)[static_cast<size_t>(j) * 32 + 4 * n + g] = w;
    if (g == 0) {
      float* fsc = reinterpret_cast<float*>(F.hq + F.fsc);
      const size_t base = (static_cast<size_t>(j) * 4 + (n >> 1)) * 4;
      fsc[base + (n & 1)] = d;
      fsc[base + 2 + (n & 1)] = sc;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
  if (lane == 0 && !F.stall) {
    __threadfence();
    atomicAdd(F.ready + (j >> 3), 1u);
  }
}

// The down projection's producer before copying super-block b of h: wait
// (bounded) until its eight 32-blocks are written.
__device__ __forceinline__ bool ffn_wait_ready(const Group& G, int b) {
  const unsigned int* f = G.ffn.ready + b;
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  if (v < 8u) {
    const long long t0 = clock64();
    for (;;) {
      __nanosleep(100);
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
      if (v >= 8u) break;
      if (clock64() - t0 > G.ffn.ready_limit) {
        atomicCAS(&g_gemv_error, 0u, 3u);
        return false;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// Tasks after each CTA's first (its own index): from the counter, which
// starts at zero, offset by the grid size; or strided by the grid size.
// A producer fetches once per task it runs, so a launch makes exactly
// G.total fetches and the one that returns G.total - 1 is the last to touch
// the counter: it puts the counter back to zero, and a later launch on the
// same workspace finds it as the quantize launch leaves it.
__device__ __forceinline__ int next_task(const Group& G, int cur) {
  if (G.counter) {
    const unsigned old = atomicAdd(G.counter, 1u);
    if (old == static_cast<unsigned>(G.total - 1)) atomicExch(G.counter, 0u);
    return static_cast<int>(gridDim.x + old);
  }
  return cur + static_cast<int>(gridDim.x);
}

// ------------------------------------------------- small-M (M <= 2) form
//
// At one or two tokens the m16n8k16 MMA uses 1/8 or 2/8 of its columns but
// still pays the full fp16 unpack of every weight. The small form keeps the
// producer, ring, tasks and K-split of the grouped GEMV and replaces the
// consumer arithmetic with exact integer dot products on the CUDA cores
// (dp4a: four unsigned nibbles times four signed int8 activations):
//   - a stage holds, besides the weight boxes, each token's 256 int8
//     quants, 8 d8 and 8 s8 of the super-block (plain Q8 buffer regions,
//     bulk-copied), not the 8-token fp16 operand image;
//   - lane l of a consumer warp takes weight row l/2 of the warp's 16 and
//     half l%2 of the super-block (quant bytes 64h..64h+63: sub-blocks
//     4h..4h+3) and forms each sub-block's isum with 8 dp4a per token.
// The fp32 arithmetic is the MMA consumer's, operation for operation, so the
// two forms give bit-identical y (batch invariance across M holds):
//   - high nibbles stay in place (16q, one mask per word), as in the MMA
//     operand; the dp4a accumulator starts at the bit pattern of 0.75f,
//     whose unit in the last place is 2^-24, so the int32 result is 0.75f
//     plus isum (low nibbles) or 16 isum (high) units, and subtracting 0.75f
//     leaves exactly the MMA's D (isum * 2^-24, or isum * 2^-20);
//     |16 isum| <= 16*15*127*32 < 2^22 keeps the sum inside the binade;
//   - the coefficients carry the same 2^24 / 2^20 factors as
//     decode_scales_q4, and each sub-block adds
//     fma(RN(a*d8), D, fma(-dmin*m, s8, acc)) as compute_block_q4 does;
//   - a super-block's eight terms go into its fresh accumulator in sub-block
//     order: half 0 adds sub-blocks 0..3 from zero, passes the result to
//     half 1 (one shuffle), which adds 4..7; the running sum and total then
//     follow the MMA consumer, and half 1 stores.
// Only Q4_K takes it, at M <= 2 outside the batch-invariant entry points
// (whose activations are the 8-token operand image).

template <bool SMALL>
__device__ __forceinline__ unsigned act_bytes(const Proj& P) {
  return SMALL ? 320u * static_cast<unsigned>(P.M) : 8u * 512u + 8u * 64u;
}

// The activation part of a stage for super-block b: the operand image (fp16
// fragments and scale quads), or in the small form each token's quants
// (256 bytes at +256m), d8 (32 bytes at +512+32m) and s8 (at +576+32m).
template <int TYPE, bool SMALL>
__device__ __forceinline__ void act_load(uint32_t st, const Proj& P, int b, uint32_t bar) {
  constexpr int kFragOff = GLay<TYPE>::kFragOff, kFscOff = GLay<TYPE>::kFscOff;
  // (checked builds: every source range inside the Q8 buffer, 16-byte aligned)
  auto in_q8 = [&](const void* src, unsigned n) {
    const uint8_t* p = static_cast<const uint8_t*>(src);
    return XQ_CHECKED(p >= P.xq0 && p + n <= P.xq0 + P.xq_bytes && (reinterpret_cast<uintptr_t>(p) & 15) == 0,
                      kChkGemvAct);
  };
  if (SMALL) {
    const int nsub = P.K >> 5;
    for (int m = 0; m < P.M; ++m) {
      const uint8_t* q = P.aq + static_cast<size_t>(m) * P.K + 256 * static_cast<size_t>(b);
      const float* d = P.ad8 + static_cast<size_t>(m) * nsub + 8 * b;
      const float* s8 = P.as8 + static_cast<size_t>(m) * nsub + 8 * b;
      if (in_q8(q, 256)) bulk_load(st + kFragOff + 256 * m, q, 256, bar);
      if (in_q8(d, 32)) bulk_load(st + kFragOff + 512 + 32 * m, d, 32, bar);
      if (in_q8(s8, 32)) bulk_load(st + kFragOff + 576 + 32 * m, s8, 32, bar);
    }
  } else {
    const uint8_t* f = P.frag + static_cast<size_t>(b) * 8 * 512;
    const uint8_t* c = P.fsc + static_cast<size_t>(b) * 8 * 64;
    if (in_q8(f, 8 * 512)) bulk_load(st + kFragOff, f, 8 * 512, bar);
    if (in_q8(c, 8 * 64)) bulk_load(st + kFscOff, c, 8 * 64, bar);
  }
}

constexpr int kMagicLo = 0x3F400000;  // 0.75f: unit in the last place 2^-24

// One super-block of the lane's row (small form): acc[m] = the super-block's
// fresh accumulator for token m < P.M, complete in the lanes of half 1.
template <bool ISUM>
__device__ __forceinline__ void compute_small_q4(const uint8_t* blk, const uint8_t* act, const Proj& P, int row, int b,
                                                 int r, int h, int lane, float (&acc)[2]) {
  const uint8_t* rp = blk + r * kQ4kBytes;
  const uint4 hd = *reinterpret_cast<const uint4*>(rp);
  const uint4* qp = reinterpret_cast<const uint4*>(rp + 16 + 64 * h);
  const uint4 q0 = qp[0], q1 = qp[1], q2 = qp[2], q3 = qp[3];
  const uint32_t w[16] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w,
                          q2.x, q2.y, q2.z, q2.w, q3.x, q3.y, q3.z, q3.w};
  // (sc, m) of sub-blocks 4h..4h+3 (public Q4_K packing) and the MMA form's
  // coefficients: a = d*sc*2^24 (even sub-blocks) or d*sc*2^20 (odd), and
  // -dmin*m, each an exact product
  const unsigned scw = h ? ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u)) : (hd.y & 0x3F3F3F3Fu);
  const unsigned mnw = h ? (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u)) : (hd.z & 0x3F3F3F3Fu);
  const float d = half_bits_to_float(hd.x);
  const float dl = d * 16777216.0f, dh = d * 1048576.0f;
  const float dm = -half_bits_to_float(hd.x >> 16);
  const float cl = -8388608.0f * dl, ch = -8388608.0f * dh, cm = -8388608.0f * dm;
  float al[4], be[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    al[k] = (k & 1) ? fmaf(byte_plus_2p23(scw, k), dh, ch) : fmaf(byte_plus_2p23(scw, k), dl, cl);
    be[k] = fmaf(byte_plus_2p23(mnw, k), dm, cm);
  }
  // sub-block 4h+k: group k/2 of the lane's 64 bytes, low nibbles for even k
  uint32_t nib[4][8];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t x = w[8 * (k >> 1) + i];
      // high nibbles stay in place (16q): one mask, no shift
      nib[k][i] = x & ((k & 1) ? 0xF0F0F0F0u : 0x0F0F0F0Fu);
    }
  const int nsub = P.K >> 5;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    if (m < P.M) {
      const uint4* ap = reinterpret_cast<const uint4*>(act + 256 * m + 128 * h);
      const float4 dv = *reinterpret_cast<const float4*>(act + 512 + 32 * m + 16 * h);
      const float4 sv = *reinterpret_cast<const float4*>(act + 576 + 32 * m + 16 * h);
      const float d8[4] = {dv.x, dv.y, dv.z, dv.w}, s8[4] = {sv.x, sv.y, sv.z, sv.w};
      float D[4], cf[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 a0 = ap[2 * k], a1 = ap[2 * k + 1];
        const int magic = kMagicLo;
        int v = dp4a_us(nib[k][0], a0.x, magic);
        v = dp4a_us(nib[k][1], a0.y, v);
        v = dp4a_us(nib[k][2], a0.z, v);
        v = dp4a_us(nib[k][3], a0.w, v);
        v = dp4a_us(nib[k][4], a1.x, v);
        v = dp4a_us(nib[k][5], a1.y, v);
        v = dp4a_us(nib[k][6], a1.z, v);
        v = dp4a_us(nib[k][7], a1.w, v);
        if (ISUM && row < P.N) {
          const size_t ii = (static_cast<size_t>(m) * P.N + row) * nsub + 8 * b + 4 * h + k;
          if (XQ_IN(ii, static_cast<size_t>(P.M) * P.N * nsub, kChkGemvIsum))
            P.isum[ii] = (k & 1) ? (v - magic) >> 4 : v - magic;
        }
        D[k] = __int_as_float(v) - 0.75f;
        cf[k] = al[k] * d8[k];
      }
      // sub-blocks 0..3 from zero (half 0), then 4..7 from half 0's result
      float c = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) c = fmaf(cf[k], D[k], fmaf(be[k], s8[k], c));
      const float c0 = __shfl_sync(0xffffffffu, c, lane & ~1);
      if (h) {
        c = c0;
#pragma unroll
        for (int k = 0; k < 4; ++k) c = fmaf(cf[k], D[k], fmaf(be[k], s8[k], c));
      }
      acc[m] = c;
    }
  }
}

// Q6_K in the small form: one super-block of the lane's row, half h (weights
// 128h..128h+127: 32-blocks p = 4h + k, ql bytes 64h.., qh bytes 128 + 32h..,
// scales 192 + 8h..), the super-block starting `off` bytes into its window.
// The MMA form's arithmetic, operation for operation:
//   - a byte's 6-bit q (low nibble from ql, two bits from qh) becomes
//     4 (q - 32) as a signed byte, (q ^ 0x20) << 2, and one dp4a per word
//     sums 4 (q - 32) * a;
//   - the dp4a accumulator starts at the bits of 3145728.0f, whose unit in
//     the last place is 0.25, so subtracting that float leaves each 16-group's
//     exact integer sum (|4 isum| < 2^22 keeps it in the binade): Da = the
//     32-block's sum, D1 = its second group's, as the MMA form's D;
//   - alpha = d * s_2p and delta = d * (s_2p+1 - s_2p) as decode_scales_q6,
//     and acc = fma(alpha d8, Da, fma(delta d8, D1, acc)) in 32-block order.
constexpr int kMagicQ6 = 0x4A400000;  // 3145728.0f: unit in the last place 0.25

template <bool ISUM>
__device__ __forceinline__ void compute_small_q6(const uint8_t* blk, int off, const uint8_t* act, const Proj& P, int row,
                                                 int b, int r, int h, int lane, float (&acc)[2]) {
  const uint8_t* sb = blk + r * GLay<14>::kBoxRow + off;
  uint32_t ql[16], qh[8], sw[2];
  load_words<16>(sb + 64 * h, ql);
  load_words<8>(sb + 128 + 32 * h, qh);
  load_words<2>(sb + 192 + 8 * h, sw);
  const float d = half_bits_to_float(*reinterpret_cast<const unsigned short*>(sb + 208));
  float al[4], de[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w = sw[k >> 1];
    const int b0 = 2 * (k & 1);
    const int s0 = static_cast<int8_t>((w >> (8 * b0)) & 0xFFu);
    const int s1 = static_cast<int8_t>((w >> (8 * b0 + 8)) & 0xFFu);
    al[k] = d * static_cast<float>(s0);
    de[k] = d * static_cast<float>(s1 - s0);
  }
  // 4 (q - 32) of weights 4i..4i+3 of 32-block k
  uint32_t y[4][8];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t Lw = (k & 1) ? ql[8 + i] : ql[i];
      const uint32_t L = ((k >> 1) ? (Lw >> 4) : Lw) & 0x0F0F0F0Fu;
      const uint32_t H = (k == 0 ? (qh[i] << 4) : (k == 1 ? (qh[i] << 2) : (k == 2 ? qh[i] : (qh[i] >> 2)))) & 0x30303030u;
      y[k][i] = ((L | H) ^ 0x20202020u) << 2;
    }
  const int ngrp = P.K >> 4;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    if (m < P.M) {
      const uint4* ap = reinterpret_cast<const uint4*>(act + 256 * m + 128 * h);
      const float4 dv = *reinterpret_cast<const float4*>(act + 512 + 32 * m + 16 * h);
      const float d8[4] = {dv.x, dv.y, dv.z, dv.w};
      float Da[4], D1[4], ca[4], cd[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 a0 = ap[2 * k], a1 = ap[2 * k + 1];
        int v0 = dp4a_ss(y[k][0], a0.x, kMagicQ6);
        v0 = dp4a_ss(y[k][1], a0.y, v0);
        v0 = dp4a_ss(y[k][2], a0.z, v0);
        v0 = dp4a_ss(y[k][3], a0.w, v0);
        int v1 = dp4a_ss(y[k][4], a1.x, kMagicQ6);
        v1 = dp4a_ss(y[k][5], a1.y, v1);
        v1 = dp4a_ss(y[k][6], a1.z, v1);
        v1 = dp4a_ss(y[k][7], a1.w, v1);
        const float g0 = __int_as_float(v0) - 3145728.0f, g1 = __int_as_float(v1) - 3145728.0f;
        D1[k] = g1;
        Da[k] = g0 + g1;
        if (ISUM && row < P.N) {
          const size_t ii = (static_cast<size_t>(m) * P.N + row) * ngrp + 16 * b + 8 * h + 2 * k;
          if (XQ_IN(ii + 1, static_cast<size_t>(P.M) * P.N * ngrp, kChkGemvIsum)) {
            P.isum[ii] = static_cast<int32_t>(g0);
            P.isum[ii + 1] = static_cast<int32_t>(g1);
          }
        }
        ca[k] = al[k] * d8[k];
        cd[k] = de[k] * d8[k];
      }
      // 32-blocks 0..3 from zero (half 0), then 4..7 from half 0's result
      float c = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) c = fmaf(ca[k], Da[k], fmaf(cd[k], D1[k], c));
      const float c0 = __shfl_sync(0xffffffffu, c, lane & ~1);
      if (h) {
        c = c0;
#pragma unroll
        for (int k = 0; k < 4; ++k) c = fmaf(ca[k], Da[k], fmaf(cd[k], D1[k], c));
      }
      acc[m] = c;
    }
  }
}

// The last warp to finish a split 16-row group (small form): lane 2r+1 adds
// row r's chunk partials in chunk order (as reduce_chunks does).
__device__ __forceinline__ void reduce_chunks_small(const Proj& P, int rg, int r, int h) {
  const int rows_pad = gemv_row_blocks(P.N) * kGemvRows;
  const int row = group_row(P, rg, r);
  if (h == 0 || row >= P.N) return;
  for (int m = 0; m < P.M; ++m) {
    float v = 0.0f;
    for (int c = 0; c < P.nch; ++c) {
      const size_t i = (static_cast<size_t>(c) * 8 + m) * rows_pad + row;
      if (XQ_IN(i, static_cast<size_t>(P.nch) * 8 * rows_pad, kChkGemvPartial)) v += __ldcg(P.partial + i);
    }
    if (XQ_IN(static_cast<size_t>(m) * P.N + row, P.y_elems, kChkGemvY))
      P.y[static_cast<size_t>(m) * P.N + row] = v;
  }
}

__device__ __forceinline__ TaskPos task_pos(const Group& G, int task);

// Consumer loop of the small form (the same ring, meta, task and split
// protocol as the MMA consumers).
template <int TYPE, bool ISUM, bool FFN>
__device__ __forceinline__ void small_consumer(const Group& G, const uint8_t* ring, const int4* meta, uint32_t full_s,
                                               uint32_t empty_s, int kStages, int kStageBytes, int kBlockBytes,
                                               int kFragOff, int warp, int lane) {
  const int r = lane >> 1, h = lane & 1;
  float run[2] = {0.0f, 0.0f}, tot[2] = {0.0f, 0.0f};
  int nrun = 0;
  int slot = 0;
  unsigned fills = 0;
  int cur_task = -1;
  TaskPos tp = {0, 0, 0, 0, 0};
  int pend_p = -1, pend_rg = 0;
  unsigned pend_old = 0;
  auto resolve = [&]() {
    if (pend_p < 0) return;
    const Proj& Q = G.p[pend_p];
    const unsigned old = __shfl_sync(0xffffffffu, pend_old, 0);
    if (old == static_cast<unsigned>(Q.nch - 1)) {
      __syncwarp();  // lane 0's acquiring increment, a stage ago, covers the partials
      if (lane == 0) Q.arrive[pend_rg] = 0u;
      reduce_chunks_small(Q, pend_rg, r, h);
      if (FFN && (pend_p == G.ffn.gate || pend_p == G.ffn.up)) ffn_arrive(G, pend_rg, lane);
    }
    pend_p = -1;
  };
  for (;;) {
    if (!mbar_wait(full_s + 8 * slot, fills & 1, 2, G.wait_limit)) return;
    const int4 m = meta[slot];
    if (m.x < 0) {
      resolve();
      return;
    }
    if (m.x != cur_task) {
      cur_task = m.x;
      tp = task_pos(G, m.x);
    }
    const Proj& P = G.p[tp.p];
    const int rg = tp.rb * kGemvWarps + warp;
    const int row = group_row(P, rg, r);
    const uint8_t* st = ring + slot * kStageBytes;
    float acc[2] = {0.0f, 0.0f};
    if (rg * 16 < P.N) {
      if constexpr (TYPE == 12) {
        compute_small_q4<ISUM>(st + warp * kBlockBytes, st + kFragOff, P, row, m.y, r, h, lane, acc);
      } else {
        // the same in-window offset for every row of the group (as the MMA form)
        const int off = (kQ6kBytes * ((P.K >> 8) * (rg & ((1 << P.gs) - 1)) + m.y)) & 15;
        compute_small_q6<ISUM>(st + warp * kBlockBytes, off, st + kFragOff, P, row, m.y, r, h, lane, acc);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_s + 8 * slot);
    run[0] += acc[0];
    run[1] += acc[1];
    if (++nrun == 32) {
      tot[0] += run[0];
      tot[1] += run[1];
      run[0] = run[1] = 0.0f;
      nrun = 0;
    }
    resolve();
    if (m.z) {
      const float v[2] = {tot[0] + run[0], tot[1] + run[1]};
      run[0] = run[1] = tot[0] = tot[1] = 0.0f;
      nrun = 0;
      if (P.nch == 1) {
        if (h == 1 && row < P.N)
          for (int t = 0; t < P.M; ++t)
            if (XQ_IN(static_cast<size_t>(t) * P.N + row, P.y_elems, kChkGemvY))
              P.y[static_cast<size_t>(t) * P.N + row] = v[t];
        if (FFN && rg * 16 < P.N && (tp.p == G.ffn.gate || tp.p == G.ffn.up)) ffn_arrive(G, rg, lane);
      } else if (rg * 16 < P.N) {
        const int rows_pad = gemv_row_blocks(P.N) * kGemvRows;
        float* part = P.partial + static_cast<size_t>(tp.c) * 8 * rows_pad;
        if (h == 1)
          for (int t = 0; t < P.M; ++t)
            if (XQ_IN((static_cast<size_t>(tp.c) * 8 + t) * rows_pad + row, static_cast<size_t>(P.nch) * 8 * rows_pad,
                      kChkGemvPartial))
              part[static_cast<size_t>(t) * rows_pad + row] = v[t];
        __syncwarp();
        if (lane == 0 && XQ_IN(rg, gemv_row_blocks(P.N) * kGemvWarps, kChkGemvArrive))
          pend_old = arrive_acq_rel(P.arrive + rg);
        pend_p = tp.p;
        pend_rg = rg;
      }
    }
    if (++slot == kStages) {
      slot = 0;
      ++fills;
    }
  }
}

template <int TYPE, bool ISUM, bool SMALL, bool FFN>
__device__ __forceinline__ void gemv_mma_body(const Group& G) {
  // Body of gemv_mma_kernel: a return here leaves through the kernel's
  // deferred dependency wait.
  using Lay = GLay<TYPE>;
  constexpr int kStages = Lay::kStages, kStageBytes = Lay::kStageBytes, kBlockBytes = Lay::kBlockBytes;
  constexpr int kFragOff = Lay::kFragOff;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float4* dec_all = reinterpret_cast<float4*>(smem + kStages * kStageBytes);
  int4* meta = reinterpret_cast<int4*>(smem + kStages * kStageBytes + kGemvWarps * kDecBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kGemvWarps * kDecBytes + kStages * 16);
  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const uint32_t full_s = static_cast<uint32_t>(__cvta_generic_to_shared(bars));
  const uint32_t empty_s = full_s + kStages * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_s + 8 * s, 1);
      mbar_init(empty_s + 8 * s, kGemvWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();
  if (warp == kGemvWarps) {
    // ------------------------------------------------------- producer
    if (lane != 0) return;
    if (G.stall) {
      if (G.wait_prev) cudaGridDependencySynchronize();
      cudaTriggerProgrammaticLaunchCompletion();
      return;
    }
    // Each CTA's first task is its own index; later tasks come from the
    // counter (or a stride). The weights do not depend on the previous grid
    // on the stream, so the weight boxes of the first task's first stages are
    // requested before waiting for it; the activation image, the task
    // counter and the arrival counts may be written by that grid.
    int task = static_cast<int>(blockIdx.x);
    int slot = 0;
    unsigned fills = 0;  // completed passes over the ring
    int bresume = -1;    // first super-block of the first task not yet requested
    if (task < G.total) {
      const TaskPos tp = task_pos(G, task);
      const Proj& P = G.p[tp.p];
      const int rows = P.N - tp.rb * kGemvRows;
      const int nblk = rows >= kGemvRows ? kGemvWarps : (rows + 15) / 16;
      int b = tp.b0;
      for (; b < tp.b1 && slot < kStages; ++b, ++slot) {
        meta[slot] = make_int4(task, b, (b == tp.b1 - 1) ? 1 : 0, 0);
        mbar_expect_tx(full_s + 8 * slot, static_cast<unsigned>(nblk * kBlockBytes) + act_bytes<SMALL>(P));
        const uint32_t st = ring_s + slot * kStageBytes;
        for (int w = 0; w < nblk; ++w) {
          int bx, by;
          weight_box<TYPE>(P, tp.rb * kGemvWarps + w, b, bx, by);
          tma_load_2d(st + w * kBlockBytes, &P.map, bx, by, full_s + 8 * slot);
        }
      }
      bresume = b;
    }
    if (G.wait_prev) cudaGridDependencySynchronize();
    cudaTriggerProgrammaticLaunchCompletion();
    if (task < G.total) {
      const TaskPos tp = task_pos(G, task);
      const Proj& P = G.p[tp.p];
      for (int k = 0; k < slot; ++k) {
        const uint32_t st = ring_s + k * kStageBytes;
        if (FFN && tp.p == G.ffn.down && !ffn_wait_ready(G, tp.b0 + k)) return;
        act_load<TYPE, SMALL>(st, P, tp.b0 + k, full_s + 8 * k);
      }
    }
    if (slot == kStages) {
      slot = 0;
      fills = 1;
    }
    for (;;) {
      const bool valid = task < G.total;
      TaskPos tp = {0, 0, 0, 1, 0};
      if (valid) tp = task_pos(G, task);
      const int nxt = valid ? next_task(G, task) : task;
      const int bfirst = bresume >= 0 ? bresume : tp.b0;
      bresume = -1;
      for (int b = bfirst; b < tp.b1; ++b) {
        if (fills > 0 && !mbar_wait(empty_s + 8 * slot, (fills - 1) & 1, 1, G.wait_limit)) return;
        meta[slot] = make_int4(valid ? task : -1, b, (b == tp.b1 - 1) ? 1 : 0, 0);
        if (!valid) {
          mbar_arrive(full_s + 8 * slot);
          return;
        }
        const Proj& P = G.p[tp.p];
        const int rows = P.N - tp.rb * kGemvRows;  // > 0
        const int nblk = rows >= kGemvRows ? kGemvWarps : (rows + 15) / 16;
        mbar_expect_tx(full_s + 8 * slot, static_cast<unsigned>(nblk * kBlockBytes) + act_bytes<SMALL>(P));
        const uint32_t st = ring_s + slot * kStageBytes;
        for (int w = 0; w < nblk; ++w) {
          int bx, by;
          weight_box<TYPE>(P, tp.rb * kGemvWarps + w, b, bx, by);
          tma_load_2d(st + w * kBlockBytes, &P.map, bx, by, full_s + 8 * slot);
        }
        if (FFN && tp.p == G.ffn.down && !ffn_wait_ready(G, b)) return;
        act_load<TYPE, SMALL>(st, P, b, full_s + 8 * slot);
        if (++slot == kStages) {
          slot = 0;
          ++fills;
        }
      }
      task = nxt;
    }
  }

  // --------------------------------------------------------- consumers
  if (G.wait_prev) cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();
  if constexpr (SMALL) {
    small_consumer<TYPE, ISUM, FFN>(G, ring, meta, full_s, empty_s, kStages, kStageBytes, kBlockBytes, kFragOff, warp,
                                    lane);
    return;
  }
  const int n8 = lane >> 2, t = lane & 3;
  float4* dec = dec_all + warp * (kDecBytes / 16);
  // Accumulation bounded by construction: one super-block's terms (at most
  // 16 fp32 roundings) go into a fresh accumulator, added once to a running
  // sum; every 32 super-blocks the running sum is added to a total.
  f2 run[2] = {0ull, 0ull}, tot[2] = {0ull, 0ull};
  int nrun = 0;
  int slot = 0;
  unsigned fills = 0;
  int cur_task = -1;
  TaskPos tp = {0, 0, 0, 0, 0};
  // Split tasks: each warp owns one arrival count per 16-row group. Lane 0
  // increments it once the warp's partials are stored; the warp examines the
  // count it got one stage later, so the atomic's round trip overlaps that
  // stage's compute, and no barrier couples the four warps. pend_p >= 0
  // marks a pending hand-off (projection and row group; pend_old is lane 0's
  // count before the increment).
  int pend_p = -1, pend_rg = 0;
  unsigned pend_old = 0;
  auto resolve = [&]() {
    if (pend_p < 0) return;
    const Proj& Q = G.p[pend_p];
    const unsigned old = __shfl_sync(0xffffffffu, pend_old, 0);
    if (old == static_cast<unsigned>(Q.nch - 1)) {  // every chunk has arrived
      __syncwarp();  // lane 0's acquiring increment, a stage ago, covers the partials
      if (lane == 0) Q.arrive[pend_rg] = 0u;  // ready for the next launch
      reduce_chunks(Q, pend_rg, n8, t);
      if (FFN && (pend_p == G.ffn.gate || pend_p == G.ffn.up)) ffn_arrive(G, pend_rg, lane);
    }
    pend_p = -1;
  };
  for (;;) {
    if (!mbar_wait(full_s + 8 * slot, fills & 1, 2, G.wait_limit)) return;
    const int4 m = meta[slot];
    if (m.x < 0) {
      resolve();
      return;
    }
    if (m.x != cur_task) {  // task geometry, once per task
      cur_task = m.x;
      tp = task_pos(G, m.x);
    }
    const Proj& P = G.p[tp.p];
    const int rg = tp.rb * kGemvWarps + warp;  // this warp's 16-row group
    const uint8_t* st = ring + slot * kStageBytes;
    const bool rows_ok = rg * 16 < P.N;
    f2 acc[2] = {0ull, 0ull};
    if (rows_ok) {
      if constexpr (TYPE == 12) {
        decode_scales_q4(st + warp * kBlockBytes, dec, lane);
        __syncwarp();
        compute_block_q4<ISUM>(st + warp * kBlockBytes, st + kFragOff, dec, P, rg, m.y, n8, t, lane, acc);
      } else if constexpr (TYPE == 8) {
        decode_scales_q8_0(st + warp * kBlockBytes, dec, lane);
        __syncwarp();
        compute_block_q8_0<ISUM>(st + warp * kBlockBytes, st + kFragOff, dec, P, rg, m.y, n8, t, lane, acc);
      } else if constexpr (TYPE == 23) {
        const int off = (kIq4xsBytes * m.y) & 15;  // 0 or 8, the same for every row (rows are 16-byte multiples)
        decode_scales_iq4xs(st + warp * kBlockBytes, off, dec, lane);
        __syncwarp();
        compute_block_iq4xs<ISUM>(st + warp * kBlockBytes, off, st + kFragOff, dec, P, rg, m.y, n8, t, lane, acc);
      } else {
        // the same for every row of the group: rows are 16-byte multiples, or
        // (grouped view) the group's rows share their position in the view
        const int off = (kQ6kBytes * ((P.K >> 8) * (rg & ((1 << P.gs) - 1)) + m.y)) & 15;
        decode_scales_q6(st + warp * kBlockBytes, off, dec, lane);
        __syncwarp();
        compute_block_q6<ISUM>(st + warp * kBlockBytes, off, st + kFragOff, dec, P, rg, m.y, n8, t, lane, acc);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_s + 8 * slot);
    run[0] = add2(run[0], acc[0]);
    run[1] = add2(run[1], acc[1]);
    if (++nrun == 32) {
      tot[0] = add2(tot[0], run[0]);
      tot[1] = add2(tot[1], run[1]);
      run[0] = run[1] = 0ull;
      nrun = 0;
    }
    resolve();  // a split hand-off from an earlier task, one stage later
    if (m.z) {
      acc[0] = add2(tot[0], run[0]);
      acc[1] = add2(tot[1], run[1]);
      run[0] = run[1] = tot[0] = tot[1] = 0ull;
      nrun = 0;
      if (P.nch == 1) {
        if (rows_ok) {
          store_y(P, rg, n8, t, lo32(acc[0]), hi32(acc[0]), lo32(acc[1]), hi32(acc[1]));
          if (FFN && (tp.p == G.ffn.gate || tp.p == G.ffn.up)) ffn_arrive(G, rg, lane);
        }
      } else if (rows_ok) {
        // K-chunk partial of a split task; the last warp to finish the row
        // group adds the chunks in chunk order (arrive_acq_rel orders the
        // stores and the reads).
        const int rows_pad = gemv_row_blocks(P.N) * kGemvRows;
        float* part = P.partial + static_cast<size_t>(tp.c) * 8 * rows_pad;
        const int r0 = rg * 16 + mma_row(n8), r1 = r0 + 8, c0 = 2 * t, c1 = c0 + 1;
        if (XQ_IN((static_cast<size_t>(tp.c) * 8 + c1) * rows_pad + (r0 > r1 ? r0 : r1),
                  static_cast<size_t>(P.nch) * 8 * rows_pad, kChkGemvPartial)) {
          part[static_cast<size_t>(c0) * rows_pad + r0] = lo32(acc[0]);
          part[static_cast<size_t>(c1) * rows_pad + r0] = hi32(acc[0]);
          part[static_cast<size_t>(c0) * rows_pad + r1] = lo32(acc[1]);
          part[static_cast<size_t>(c1) * rows_pad + r1] = hi32(acc[1]);
        }
        __syncwarp();
        if (lane == 0 && XQ_IN(rg, gemv_row_blocks(P.N) * kGemvWarps, kChkGemvArrive))
          pend_old = arrive_acq_rel(P.arrive + rg);
        pend_p = tp.p;
        pend_rg = rg;
      }
    }
    if (++slot == kStages) {
      slot = 0;
      ++fills;
    }
  }
}

template <int TYPE, bool ISUM, bool SMALL, bool FFN>
__global__ void __launch_bounds__(32 * (kGemvWarps + 1), kGemvCtasPerSM)
gemv_mma_kernel(const __grid_constant__ Group G) {
  gemv_mma_body<TYPE, ISUM, SMALL, FFN>(G);
  // A launch that did not wait for the previous grid on entry waits before
  // its threads exit, so that its completion still implies the completion of
  // every earlier kernel on the stream (the next kernel's dependency wait
  // relies on that).
  if (!G.wait_prev) cudaGridDependencySynchronize();
}

template <int TYPE, bool ISUM, bool SMALL = false, bool FFN = false>
int max_ctas() {
  static int per_sm = -1;
  if (per_sm < 0) {
    int n = 0;
    constexpr int kSmemBytes = GLay<TYPE>::kSmemBytes;
    cudaFuncSetAttribute(gemv_mma_kernel<TYPE, ISUM, SMALL, FFN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSmemBytes);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_mma_kernel<TYPE, ISUM, SMALL, FFN>, 32 * (kGemvWarps + 1),
                                                      kSmemBytes) != cudaSuccess ||
        n < 1)
      n = 1;
    per_sm = n;
  }
  return per_sm * kNumSMs;
}

// Weight rows as a 2D tensor, boxes of 16 rows: Q4_K as 8-byte elements
// {row_bytes/8, N} with one super-block per box row; Q6_K and IQ4_XS as
// bytes {row_bytes, N} with 240- and 144-byte box rows (rows must be 16-byte
// multiples).
bool encode_weight_map(int type, CUtensorMap* map, const uint8_t* W, int N, int K) {
  const unsigned long long nsb = static_cast<unsigned long long>(K / 256);
  if (type == 14 && q6k_row_shift(K) > 0) {
    // grouped view: 2^gs rows per tensor-map row
    const int gs = q6k_row_shift(K);
    const unsigned long long vrow = (nsb * kQ6kBytes) << gs;
    return encode_tma_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, vrow, static_cast<unsigned long long>(N >> gs), vrow,
                         GLay<14>::kBoxRow, 16);
  }
  if (type == 12)
    return encode_tma_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, W, nsb * kQ4kBytes / 8, static_cast<unsigned long long>(N),
                         nsb * kQ4kBytes, kQ4kBytes / 8, 16);
  if (type == 8)
    return encode_tma_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, W, nsb * kQ80Group / 8, static_cast<unsigned long long>(N),
                         nsb * kQ80Group, kQ80Group / 8, 16);
  if (type == 23)
    return encode_tma_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, nsb * kIq4xsBytes, static_cast<unsigned long long>(N),
                         nsb * kIq4xsBytes, GLay<23>::kBoxRow, 16);
  return encode_tma_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, nsb * kQ6kBytes, static_cast<unsigned long long>(N),
                       nsb * kQ6kBytes, GLay<14>::kBoxRow, 16);
}

}  // namespace

cudaError_t take_gemv_check(unsigned int* code) { return take_check_word(code); }

cudaError_t take_gemv_error(unsigned int* code) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_gemv_error, &z, sizeof(z));
  *code = v;
  return e;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, unsigned long long dim0,
                   unsigned long long dim1, unsigned long long stride1, unsigned box0, unsigned box1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int q6k_row_shift(int K) {
  const int row = (K / 256) * kQ6kBytes;
  int gs = 0;
  while (gs < 3 && ((row << gs) & 15) != 0) ++gs;
  return gs;
}

bool gemv_mma_supports(int type, int N, int K) {
  if (type == 14) {
    const int gs = q6k_row_shift(K);
    return gs == 0 || (N % (16 << gs)) == 0;
  }
  return type == 12 || type == 8 || (type == 23 && ((K / 256) % 2) == 0);
}

cudaError_t launch_gemv_mma(int type, const MmaProj* projs, int n, cudaStream_t s, bool pdl, unsigned int* counter,
                            uint8_t* arrive_ws, uint8_t* partial_ws, bool wait_prev, bool stall_test,
                            const FfnFuse* ffn) {
  if (n <= 0 || n > kMaxProj || (type != 12 && type != 14 && type != 8 && type != 23)) return cudaErrorInvalidValue;
  if (ffn) {
    const bool ok = ffn->gate >= 0 && ffn->gate < n && ffn->up >= 0 && ffn->up < n && ffn->gate != ffn->up &&
                    ffn->down < n && ffn->down != ffn->gate && ffn->down != ffn->up && ffn->arrive && ffn->ready &&
                    ffn->hq && ffn->M >= 1 && ffn->M <= 8 && (ffn->F % 256) == 0 && projs[ffn->gate].N == ffn->F &&
                    projs[ffn->up].N == ffn->F && projs[ffn->gate].M_total == ffn->M &&
                    projs[ffn->up].M_total == ffn->M && projs[ffn->gate].chunk == 0 && projs[ffn->up].chunk == 0 &&
                    (ffn->down < 0 || (projs[ffn->down].K == ffn->F && projs[ffn->down].xq == ffn->hq &&
                                       projs[ffn->down].M_total == ffn->M));
    if (!ok) return cudaErrorInvalidValue;
  }
  // Per-projection K-chunking (only with split workspaces) and task cost.
  const bool split = arrive_ws != nullptr && partial_ws != nullptr;
  int nch[kMaxProj], cost[kMaxProj];
  for (int k = 0; k < n; ++k) {
    nch[k] = (split && projs[k].nch > 1) ? projs[k].nch : 1;
    cost[k] = ((projs[k].K >> 8) + nch[k] - 1) / nch[k];
  }
  // With a fused feed, gate and up go first, so that h is complete about when
  // the first wave of tasks ends, and down goes last: its tasks wait for h.
  if (ffn) {
    cost[ffn->gate] = cost[ffn->up] = 1 << 30;
    if (ffn->down >= 0) cost[ffn->down] = -1;
  }
  // Most expensive tasks first (dynamic scheduling takes them in order).
  int order[kMaxProj];
  for (int k = 0; k < n; ++k) order[k] = k;
  for (int a = 1; a < n; ++a)
    for (int b = a; b > 0 && cost[order[b]] > cost[order[b - 1]]; --b) {
      const int tmp = order[b];
      order[b] = order[b - 1];
      order[b - 1] = tmp;
    }
  // Split workspaces: arrival counts and partial buffers, in item order.
  size_t arrive_off[kMaxProj], partial_off[kMaxProj];
  {
    size_t a = 0, p = 0;
    for (int k = 0; k < n; ++k)
      if (nch[k] > 1) {
        arrive_off[k] = a;
        a += gemv_split_arrive_bytes(projs[k].N);
        partial_off[k] = p;
        p += gemv_split_partial_bytes(projs[k].N, nch[k]);
      }
  }
  Group G;
  G.n = n;
  G.counter = counter;
  G.ffn = Ffn{};
  G.ffn.gate = G.ffn.up = G.ffn.down = -1;
  if (ffn) {
    const Q8Layout H = q8_layout(ffn->M, ffn->F, false);
    G.ffn.arrive = ffn->arrive;
    G.ffn.ready = ffn->ready;
    G.ffn.hq = ffn->hq;
    G.ffn.h_out = ffn->h_out;
    G.ffn.qs = H.qs;
    G.ffn.d8 = H.d8;
    G.ffn.s8 = H.s8;
    G.ffn.frag = H.frag;
    G.ffn.fsc = H.fsc;
    G.ffn.F = ffn->F;
    G.ffn.M = ffn->M;
    G.ffn.hq_bytes = H.total;
    G.ffn.stall = ffn->stall ? 1 : 0;
    G.ffn.ready_limit = ffn->stall ? kStallWaitClocks : kWaitClocks;
    for (int k = 0; k < n; ++k) {
      if (order[k] == ffn->gate) G.ffn.gate = k;
      if (order[k] == ffn->up) G.ffn.up = k;
      if (order[k] == ffn->down) G.ffn.down = k;
    }
  }
  G.wait_prev = (wait_prev || !pdl) ? 1 : 0;
  G.stall = stall_test ? 1 : 0;
  G.wait_limit = stall_test ? kStallWaitClocks : kWaitClocks;
  // With h withheld, down's stage waits outlast the producer's wait for h,
  // so that code 3 is the first error recorded.
  if (ffn && ffn->stall) G.wait_limit = 4 * kStallWaitClocks;
  int total = 0;
  bool isum = false;
  // Q4_K and Q6_K at one or two tokens take the small-M (dp4a) form, except
  // in the batch-invariant layout.
  bool small = type == 12 || type == 14;
  for (int k = 0; k < n; ++k)
    small = small && projs[k].M_total <= 2 && projs[k].chunk == 0 && !projs[k].gemv_image;
  for (int k = 0; k < n; ++k) {
    const int src = order[k];
    const MmaProj& q = projs[src];
    const Q8Layout L = q8_layout(q.M_total, q.K, q.gemv_image);
    const int m0 = 8 * q.chunk;
    Proj& P = G.p[k];
    if (!gemv_mma_supports(type, q.N, q.K) || !encode_weight_map(type, &P.map, q.W, q.N, q.K)) return cudaErrorInvalidValue;
    P.gs = type == 14 ? q6k_row_shift(q.K) : 0;
    P.frag = q.xq + L.frag + static_cast<size_t>(q.chunk) * 16 * q.K;
    P.fsc = q.xq + L.fsc + static_cast<size_t>(q.chunk) * 2 * q.K;
    P.aq = q.xq + L.qs;
    P.ad8 = reinterpret_cast<const float*>(q.xq + L.d8);
    P.as8 = reinterpret_cast<const float*>(q.xq + L.s8);
    P.y = q.y + static_cast<size_t>(m0) * q.N;
    P.isum = q.isum;
    P.N = q.N;
    P.K = q.K;
    P.M = (q.M_total - m0) < 8 ? (q.M_total - m0) : 8;
    P.nch = nch[src];
    P.partial = nullptr;
    P.arrive = nullptr;
    for (int i = 0; i < 4; ++i) P.cb[i] = q.codebook[i] ^ 0x80808080u;  // IQ4_XS operand bias
    const int rbs = gemv_row_blocks(q.N);
    if (P.nch > 1) {
      P.partial = reinterpret_cast<float*>(partial_ws + partial_off[src]);
      P.arrive = reinterpret_cast<unsigned int*>(arrive_ws + arrive_off[src]);
    }
    P.xq0 = q.xq;
    P.xq_bytes = L.total;
    {
      const long long full = static_cast<long long>(P.M) * q.N;
      const long long lim = q.y_limit >= 0 ? q.y_limit - static_cast<long long>(m0) * q.N : full;
      P.y_elems = static_cast<unsigned long long>(lim < 0 ? 0 : (lim < full ? lim : full));
    }
    P.task0 = total;
    total += rbs * P.nch;
    isum = isum || (q.isum != nullptr);
  }
  G.total = total;
  if (total == 0) return cudaSuccess;
  // The fused SwiGLU feed has its own instantiations (without the isum
  // hook), so that other launches carry none of its code.
  const bool fz = ffn != nullptr;
  if (fz && isum) return cudaErrorInvalidValue;
  const bool s12 = small && type == 12, s14 = small && type == 14;
  const int cap = fz ? (s12 ? max_ctas<12, false, true, true>()
                       : s14 ? max_ctas<14, false, true, true>()
                       : type == 12 ? max_ctas<12, false, false, true>()
                       : type == 8  ? max_ctas<8, false, false, true>()
                       : type == 23 ? max_ctas<23, false, false, true>()
                                    : max_ctas<14, false, false, true>())
                  : s12        ? (isum ? max_ctas<12, true, true>() : max_ctas<12, false, true>())
                  : s14        ? (isum ? max_ctas<14, true, true>() : max_ctas<14, false, true>())
                  : type == 12 ? (isum ? max_ctas<12, true>() : max_ctas<12, false>())
                  : type == 8  ? (isum ? max_ctas<8, true>() : max_ctas<8, false>())
                  : type == 23 ? (isum ? max_ctas<23, true>() : max_ctas<23, false>())
                               : (isum ? max_ctas<14, true>() : max_ctas<14, false>());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(total < cap ? total : cap));
  cfg.blockDim = dim3(32 * (kGemvWarps + 1));
  cfg.dynamicSmemBytes =
      type == 12 ? GLay<12>::kSmemBytes
                 : (type == 8 ? GLay<8>::kSmemBytes : (type == 23 ? GLay<23>::kSmemBytes : GLay<14>::kSmemBytes));
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (fz) {
    if (s12) return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<12, false, true, true>, G);
    if (s14) return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<14, false, true, true>, G);
    if (type == 12) return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<12, false, false, true>, G);
    if (type == 8) return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<8, false, false, true>, G);
    if (type == 23) return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<23, false, false, true>, G);
    return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<14, false, false, true>, G);
  }
  if (type == 8)
    return isum ? cudaLaunchKernelEx(&cfg, gemv_mma_kernel<8, true, false, false>, G)
                : cudaLaunchKernelEx(&cfg, gemv_mma_kernel<8, false, false, false>, G);
  if (type == 23)
    return isum ? cudaLaunchKernelEx(&cfg, gemv_mma_kernel<23, true, false, false>, G)
                : cudaLaunchKernelEx(&cfg, gemv_mma_kernel<23, false, false, false>, G);
  if (s12)
    return isum ? cudaLaunchKernelEx(&cfg, gemv_mma_kernel<12, true, true, false>, G)
                : cudaLaunchKernelEx(&cfg, gemv_mma_kernel<12, false, true, false>, G);
  if (s14)
    return isum ? cudaLaunchKernelEx(&cfg, gemv_mma_kernel<14, true, true, false>, G)
                : cudaLaunchKernelEx(&cfg, gemv_mma_kernel<14, false, true, false>, G);
  if (type == 12)
    return isum ? cudaLaunchKernelEx(&cfg, gemv_mma_kernel<12, true, false, false>, G)
                : cudaLaunchKernelEx(&cfg, gemv_mma_kernel<12, false, false, false>, G);
  return isum ? cudaLaunchKernelEx(&cfg, gemv_mma_kernel<14, true, false, false>, G)
              : cudaLaunchKernelEx(&cfg, gemv_mma_kernel<14, false, false, false>, G);
}

}  // namespace xq
