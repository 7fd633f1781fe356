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
// The tile is 128 tokens (MMA M, the TMEM lanes) x 128 weight rows (MMA N);
// both operands are read from shared memory.
//
// A operand (tokens): the q8 values as fp16 integers, from the tile image
// the quantizer writes (one bulk copy of 128 tokens x 32 features per item).
// B operand (weights), unpacked by four warps (thread = weight row) into the
// same K-major layout:
//   Q4_K: sc_j * q * 2^-14 in fp16 (sc*q <= 945, exact): the nibble masked in
//         place is the fp16 subnormal q * 2^-24 (16q * 2^-24 for a high
//         nibble), and one fp16 multiply by sc * 2^10 (sc * 2^6) is exact.
//   Q6_K: s * (q - 32) in fp16 when |s| <= 64 (magnitude <= 2048, exact).
//         Rows with a larger scale use two operands, 2*(s>>1)*(q - 32) (even,
//         <= 4096, exact) and (s&1)*(q - 32), multiplied by the same token
//         operand into the same accumulator; the second pair of MMAs is issued
//         only when some row of the tile needs it.
// Exactness: every product is an integer (times 2^-14 for Q4_K) and every
// partial sum of a 32-block accumulator stays below 2^24 in magnitude
// (Q4_K: 945*127*32; Q6_K, worst split: 129*32*127*32 = 16,776,192), so
// each accumulator is exact whatever the order of accumulation.
// Q4_K min term: one bf16 MMA per super-block, the three-piece bf16 split of
// s8 (exact) against mn_j (exact): exact products summed in fp32.
//
// Epilogue (thread = token, 64 weight rows): per 32-block acc[n] += d8 * D[n]
// (one fp32 FMA per output, d8 a per-thread scalar); per super-block
// run[n] += d'[n] * acc[n] (- dmin[n] * Dmin[n]), d' = d*2^14 for Q4_K and d
// for Q6_K, with run kept in TMEM and written to y after the last
// super-block. d' and -dmin reach the epilogue through a shared-memory ring.
//
// Grid: one CTA per (128-row weight tile, K range, 128-token tile). A launch
// inside a layer call may split K into ranges (TileArgs::splits); each CTA
// then writes its range's sums as a partial, and the tile's last CTA adds
// the ranges in order into y.
//
// Warp roles (512 threads): warps 0-3 unpack, warps 4-11 epilogue (warp w
// reads TMEM lane quarter w%4, weight-row half (w-4)/4), warp 12 producer
// (raw weights by TMA or row copies, token items by bulk copy), warps 13-15
// MMA issuers, one per accumulator (warp 13 also owns TMEM). TMEM columns: [0,128) running sums, then three
// 128-column accumulators, so the tensor core runs up to three 32-blocks
// ahead of the epilogue. Every mbarrier wait is bounded (about 2^32 clocks);
// on expiry the kernel records an error code, leaves its loops, waits for
// its own tensor-core work and frees TMEM.
#include <cuda.h>

#include "xq_check.cuh"
#include "xq_common.cuh"
#include "xq_ptx.cuh"

namespace xq {

__device__ unsigned int g_tile_error;  // set by a timed-out wait (never expected)

namespace {

using namespace ptx;

constexpr int kRows = 128;      // weight rows per tile (MMA N)
constexpr int kTokStages = 8;   // token item ring
constexpr int kWStages = 4;     // unpacked weight operand ring
constexpr int kNumD = 3;        // accumulators in TMEM
constexpr int kCoefStages = 4;  // per-super-block row coefficients
constexpr uint32_t kColRun = 0, kColD = 128;
constexpr long long kWaitClocks = 1LL << 32;
constexpr int kQ6Window = 224;  // bytes copied per Q6_K row and super-block
constexpr int kQ6Pitch = 240;   // their pitch in shared memory (conflict-free 16-byte reads)
constexpr int kOpBytes = kRows * 32 * 2;  // one 128-row x 32-slot fp16 operand

// Warp roles: warps 0-3 unpack, then kEpi epilogue warps (kEpi / 4 per TMEM
// lane quarter, each thread taking kCols = 512 / kEpi weight columns of its
// token), the producer, then kMma MMA issuers. The epilogue holds a
// kCols-wide fp32 accumulator per thread; at 64 columns (8 warps) it fills
// the 128-register cap of a 512-thread CTA and bounds the Q4_K tile. Sixteen
// epilogue warps of 32 columns would halve that, but 22 warps leave 80
// registers a thread, and the spills cost more than the parallelism gains
// (measured on the 12288 x 4096 x 512 up projection: 270 us against 241).
template <int TYPE>
struct Roles {
  static constexpr int kEpi = 8;
  static constexpr int kMma = 3;
  static constexpr int kCols = 512 / kEpi;
  static constexpr int kEpi0 = 4, kProd = 4 + kEpi, kMma0 = 5 + kEpi;
  static constexpr int kThreads = 32 * (5 + kEpi + kMma);
};

// Register split between the warpgroups (setmaxnreg): the kernel is built
// for 128 registers a thread (the cap of a 512-thread CTA, checked on the host
// before every launch), the producer and MMA warpgroup (warps 12-15) gives
// back down to kRegsCtl, and the two epilogue warpgroups (warps 4-11) take
// kRegsEpi, for their kCols-wide accumulators. The sum stays inside the CTA's
// launch allocation: (128 + 2 * kRegsEpi + kRegsCtl) * 128 <= 512 * 128.
constexpr int kRegsLaunch = 128, kRegsCtl = 56, kRegsEpi = 152;
static_assert(128 * (kRegsLaunch + 2 * kRegsEpi + kRegsCtl) <= 512 * kRegsLaunch, "register split exceeds the CTA");

template <int TYPE>
struct Fmt;
template <>
struct Fmt<12> {
  static constexpr int kRawRow = kQ4kBytes, kRawStages = 3;
  static constexpr int kItems = 9;             // 8 sub-blocks + the min-term item
  static constexpr int kWBytes = kOpBytes;     // one operand per item
};
template <>
struct Fmt<14> {
  // (kRawPad: room for the 128-byte gaps between the boxes of a grouped view)
  static constexpr int kRawRow = kQ6Pitch, kRawStages = 2, kRawPad = 1024;
  static constexpr int kItems = 8;
  static constexpr int kWBytes = 2 * kOpBytes;  // high and low operands
};
template <>
struct Fmt<8> {
  static constexpr int kRawRow = kQ80Group, kRawStages = 2;  // 8 Q8_0 blocks (272 bytes) per row and stage
  static constexpr int kItems = 8;
  static constexpr int kWBytes = kOpBytes;
};
template <>
struct Fmt<23> {
  static constexpr int kRawRow = 144, kRawStages = 3;  // the 136-byte super-block's 16-byte-aligned window
  static constexpr int kItems = 8;
  static constexpr int kWBytes = 2 * kOpBytes;  // high and low operands
};

// Bytes of one raw-weight stage: the 128 rows, plus the Q6_K gaps.
template <int TYPE>
constexpr int raw_stage_bytes() {
  if constexpr (TYPE == 14) return kRows * Fmt<14>::kRawRow + Fmt<14>::kRawPad;
  else return kRows * Fmt<TYPE>::kRawRow;
}

template <int TYPE>
struct Smem {
  static constexpr int kRaw = Fmt<TYPE>::kRawStages * raw_stage_bytes<TYPE>();
  static constexpr int kTok = kTokStages * kTileItem;
  static constexpr int kW = kWStages * Fmt<TYPE>::kWBytes;
  static constexpr int kCoef = kCoefStages * kRows * 8;
  // Q8_0: the scale of every 32-block of every row, [stage][block][row]
  static constexpr int kDs = TYPE == 8 ? kCoefStages * 8 * kRows * 4 : 0;
  static constexpr int kRawOff = 0, kTokOff = kRaw, kWOff = kTokOff + kTok, kCoefOff = kWOff + kW;
  static constexpr int kDsOff = kCoefOff + kCoef;
  static constexpr int kBarOff = kDsOff + kDs;
};

// barrier indices (raw ring first; its size depends on the type)
template <int TYPE>
struct Bars {
  static constexpr int RS = Fmt<TYPE>::kRawStages;
  static constexpr int kRawFull = 0, kRawEmpty = RS, kTokFull = 2 * RS, kTokEmpty = kTokFull + kTokStages,
                       kWFull = kTokEmpty + kTokStages, kWEmpty = kWFull + kWStages, kDFull = kWEmpty + kWStages,
                       kDEmpty = kDFull + kNumD, kCoefFull = kDEmpty + kNumD, kCoefEmpty = kCoefFull + kCoefStages,
                       kVote = kCoefEmpty + kCoefStages, kDone = kVote + 2, kCount = kDone + kNumD;
};

template <int TYPE>
constexpr int smem_bytes() {
  return Smem<TYPE>::kBarOff + Bars<TYPE>::kCount * 8 + 16 + (kWStages + 8) * 4;
}

struct TileArgs {
  CUtensorMap map;             // Q4_K: {row_bytes/8, N} of u64, box {18, 128}
  const uint8_t* W;
  const uint8_t* img;          // tile image of the Q8 buffer
  float* y;                    // [M][N]
  int32_t* sums;               // test hook: [M][N][K/32] per-32-block integer sums, or null
  unsigned long long w_bytes;  // N * row_bytes
  unsigned long long img_bytes;  // bytes of the tile image (bounds checks of checked builds)
  int q6_tma;                  // Q6_K by tensor map (rows of 16-byte multiples, or the grouped view below)
  int N, K, M, nsb, row_bytes, ttiles;
  uint32_t cb[4];              // IQ4_XS: codebook bytes with their sign bits flipped
  // K-split (layer calls that would leave SMs idle): each tile's super-blocks
  // in `splits` ranges, one CTA each; a CTA stores its sums in partial
  // [splits][M][N] and the last CTA of the tile to arrive (count in
  // arrive[tile], zero before the launch and left zero) adds the ranges in
  // order into y. splits = 1: y directly.
  int splits;
  float* partial;
  unsigned int* arrive;
  // 0: the launch reads nothing the previous grid on the stream writes (a
  // later launch of the same layer): it waits for that grid only before its
  // threads exit, so that its completion still implies the earlier ones.
  int wait_prev;
  // Q6_K grouped view (kernels with GV set): 2^q6_gs consecutive rows per map
  // row (map {row_bytes << gs, N >> gs} of u8), 2^gs boxes of 240 x (128 >> gs)
  // a super-block, box i holding rows i, i + 2^gs, ... of the tile, each at
  // its own 128-byte-aligned place in the stage. Without GV: map {row_bytes,
  // N}, one box of 240 x 128.
  int q6_gs;
};

// Waits of the producer, unpack and epilogue warps suspend between polls;
// the MMA issuer, on the critical path, polls without suspending.
__device__ __forceinline__ bool wait_bar(uint32_t bar, unsigned parity, unsigned code) {
  return mbar_wait_sleep(bar, parity, &g_tile_error, code, kWaitClocks);
}
__device__ __forceinline__ bool wait_bar_spin(uint32_t bar, unsigned parity, unsigned code) {
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

__device__ __forceinline__ uint32_t half2_of(float v) {
  const uint32_t h = __half_as_ushort(__float2half_rn(v));
  return h | (h << 16);
}

// IQ4_XS: the codebook bytes (sign bits flipped) of four 4-bit indices, one
// per byte of x. The indices' low 3 bits, compacted into permute selectors,
// pick from each codebook half; a sign-replicating permute of x << 4 turns
// index bit 3 into a byte mask that chooses between the halves.
__device__ __forceinline__ uint32_t iq4_codes(uint32_t x, const uint32_t (&cb)[4]) {
  const uint32_t sel = prmt(x | (x >> 4), 0u, 0x4420u) & 0x7777u;
  const uint32_t lo = prmt(cb[0], cb[1], sel), hi = prmt(cb[2], cb[3], sel);
  const uint32_t m = prmt(x << 4, 0u, 0xBA98u);
  return (hi & m) | (lo & ~m);
}

// Store one row's 32 k-slots (16 words: word c holds slots 2c, 2c+1) into a
// 128-row K-major operand: slot group q (8 slots, 16 bytes) of row r at
// (r/8)*512 + q*128 + (r%8)*16.
__device__ __forceinline__ void store_row(uint8_t* op, int r, const uint32_t (&v)[16]) {
  uint8_t* p = op + (r >> 3) * 512 + (r & 7) * 16;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(p + q * 128) = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// GV: the Q6_K grouped tensor-map view; SPLIT: a launch with K ranges
// (splits > 1). Each is a kernel of its own so that the plain kernel carries
// none of their code: compiled into it, the two cost the 512-token Qwen3-8B
// FFN tiles 7% (grouped view, down) and 5% (K ranges, up and down).
template <int TYPE, bool SUMS, bool GV, bool SPLIT>
__global__ void __launch_bounds__(Roles<TYPE>::kThreads, 1) tile_mma_kernel(const __grid_constant__ TileArgs A) {
  using R = Roles<TYPE>;
  using F = Fmt<TYPE>;
  using S = Smem<TYPE>;
  using B = Bars<TYPE>;
  constexpr int kRawBytes = kRows * F::kRawRow;     // bytes a stage's copies deliver
  constexpr int kRawStage = GV ? raw_stage_bytes<TYPE>() : kRawBytes;  // stage stride in the ring
  constexpr int kItems = F::kItems;
  constexpr int RS = F::kRawStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* raw_ring = smem + S::kRawOff;
  uint8_t* tok_ring = smem + S::kTokOff;
  uint8_t* w_ring = smem + S::kWOff;
  float2* coef_ring = reinterpret_cast<float2*>(smem + S::kCoefOff);
  float* ds_ring = reinterpret_cast<float*>(smem + S::kDsOff);  // Q8_0 only
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B::kCount);
  int* split_flag = reinterpret_cast<int*>(tmem_slot + 4);  // [kWStages]: tile uses the two-operand form
  int* split_vote = split_flag + kWStages;                  // [2][4 unpack warps]
  const uint32_t bar0 = smem_addr(bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA = (weight tile, K range, token tile), token tile fastest so that the
  // CTAs of one weight tile run side by side
  const int tt = blockIdx.x % A.ttiles, wks = blockIdx.x / A.ttiles;
  const int ks = SPLIT ? wks % A.splits : 0, wt = SPLIT ? wks / A.splits : wks;
  const int kb0 = SPLIT ? A.nsb * ks / A.splits : 0;                 // first super-block of this CTA
  const int nb = SPLIT ? A.nsb * (ks + 1) / A.splits - kb0 : A.nsb;  // super-blocks of this CTA
  const int nitems = nb * kItems;
#define BAR(i) (bar0 + 8u * static_cast<uint32_t>(i))

  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(BAR(B::kRawFull + s), 1);
      mbar_init(BAR(B::kRawEmpty + s), 4);
    }
    for (int s = 0; s < kTokStages; ++s) {
      mbar_init(BAR(B::kTokFull + s), 1);
      mbar_init(BAR(B::kTokEmpty + s), R::kEpi);
    }
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(BAR(B::kWFull + s), 4);
      mbar_init(BAR(B::kWEmpty + s), 1);
    }
    for (int s = 0; s < kNumD; ++s) {
      mbar_init(BAR(B::kDFull + s), 1);
      mbar_init(BAR(B::kDEmpty + s), R::kEpi);
    }
    for (int s = 0; s < kCoefStages; ++s) {
      mbar_init(BAR(B::kCoefFull + s), 4);
      mbar_init(BAR(B::kCoefEmpty + s), R::kEpi);
    }
    for (int s = 0; s < 2; ++s) mbar_init(BAR(B::kVote + s), 4);
    for (int s = 0; s < kNumD; ++s) mbar_init(BAR(B::kDone + s), 1);
    mbar_init_fence();
  }
  if (warp == R::kMma0) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The tile image is written by the previous kernel on the stream (or, for
  // a later launch of a layer, before the first launch's wait).
  if (A.wait_prev) cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();

  // Register split (setmaxnreg): warpgroup 3 (producer and MMA issuers,
  // warps 12-15) gives registers back at one instruction before its roles
  // split; the epilogue warpgroups (warps 4-11) then take them.
  static_assert(R::kProd == 12 && R::kThreads == 512, "the register split assumes warpgroups 0 / 1-2 / 3");
  if (warp >= R::kProd) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == R::kProd) {
      // ------------------------------------------------------- producer
      const uint8_t* rec = A.img + static_cast<size_t>(tt) * A.nsb * kTileRecord;
      const int row0 = wt * kRows;
      const int rows = min(kRows, A.N - row0);
      unsigned tf = 0;  // token items issued
      bool ok = true;
      for (int b = 0; b < nb && ok; ++b) {
        const int gb = kb0 + b;  // super-block in the row
        const int rs = b % RS;
        if (b >= RS && !warp_wait(BAR(B::kRawEmpty + rs), ((b / RS) - 1) & 1, 1)) break;
        const uint32_t dst = smem_addr(raw_ring + rs * kRawStage);
        if (TYPE == 12 || TYPE == 23 || TYPE == 8) {
          if (lane == 0) {
            mbar_expect_tx(BAR(B::kRawFull + rs), kRawBytes);  // rows past N arrive zero-filled
            const int x = TYPE == 12 ? gb * (kQ4kBytes / 8) : (TYPE == 8 ? gb * (kQ80Group / 8) : (kIq4xsBytes * gb) & ~15);
            // x in map elements: 8 bytes for Q4_K and Q8_0, 1 byte for IQ4_XS
            if (XQ_CHECKED((((TYPE == 23) ? x : 8 * x) & 15) == 0 && x >= 0, kChkTileBox))
              tma_load_2d(dst, &A.map, x, row0, BAR(B::kRawFull + rs));
          }
        } else if (A.q6_tma) {
          // Q6_K by tensor map: boxes of 240 bytes from the 16-byte boundary
          // at or below the super-block. Rows of 16-byte multiples: one box
          // of the 128 rows (the same offset in every row). Grouped view
          // (2^gs rows per map row): box i takes rows i, i + 2^gs, ... of the
          // tile, whose windows all start at the same position in their map
          // rows. Rows past N and bytes past a map row arrive zero-filled.
          if (lane == 0) {
            mbar_expect_tx(BAR(B::kRawFull + rs), kRawBytes);
            if constexpr (GV) {
              const int gs = A.q6_gs, rb = kRows >> gs;
              for (int i = 0; i < (1 << gs); ++i) {
                const int x = (i * A.row_bytes + kQ6kBytes * gb) & ~15;
                if (XQ_CHECKED((x & 15) == 0 && x >= 0, kChkTileBox))
                  tma_load_2d(dst + i * (rb * kQ6Pitch + 128), &A.map, x, row0 >> gs, BAR(B::kRawFull + rs));
              }
            } else {
              const int x = (kQ6kBytes * gb) & ~15;
              if (XQ_CHECKED((x & 15) == 0 && x >= 0, kChkTileBox))
                tma_load_2d(dst, &A.map, x, row0, BAR(B::kRawFull + rs));
            }
          }
        } else {
          unsigned mine = 0;
          for (int r = lane; r < rows; r += 32) mine += q6_window(A, row0 + r, gb);
          const unsigned total = __reduce_add_sync(0xffffffffu, mine);
          if (lane == 0) mbar_expect_tx(BAR(B::kRawFull + rs), total);
          __syncwarp();
          for (int r = lane; r < rows; r += 32) {
            const unsigned long long start = static_cast<unsigned long long>(row0 + r) * A.row_bytes + 210ull * gb;
            const unsigned win = q6_window(A, row0 + r, gb);
            if (XQ_CHECKED((start & ~15ull) + win <= A.w_bytes && (win & 15) == 0 &&
                               ((reinterpret_cast<uintptr_t>(A.W) + (start & ~15ull)) & 15) == 0,
                           kChkTileQ6Window))
              bulk_load(dst + r * kQ6Pitch, A.W + (start & ~15ull), win, BAR(B::kRawFull + rs));
          }
        }
        for (int it = 0; it < kItems; ++it, ++tf) {
          const int ts = tf % kTokStages;
          if (tf >= kTokStages && !warp_wait(BAR(B::kTokEmpty + ts), ((tf / kTokStages) - 1) & 1, 2)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const unsigned bytes = it < 8 ? kTileItem : kTileItemOp;
            mbar_expect_tx(BAR(B::kTokFull + ts), bytes);
            const size_t off = (static_cast<size_t>(tt) * A.nsb + gb) * kTileRecord + static_cast<size_t>(it) * kTileItem;
            if (XQ_CHECKED(off + bytes <= A.img_bytes && ((reinterpret_cast<uintptr_t>(A.img) + off) & 15) == 0,
                           kChkTileItem))
              bulk_load(smem_addr(tok_ring + ts * kTileItem), rec + static_cast<size_t>(gb) * kTileRecord + it * kTileItem,
                        bytes, BAR(B::kTokFull + ts));
          }
        }
      }
      // No copy may still be landing when the CTA exits: wait for the last
      // fill of every stage (already complete on the normal path).
      if (lane == 0) {
        for (int b = nb > RS ? nb - RS : 0; b < nb; ++b) wait_bar(BAR(B::kRawFull + b % RS), (b / RS) & 1, 11);
        for (unsigned f = tf > kTokStages ? tf - kTokStages : 0; f < tf; ++f)
          wait_bar(BAR(B::kTokFull + f % kTokStages), (f / kTokStages) & 1, 12);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------- MMA
      // kMma issuing threads: thread k issues items f = k, k + kMma, ... in
      // order, item f into accumulator f % kNumD. Each thread's chain of waits,
      // MMAs and commits is serial; the epilogue frees the accumulators in item
      // order, so one issuer keeps the same order as several.
      const int k = warp - R::kMma0;
      if (lane == 0 && k < nitems) {
        constexpr uint32_t kIdH = idesc_f16(kTileTokens, kRows, false);
        constexpr uint32_t kIdB = idesc_f16(kTileTokens, kRows, true);
        const uint32_t tok0 = smem_addr(tok_ring), w0 = smem_addr(w_ring);
        for (int f = k; f < nitems; f += R::kMma) {
          const int ts = f % kTokStages, ws = f % kWStages, d = f % kNumD, it = f % kItems;
          if (!wait_bar_spin(BAR(B::kTokFull + ts), (f / kTokStages) & 1, 6)) break;
          if (!wait_bar_spin(BAR(B::kWFull + ws), (f / kWStages) & 1, 7)) break;
          if (f >= kNumD && !wait_bar_spin(BAR(B::kDEmpty + d), ((f / kNumD) - 1) & 1, 8)) break;
          tc_fence_after();
          const uint32_t dt = tmem + kColD + 128u * d;
          const uint32_t as = tok0 + ts * kTileItem, bs = w0 + ws * F::kWBytes;
          const uint64_t a0 = smem_desc(as, 128, 512), a1 = smem_desc(as + 256, 128, 512);
          const uint32_t id = (TYPE == 12 && it == 8) ? kIdB : kIdH;
          mma_f16_ss(dt, a0, smem_desc(bs, 128, 512), id, false);
          mma_f16_ss(dt, a1, smem_desc(bs + 256, 128, 512), id, true);
          if ((TYPE == 14 || TYPE == 23) && split_flag[ws]) {
            mma_f16_ss(dt, a0, smem_desc(bs + kOpBytes, 128, 512), id, true);
            mma_f16_ss(dt, a1, smem_desc(bs + kOpBytes + 256, 128, 512), id, true);
          }
          tc_commit(BAR(B::kWEmpty + ws));
          tc_commit(BAR(B::kDFull + d));
        }
      }
      // all issued MMAs complete before TMEM is freed
      if (lane == 0) {
        tc_commit(BAR(B::kDone + k));
        wait_bar_spin(BAR(B::kDone + k), 0, 9);
      }
      __syncwarp();
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- unpack
    const int r = threadIdx.x;  // tile row
    const int n = wt * kRows + r;
    const bool row_ok = n < A.N;
    unsigned wf = 0;  // weight operands filled
    bool ok = true;
    for (int b = 0; b < nb && ok; ++b) {
      const int gb = kb0 + b;  // super-block in the row
      const int rs = b % RS, cs = b % kCoefStages;
      if (!warp_wait(BAR(B::kRawFull + rs), (b / RS) & 1, 3)) break;
      if (b >= kCoefStages && !warp_wait(BAR(B::kCoefEmpty + cs), ((b / kCoefStages) - 1) & 1, 4)) break;
      // this row's window: row r of the stage, or in a Q6_K grouped view row
      // r >> gs of box r mod 2^gs (boxes 128-byte aligned, see the producer)
      const uint8_t* raw = GV ? raw_ring + rs * kRawStage +
                                     (r & ((1 << A.q6_gs) - 1)) * ((kRows >> A.q6_gs) * F::kRawRow + 128) +
                                     (r >> A.q6_gs) * F::kRawRow
                               : raw_ring + rs * kRawStage + r * F::kRawRow;
      if (TYPE == 12) {
        // Scales and mins (public Q4_K packing): j < 4: sc = s[j] & 63,
        // m = s[j+4] & 63; j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
        // m = (s[j+4] >> 4) | (s[j] >> 6) << 4. Rows past N are zero-filled.
        const uint4 h = *reinterpret_cast<const uint4*>(raw);
        const uint32_t sc_lo = h.y & 0x3F3F3F3Fu, mn_lo = h.z & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
        const uint32_t mn_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
        coef_ring[cs * kRows + r] =
            make_float2(half_bits_to_float(h.x) * 16384.0f, -half_bits_to_float(h.x >> 16));
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B::kCoefFull + cs));
#pragma unroll
        for (int it = 0; it < 9; ++it, ++wf) {
          const int ws = wf % kWStages;
          if (wf >= kWStages && !warp_wait(BAR(B::kWEmpty + ws), ((wf / kWStages) - 1) & 1, 5)) {
            ok = false;
            break;
          }
          uint32_t v[16];
          if (it < 8) {
            const int g = it >> 1;
            const bool hi = (it & 1) != 0;
            const uint32_t sc = ((it < 4 ? sc_lo : sc_hi) >> (8 * (it & 3))) & 0xFFu;
            const uint32_t S2 = half2_of(static_cast<float>(sc) * (hi ? 64.0f : 1024.0f));
            const uint4* qp = reinterpret_cast<const uint4*>(raw + 16 + 32 * g);
            const uint4 q0 = qp[0], q1 = qp[1];
            const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            const uint32_t mk = hi ? 0x00F000F0u : 0x000F000Fu;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              // words 2i, 2i+1 = k-slots 4i..4i+3 = weights 4i, 4i+2, 4i+1, 4i+3
              v[2 * i] = hmul2(w[i] & mk, S2);
              v[2 * i + 1] = hmul2((w[i] >> 8) & mk, S2);
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
          store_row(w_ring + ws * F::kWBytes, r, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B::kWFull + ws));
        }
      } else if (TYPE == 8) {
        // Q8_0: 8 blocks of 34 bytes (fp16 d, 32 int8 quants). Each block's
        // d goes to the scale ring for the epilogue (it scales that block's
        // accumulator per row); the super-block coefficient is 1.
        coef_ring[cs * kRows + r] = make_float2(1.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          ds_ring[(cs * 8 + i) * kRows + r] = half_bits_to_float(*reinterpret_cast<const unsigned short*>(raw + 34 * i));
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B::kCoefFull + cs));
#pragma unroll
        for (int it = 0; it < 8; ++it, ++wf) {
          const int ws = wf % kWStages;
          if (wf >= kWStages && !warp_wait(BAR(B::kWEmpty + ws), ((wf / kWStages) - 1) & 1, 5)) {
            ok = false;
            break;
          }
          uint32_t qw[8];
          load_words<8>(raw + 34 * it + 2, qw);  // 2-byte aligned quants
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // weights 4i..4i+3: the int8 q with its sign bit flipped under the
            // exponent of 1024, minus 1152, is the exact fp16 q
            const uint32_t x = qw[i] ^ 0x80808080u;
            v[2 * i] = hsub2(prmt(x, 0x64646464u, 0x4240u), 0x64806480u);      // weights 4i, 4i+2
            v[2 * i + 1] = hsub2(prmt(x, 0x64646464u, 0x4341u), 0x64806480u);  // weights 4i+1, 4i+3
          }
          store_row(w_ring + ws * F::kWBytes, r, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B::kWFull + ws));
        }
      } else if (TYPE == 23) {
        // IQ4_XS: d at 0, scales_h at 2, scales_l[4] at 4, 128 index bytes
        // at 8, starting off = 136b mod 16 (0 or 8) bytes into the window.
        // Sub-block j's weight is codebook[index] * s_j, s_j = ls_j - 32 in
        // [-32, 31]; |value * s| reaches 4096, so as for Q6_K the operand is
        // split into 2*(s>>1)*value (even, exact) and (s&1)*value when some
        // row of the tile has |s| > 16, and the tile then reads both.
        const uint8_t* sb = raw + ((kIq4xsBytes * gb) & 15);
        const uint2 h = *reinterpret_cast<const uint2*>(sb);  // d | scales_h, scales_l (zero past N)
        coef_ring[cs * kRows + r] = make_float2(half_bits_to_float(h.x), 0.0f);
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B::kCoefFull + cs));
        int sj[8];
        bool big = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sj[j] = static_cast<int>(((h.y >> (4 * j)) & 15u) | (((h.x >> (16 + 2 * j)) & 3u) << 4)) - 32;
          big = big || (row_ok && (sj[j] > 16 || sj[j] < -16));
        }
        const bool any = __any_sync(0xffffffffu, big);
        int* vote = split_vote + 4 * (b & 1);
        if (lane == 0) {
          vote[warp] = any ? 1 : 0;
          mbar_arrive(BAR(B::kVote + (b & 1)));
        }
        if (!warp_wait(BAR(B::kVote + (b & 1)), (b >> 1) & 1, 15)) break;
        const bool split = (vote[0] | vote[1] | vote[2] | vote[3]) != 0;
        const uint32_t cb[4] = {A.cb[0], A.cb[1], A.cb[2], A.cb[3]};
#pragma unroll
        for (int it = 0; it < 8; ++it, ++wf) {
          const int ws = wf % kWStages;
          if (wf >= kWStages && !warp_wait(BAR(B::kWEmpty + ws), ((wf / kWStages) - 1) & 1, 5)) {
            ok = false;
            break;
          }
          const int s = sj[it];
          const bool wide = s > 16 || s < -16;
          const uint32_t Shi = half2_of(static_cast<float>(wide ? 2 * (s >> 1) : s));
          const uint32_t Slo = half2_of(static_cast<float>(wide ? (s & 1) : 0));
          // 16 index bytes, 8-byte aligned only (the window offset is 0 or 8)
          const uint2 qa = *reinterpret_cast<const uint2*>(sb + 8 + 16 * it);
          const uint2 qc = *reinterpret_cast<const uint2*>(sb + 16 + 16 * it);
          const uint32_t qw[4] = {qa.x, qa.y, qc.x, qc.y};
          uint32_t v[16], u[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // weights 4i..4i+3: low nibbles of bytes 4i.. for i < 4, high nibbles of bytes 4(i-4).. after
            const uint32_t x = iq4_codes((i < 4 ? qw[i] : (qw[i - 4] >> 4)) & 0x0F0F0F0Fu, cb);
            const uint32_t x0 = hsub2(prmt(x, 0x64646464u, 0x4240u), 0x64806480u);  // weights 4i, 4i+2
            const uint32_t x1 = hsub2(prmt(x, 0x64646464u, 0x4341u), 0x64806480u);  // weights 4i+1, 4i+3
            v[2 * i] = row_ok ? hmul2(x0, Shi) : 0u;
            v[2 * i + 1] = row_ok ? hmul2(x1, Shi) : 0u;
            u[2 * i] = row_ok ? hmul2(x0, Slo) : 0u;
            u[2 * i + 1] = row_ok ? hmul2(x1, Slo) : 0u;
          }
          uint8_t* op = w_ring + ws * F::kWBytes;
          store_row(op, r, v);
          if (split) store_row(op + kOpBytes, r, u);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (warp == 0) split_flag[ws] = split ? 1 : 0;
            mbar_arrive(BAR(B::kWFull + ws));
          }
        }
      } else {
        // Q6_K: ql[128] at 0, qh[64] at 128, scales int8[16] at 192, d at
        // 208. The row's window starts `off` (even, 0..14) bytes before the
        // super-block.
        const unsigned long long start = static_cast<unsigned long long>(n) * A.row_bytes + 210ull * gb;
        const uint8_t* sb = raw + (start & 15);
        const bool cut = (start & ~15ull) + kQ6Window > A.w_bytes;  // scales and d not all in the window
        uint32_t sw[4] = {0u, 0u, 0u, 0u};
        float d = 0.0f;
        if (row_ok) {
          if (!cut) {
            load_words<4>(sb + 192, sw);
            d = half_bits_to_float(*reinterpret_cast<const unsigned short*>(sb + 208));
          } else if (XQ_CHECKED(start + 210 <= A.w_bytes, kChkTileQ6Cut)) {
            const unsigned short* gs = reinterpret_cast<const unsigned short*>(A.W + start + 192);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              sw[k] = static_cast<uint32_t>(__ldg(gs + 2 * k)) | (static_cast<uint32_t>(__ldg(gs + 2 * k + 1)) << 16);
            d = half_bits_to_float(__ldg(gs + 8));
          }
        }
        coef_ring[cs * kRows + r] = make_float2(d, 0.0f);
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B::kCoefFull + cs));
        // |s| > 64 in any row of the tile needs the two-operand form for the
        // whole tile (the low operand is read for all 128 rows): the four
        // unpack warps vote, double-buffered by super-block parity, through
        // an mbarrier per buffer (a warp reuses a buffer only after every
        // warp has passed the next super-block's vote, hence read this one).
        bool big = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) big = big || (__vcmpgtu4(__vabsss4(sw[k]), 0x40404040u) != 0u);
        const bool any = __any_sync(0xffffffffu, big);
        int* vote = split_vote + 4 * (b & 1);
        if (lane == 0) {
          vote[warp] = any ? 1 : 0;
          mbar_arrive(BAR(B::kVote + (b & 1)));
        }
        if (!warp_wait(BAR(B::kVote + (b & 1)), (b >> 1) & 1, 15)) break;
        const bool split = (vote[0] | vote[1] | vote[2] | vote[3]) != 0;
        uint32_t ql[16], qh[8];
#pragma unroll
        for (int it = 0; it < 8; ++it, ++wf) {
          const int hh = it >> 2, rr = it & 3;
          if (rr == 0 && row_ok) {
            load_words<16>(sb + 64 * hh, ql);
            load_words<8>(sb + 128 + 32 * hh, qh);
          }
          const int ws = wf % kWStages;
          if (wf >= kWStages && !warp_wait(BAR(B::kWEmpty + ws), ((wf / kWStages) - 1) & 1, 5)) {
            ok = false;
            break;
          }
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
          uint8_t* op = w_ring + ws * F::kWBytes;
          store_row(op, r, v);
          if (split) store_row(op + kOpBytes, r, u);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (warp == 0) split_flag[ws] = split ? 1 : 0;
            mbar_arrive(BAR(B::kWFull + ws));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B::kRawEmpty + rs));
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    // -------------------------------------------------------- epilogue
    const int quarter = warp & 3, part = (warp - R::kEpi0) >> 2;
    constexpr int kCols = R::kCols;           // weight columns of this thread
    const int r = quarter * 32 + lane;        // token of the tile = TMEM lane
    const int m = tt * kTileTokens + r;
    const int n0 = wt * kRows + kCols * part;  // first weight row of this thread's columns
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    f2 acc[kCols / 2];                        // weight-row pairs (2i, 2i+1) of the current super-block
#pragma unroll
    for (int i = 0; i < kCols / 2; ++i) acc[i] = 0ull;
    bool ok = true;
    int f = 0;
    for (int b = 0; b < nb && ok; ++b) {
      const int gb = kb0 + b;  // super-block in the row
      for (int it = 0; it < kItems; ++it, ++f) {
        const int d = f % kNumD, ts = f % kTokStages;
        // Both phases tested at once, so that their latencies overlap (the
        // token stage's is long complete); a phase not yet complete falls
        // back to the bounded wait. Every lane acquires both.
        const bool d_now = mbar_try_wait(BAR(B::kDFull + d), (f / kNumD) & 1);
        const bool t_now = mbar_try_wait(BAR(B::kTokFull + ts), (f / kTokStages) & 1);
        bool got = d_now || wait_bar(BAR(B::kDFull + d), (f / kNumD) & 1, 10);
        got = got && (t_now || wait_bar(BAR(B::kTokFull + ts), (f / kTokStages) & 1, 13));
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dcol = tl + kColD + 128u * d + static_cast<uint32_t>(kCols * part);
        if (TYPE == 8 && it == 0 && !warp_wait(BAR(B::kCoefFull + b % kCoefStages), (b / kCoefStages) & 1, 14)) {
          ok = false;
          break;
        }
        if (it < 8) {
          const float d8 = reinterpret_cast<const float*>(tok_ring + ts * kTileItem + kTileItemOp)[r];
          const f2 d82 = pk(d8, d8);
          // Q8_0: this block's per-row scales (pairs of this thread's rows)
          const float2* dsp =
              reinterpret_cast<const float2*>(ds_ring + ((b % kCoefStages) * 8 + it) * kRows + kCols * part);
          // two 16-column loads in flight per wait
#pragma unroll
          for (int c = 0; c < kCols / 16; c += 2) {
            uint32_t v[16], w[16];
            tmem_ld16(dcol + 16 * c, v);
            tmem_ld16(dcol + 16 * c + 16, w);
            tmem_wait_ld();
            if (SUMS && m < A.M) {
              // test hook: the 32-block's exact integer (Q4_K sc*isum, from
              // the operand's 2^-14 scale; Q6_K and IQ4_XS scale*isum summed
              // over the block's groups; Q8_0 isum)
              const int nsub = A.K >> 5;
              const float sc = TYPE == 12 ? 16384.0f : 1.0f;
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int n1 = n0 + 16 * c + e, n2 = n1 + 16;
                const size_t ns = static_cast<size_t>(A.M) * A.N * nsub;
                const size_t i1 = (static_cast<size_t>(m) * A.N + n1) * nsub + 8 * gb + it;
                const size_t i2 = (static_cast<size_t>(m) * A.N + n2) * nsub + 8 * gb + it;
                if (n1 < A.N && XQ_IN(i1, ns, kChkTileSums)) A.sums[i1] = static_cast<int32_t>(__uint_as_float(v[e]) * sc);
                if (n2 < A.N && XQ_IN(i2, ns, kChkTileSums)) A.sums[i2] = static_cast<int32_t>(__uint_as_float(w[e]) * sc);
              }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              f2 s0 = d82, s1 = d82;
              if (TYPE == 8) {
                const float2 a = dsp[8 * c + k], e = dsp[8 * c + 8 + k];
                s0 = mul2(d82, pk(a.x, a.y));
                s1 = mul2(d82, pk(e.x, e.y));
              }
              acc[8 * c + k] = fma2(s0, pk(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), acc[8 * c + k]);
              acc[8 * c + 8 + k] =
                  fma2(s1, pk(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1])), acc[8 * c + 8 + k]);
            }
          }
        }
        if (it == kItems - 1) {
          // super-block end: run += d' * acc (- dmin * Dmin)
          const int cs = b % kCoefStages;
          if (TYPE != 8 && !warp_wait(BAR(B::kCoefFull + cs), (b / kCoefStages) & 1, 14)) {  // Q8_0 waited at item 0
            ok = false;
            break;
          }
          const float4* cf = reinterpret_cast<const float4*>(coef_ring + cs * kRows + kCols * part);
          const bool last = b == nb - 1;
#pragma unroll
          for (int c = 0; c < kCols / 16; ++c) {
            uint32_t run[16], dmin[16];
            if (b > 0) tmem_ld16(tl + kColRun + static_cast<uint32_t>(kCols * part) + 16u * c, run);
            if (TYPE == 12) tmem_ld16(dcol + 16 * c, dmin);
            tmem_wait_ld();
            uint32_t out[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float4 q = cf[8 * c + k];  // (d', -dmin) of rows 2k, 2k+1 of this chunk
              f2 rv = b > 0 ? pk(__uint_as_float(run[2 * k]), __uint_as_float(run[2 * k + 1])) : 0ull;
              rv = fma2(pk(q.x, q.z), acc[8 * c + k], rv);
              if (TYPE == 12)
                rv = fma2(pk(q.y, q.w), pk(__uint_as_float(dmin[2 * k]), __uint_as_float(dmin[2 * k + 1])), rv);
              out[2 * k] = static_cast<uint32_t>(rv);
              out[2 * k + 1] = static_cast<uint32_t>(rv >> 32);
              acc[8 * c + k] = 0ull;
            }
            if (last) {
              if (m < A.M) {
                const int nc = n0 + 16 * c;
                // y, or this K range's partial sums (same [M][N] layout)
                float* yr = (SPLIT ? A.partial + static_cast<size_t>(ks) * A.M * A.N : A.y) +
                            static_cast<size_t>(m) * A.N;
                if (!XQ_IN(static_cast<size_t>(m) * A.N + (nc < A.N ? nc : 0), static_cast<size_t>(A.M) * A.N,
                           kChkTileY)) {
                } else if ((A.N & 3) == 0 && nc + 16 <= A.N) {
#pragma unroll
                  for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4*>(yr + nc + 4 * k) =
                        make_uint4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
                } else {
#pragma unroll
                  for (int k = 0; k < 16; ++k)
                    if (nc + k < A.N) yr[nc + k] = __uint_as_float(out[k]);
                }
              }
            } else {
              tmem_st16(tl + kColRun + static_cast<uint32_t>(kCols * part) + 16u * c, out);
            }
          }
          if (!last) tmem_wait_st();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B::kCoefEmpty + cs));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(BAR(B::kDEmpty + d));
          mbar_arrive(BAR(B::kTokEmpty + ts));
        }
      }
    }
    if constexpr (SPLIT) {
      // K-split: once every epilogue thread has stored its partial sums
      // (named barrier 1, the epilogue warps only), one thread counts the CTA
      // in with an acquire-release increment (its release publishes the
      // stores the barrier ordered before it; its acquire, in the last CTA,
      // covers every other CTA's). The last CTA of the tile adds the K
      // ranges in order into y and leaves the count at zero.
      asm volatile("bar.sync 1, %0;" ::"n"(32 * R::kEpi) : "memory");
      const int tile = wt * A.ttiles + tt;
      if (threadIdx.x == 32 * R::kEpi0) {
        unsigned old = 0;
        if (XQ_IN(tile, (A.N + kRows - 1) / kRows * A.ttiles, kChkTileSplit))
          asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(A.arrive + tile) : "memory");
        const bool last_cta = old == static_cast<unsigned>(A.splits - 1);
        if (last_cta) A.arrive[tile] = 0u;
        tmem_slot[1] = last_cta ? 1u : 0u;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * R::kEpi) : "memory");
      if (tmem_slot[1] != 0u && m < A.M) {
        const size_t plane = static_cast<size_t>(A.M) * A.N;
        const size_t row = static_cast<size_t>(m) * A.N;
        for (int c = 0; c < kCols; c += 4) {
          const int nc = n0 + c;
          if (nc >= A.N) break;
          if ((A.N & 3) == 0) {
            float4 v = __ldcg(reinterpret_cast<const float4*>(A.partial + row + nc));
            for (int k = 1; k < A.splits; ++k) {
              const float4 w = __ldcg(reinterpret_cast<const float4*>(A.partial + k * plane + row + nc));
              v.x += w.x;
              v.y += w.y;
              v.z += w.z;
              v.w += w.w;
            }
            if (XQ_IN(row + nc + 3, plane, kChkTileY)) *reinterpret_cast<float4*>(A.y + row + nc) = v;
          } else {
            for (int e = 0; e < 4 && nc + e < A.N; ++e) {
              float v = __ldcg(A.partial + row + nc + e);
              for (int k = 1; k < A.splits; ++k) v += __ldcg(A.partial + k * plane + row + nc + e);
              if (XQ_IN(row + nc + e, plane, kChkTileY)) A.y[row + nc + e] = v;
            }
          }
        }
      }
    }
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == R::kMma0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // A launch that did not wait for the previous grid on entry waits before
  // its threads exit (the next kernel's dependency wait relies on that).
  if (!A.wait_prev) cudaGridDependencySynchronize();
}

template <int TYPE, bool SUMS, bool GV, bool SPLIT>
cudaError_t launch_tile(const TileArgs& A, int grid, cudaStream_t s, bool pdl) {
  // The register split inside the kernel is sized for a launch allocation
  // of exactly kRegsLaunch registers a thread; anything else is refused
  // before launch (a split larger than the allocation would never complete).
  static int regs_ok = -1;
  if (regs_ok < 0) {
    cudaFuncAttributes fa;
    regs_ok = (cudaFuncGetAttributes(&fa, tile_mma_kernel<TYPE, SUMS, GV, SPLIT>) == cudaSuccess &&
               fa.numRegs == kRegsLaunch)
                  ? 1
                  : 0;
  }
  if (!regs_ok) return cudaErrorInvalidConfiguration;
  static bool smem_set = false;
  if (!smem_set) {
    const cudaError_t e = cudaFuncSetAttribute(tile_mma_kernel<TYPE, SUMS, GV, SPLIT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<TYPE>());
    if (e != cudaSuccess) return e;
    smem_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Roles<TYPE>::kThreads);
  cfg.dynamicSmemBytes = smem_bytes<TYPE>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tile_mma_kernel<TYPE, SUMS, GV, SPLIT>, A);
}

}  // namespace

cudaError_t take_tile_check(unsigned int* code) { return take_check_word(code); }

cudaError_t take_tile_error(unsigned int* code) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tile_error, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tile_error, &z, sizeof(z));
  *code = v;
  return e;
}

// The instantiation for a launch: K ranges (never with the sums hook, which
// the caller refuses), else with or without the hook.
template <int TYPE, bool GV = false>
cudaError_t launch_tile_for(const TileArgs& A, int grid, cudaStream_t s, bool pdl) {
  if (A.splits > 1) return launch_tile<TYPE, false, GV, true>(A, grid, s, pdl);
  return A.sums ? launch_tile<TYPE, true, GV, false>(A, grid, s, pdl)
                : launch_tile<TYPE, false, GV, false>(A, grid, s, pdl);
}

cudaError_t launch_tile_mma(int type, const uint8_t* W, const uint8_t* xq, int M, int N, int K, float* y,
                            cudaStream_t s, bool pdl, const uint32_t* codebook, int32_t* sums, const TileSplit* split,
                            bool wait_prev) {
  if (M <= kGemvMaxTokens || N <= 0 || K <= 0 || (K & 255) != 0 ||
      (type != 12 && type != 14 && type != 23 && type != 8))
    return cudaErrorInvalidValue;
  const int splits = split ? split->splits : 1;
  if (splits < 1 || splits > (K >> 8) || (splits > 1 && (!split->partial || !split->arrive || sums)) ||
      (!wait_prev && !pdl))
    return cudaErrorInvalidValue;
  if (type == 23 && (!codebook || (K & 511) != 0)) return cudaErrorInvalidValue;
  const Q8Layout L = q8_layout(M, K);
  TileArgs A = {};
  A.W = W;
  A.img = xq + L.tile;
  A.y = y;
  A.sums = sums;
  A.N = N;
  A.K = K;
  A.M = M;
  A.nsb = K >> 8;
  A.row_bytes = A.nsb * (type == 12 ? kQ4kBytes : (type == 23 ? kIq4xsBytes : (type == 8 ? kQ80Group : kQ6kBytes)));
  for (int i = 0; i < 4; ++i) A.cb[i] = codebook ? (codebook[i] ^ 0x80808080u) : 0u;
  A.w_bytes = static_cast<unsigned long long>(N) * A.row_bytes;
  A.img_bytes = L.total - L.tile;
  A.ttiles = L.ttiles;
  A.splits = splits;
  A.partial = splits > 1 ? split->partial : nullptr;
  A.arrive = splits > 1 ? split->arrive : nullptr;
  A.wait_prev = wait_prev ? 1 : 0;
  const int grid = ((N + kRows - 1) / kRows) * L.ttiles * splits;
  if (type == 12) {
    if (!encode_tma_2d(&A.map, CU_TENSOR_MAP_DATA_TYPE_UINT64, W, A.row_bytes / 8, static_cast<unsigned long long>(N),
                       A.row_bytes, kQ4kBytes / 8, kRows))
      return cudaErrorInvalidValue;
    return launch_tile_for<12>(A, grid, s, pdl);
  }
  if (type == 23) {
    if (!encode_tma_2d(&A.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, A.row_bytes, static_cast<unsigned long long>(N),
                       A.row_bytes, Fmt<23>::kRawRow, kRows))
      return cudaErrorInvalidValue;
    return launch_tile_for<23>(A, grid, s, pdl);
  }
  if (type == 8) {
    if (!encode_tma_2d(&A.map, CU_TENSOR_MAP_DATA_TYPE_UINT64, W, A.row_bytes / 8, static_cast<unsigned long long>(N),
                       A.row_bytes, kQ80Group / 8, kRows))
      return cudaErrorInvalidValue;
    return launch_tile_for<8>(A, grid, s, pdl);
  }
  // Q6_K by tensor map: one box per super-block when rows are 16-byte
  // multiples (K a multiple of 2048); else 2^gs rows per map row (the fewest
  // whose bytes are a multiple of 16) and 2^gs boxes, when N is a multiple of
  // 2^gs; else a bulk copy per row
  A.q6_gs = q6k_row_shift(K);
  A.q6_tma = (N % (1 << A.q6_gs)) == 0 ? 1 : 0;
  if (A.q6_tma) {
    const unsigned long long vrow = static_cast<unsigned long long>(A.row_bytes) << A.q6_gs;
    if (!encode_tma_2d(&A.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, vrow, static_cast<unsigned long long>(N >> A.q6_gs),
                       vrow, kQ6Pitch, kRows >> A.q6_gs))
      return cudaErrorInvalidValue;
  }
  return A.q6_tma && A.q6_gs ? launch_tile_for<14, true>(A, grid, s, pdl) : launch_tile_for<14>(A, grid, s, pdl);
}

}  // namespace xq
