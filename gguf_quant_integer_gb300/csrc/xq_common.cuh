// Device helpers and internal launcher declarations for the xq library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace xq {

constexpr int kQ4kBytes = 144;  // GGUF Q4_K super-block: 256 weights
constexpr int kQ6kBytes = 210;  // GGUF Q6_K super-block: 256 weights
constexpr int kIq4xsBytes = 136;  // GGUF IQ4_XS super-block: 256 weights
constexpr int kQ80Bytes = 34;   // GGUF Q8_0 block: 32 weights
constexpr int kQ80Group = 8 * kQ80Bytes;  // 8 Q8_0 blocks: 256 weights, 16-byte multiple
constexpr int kNumSMs = 152;    // GB300: 2 dies x 76 SMs

// ---------------------------------------------------------------- loads

// Streaming 16-byte load for weight bytes: read once per launch, so it skips
// L1 allocation (the read-only path still goes through L2).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned ld_stream4(const void* p) {
  unsigned v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Activation loads: small, re-read by every row of the CTA, so they stay
// cacheable in L1.
__device__ __forceinline__ uint4 ld_act16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ----------------------------------------------------------- integer ops

// Four-way byte dot product: unsigned bytes of a times signed bytes of b,
// accumulated into c.
__device__ __forceinline__ int dp4a_us(unsigned a, unsigned b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// Four signed bytes of a times four signed bytes of b, plus c.
__device__ __forceinline__ int dp4a_ss(unsigned a, unsigned b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Byte permute of the 8-byte pair (hi:lo).
__device__ __forceinline__ unsigned prmt(unsigned lo, unsigned hi, unsigned sel) {
  unsigned d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(lo), "r"(hi), "r"(sel));
  return d;
}

__device__ __forceinline__ float half_bits_to_float(unsigned bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// ------------------------------------------------------- Q8 buffer layout
//
// The Q8 activation buffer of M tokens x K features holds, in order:
//   qs   int8 [M][K]                      at 0
//   d8   fp32 [M][K/32]                   at M*K
//   s8   fp32 [M][K/32]                   at M*K + 4*M*K/32
// followed, at F = round_up(1.25*M*K, 256), by the tensor-core operand image
// of the matmul path that serves this M.
//
// M <= kGemvMaxTokens (warp-level MMA GEMV, 8-token chunks):
//   frag fp16 [C][K/32][32][8]            at F
//   fsc  fp32 [C][K/32][4][4]             at F + C*16*K
// with C = ceil(M/8) chunks of 8 tokens, laid out as the B operand of an
// m16n8k16 MMA with 8 token columns: for chunk c, 32-block j, lane = 4n + t
// (token n, quad t), slot s: frag = (half) qs[8c+n][32j + 8t + perm[s]],
// perm = 0,2,1,3,4,6,5,7; fsc[c][j][t] = (d8[8c+2t][j], d8[8c+2t+1][j],
// s8[8c+2t][j], s8[8c+2t+1][j]). Tokens past M in the last chunk are zero.
//
// M > kGemvMaxTokens (tensor-memory tile kernel), T = ceil(M/128) token tiles:
//   tile [T][K/256] records of kTileRecord bytes at F. Record (t, b) holds,
//   for the 128 tokens 128t .. 128t+127 and super-block b:
//     8 items, one per 32-block j = 8b + i (kTileItem bytes each):
//       op  fp16 [128 tokens][32 k-slots] in the K-major no-swizzle layout of
//           the MMA B operand: token r, slot s at byte
//           (r/8)*512 + (s/8)*128 + (r%8)*16 + (s%8)*2, holding
//           qs[128t+r][32j + 4(s/4) + pr[s%4]], pr = 0,2,1,3;
//       d8  fp32 [128] at byte kTileItemOp: d8[128t+r][j];
//     then one bf16 operand (kTileItemOp bytes, same layout) whose slot
//     3i + p (i < 8, p < 3) holds piece p of s8[128t+r][8b+i] split into
//     three bf16 numbers by truncation (their sum is s8 exactly); slots
//     24..31 are zero.
//   Tokens past M are zero.
constexpr int kTileTokens = 128;
constexpr int kTileItemOp = 8192;                         // 128 tokens x 32 slots x 2 B
constexpr int kTileItem = kTileItemOp + 4 * kTileTokens;  // 8704
constexpr int kTileRecord = 8 * kTileItem + kTileItemOp;  // 77824

struct Q8Layout {
  size_t qs, d8, s8, frag, fsc, tile, total;
  int chunks;  // 8-token chunks of the GEMV image (M <= kGemvMaxTokens), else 0
  int ttiles;  // 128-token tiles of the tile image (M > kGemvMaxTokens), else 0
};

// Up to this many tokens a matmul runs the GEMV over 8-token chunks (up to 8
// chunks in one launch, which then read each weight tile from HBM about once),
// above it the tile kernel. Measured on GB300 (weights past L2): a Q4_K
// 12288 x 4096 matmul takes 18 us at M = 9..16, 34 us at 32 and 65 us at 64
// as GEMV chunks against 80 us on the tile kernel at any M <= 128; a Q6_K
// 4096 x 12288 one 45 / 82 / 118 us against 323 us.
constexpr int kGemvMaxTokens = 64;

// gemv_image: the GEMV layout (8-token chunks) for any M; the batch-invariant
// entry points use it.
__host__ __device__ inline Q8Layout q8_layout(int M, int K, bool gemv_image = false) {
  Q8Layout L;
  const size_t mk = static_cast<size_t>(M) * K;
  L.qs = 0;
  L.d8 = mk;
  L.s8 = mk + 4 * (mk / 32);
  const size_t F = (mk + 8 * (mk / 32) + 255) & ~static_cast<size_t>(255);
  if (M <= kGemvMaxTokens || gemv_image) {
    L.chunks = (M + 7) / 8;
    L.ttiles = 0;
    L.frag = F;
    L.fsc = L.frag + static_cast<size_t>(L.chunks) * 16 * K;
    L.tile = L.total = L.fsc + static_cast<size_t>(L.chunks) * 2 * K;
  } else {
    L.chunks = 0;
    L.ttiles = (M + kTileTokens - 1) / kTileTokens;
    L.frag = L.fsc = L.tile = F;
    L.total = F + static_cast<size_t>(L.ttiles) * (K / 256) * kTileRecord;
  }
  return L;
}

constexpr int kMaxProj = 8;  // projections per grouped launch

// --------------------------------------------------------- launchers

struct GemvArgs {
  const uint8_t* W;     // weight super-blocks
  const int8_t* qs;     // Q8 quants [M][K]
  const float* d8;      // Q8 scales [M][K/32]
  const float* s8;      // Q8 scale*sum [M][K/32]
  int M, N, K;          // M in 1..8 for one launch
  float* y;             // [M][N], row stride ldy (floats)
  long long ldy;
  int32_t* isum;        // optional sub-block sums (test hook)
};

struct QuantJob {
  const float* x;   // fp32 [M][K]
  uint8_t* xq;      // Q8 buffer (layout above)
  int M, K;
  bool gemv_image = false;  // 8-token GEMV image for any M (batch-invariant layout)
  // With up: the quantized value is h = silu(x) * up (x the gate output, up
  // the up output, both fp32 [M][K]), optionally written to h_out.
  const float* up = nullptr;
  float* h_out = nullptr;
};

// One launch quantizing up to kMaxProj activations; also zeroes the
// zero_count words at zero_words when given (the next grouped matmul's task
// counter and arrival counts).
cudaError_t launch_quantize_q8(const QuantJob* jobs, int n, cudaStream_t s, bool pdl,
                               unsigned int* zero_words = nullptr, int zero_count = 0);

struct MmaProj {
  int nch;             // K-chunks when split workspaces are given (0 or 1: none)
  bool gemv_image = false;  // the Q8 buffer uses the GEMV image for M_total > 8 too
  const uint8_t* W;    // super-blocks [N][K/256]
  const uint8_t* xq;   // Q8 buffer of this projection's input (M_total tokens)
  float* y;            // [M_total][N]; this launch writes tokens 8*chunk .. 8*chunk+7
  int32_t* isum;       // optional [M_total][N][K/32], only with M_total <= 8
  int N, K, M_total, chunk;
  uint32_t codebook[4] = {0u, 0u, 0u, 0u};  // IQ4_XS: the 16 int8 values, little-endian bytes
  // Elements of y [M_total][N] the launch may write (bounds checks of checked
  // builds; -1: all of them). The check probe declares fewer.
  long long y_limit = -1;
};

// K-chunks a projection's rows are split into when a split workspace is
// available, for a chunk length of `chunk` super-blocks: rows longer than
// 24 super-blocks (or than `chunk`, once the chunk length drops below 16)
// go in ceil(nsb / chunk) chunks.
__host__ __device__ inline int gemv_split_chunks(int K, int M_total, int chunk = 16) {
  const int nsb = K >> 8;
  if (M_total > 8) return 1;
  const int limit = chunk >= 16 ? 24 : chunk;
  return nsb > limit ? (nsb + chunk - 1) / chunk : 1;
}
// Grouped GEMV geometry: consumer warps per CTA (16 weight rows each, so a
// task covers kGemvRows rows), and resident CTAs per SM.
constexpr int kGemvWarps = 4;
constexpr int kGemvRows = 16 * kGemvWarps;
constexpr int kGemvCtasPerSM = 3;
constexpr int kGemvSlots = kGemvCtasPerSM * kNumSMs;
// Workspace of a split projection: partial sums [nch][8][rows padded to
// kGemvRows] and one arrival count per 16-row group (both rounded to 256 bytes).
__host__ __device__ inline int gemv_row_blocks(int N) { return (N + kGemvRows - 1) / kGemvRows; }
__host__ __device__ inline size_t gemv_split_partial_bytes(int N, int nch) {
  return ((static_cast<size_t>(nch) * 8 * gemv_row_blocks(N) * kGemvRows * 4) + 255) & ~static_cast<size_t>(255);
}
__host__ __device__ inline size_t gemv_split_arrive_bytes(int N) {
  return ((static_cast<size_t>(gemv_row_blocks(N)) * kGemvWarps * 4) + 255) & ~static_cast<size_t>(255);
}

// Whether the tensor-core GEMV takes this weight: every Q4_K and Q8_0
// shape; IQ4_XS when K is a multiple of 512; Q6_K when its rows are 16-byte
// multiples (K/256 a multiple of 8), or else when N is a multiple of 16 * 2^gs
// with 2^gs (2, 4 or 8) the number of consecutive rows whose bytes are a
// multiple of 16 (q6k_row_shift): the tensor map then takes 2^gs rows per
// map row.
int q6k_row_shift(int K);
bool gemv_mma_supports(int type, int N, int K);

// One launch for up to kMaxProj projection chunks of <= 8 tokens, all of one
// type (12 = Q4_K, 14 = Q6_K, the latter only where gemv_mma_supports). With
// a counter (zeroed by the previous kernel on the stream) tasks are fetched
// dynamically, most expensive first; without one they are strided. With a
// split workspace (arrival counts, zeroed before the first use, at arrive_ws;
// partial sums at partial_ws; sizes from the gemv_split_* helpers in item
// order) long rows are split into K-chunks across CTAs.
// stall_test (a test hook): the producer issues no stage and every wait is
// limited to about 10^5 clocks, so the consumers' first waits run out,
// record their error code and return; y is left unwritten.
//
// ffn (optional): the launch runs the gate and up projections of a SwiGLU
// FFN (items ffn->gate and ffn->up, N = F, M <= 8, one chunk) and writes
// h = silu(y_gate) * y_up as Q8 (layout q8_layout(M, F, false)) at ffn->hq,
// counting each completed 32-block in ffn->arrive (F/32 words) and each
// completed super-block's blocks in ffn->ready (F/256 words), both zero
// before the launch. ffn->down >= 0: that item is the down projection (K =
// F, reading ffn->hq); its tasks are placed after every other task, and its
// activation copies wait for the ready counts. ffn->down < 0: down runs in a
// later launch, which must wait for this grid's completion.
struct FfnFuse {
  int gate, up, down;
  unsigned int* arrive;
  unsigned int* ready;
  uint8_t* hq;
  float* h_out;  // optional fp32 copy of h [M][F]
  int F, M;
  bool stall = false;  // test hook: h never counted ready; every wait limited to about 10^5 clocks
};
cudaError_t launch_gemv_mma(int type, const MmaProj* projs, int n, cudaStream_t s, bool pdl,
                            unsigned int* counter = nullptr, uint8_t* arrive_ws = nullptr,
                            uint8_t* partial_ws = nullptr, bool wait_prev = true, bool stall_test = false,
                            const FfnFuse* ffn = nullptr);

// Read and clear the error word each waiting kernel sets when a bounded wait
// runs out (0: none since the last read). Synchronous device reads/writes.
cudaError_t take_gemv_error(unsigned int* code);
cudaError_t take_tile_error(unsigned int* code);
// Checked builds: read and clear the bounds-check word of each kernel file
// (the site number of the first failed check; always 0 in normal builds).
cudaError_t take_gemv_check(unsigned int* code);
cudaError_t take_tile_check(unsigned int* code);
cudaError_t take_quant_check(unsigned int* code);
cudaError_t take_q6k_check(unsigned int* code);

// 2D tensor map (no interleave, no swizzle, zero fill): dims {dim0, dim1}
// elements of type dt, rows stride1 bytes apart, boxes box0 x box1. False
// if the driver entry point is missing or rejects the arguments.
bool encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, unsigned long long dim0,
                   unsigned long long dim1, unsigned long long stride1, unsigned box0, unsigned box1);

// y = x W^T for M > 64 tokens on the tensor-memory tile kernel; type is 12
// (Q4_K), 14 (Q6_K), 8 (Q8_0) or 23 (IQ4_XS, with its codebook as 4
// little-endian words; K a multiple of 512), xq the Q8 buffer of M tokens
// (tile image present).
// sums (test hook, or null): [M][N][K/32] int32, each 32-block's exact
// integer as the kernel accumulates it (Q4_K sc_j * isum_j; Q6_K
// s_2p * isum_2p + s_2p+1 * isum_2p+1; Q8_0 isum_j; IQ4_XS (ls_j - 32) * isum_j).
// split (layer calls, or null): the K-split of tile_split_count, with
// partial [splits][M][N] fp32 and one arrival count per 128 x 128 tile,
// zeroed before the launch (the kernel leaves them zero). wait_prev false:
// a later launch of a layer, which reads nothing the previous grid writes
// and waits for it only before exiting (needs pdl).
struct TileSplit {
  int splits;
  float* partial;
  unsigned int* arrive;
};
// K ranges per tile for a layer's tile launch: 1 when the launch's 128 x 128
// tiles already cover the SMs, else as many as fill them (one CTA per SM),
// at most 8 and at most one per two super-blocks.
inline int tile_split_count(int N, int K, int M) {
  const long long tiles = static_cast<long long>((N + 127) / 128) * ((M + kTileTokens - 1) / kTileTokens);
  if (tiles <= 0 || tiles >= kNumSMs) return 1;
  long long s = kNumSMs / tiles;
  const int nsb = K >> 8;
  if (s > nsb / 2) s = nsb / 2;
  if (s > 8) s = 8;
  return s < 1 ? 1 : static_cast<int>(s);
}
inline size_t tile_split_arrive_bytes(int N, int M) {
  return ((static_cast<size_t>((N + 127) / 128) * ((M + kTileTokens - 1) / kTileTokens) * 4) + 255) &
         ~static_cast<size_t>(255);
}
inline size_t tile_split_partial_bytes(int N, int M, int splits) {
  return ((static_cast<size_t>(splits) * M * N * 4) + 255) & ~static_cast<size_t>(255);
}
cudaError_t launch_tile_mma(int type, const uint8_t* W, const uint8_t* xq, int M, int N, int K, float* y,
                            cudaStream_t s, bool pdl, const uint32_t* codebook = nullptr, int32_t* sums = nullptr,
                            const TileSplit* split = nullptr, bool wait_prev = true);
cudaError_t launch_gemv_q6k(const GemvArgs& a, cudaStream_t s);

}  // namespace xq
