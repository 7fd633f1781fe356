// Q4_K x Q8 -> fp32 for M <= 8 tokens on the fifth-generation tensor cores
// (tcgen05.mma kind::f16, operands holding exact integers, fp32 accumulators
// in tensor memory).
//
// What it computes (xLLM v0.7 long-context article, section 一; the M
// template of section B2): for output row n and token m,
//   y[m][n] = sum over super-blocks b, sub-blocks j of
//             d*sc_j*d8[m][8b+j]*isum_j  -  dmin*m_j*s8[m][8b+j]
//   isum_j  = sum_{i<32} q[32j+i] * q8[m][256b+32j+i]        (exact)
//
// Rows on the tensor-memory lanes. A CTA takes 128 weight rows (the MMA M
// side) and one super-block per pipeline step. Thread r of the four unpack
// warps masks its own row's 128 quant bytes into fp16 operands and stores
// them in tensor memory as the A operand: a low nibble masked in place,
// q & 0x000F000F, is the fp16 subnormal q * 2^-24, a high nibble masked in
// place is 16q * 2^-24 (one AND per two weights, no conversion). The B
// operand is the activation image the quantizer writes: the 8 tokens' int8
// values as fp16 integers, one 256-byte slice of 8 tokens x 16 k-slots per
// MMA (K-major core matrices).
//
// One accumulator per super-block. The MMA N side is 16 columns: sub-blocks
// 2p and 2p+1 (the low and high nibbles of the same 32 quant bytes) share
// columns 16p .. 16p+15, sub-block 2p's tokens in the first 8 and 2p+1's in
// the last 8. Their B tiles are block-diagonal: the MMAs of sub-block 2p read
// the token slice as n-rows 0..7 and a zero block as rows 8..15, those of 2p+1
// the other way round (the two halves are separate core-matrix groups of the
// shared-memory descriptor, so the zeros are two fixed 256-byte blocks of
// each stage, never copied). Sixteen MMAs (K = 16 each) leave all 64 exact
// sub-block sums of the super-block, 8 sub-blocks x 8 tokens, in 64 columns:
// every product and partial sum is an integer multiple of 2^-24 below 2^-2,
// so the fp32 accumulation is exact and D * 2^24 (low) or D * 2^20 (high) is
// the integer sum, bit for bit.
//
// Epilogue (thread = row): the thread decodes its own row's d, dmin and the
// eight 6-bit (sc, m) pairs, reads its 64 sums from tensor memory, and adds
//   acc[t] += (alpha_j * d8_j[t]) * D_j[t] + beta_j * s8_j[t]
// with alpha_j = d * sc_j * 2^24 (2^20 for a high nibble), beta_j = -dmin *
// m_j, packed over token pairs. Accumulation is bounded by construction: a
// super-block's 16 fp32 roundings go into a fresh accumulator, which is then
// added once to a running sum; every 32 super-blocks the running sum is
// added to a total.
//
// Pipeline. One CTA per SM (320 threads): warps 0-3 unpack, 4-7 epilogue,
// 8 the producer (one lane: 2D TMA of 128 rows x 144 bytes, and bulk copies
// of the super-block's activation slices and scale quads, into an 8-stage
// ring), 9 the MMA issuer (one lane; it also owns tensor memory). Tensor
// memory holds three A buffers (128 columns each) and two accumulators (64
// columns each), so unpacking, MMAs and the epilogue of consecutive
// super-blocks overlap. Tasks are 128 rows x a range of super-blocks, taken
// dynamically from a counter (most expensive first) or strided; long rows
// can be split over K, each epilogue warp publishing its 32 rows' partial
// sums and an arrival count, the last arrival adding the chunks in chunk
// order. Every mbarrier wait is bounded (about 2^32 clocks); on expiry the
// kernel records an error code, leaves its loops, waits for its own copies
// and tensor-core work, and frees tensor memory.
#include <cuda.h>

#include "xq_common.cuh"
#include "xq_ptx.cuh"

namespace xq {

__device__ unsigned int g_gemv_tc_error;  // set by a timed-out wait (never expected)

namespace {

using namespace ptx;

constexpr int kRows = kTcRows;               // weight rows per task = TMEM lanes
constexpr int kStages = 8;
constexpr int kRaw = kRows * kQ4kBytes;      // 18432: 128 rows x one super-block
constexpr int kZlo = kRaw;                   // 256 zero bytes
constexpr int kSlices = kZlo + 256;          // 16 activation slices of 256 bytes
constexpr int kZhi = kSlices + kTcImgSb;     // 256 zero bytes
constexpr int kFsc = kZhi + 256;             // 512 bytes of scale quads
constexpr int kStageBytes = kFsc + 512;      // 23552
constexpr unsigned kStageTx = kRaw + kTcImgSb + 512;
constexpr int kABufs = 3, kDBufs = 2;
constexpr uint32_t kColA = 0, kColD = 128 * kABufs;  // A: 3 x 128 columns, D: 2 x 64
constexpr int kThreads = 320;
constexpr int kWarpEpi = 4, kWarpProd = 8, kWarpMma = 9;
constexpr long long kWaitClocks = 1LL << 32;
constexpr long long kStallWaitClocks = 100000;  // the test hook's short limit (about 50 us)

// mbarriers
constexpr int kFull = 0, kEmpty = kStages, kAFull = 2 * kStages, kAEmpty = kAFull + kABufs, kDFull = kAEmpty + kABufs,
              kDEmpty = kDFull + kDBufs, kDone = kDEmpty + kDBufs, kNumBars = kDone + 1;
constexpr int kMetaOff = kStages * kStageBytes;
constexpr int kBarOff = kMetaOff + kStages * 16;
constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16;
static_assert(kSmemBytes + 1024 <= 227 * 1024, "shared memory of one CTA");
static_assert(kColD + 64 * kDBufs <= 512, "tensor memory columns");
static_assert(kStageBytes % 128 == 0, "stage alignment");

struct TProj {
  CUtensorMap map;       // {row_bytes/8 u64, N}, box {18, 128}
  const uint8_t* tcb;    // activation slices [K/256][4096]
  const uint8_t* fsc;    // scale quads [K/32][64 B]
  float* y;
  int32_t* isum;
  float* partial;        // split: [nch][8][128 * row blocks]
  unsigned int* arrive;  // split: one count per 32-row group
  int N, K, M, task0, nch;
};

struct TGroup {
  TProj p[kMaxProj];
  unsigned int* counter;  // dynamic task counter (zeroed before launch) or null
  long long wait_limit;   // clocks a wait may take before it records an error and gives up
  int n, total;
  int wait_prev;  // 0: nothing this launch reads is written by the previous grid on the stream
  int stall;      // test hook: the producer issues no stage, so every first wait runs out
};

struct TaskPos {
  int p, rb, b0, b1, c;
};

__device__ __forceinline__ TaskPos task_pos(const TGroup& G, int task) {
  int p = 0;
#pragma unroll 1
  while (p + 1 < G.n && task >= G.p[p + 1].task0) ++p;
  const TProj& P = G.p[p];
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

__device__ __forceinline__ int next_task(const TGroup& G, int cur) {
  if (G.counter) return static_cast<int>(gridDim.x + atomicAdd(G.counter, 1u));
  return cur + static_cast<int>(gridDim.x);
}

__device__ __forceinline__ bool wait_sleep(uint32_t bar, unsigned parity, unsigned code, long long limit) {
  return mbar_wait_sleep(bar, parity, &g_gemv_tc_error, code, limit);
}
__device__ __forceinline__ bool wait_spin(uint32_t bar, unsigned parity, unsigned code, long long limit) {
  return mbar_wait(bar, parity, &g_gemv_tc_error, code, limit);
}
// Every lane waits (suspending between polls, so that waiting warps leave
// the issue slots to the working ones); the warp goes on only if all of them
// saw the phase.
__device__ __forceinline__ bool warp_wait(uint32_t bar, unsigned parity, unsigned code, long long limit) {
  const bool ok = wait_sleep(bar, parity, code, limit);
  return __all_sync(0xffffffffu, ok);
}

// Byte k of a packed word as 2^23 + byte, an exact fp32 (0x4B0000xx).
__device__ __forceinline__ float byte_plus_2p23(unsigned w, int k) {
  return __uint_as_float(prmt(w, 0x4B000000u, 0x7540u | static_cast<unsigned>(k)));
}

__device__ __forceinline__ void act_load(uint32_t st, const TProj& P, int b, uint32_t bar) {
  bulk_load(st + kSlices, P.tcb + static_cast<size_t>(b) * kTcImgSb, kTcImgSb, bar);
  bulk_load(st + kFsc, P.fsc + static_cast<size_t>(b) * 512, 512, bar);
}

// The last epilogue warp of a split 32-row group: y = the group's K-chunk
// partials added in chunk order.
__device__ __forceinline__ void reduce_chunks(const TProj& P, int rb, int r) {
  const int rows_pad = tc_row_blocks(P.N) * kRows;
  const int n = rb * kRows + r;
  if (n >= P.N) return;
  for (int t = 0; t < P.M; ++t) {
    float v = 0.0f;
    for (int c = 0; c < P.nch; ++c) v += __ldcg(P.partial + (static_cast<size_t>(c) * 8 + t) * rows_pad + n);
    P.y[static_cast<size_t>(t) * P.N + n] = v;
  }
}

template <bool ISUM>
__global__ void __launch_bounds__(kThreads, 1) gemv_tc_kernel(const __grid_constant__ TGroup G) {
  extern __shared__ __align__(1024) uint8_t smem[];
  int4* meta = reinterpret_cast<int4*>(smem + kMetaOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  const uint32_t smem0 = smem_addr(smem);
  const uint32_t bar0 = smem_addr(bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#define BAR(i) (bar0 + 8u * static_cast<uint32_t>(i))
#define STAGE_S(s) (smem0 + static_cast<uint32_t>(s) * kStageBytes)
#define STAGE(s) (smem + static_cast<size_t>(s) * kStageBytes)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(BAR(kFull + s), 1);
      mbar_init(BAR(kEmpty + s), 9);  // 4 unpack warps, 4 epilogue warps, the MMA commit
    }
    for (int s = 0; s < kABufs; ++s) {
      mbar_init(BAR(kAFull + s), 4);
      mbar_init(BAR(kAEmpty + s), 1);
    }
    for (int s = 0; s < kDBufs; ++s) {
      mbar_init(BAR(kDFull + s), 1);
      mbar_init(BAR(kDEmpty + s), 4);
    }
    mbar_init(BAR(kDone), 1);
    mbar_init_fence();
  }
  // The zero blocks of every stage: written once, never copied over.
  for (int i = threadIdx.x; i < kStages * 32; i += kThreads) {
    const int s = i >> 5, k = i & 31;
    *reinterpret_cast<uint4*>(STAGE(s) + (k < 16 ? kZlo : kZhi) + 16 * (k & 15)) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  if (warp == kWarpMma) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long lim = G.wait_limit;

  if (warp == kWarpProd) {
    // ------------------------------------------------------- producer
    // Each CTA's first task is its own index; later ones come from the
    // counter (or a stride). Weights do not depend on the previous grid on
    // the stream, so the first task's first stages are requested before the
    // dependency wait; the activation image, the counter and the arrival
    // counts may be written by that grid.
    if (lane == 0 && G.stall) {
      if (G.wait_prev) cudaGridDependencySynchronize();
      cudaTriggerProgrammaticLaunchCompletion();
    } else if (lane == 0) {
      int task = static_cast<int>(blockIdx.x);
      int g = 0;          // stages issued
      int bresume = -1;   // first super-block of the first task not yet requested
      if (task < G.total) {
        const TaskPos tp = task_pos(G, task);
        const TProj& P = G.p[tp.p];
        int b = tp.b0;
        for (; b < tp.b1 && g < kStages; ++b, ++g) {
          meta[g] = make_int4(task, b, (b == tp.b1 - 1) ? 1 : 0, 0);
          mbar_expect_tx(BAR(kFull + g), kStageTx);
          tma_load_2d(STAGE_S(g), &P.map, b * (kQ4kBytes / 8), tp.rb * kRows, BAR(kFull + g));
        }
        bresume = b;
      }
      if (G.wait_prev) cudaGridDependencySynchronize();
      cudaTriggerProgrammaticLaunchCompletion();
      if (task < G.total) {
        const TaskPos tp = task_pos(G, task);
        for (int k = 0; k < g; ++k) act_load(STAGE_S(k), G.p[tp.p], tp.b0 + k, BAR(kFull + k));
      }
      bool ok = true;
      for (;;) {
        const bool valid = task < G.total;
        if (!valid) {
          const int slot = g % kStages;
          if (g >= kStages && !wait_sleep(BAR(kEmpty + slot), ((g / kStages) - 1) & 1, 1, lim)) break;
          meta[slot] = make_int4(-1, 0, 0, 0);
          mbar_arrive(BAR(kFull + slot));
          ++g;  // the final wait below covers this stage (its arrival moved the slot's phase)
          break;
        }
        const TaskPos tp = task_pos(G, task);
        const TProj& P = G.p[tp.p];
        const int nxt = next_task(G, task);
        const int bfirst = bresume >= 0 ? bresume : tp.b0;
        bresume = -1;
        for (int b = bfirst; b < tp.b1; ++b, ++g) {
          const int slot = g % kStages;
          if (g >= kStages && !wait_sleep(BAR(kEmpty + slot), ((g / kStages) - 1) & 1, 1, lim)) {
            ok = false;
            break;
          }
          meta[slot] = make_int4(task, b, (b == tp.b1 - 1) ? 1 : 0, 0);
          mbar_expect_tx(BAR(kFull + slot), kStageTx);
          tma_load_2d(STAGE_S(slot), &P.map, b * (kQ4kBytes / 8), tp.rb * kRows, BAR(kFull + slot));
          act_load(STAGE_S(slot), P, b, BAR(kFull + slot));
        }
        if (!ok) break;
        task = nxt;
      }
      // No copy may still be landing when the CTA exits (already complete on
      // the normal path).
      for (int k = g > kStages ? g - kStages : 0; k < g; ++k) wait_sleep(BAR(kFull + k % kStages), (k / kStages) & 1, 2, lim);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------------------------------- unpack
    const int r = threadIdx.x;  // row of the task = TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int g = 0;; ++g) {
      const int slot = g % kStages;
      if (!warp_wait(BAR(kFull + slot), (g / kStages) & 1, 3, lim)) break;
      if (meta[slot].x < 0) break;
      const int ab = g % kABufs;
      if (g >= kABufs && !warp_wait(BAR(kAEmpty + ab), ((g / kABufs) - 1) & 1, 4, lim)) break;
      tc_fence_after();
      const uint4* q = reinterpret_cast<const uint4*>(STAGE(slot) + r * kQ4kBytes + 16);
      const uint32_t acol = tl + kColA + 128u * ab;
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        // quant bytes 32*g4 .. +31: low nibbles are sub-block 2*g4, high
        // nibbles sub-block 2*g4+1; word i holds weights 4i..4i+3, and the
        // two fp16 of a column are weights (4i, 4i+2) or (4i+1, 4i+3)
        const uint4 a = q[2 * g4], c = q[2 * g4 + 1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t s = w[i] >> 8;
          lo[2 * i] = w[i] & 0x000F000Fu;
          lo[2 * i + 1] = s & 0x000F000Fu;
          hi[2 * i] = w[i] & 0x00F000F0u;
          hi[2 * i + 1] = s & 0x00F000F0u;
        }
        tmem_st16(acol + 32u * g4, lo);
        tmem_st16(acol + 32u * g4 + 16u, hi);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(BAR(kAFull + ab));
        mbar_arrive(BAR(kEmpty + slot));
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t kId = idesc_f16(kRows, 16, false);
      for (int g = 0;; ++g) {
        const int slot = g % kStages;
        if (!wait_spin(BAR(kFull + slot), (g / kStages) & 1, 5, lim)) break;
        if (meta[slot].x < 0) break;
        const int ab = g % kABufs, db = g % kDBufs;
        if (!wait_spin(BAR(kAFull + ab), (g / kABufs) & 1, 6, lim)) break;
        if (g >= kDBufs && !wait_spin(BAR(kDEmpty + db), ((g / kDBufs) - 1) & 1, 7, lim)) break;
        tc_fence_after();
        const uint32_t st = STAGE_S(slot);
        const uint32_t zlo = st + kZlo, zhi = st + kZhi;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          // MMA i: sub-block j = i/2, k-slots 16*(i%2) .. +15
          const uint32_t sl = st + kSlices + 256u * i;
          const int j = i >> 1;
          const uint64_t bd = (j & 1) ? smem_desc(zlo, 128, sl - zlo) : smem_desc(sl, 128, zhi - sl);
          mma_f16_ts(tmem + kColD + 64u * db + 16u * (j >> 1), tmem + kColA + 128u * ab + 8u * i, bd, kId,
                     (i & 3) != 0);
        }
        tc_commit(BAR(kAEmpty + ab));
        tc_commit(BAR(kDFull + db));
        tc_commit(BAR(kEmpty + slot));
      }
      // every issued MMA completes before tensor memory is freed
      tc_commit(BAR(kDone));
      wait_spin(BAR(kDone), 0, 8, lim);
    }
    __syncwarp();
  } else if (warp >= kWarpEpi && warp < kWarpProd) {
    // -------------------------------------------------------- epilogue
    const int quarter = warp - kWarpEpi;
    const int r = quarter * 32 + lane;  // row of the task = TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    f2 run[4] = {0ull, 0ull, 0ull, 0ull}, tot[4] = {0ull, 0ull, 0ull, 0ull};
    int nrun = 0;
    int cur_task = -1;
    TaskPos tp = {0, 0, 0, 0, 0};
    // Split tasks: each warp owns one arrival count per 32-row group; lane 0
    // increments it once the warp's partials are stored, and the warp
    // examines the count it got one stage later.
    int pend_p = -1, pend_rb = 0;
    unsigned pend_old = 0;
    auto resolve = [&]() {
      if (pend_p < 0) return;
      const TProj& Q = G.p[pend_p];
      const unsigned old = __shfl_sync(0xffffffffu, pend_old, 0);
      if (old == static_cast<unsigned>(Q.nch - 1)) {  // every chunk has arrived
        __threadfence();
        __syncwarp();
        if (lane == 0) Q.arrive[pend_rb * 4 + quarter] = 0u;  // ready for the next launch
        reduce_chunks(Q, pend_rb, r);
      }
      pend_p = -1;
    };
    for (int g = 0;; ++g) {
      const int slot = g % kStages;
      if (!warp_wait(BAR(kFull + slot), (g / kStages) & 1, 9, lim)) break;
      const int4 m = meta[slot];
      if (m.x < 0) {
        resolve();
        break;
      }
      if (m.x != cur_task) {
        cur_task = m.x;
        tp = task_pos(G, m.x);
      }
      const TProj& P = G.p[tp.p];
      // This row's scales and mins (public Q4_K packing): j < 4: sc = s[j] & 63,
      // m = s[j+4] & 63; j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
      // m = (s[j+4] >> 4) | (s[j] >> 6) << 4. alpha = d*sc*2^24 (2^20 for
      // the high nibbles of odd j) and beta = -dmin*m, each (2^23 + byte)*x -
      // 2^23*x: one rounding of an exact product.
      f2 al[8], be[8];
      {
        const uint4 hd = *reinterpret_cast<const uint4*>(STAGE(slot) + r * kQ4kBytes);
        const uint32_t scw[2] = {hd.y & 0x3F3F3F3Fu, (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u)};
        const uint32_t mnw[2] = {hd.z & 0x3F3F3F3Fu, ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u)};
        const float d = half_bits_to_float(hd.x);
        const float dl = d * 16777216.0f, dh = d * 1048576.0f;
        const float dm = -half_bits_to_float(hd.x >> 16);
        const float cl = -8388608.0f * dl, ch = -8388608.0f * dh, cm = -8388608.0f * dm;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float a = (j & 1) ? fmaf(byte_plus_2p23(scw[j >> 2], j & 3), dh, ch)
                                  : fmaf(byte_plus_2p23(scw[j >> 2], j & 3), dl, cl);
          const float bm = fmaf(byte_plus_2p23(mnw[j >> 2], j & 3), dm, cm);
          al[j] = pk(a, a);
          be[j] = pk(bm, bm);
        }
      }
      const int db = g % kDBufs;
      if (!warp_wait(BAR(kDFull + db), (g / kDBufs) & 1, 10, lim)) break;
      tc_fence_after();
      uint32_t v[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld16(tl + kColD + 64u * db + 16u * c, v[c]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(kDEmpty + db));
      const int n = tp.rb * kRows + r;
      if (ISUM && n < P.N) {
        const int nsub = P.K >> 5;
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int t = 0; t < 8; ++t)
            if (t < P.M)
              P.isum[(static_cast<size_t>(t) * P.N + n) * nsub + 8 * m.y + j] = static_cast<int32_t>(
                  __uint_as_float(v[j >> 1][8 * (j & 1) + t]) * ((j & 1) ? 1048576.0f : 16777216.0f));
      }
      // this super-block's terms, token pairs (2q, 2q+1)
      const ulonglong2* fs = reinterpret_cast<const ulonglong2*>(STAGE(slot) + kFsc);  // [j][q]: (d8 pair, s8 pair)
      const int nq = (P.M + 1) >> 1;
      f2 acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < nq) {
            const ulonglong2 f = fs[4 * j + q];
            const uint32_t* vj = v[j >> 1] + 8 * (j & 1) + 2 * q;
            acc[q] = fma2(mul2(al[j], f.x), pk(__uint_as_float(vj[0]), __uint_as_float(vj[1])),
                          fma2(be[j], f.y, acc[q]));
          }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(kEmpty + slot));
#pragma unroll
      for (int q = 0; q < 4; ++q) run[q] = add2(run[q], acc[q]);
      if (++nrun == 32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          tot[q] = add2(tot[q], run[q]);
          run[q] = 0ull;
        }
        nrun = 0;
      }
      resolve();  // a split hand-off from an earlier task, one stage later
      if (m.z) {
        f2 out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          out[q] = add2(tot[q], run[q]);
          run[q] = 0ull;
          tot[q] = 0ull;
        }
        nrun = 0;
        if (P.nch == 1) {
          if (n < P.N) {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (t < P.M) P.y[static_cast<size_t>(t) * P.N + n] = (t & 1) ? hi32(out[t >> 1]) : lo32(out[t >> 1]);
          }
        } else {
          // K-chunk partial of a split task: lane 0's fence, after the warp
          // barrier, publishes the warp's stores ahead of its relaxed
          // increment; the last warp fences again before its reads.
          const int rows_pad = tc_row_blocks(P.N) * kRows;
          float* part = P.partial + static_cast<size_t>(tp.c) * 8 * rows_pad + n;
#pragma unroll
          for (int t = 0; t < 8; ++t)
            if (t < P.M) part[static_cast<size_t>(t) * rows_pad] = (t & 1) ? hi32(out[t >> 1]) : lo32(out[t >> 1]);
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            pend_old = atomicAdd(P.arrive + tp.rb * 4 + quarter, 1u);
          }
          pend_p = tp.p;
          pend_rb = tp.rb;
        }
      }
    }
  }
#undef STAGE
#undef STAGE_S
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // A launch that did not wait for the previous grid on entry waits before
  // its threads exit, so that its completion still implies the completion of
  // every earlier kernel on the stream.
  if (!G.wait_prev) cudaGridDependencySynchronize();
}

template <bool ISUM>
cudaError_t set_smem() {
  static bool done = false;
  if (done) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel<ISUM>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess) done = true;
  return e;
}

}  // namespace

cudaError_t take_gemv_tc_error(unsigned int* code) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_tc_error, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_gemv_tc_error, &z, sizeof(z));
  *code = v;
  return e;
}

cudaError_t launch_gemv_tc(const MmaProj* projs, int n, cudaStream_t s, bool pdl, unsigned int* counter,
                           uint8_t* arrive_ws, uint8_t* partial_ws, bool wait_prev, bool stall_test) {
  if (n <= 0 || n > kMaxProj) return cudaErrorInvalidValue;
  const bool split = arrive_ws != nullptr && partial_ws != nullptr;
  int nch[kMaxProj], cost[kMaxProj];
  for (int k = 0; k < n; ++k) {
    nch[k] = (split && projs[k].nch > 1) ? projs[k].nch : 1;
    cost[k] = ((projs[k].K >> 8) + nch[k] - 1) / nch[k];
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
  size_t arrive_off[kMaxProj], partial_off[kMaxProj];
  {
    size_t a = 0, p = 0;
    for (int k = 0; k < n; ++k)
      if (nch[k] > 1) {
        arrive_off[k] = a;
        a += tc_split_arrive_bytes(projs[k].N);
        partial_off[k] = p;
        p += tc_split_partial_bytes(projs[k].N, nch[k]);
      }
  }
  TGroup G;
  G.n = n;
  G.counter = counter;
  G.wait_prev = (wait_prev || !pdl) ? 1 : 0;
  G.stall = stall_test ? 1 : 0;
  G.wait_limit = stall_test ? kStallWaitClocks : kWaitClocks;
  int total = 0;
  bool isum = false;
  for (int k = 0; k < n; ++k) {
    const int src = order[k];
    const MmaProj& q = projs[src];
    if (q.M_total < 1 || q.M_total > 8 || q.chunk != 0 || q.gemv_image || (q.K & 255) != 0 || q.N <= 0)
      return cudaErrorInvalidValue;
    const Q8Layout L = q8_layout(q.M_total, q.K);
    if (L.tcb == 0) return cudaErrorInvalidValue;
    TProj& P = G.p[k];
    const unsigned long long nsb = static_cast<unsigned long long>(q.K / 256);
    if (!encode_tma_2d(&P.map, CU_TENSOR_MAP_DATA_TYPE_UINT64, q.W, nsb * kQ4kBytes / 8,
                       static_cast<unsigned long long>(q.N), nsb * kQ4kBytes, kQ4kBytes / 8, kTcRows))
      return cudaErrorInvalidValue;
    P.tcb = q.xq + L.tcb;
    P.fsc = q.xq + L.fsc;
    P.y = q.y;
    P.isum = q.isum;
    P.N = q.N;
    P.K = q.K;
    P.M = q.M_total;
    P.nch = nch[src];
    P.partial = nullptr;
    P.arrive = nullptr;
    if (P.nch > 1) {
      P.partial = reinterpret_cast<float*>(partial_ws + partial_off[src]);
      P.arrive = reinterpret_cast<unsigned int*>(arrive_ws + arrive_off[src]);
    }
    P.task0 = total;
    total += tc_row_blocks(q.N) * P.nch;
    isum = isum || (q.isum != nullptr);
  }
  G.total = total;
  if (total == 0) return cudaSuccess;
  const cudaError_t e = isum ? set_smem<true>() : set_smem<false>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(total < kNumSMs ? total : kNumSMs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return isum ? cudaLaunchKernelEx(&cfg, gemv_tc_kernel<true>, G) : cudaLaunchKernelEx(&cfg, gemv_tc_kernel<false>, G);
}

}  // namespace xq
