// The C ABI of include/xq.h: argument checks, buffer layout and dispatch.
// Every check runs before anything is enqueued; nothing here allocates.
#include <cstdint>

#include "xq.h"
#include "xq_common.cuh"

namespace {

using xq::GemvArgs;

constexpr int kMaxGemvM = 8;  // tokens per GEMV launch (the kernels' M template)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int block_bytes(int type) {
  // bytes per 256 weights
  return type == XQ_TYPE_Q4_K    ? xq::kQ4kBytes
         : type == XQ_TYPE_Q6_K  ? xq::kQ6kBytes
         : type == XQ_TYPE_Q8_0  ? xq::kQ80Group
         : type == XQ_TYPE_IQ4_XS ? xq::kIq4xsBytes
                                 : 0;
}

xq_status check_shape(int M, int N, int K) {
  if (M < 0 || N < 0 || K <= 0 || (K % 256) != 0) return XQ_ERR_SHAPE;
  return XQ_OK;
}

// Enqueue y = x W^T. M > 64 (the buffer holds the tile image): the
// tensor-memory tile kernel. M <= 64: the warp-level MMA GEMV in 8-token
// chunks (up to kMaxProj chunks per launch, which share each weight tile
// through L2) for Q4_K, Q8_0, IQ4_XS and Q6_K rows that are 16-byte
// multiples; the dp4a GEMV for the other Q6_K shapes. invariant: every M in
// 8-token GEMV chunks from the GEMV-image layout, never split over K, so
// that each token's row of y is computed by the same operations whatever M.
//
// A single matmul has no workspace for split-K partial sums, so its GEMV
// launch has one task per 64 rows over the whole of K. Q6_K weights in the
// grouped view (rows that are not 16-byte multiples) take the tensor-core
// GEMV only when that gives at least 128 tasks; narrower ones run faster on
// the dp4a kernel, whose warps take a few rows each (measured on GB300, M = 8,
// weights past L2: 1536 x 8960 24.7 us on dp4a against 35.1 us; 8960 x 1536
// 16.5 us against 9.9 us). The choice depends on the shape only, never on M.
bool single_gemv(int type, int N, int K) {
  if (!xq::gemv_mma_supports(type, N, K)) return false;
  return type != XQ_TYPE_Q6_K || xq::q6k_row_shift(K) == 0 || xq::gemv_row_blocks(N) >= 128;
}

xq_status run_matmul(int type, const void* W, const void* xq, int M, int N, int K, float* y,
                     int32_t* isum, cudaStream_t s, bool invariant = false, const uint32_t* codebook = nullptr) {
  const xq::Q8Layout L = xq::q8_layout(M, K, invariant);
  const uint8_t* base = static_cast<const uint8_t*>(xq);
  if (L.ttiles > 0) {
    const cudaError_t e = xq::launch_tile_mma(type, static_cast<const uint8_t*>(W), base, M, N, K, y, s, true, codebook);
    return e == cudaSuccess ? XQ_OK : XQ_ERR_CUDA;
  }
  if (single_gemv(type, N, K)) {
    xq::MmaProj items[xq::kMaxProj];
    int n = 0;
    for (int c = 0; c < L.chunks; ++c) {
      xq::MmaProj& q = items[n++];
      q.W = static_cast<const uint8_t*>(W);
      q.xq = base;
      q.y = y;
      q.isum = isum;
      q.N = N;
      q.K = K;
      q.M_total = M;
      q.chunk = c;
      q.nch = 1;
      q.gemv_image = invariant;
      if (codebook)
        for (int i = 0; i < 4; ++i) q.codebook[i] = codebook[i];
      if (n == xq::kMaxProj || c + 1 == L.chunks) {
        if (xq::launch_gemv_mma(type, items, n, s, true) != cudaSuccess) return XQ_ERR_CUDA;
        n = 0;
      }
    }
    return XQ_OK;
  }
  for (int m0 = 0; m0 < M; m0 += kMaxGemvM) {
    const int mc = (M - m0) < kMaxGemvM ? (M - m0) : kMaxGemvM;
    GemvArgs a;
    a.W = static_cast<const uint8_t*>(W);
    a.qs = reinterpret_cast<const int8_t*>(base + L.qs) + static_cast<size_t>(m0) * K;
    a.d8 = reinterpret_cast<const float*>(base + L.d8) + static_cast<size_t>(m0) * (K / 32);
    a.s8 = reinterpret_cast<const float*>(base + L.s8) + static_cast<size_t>(m0) * (K / 32);
    a.M = mc;
    a.N = N;
    a.K = K;
    a.y = y + static_cast<size_t>(m0) * N;
    a.ldy = N;
    a.isum = isum;
    if (xq::launch_gemv_q6k(a, s) != cudaSuccess) return XQ_ERR_CUDA;
  }
  return XQ_OK;
}

xq_status matmul_entry(int type, const void* W, const void* xq, int M, int N, int K, float* y,
                       int32_t* isum, xq_stream stream) {
  xq_status st = check_shape(M, N, K);
  if (st != XQ_OK) return st;
  if (M == 0 || N == 0) return XQ_OK;
  if (!W || !xq || !y) return XQ_ERR_ARG;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(y)) return XQ_ERR_ALIGN;
  if (isum) {
    if (M > kMaxGemvM) return XQ_ERR_UNSUPPORTED;
    if (!aligned16(isum)) return XQ_ERR_ALIGN;
  }
  return run_matmul(type, W, xq, M, N, K, y, isum, reinterpret_cast<cudaStream_t>(stream));
}

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// The layer workspace ends with the grouped matmuls' scheduling state (for
// M <= 8): one 256-byte task counter per weight type, then the arrival
// counts of split projections of both types, then their partial sums (sizes
// from the same helpers the launcher uses). The counters and arrival counts
// form one range that the quantize launch zeroes.
constexpr size_t kCounterBytes = 256;
constexpr int kTypes = 4;  // 0: Q4_K, 1: Q6_K, 2: Q8_0, 3: IQ4_XS
constexpr int kTypeIds[kTypes] = {XQ_TYPE_Q4_K, XQ_TYPE_Q6_K, XQ_TYPE_Q8_0, XQ_TYPE_IQ4_XS};

int type_index(int type) {
  return type == XQ_TYPE_Q4_K ? 0 : (type == XQ_TYPE_Q6_K ? 1 : (type == XQ_TYPE_Q8_0 ? 2 : 3));
}

// The 16 int8 codebook values of an IQ4_XS weight as 4 little-endian words.
void pack_codebook(const int8_t* codebook, uint32_t (&cb)[4]) {
  for (int i = 0; i < 4; ++i)
    cb[i] = static_cast<uint32_t>(static_cast<uint8_t>(codebook[4 * i])) |
            (static_cast<uint32_t>(static_cast<uint8_t>(codebook[4 * i + 1])) << 8) |
            (static_cast<uint32_t>(static_cast<uint8_t>(codebook[4 * i + 2])) << 16) |
            (static_cast<uint32_t>(static_cast<uint8_t>(codebook[4 * i + 3])) << 24);
}

// A projection's MmaProj fields that do not depend on the chunk.
void set_codebook(const xq_proj& q, xq::MmaProj& it) {
  if (q.type == XQ_TYPE_IQ4_XS && q.codebook) {
    uint32_t cb[4];
    pack_codebook(q.codebook, cb);
    for (int i = 0; i < 4; ++i) it.codebook[i] = cb[i];
  }
}

struct Sched {
  bool dynamic[kTypes];  // the type's grouped GEMV fits one launch: counter and K-split
  size_t arrive[kTypes], partial[kTypes];
  int nch[64];           // K-chunks per projection (1: not split)
  int tsplit[64];        // M > 64: K ranges per tile of each projection's tile launch (1: not split)
};

// Projections that go to the grouped tensor-core GEMV at M <= 8.
bool in_group(const xq_proj& q, int M) {
  return q.N > 0 && M <= kMaxGemvM && xq::gemv_mma_supports(q.type, q.N, q.K);
}


// K-chunking of a grouped launch: chunks of ~16 super-blocks for long rows;
// while the group has fewer 64-row tasks than resident CTAs, halve the chunk
// length once, to 8 (4-super-block chunks cost more in hand-offs and pipeline
// refills than the idle CTAs they put to work).
void choose_chunks(const xq_proj* proj, int n_proj, int M, int type, int* nch) {
  for (int chunk = 16;; chunk /= 2) {
    long long tasks = 0;
    for (int p = 0; p < n_proj; ++p) {
      if (!in_group(proj[p], M) || proj[p].type != type) continue;
      nch[p] = xq::gemv_split_chunks(proj[p].K, M, chunk);
      tasks += static_cast<long long>(xq::gemv_row_blocks(proj[p].N)) * nch[p];
    }
    if (tasks >= xq::kGemvSlots || chunk <= 8) return;
  }
}

Sched sched_layout(const xq_proj* proj, int n_proj, int M) {
  Sched sc = {};
  if (M > kMaxGemvM) {
    // 8 < M <= 64: every (projection, 8-token chunk) pair of a long row is
    // split over K with its own arrival counts and partial sums (the pairs
    // are spread over several launches that may run at once); no counters.
    for (int p = 0; p < n_proj && p < 64; ++p) sc.nch[p] = sc.tsplit[p] = 1;
    if (M > xq::kGemvMaxTokens) {
      // tile launches: K-split where a projection's tiles leave SMs idle,
      // with one arrival count per tile and the partial sums of every range
      for (int p = 0; p < n_proj && p < 64; ++p) {
        const xq_proj& q = proj[p];
        if (q.N <= 0) continue;
        sc.tsplit[p] = xq::tile_split_count(q.N, q.K, M);
        if (sc.tsplit[p] <= 1) continue;
        const int g = type_index(q.type);
        sc.arrive[g] += xq::tile_split_arrive_bytes(q.N, M);
        sc.partial[g] += xq::tile_split_partial_bytes(q.N, M, sc.tsplit[p]);
      }
      return sc;
    }
    const int chunks = (M + 7) / 8;
    for (int p = 0; p < n_proj && p < 64; ++p) {
      const xq_proj& q = proj[p];
      if (q.N <= 0 || !xq::gemv_mma_supports(q.type, q.N, q.K)) continue;
      sc.nch[p] = xq::gemv_split_chunks(q.K, kMaxGemvM, 16);
      if (sc.nch[p] <= 1) continue;
      const int g = type_index(q.type);
      sc.arrive[g] += chunks * xq::gemv_split_arrive_bytes(q.N);
      sc.partial[g] += chunks * xq::gemv_split_partial_bytes(q.N, sc.nch[p]);
    }
    return sc;
  }
  int items[kTypes] = {0, 0, 0, 0};
  for (int p = 0; p < n_proj && p < 64; ++p) {
    sc.nch[p] = 1;
    if (in_group(proj[p], M)) ++items[type_index(proj[p].type)];
  }
  for (int g = 0; g < kTypes; ++g) {
    sc.dynamic[g] = items[g] > 0 && items[g] <= xq::kMaxProj;
    if (sc.dynamic[g]) choose_chunks(proj, n_proj, M, kTypeIds[g], sc.nch);
  }
  for (int p = 0; p < n_proj; ++p) {
    if (!in_group(proj[p], M) || !sc.dynamic[type_index(proj[p].type)] || sc.nch[p] <= 1) continue;
    const int g = type_index(proj[p].type);
    sc.arrive[g] += xq::gemv_split_arrive_bytes(proj[p].N);
    sc.partial[g] += xq::gemv_split_partial_bytes(proj[p].N, sc.nch[p]);
  }
  return sc;
}

size_t sched_bytes(const Sched& sc) {
  size_t b = kTypes * kCounterBytes;
  for (int g = 0; g < kTypes; ++g) b += sc.arrive[g] + sc.partial[g];
  return b;
}

// Validate a layer description and find each input's K (0 = unused).
xq_status layer_inputs(const xq_proj* proj, int n_proj, int n_inputs, int M, int* in_k) {
  if (!proj || n_proj < 0 || n_proj > 64 || n_inputs < 0 || n_inputs > 64) return XQ_ERR_ARG;
  if (M < 0) return XQ_ERR_SHAPE;
  for (int i = 0; i < n_inputs; ++i) in_k[i] = 0;
  for (int p = 0; p < n_proj; ++p) {
    const xq_proj& q = proj[p];
    if (block_bytes(q.type) == 0) return XQ_ERR_ARG;
    if (q.type == XQ_TYPE_IQ4_XS && !q.codebook) return XQ_ERR_ARG;
    if (q.input < 0 || q.input >= n_inputs) return XQ_ERR_ARG;
    const xq_status st = check_shape(M, q.N, q.K);
    if (st != XQ_OK) return st;
    if (q.type == XQ_TYPE_IQ4_XS && (q.K % 512) != 0) return XQ_ERR_SHAPE;
    if (in_k[q.input] == 0) in_k[q.input] = q.K;
    if (in_k[q.input] != q.K) return XQ_ERR_SHAPE;
  }
  return XQ_OK;
}

// The matmul launches of a layer whose inputs are already quantized: q8[p]
// is projection p's Q8 buffer, sched the scheduling state sc describes
// (zeroed by the kernel before). M <= 8: one grouped tensor-core GEMV launch
// per weight type (kMaxProj items per launch), then the dp4a GEMV for the
// Q6_K rows that are not 16-byte multiples; 8 < M <= 64: grouped launches
// over (projection, 8-token chunk) pairs; M > 64: the tile kernel per
// projection, in the order given.
// One projection on its own (run_matmul), with its codebook for IQ4_XS.
xq_status run_one(const xq_proj& q, const uint8_t* q8, int M, cudaStream_t s) {
  uint32_t cb[4];
  const uint32_t* cbp = nullptr;
  if (q.type == XQ_TYPE_IQ4_XS) {
    pack_codebook(q.codebook, cb);
    cbp = cb;
  }
  return run_matmul(q.type, q.W, q8, M, q.N, q.K, q.y, nullptr, s, false, cbp);
}

// The SwiGLU feed fused into a layer's matmul launches (M <= 8): gate, up and
// down index proj; arrive and ready are zeroed counters (F/32 and F/256
// words), hq is h's Q8 buffer, which down reads.
struct FfnSpec {
  int gate, up, down;
  unsigned int* arrive;
  unsigned int* ready;
  uint8_t* hq;
  int F;
  bool stall;  // test hook (xq_debug_stalled_ffn_layer)
};

xq_status layer_matmuls(const xq_proj* proj, int n_proj, const uint8_t* const* q8, int M, const Sched& sc,
                        uint8_t* sched, cudaStream_t s, const FfnSpec* ffn = nullptr) {
  if (M > kMaxGemvM) {
    // 8 < M <= 64: per weight type, grouped GEMV launches over every
    // (projection, 8-token chunk) pair, kMaxProj pairs per launch, the chunks
    // of one projection side by side so that they share its weight tiles
    // through L2; rows longer than 24 super-blocks split over K (no task
    // counter). The other projections (and all of them above 64 tokens) run
    // on their own.
    const bool chunked = M <= xq::kGemvMaxTokens;
    const int chunks = (M + 7) / 8;
    // split workspaces: per type, the arrival counts (zeroed by the quantize
    // launch), then the partial sums, consumed launch by launch in item order
    // (8 < M <= 64: GEMV chunks; M > 64: tile K ranges)
    uint8_t* arr_cur[kTypes];
    uint8_t* part_cur[kTypes];
    {
      uint8_t* a = sched + kTypes * kCounterBytes;
      uint8_t* pt = a;
      for (int g = 0; g < kTypes; ++g) pt += sc.arrive[g];
      for (int g = 0; g < kTypes; ++g) {
        arr_cur[g] = a;
        part_cur[g] = pt;
        a += sc.arrive[g];
        pt += sc.partial[g];
      }
    }
    bool first_launch = true;
    for (int g = 0; chunked && g < kTypes; ++g) {
      const int type = kTypeIds[g];
      xq::MmaProj items[xq::kMaxProj];
      int n = 0;
      auto launch = [&]() -> bool {
        size_t ab = 0, pb = 0;
        for (int k = 0; k < n; ++k)
          if (items[k].nch > 1) {
            ab += xq::gemv_split_arrive_bytes(items[k].N);
            pb += xq::gemv_split_partial_bytes(items[k].N, items[k].nch);
          }
        const bool split = ab > 0;
        if (xq::launch_gemv_mma(type, items, n, s, true, nullptr, split ? arr_cur[g] : nullptr,
                                split ? part_cur[g] : nullptr, first_launch) != cudaSuccess)
          return false;
        arr_cur[g] += ab;
        part_cur[g] += pb;
        first_launch = false;
        n = 0;
        return true;
      };
      for (int p = 0; p < n_proj; ++p) {
        const xq_proj& q = proj[p];
        if (q.N == 0 || q.type != type || !xq::gemv_mma_supports(q.type, q.N, q.K)) continue;
        for (int c = 0; c < chunks; ++c) {
          xq::MmaProj& it = items[n++];
          it.W = static_cast<const uint8_t*>(q.W);
          it.xq = q8[p];
          it.y = q.y;
          it.isum = nullptr;
          it.N = q.N;
          it.K = q.K;
          it.M_total = M;
          it.chunk = c;
          it.nch = sc.nch[p];
          set_codebook(q, it);
          if (n == xq::kMaxProj && !launch()) return XQ_ERR_CUDA;
        }
      }
      if (n > 0 && !launch()) return XQ_ERR_CUDA;
    }
    if (!chunked) {
      // M > 64: one tile launch per projection, in order, K-split where its
      // tiles would leave SMs idle. Only the first launch waits for the
      // previous grid (the quantizer) on entry: the later ones read nothing
      // an earlier one writes and start as its CTAs drain, and wait for it
      // before their threads exit, which keeps the stream's order.
      bool first = true;
      for (int p = 0; p < n_proj; ++p) {
        const xq_proj& q = proj[p];
        if (q.N == 0) continue;
        uint32_t cb[4];
        const uint32_t* cbp = nullptr;
        if (q.type == XQ_TYPE_IQ4_XS) {
          pack_codebook(q.codebook, cb);
          cbp = cb;
        }
        const int g = type_index(q.type);
        xq::TileSplit ts;
        ts.splits = sc.tsplit[p];
        ts.partial = reinterpret_cast<float*>(part_cur[g]);
        ts.arrive = reinterpret_cast<unsigned int*>(arr_cur[g]);
        if (xq::launch_tile_mma(q.type, static_cast<const uint8_t*>(q.W), q8[p], M, q.N, q.K, q.y, s, true, cbp,
                                nullptr, ts.splits > 1 ? &ts : nullptr, first) != cudaSuccess)
          return XQ_ERR_CUDA;
        if (ts.splits > 1) {
          arr_cur[g] += xq::tile_split_arrive_bytes(q.N, M);
          part_cur[g] += xq::tile_split_partial_bytes(q.N, M, ts.splits);
        }
        first = false;
      }
      return XQ_OK;
    }
    for (int p = 0; p < n_proj; ++p) {
      const xq_proj& q = proj[p];
      if (q.N == 0 || xq::gemv_mma_supports(q.type, q.N, q.K)) continue;
      const xq_status st = run_one(q, q8[p], M, s);
      if (st != XQ_OK) return st;
    }
    return XQ_OK;
  }
  unsigned int* counter[kTypes];
  uint8_t* arrive[kTypes];
  uint8_t* partial[kTypes];
  {
    uint8_t* a = sched + kTypes * kCounterBytes;
    uint8_t* pt = a;
    for (int g = 0; g < kTypes; ++g) pt += sc.arrive[g];
    for (int g = 0; g < kTypes; ++g) {
      counter[g] = sc.dynamic[g] ? reinterpret_cast<unsigned int*>(sched + g * kCounterBytes) : nullptr;
      arrive[g] = sc.dynamic[g] ? a : nullptr;
      partial[g] = sc.dynamic[g] ? pt : nullptr;
      a += sc.arrive[g];
      pt += sc.partial[g];
    }
  }
  // Only the first grouped launch waits for the previous grid on the stream
  // (the quantizer). The later ones start as its CTAs drain: they read
  // nothing it writes, and its CTAs trigger their launch only after their own
  // wait for the quantizer. They wait for the earlier grids before exiting,
  // which keeps the stream's order for the kernels that follow.
  // With a fused SwiGLU feed, gate and up's weight type launches first; the
  // launch that holds them writes h, and a down projection of another type
  // waits for that grid. Otherwise a type whose 64-row tasks fill at most
  // half the resident CTA slots launches first: its CTAs all start at once
  // and trigger the next launch, which then runs beside it on the free SMs.
  // After a full grid it would start only as that grid drains, and its long
  // rows would end the layer (the Qwen2.5-1.5B Q4_K_M layer, whose Q6_K
  // group is about 120 tasks, takes 24.8 instead of 26.8 us at M = 8).
  int type_order[kTypes];
  {
    int k = 0;
    if (ffn) {
      const int first = type_index(proj[ffn->gate].type);
      type_order[k++] = first;
      for (int g = 0; g < kTypes; ++g)
        if (g != first) type_order[k++] = g;
    } else {
      long long tasks[kTypes] = {0, 0, 0, 0};
      for (int p = 0; p < n_proj && p < 64; ++p)
        if (in_group(proj[p], M))
          tasks[type_index(proj[p].type)] += static_cast<long long>(xq::gemv_row_blocks(proj[p].N)) * sc.nch[p];
      for (int g = 0; g < kTypes; ++g)
        if (tasks[g] > 0 && 2 * tasks[g] <= xq::kGemvSlots) type_order[k++] = g;
      for (int g = 0; g < kTypes; ++g)
        if (!(tasks[g] > 0 && 2 * tasks[g] <= xq::kGemvSlots)) type_order[k++] = g;
    }
  }
  bool first_launch = true;
  for (int gi = 0; gi < kTypes; ++gi) {
    const int g = type_order[gi];
    const int type = kTypeIds[g];
    xq::MmaProj items[xq::kMaxProj];
    int item_proj[xq::kMaxProj];
    int n = 0;
    for (int p = 0; p <= n_proj; ++p) {
      if (p < n_proj) {
        const xq_proj& q = proj[p];
        if (!in_group(q, M) || q.type != type) continue;
        item_proj[n] = p;
        xq::MmaProj& it = items[n++];
        it.W = static_cast<const uint8_t*>(q.W);
        it.xq = q8[p];
        it.y = q.y;
        it.isum = nullptr;
        it.N = q.N;
        it.K = q.K;
        it.M_total = M;
        it.chunk = 0;
        it.nch = sc.nch[p];
        set_codebook(q, it);
      }
      if (n > 0 && (n == xq::kMaxProj || p == n_proj)) {
        xq::FfnFuse fz;
        const xq::FfnFuse* fzp = nullptr;
        bool wait = first_launch;
        if (ffn) {
          int ig = -1, iu = -1, id = -1;
          for (int k = 0; k < n; ++k) {
            if (item_proj[k] == ffn->gate) ig = k;
            if (item_proj[k] == ffn->up) iu = k;
            if (item_proj[k] == ffn->down) id = k;
          }
          if ((ig >= 0) != (iu >= 0)) return XQ_ERR_UNSUPPORTED;  // excluded by the plan
          if (ig >= 0) {
            fz.gate = ig;
            fz.up = iu;
            fz.down = id;
            fz.arrive = ffn->arrive;
            fz.ready = ffn->ready;
            fz.hq = ffn->hq;
            fz.h_out = nullptr;
            fz.F = ffn->F;
            fz.M = M;
            fz.stall = ffn->stall;
            fzp = &fz;
          } else if (id >= 0) {
            wait = true;  // h comes from an earlier grid
          }
        }
        if (xq::launch_gemv_mma(type, items, n, s, true, counter[g], arrive[g], partial[g], wait, false, fzp) !=
            cudaSuccess)
          return XQ_ERR_CUDA;
        first_launch = false;
        n = 0;
      }
    }
  }
  for (int p = 0; p < n_proj; ++p) {
    const xq_proj& q = proj[p];
    if (q.N == 0 || in_group(q, M)) continue;
    const xq_status st = run_one(q, q8[p], M, s);
    if (st != XQ_OK) return st;
  }
  return XQ_OK;
}

// Bytes of the scheduling state sc describes, all of it zeroed before the
// matmuls (counters and arrival counts) or written before it is read.
size_t sched_zero_bytes(const Sched& sc) {
  size_t z = kTypes * kCounterBytes;
  for (int g = 0; g < kTypes; ++g) z += sc.arrive[g];
  return z;
}

}  // namespace

extern "C" {


const char* xq_status_str(xq_status s) {
  switch (s) {
    case XQ_OK: return "ok";
    case XQ_ERR_ARG: return "invalid argument";
    case XQ_ERR_SHAPE: return "invalid shape";
    case XQ_ERR_ALIGN: return "pointer not 16-byte aligned";
    case XQ_ERR_WORKSPACE: return "workspace too small";
    case XQ_ERR_CUDA: return "CUDA launch failed";
    case XQ_ERR_UNSUPPORTED: return "unsupported";
  }
  return "unknown status";
}

size_t xq_q8_bytes(int M, int K) {
  if (M < 0 || K <= 0 || (K % 32) != 0) return 0;
  if (M > xq::kGemvMaxTokens && (K % 256) != 0) return 0;  // the tile image is per super-block
  return xq::q8_layout(M, K).total;
}

size_t xq_q8_bytes_invariant(int M, int K) {
  if (M < 0 || K <= 0 || (K % 32) != 0) return 0;
  return xq::q8_layout(M, K, true).total;
}

xq_status xq_quantize_q8_invariant(const float* x, int M, int K, void* xq, xq_stream stream) {
  if (M < 0 || K <= 0 || (K % 256) != 0) return XQ_ERR_SHAPE;
  if (M == 0) return XQ_OK;
  if (!x || !xq) return XQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(xq)) return XQ_ERR_ALIGN;
  xq::QuantJob job;
  job.x = x;
  job.xq = static_cast<uint8_t*>(xq);
  job.M = M;
  job.K = K;
  job.gemv_image = true;
  const cudaError_t e = xq::launch_quantize_q8(&job, 1, reinterpret_cast<cudaStream_t>(stream), true);
  return e == cudaSuccess ? XQ_OK : XQ_ERR_CUDA;
}

xq_status xq_matmul_invariant(int type, const void* W, const void* xq, int M, int N, int K, float* y,
                              xq_stream stream) {
  if (block_bytes(type) == 0) return XQ_ERR_ARG;
  if (type == XQ_TYPE_IQ4_XS) return XQ_ERR_UNSUPPORTED;  // no codebook argument here
  xq_status st = check_shape(M, N, K);
  if (st != XQ_OK) return st;
  if (M == 0 || N == 0) return XQ_OK;
  if (!W || !xq || !y) return XQ_ERR_ARG;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(y)) return XQ_ERR_ALIGN;
  return run_matmul(type, W, xq, M, N, K, y, nullptr, reinterpret_cast<cudaStream_t>(stream), true);
}

size_t xq_weight_bytes(int type, int N, int K) {
  const int bb = block_bytes(type);
  if (bb == 0 || N < 0 || K <= 0 || (K % 256) != 0) return 0;
  return static_cast<size_t>(N) * (K / 256) * bb;
}

xq_status xq_quantize_q8(const float* x, int M, int K, void* xq, xq_stream stream) {
  if (M < 0 || K <= 0 || (K % 256) != 0) return XQ_ERR_SHAPE;
  if (M == 0) return XQ_OK;
  if (!x || !xq) return XQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(xq)) return XQ_ERR_ALIGN;
  xq::QuantJob job;
  job.x = x;
  job.xq = static_cast<uint8_t*>(xq);
  job.M = M;
  job.K = K;
  const cudaError_t e = xq::launch_quantize_q8(&job, 1, reinterpret_cast<cudaStream_t>(stream), true);
  return e == cudaSuccess ? XQ_OK : XQ_ERR_CUDA;
}

xq_status xq_matmul_q4k_q8(const void* W, const void* xq, int M, int N, int K, float* y,
                           xq_stream stream) {
  return matmul_entry(XQ_TYPE_Q4_K, W, xq, M, N, K, y, nullptr, stream);
}

xq_status xq_matmul_q6k_q8(const void* W, const void* xq, int M, int N, int K, float* y,
                           xq_stream stream) {
  return matmul_entry(XQ_TYPE_Q6_K, W, xq, M, N, K, y, nullptr, stream);
}

xq_status xq_matmul_q8_0_q8(const void* W, const void* xq, int M, int N, int K, float* y,
                            xq_stream stream) {
  return matmul_entry(XQ_TYPE_Q8_0, W, xq, M, N, K, y, nullptr, stream);
}

xq_status xq_debug_isums_q8_0(const void* W, const void* xq, int M, int N, int K, float* y,
                              int32_t* isum, xq_stream stream) {
  if (!isum) return XQ_ERR_ARG;
  return matmul_entry(XQ_TYPE_Q8_0, W, xq, M, N, K, y, isum, stream);
}

// IQ4_XS: M <= 64 on the tensor-core GEMV, M > 64 on the tile kernel; rows
// that are 16-byte multiples (K a multiple of 512); the codebook is read
// from the host during the call.
static xq_status iq4xs_entry(const void* W, const int8_t* codebook, const void* xq, int M, int N, int K, float* y,
                             int32_t* isum, xq_stream stream) {
  xq_status st = check_shape(M, N, K);
  if (st != XQ_OK) return st;
  if ((K % 512) != 0) return XQ_ERR_SHAPE;
  if (M == 0 || N == 0) return XQ_OK;
  if (!W || !xq || !y || !codebook) return XQ_ERR_ARG;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(y) || (isum && !aligned16(isum))) return XQ_ERR_ALIGN;
  if (isum && M > kMaxGemvM) return XQ_ERR_UNSUPPORTED;
  uint32_t cb[4];
  pack_codebook(codebook, cb);
  return run_matmul(XQ_TYPE_IQ4_XS, W, xq, M, N, K, y, isum, reinterpret_cast<cudaStream_t>(stream), false, cb);
}

xq_status xq_matmul_iq4xs_q8(const void* W, const int8_t* codebook, const void* xq, int M, int N, int K, float* y,
                             xq_stream stream) {
  return iq4xs_entry(W, codebook, xq, M, N, K, y, nullptr, stream);
}

xq_status xq_debug_isums_iq4xs(const void* W, const int8_t* codebook, const void* xq, int M, int N, int K, float* y,
                               int32_t* isum, xq_stream stream) {
  if (!isum) return XQ_ERR_ARG;
  return iq4xs_entry(W, codebook, xq, M, N, K, y, isum, stream);
}

xq_status xq_debug_isums_q4k(const void* W, const void* xq, int M, int N, int K, float* y,
                             int32_t* isum, xq_stream stream) {
  if (!isum) return XQ_ERR_ARG;
  return matmul_entry(XQ_TYPE_Q4_K, W, xq, M, N, K, y, isum, stream);
}

xq_status xq_debug_isums_q6k(const void* W, const void* xq, int M, int N, int K, float* y,
                             int32_t* isum, xq_stream stream) {
  if (!isum) return XQ_ERR_ARG;
  return matmul_entry(XQ_TYPE_Q6_K, W, xq, M, N, K, y, isum, stream);
}

size_t xq_layer_workspace_bytes(const xq_proj* proj, int n_proj, int n_inputs, int M) {
  int in_k[64];
  if (layer_inputs(proj, n_proj, n_inputs, M, in_k) != XQ_OK) return 0;
  size_t total = 0;
  for (int i = 0; i < n_inputs; ++i)
    if (in_k[i]) total += round256(xq_q8_bytes(M, in_k[i]));
  return total + sched_bytes(sched_layout(proj, n_proj, M));
}

xq_status xq_layer_mixed(const xq_proj* proj, int n_proj, const float* const* inputs, int n_inputs,
                         int M, void* workspace, size_t ws_bytes, xq_stream stream) {
  int in_k[64];
  xq_status st = layer_inputs(proj, n_proj, n_inputs, M, in_k);
  if (st != XQ_OK) return st;
  if (M == 0) return XQ_OK;
  if (n_inputs > 0 && !inputs) return XQ_ERR_ARG;
  size_t need = 0;
  size_t off[64];
  for (int i = 0; i < n_inputs; ++i) {
    off[i] = need;
    if (in_k[i]) {
      if (!inputs[i]) return XQ_ERR_ARG;
      if (!aligned16(inputs[i])) return XQ_ERR_ALIGN;
      need += round256(xq_q8_bytes(M, in_k[i]));
    }
  }
  const size_t sched_off = need;
  const Sched sc = sched_layout(proj, n_proj, M);
  need += sched_bytes(sc);
  if (!workspace) return XQ_ERR_ARG;
  if (ws_bytes < need) return XQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return XQ_ERR_ALIGN;
  for (int p = 0; p < n_proj; ++p) {
    if (proj[p].N == 0) continue;
    if (!proj[p].W || !proj[p].y) return XQ_ERR_ARG;
    if (!aligned16(proj[p].W) || !aligned16(proj[p].y)) return XQ_ERR_ALIGN;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // scheduling state: counters and arrival counts, zeroed by the quantize
  // launch (the matmuls leave them at zero), then partial sums
  const int zero_words = static_cast<int>(sched_zero_bytes(sc) / 4);
  // One launch quantizes every input that is read (up to kMaxProj per launch).
  {
    xq::QuantJob jobs[xq::kMaxProj];
    int n = 0, left = 0;
    for (int i = 0; i < n_inputs; ++i) left += in_k[i] ? 1 : 0;
    for (int i = 0; i < n_inputs; ++i) {
      if (!in_k[i]) continue;
      xq::QuantJob& j = jobs[n++];
      j.x = inputs[i];
      j.xq = ws + off[i];
      j.M = M;
      j.K = in_k[i];
      --left;
      if (n == xq::kMaxProj || left == 0) {
        unsigned int* zero = left == 0 ? reinterpret_cast<unsigned int*>(ws + sched_off) : nullptr;
        if (xq::launch_quantize_q8(jobs, n, s, true, zero, zero_words) != cudaSuccess) return XQ_ERR_CUDA;
        n = 0;
      }
    }
  }
  const uint8_t* q8[64];
  for (int p = 0; p < n_proj; ++p) q8[p] = ws + off[proj[p].input];
  return layer_matmuls(proj, n_proj, q8, M, sc, ws + sched_off, s);
}

xq_status xq_debug_layer_matmuls(const xq_proj* proj, int n_proj, int n_inputs, int M, void* workspace,
                                 size_t ws_bytes, xq_stream stream) {
  int in_k[64];
  const xq_status st = layer_inputs(proj, n_proj, n_inputs, M, in_k);
  if (st != XQ_OK) return st;
  if (M == 0) return XQ_OK;
  // the workspace layout of xq_layer_mixed: the used inputs' Q8 buffers in
  // input order, then the scheduling state
  size_t off[64];
  size_t need = 0;
  for (int i = 0; i < n_inputs; ++i) {
    off[i] = need;
    if (in_k[i]) need += round256(xq_q8_bytes(M, in_k[i]));
  }
  const size_t sched_off = need;
  const Sched sc = sched_layout(proj, n_proj, M);
  need += sched_bytes(sc);
  if (!workspace) return XQ_ERR_ARG;
  if (ws_bytes < need) return XQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return XQ_ERR_ALIGN;
  for (int p = 0; p < n_proj; ++p) {
    if (proj[p].N == 0) continue;
    if (!proj[p].W || !proj[p].y) return XQ_ERR_ARG;
    if (!aligned16(proj[p].W) || !aligned16(proj[p].y)) return XQ_ERR_ALIGN;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* q8[64];
  for (int p = 0; p < n_proj; ++p) q8[p] = ws + off[proj[p].input];
  return layer_matmuls(proj, n_proj, q8, M, sc, ws + sched_off, reinterpret_cast<cudaStream_t>(stream));
}

xq_status xq_debug_tile_sums(int type, const void* W, const int8_t* codebook, const void* xq, int M, int N, int K,
                             float* y, int32_t* sums, xq_stream stream) {
  if (block_bytes(type) == 0) return XQ_ERR_ARG;
  xq_status st = check_shape(M, N, K);
  if (st != XQ_OK) return st;
  if (M <= xq::kGemvMaxTokens) return XQ_ERR_UNSUPPORTED;  // the tile kernel serves M > 64
  if (type == XQ_TYPE_IQ4_XS && (K % 512) != 0) return XQ_ERR_SHAPE;
  if (N == 0) return XQ_OK;
  if (!W || !xq || !y || !sums || (type == XQ_TYPE_IQ4_XS && !codebook)) return XQ_ERR_ARG;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(y) || !aligned16(sums)) return XQ_ERR_ALIGN;
  uint32_t cb[4];
  if (type == XQ_TYPE_IQ4_XS) pack_codebook(codebook, cb);
  const cudaError_t e =
      xq::launch_tile_mma(type, static_cast<const uint8_t*>(W), static_cast<const uint8_t*>(xq), M, N, K, y,
                          reinterpret_cast<cudaStream_t>(stream), true, type == XQ_TYPE_IQ4_XS ? cb : nullptr, sums);
  return e == cudaSuccess ? XQ_OK : XQ_ERR_CUDA;
}

xq_status xq_device_error(xq_stream stream, unsigned int* code_out) {
  if (!code_out) return XQ_ERR_ARG;
  *code_out = 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return XQ_ERR_CUDA;
  unsigned int c[2] = {0u, 0u};
  const cudaError_t e0 = xq::take_gemv_error(&c[0]);
  const cudaError_t e1 = xq::take_tile_error(&c[1]);
  if (e0 != cudaSuccess || e1 != cudaSuccess) return XQ_ERR_CUDA;
  for (int k = 0; k < 2; ++k)
    if (c[k]) {
      *code_out = (static_cast<unsigned int>(k + 1) << 8) | (c[k] & 0xFFu);
      break;
    }
  // checked builds: the first failed bounds check of each kernel file
  unsigned int chk[4] = {0u, 0u, 0u, 0u};
  const cudaError_t c0 = xq::take_gemv_check(&chk[0]);
  const cudaError_t c1 = xq::take_tile_check(&chk[1]);
  const cudaError_t c2 = xq::take_quant_check(&chk[2]);
  const cudaError_t c3 = xq::take_q6k_check(&chk[3]);
  if (c0 != cudaSuccess || c1 != cudaSuccess || c2 != cudaSuccess || c3 != cudaSuccess) return XQ_ERR_CUDA;
  for (int k = 0; k < 4 && *code_out == 0; ++k)
    if (chk[k]) *code_out = (9u << 8) | (chk[k] & 0xFFu);
  return XQ_OK;
}

xq_status xq_debug_check_probe(const void* W, const void* xq, int M, int N, int K, float* y, xq_stream stream) {
#ifdef XQ_CHECK
  if (M < 2 || M > kMaxGemvM) return XQ_ERR_SHAPE;
  const xq_status st = check_shape(M, N, K);
  if (st != XQ_OK) return st;
  if (!W || !xq || !y) return XQ_ERR_ARG;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(y)) return XQ_ERR_ALIGN;
  xq::MmaProj q;
  q.W = static_cast<const uint8_t*>(W);
  q.xq = static_cast<const uint8_t*>(xq);
  q.y = y;
  q.isum = nullptr;
  q.N = N;
  q.K = K;
  q.M_total = M;
  q.chunk = 0;
  q.nch = 1;
  q.y_limit = static_cast<long long>(M - 1) * N;  // one token row short of what the launch writes
  return xq::launch_gemv_mma(XQ_TYPE_Q4_K, &q, 1, reinterpret_cast<cudaStream_t>(stream), true) == cudaSuccess
             ? XQ_OK
             : XQ_ERR_CUDA;
#else
  (void)W;
  (void)xq;
  (void)M;
  (void)N;
  (void)K;
  (void)y;
  (void)stream;
  return XQ_ERR_UNSUPPORTED;
#endif
}

xq_status xq_debug_stalled_matmul_q4k(const void* W, const void* xq, int M, int N, int K, float* y,
                                      xq_stream stream) {
  xq_status st = check_shape(M, N, K);
  if (st != XQ_OK) return st;
  if (M < 1 || M > kMaxGemvM || N == 0) return XQ_ERR_SHAPE;
  if (!W || !xq || !y) return XQ_ERR_ARG;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(y)) return XQ_ERR_ALIGN;
  xq::MmaProj q;
  q.W = static_cast<const uint8_t*>(W);
  q.xq = static_cast<const uint8_t*>(xq);
  q.y = y;
  q.isum = nullptr;
  q.N = N;
  q.K = K;
  q.M_total = M;
  q.chunk = 0;
  q.nch = 1;
  const cudaError_t e = xq::launch_gemv_mma(XQ_TYPE_Q4_K, &q, 1, reinterpret_cast<cudaStream_t>(stream), true, nullptr,
                                            nullptr, nullptr, true, true);
  return e == cudaSuccess ? XQ_OK : XQ_ERR_CUDA;
}

xq_status xq_silu_mul_quantize_q8(const float* gate, const float* up, int M, int K, void* xq, float* h_out,
                                  xq_stream stream) {
  if (M < 0 || K <= 0 || (K % 256) != 0) return XQ_ERR_SHAPE;
  if (M == 0) return XQ_OK;
  if (!gate || !up || !xq) return XQ_ERR_ARG;
  if (!aligned16(gate) || !aligned16(up) || !aligned16(xq)) return XQ_ERR_ALIGN;
  xq::QuantJob job;
  job.x = gate;
  job.up = up;
  job.h_out = h_out;
  job.xq = static_cast<uint8_t*>(xq);
  job.M = M;
  job.K = K;
  const cudaError_t e = xq::launch_quantize_q8(&job, 1, reinterpret_cast<cudaStream_t>(stream), true);
  return e == cudaSuccess ? XQ_OK : XQ_ERR_CUDA;
}

}  // extern "C"

namespace {

// The layer with a SwiGLU-fed down projection, in four launches: the Q8
// quantization of every input; the gate and up projections (group A);
// h = silu(y_gate) * y_up quantized to Q8; every other projection together
// with down (group C), so that the projections that do not depend on gate
// and up share down's grouped launch. Workspace: the inputs' Q8 buffers,
// h's Q8 buffer, then the scheduling state of A and of C.
//
// At M <= 8, when gate and up share one grouped launch, the feed is fused
// instead: the Q8 quantization of every input, then the layer's grouped
// launches (gate and up's type first), whose gate/up warps write h's Q8
// themselves; a down projection in the same launch waits per super-block
// for h, one in a later launch for the grid. Workspace: the inputs' Q8
// buffers, h's Q8 buffer, h's block counters, then the layer's scheduling
// state (the quantize launch zeroes the counters and the state).
struct FfnPlan {
  xq_proj a[2], c[64];
  int n_c;
  int c_input[64];  // layer input of each C projection, -1 for down (reads h)
  int in_k[64];
  size_t off[64];
  size_t h_off, sched_a, sched_c, total;
  Sched sc_a, sc_c;
  bool fused;
  xq_proj all[64];  // fused: the layer with down as it is (its input unused)
  Sched sc_all;
  size_t ffn_off, ffn_bytes, sched_all;
};

xq_status ffn_plan(const xq_proj* proj, int n_proj, int n_inputs, int M, int gate, int up, int down, FfnPlan* f) {
  if (!proj || n_proj < 3 || n_proj > 64 || n_inputs < 0 || n_inputs > 64) return XQ_ERR_ARG;
  if (gate < 0 || up < 0 || down < 0 || gate >= n_proj || up >= n_proj || down >= n_proj || gate == up ||
      gate == down || up == down)
    return XQ_ERR_ARG;
  if (proj[gate].N != proj[up].N || proj[down].K != proj[gate].N) return XQ_ERR_SHAPE;
  xq_proj rest[64];
  int n_rest = 0;
  for (int p = 0; p < n_proj; ++p)
    if (p != down) rest[n_rest++] = proj[p];
  xq_status st = layer_inputs(rest, n_rest, n_inputs, M, f->in_k);
  if (st != XQ_OK) return st;
  xq_proj d = proj[down];
  d.input = 0;
  int dk[1];
  st = layer_inputs(&d, 1, 1, M, dk);
  if (st != XQ_OK) return st;
  f->a[0] = proj[gate];
  f->a[1] = proj[up];
  f->n_c = 0;
  for (int p = 0; p < n_proj; ++p) {
    if (p == gate || p == up) continue;
    f->c_input[f->n_c] = p == down ? -1 : proj[p].input;
    f->c[f->n_c++] = p == down ? d : proj[p];
  }
  size_t need = 0;
  for (int i = 0; i < n_inputs; ++i) {
    f->off[i] = need;
    if (f->in_k[i]) need += round256(xq_q8_bytes(M, f->in_k[i]));
  }
  f->h_off = need;
  need += round256(xq_q8_bytes(M, d.K));
  // fused feed: gate and up in the GEMV group, in one launch of their type
  f->fused = false;
  // (h's blocks are counted per pair of 16-row groups of consecutive rows, so
  // Q6_K gate/up rows in the grouped view keep the separate feed launch)
  const bool grouped_rows = proj[gate].type == XQ_TYPE_Q6_K && xq::q6k_row_shift(proj[gate].K) > 0;
  if (M >= 1 && M <= kMaxGemvM && in_group(proj[gate], M) && in_group(proj[up], M) &&
      proj[gate].type == proj[up].type && !grouped_rows) {
    int same = 0;
    for (int p = 0; p < n_proj; ++p) same += (in_group(proj[p], M) && proj[p].type == proj[gate].type) ? 1 : 0;
    f->fused = same <= xq::kMaxProj;
  }
  if (f->fused) {
    for (int p = 0; p < n_proj; ++p) f->all[p] = proj[p];
    f->sc_all = sched_layout(f->all, n_proj, M);
    f->ffn_off = need;
    f->ffn_bytes = round256(4 * static_cast<size_t>(d.K / 32 + d.K / 256));
    need += f->ffn_bytes;
    f->sched_all = need;
    need += sched_bytes(f->sc_all);
    f->total = need;
    return XQ_OK;
  }
  f->sc_a = sched_layout(f->a, 2, M);
  f->sc_c = sched_layout(f->c, f->n_c, M);
  f->sched_a = need;
  need += round256(sched_bytes(f->sc_a));
  f->sched_c = need;
  need += sched_bytes(f->sc_c);
  f->total = need;
  return XQ_OK;
}

xq_status layer_ffn(const xq_proj* proj, int n_proj, int gate, int up, int down, const float* const* inputs,
                    int n_inputs, int M, void* workspace, size_t ws_bytes, xq_stream stream, bool stall) {
  FfnPlan f;
  xq_status st = ffn_plan(proj, n_proj, n_inputs, M, gate, up, down, &f);
  if (st != XQ_OK) return st;
  if (M == 0) return XQ_OK;
  if (stall && !f.fused) return XQ_ERR_UNSUPPORTED;
  if (n_inputs > 0 && !inputs) return XQ_ERR_ARG;
  for (int i = 0; i < n_inputs; ++i)
    if (f.in_k[i]) {
      if (!inputs[i]) return XQ_ERR_ARG;
      if (!aligned16(inputs[i])) return XQ_ERR_ALIGN;
    }
  if (!workspace) return XQ_ERR_ARG;
  if (ws_bytes < f.total) return XQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return XQ_ERR_ALIGN;
  for (int p = 0; p < n_proj; ++p) {
    if (proj[p].N == 0) continue;
    if (!proj[p].W || !proj[p].y) return XQ_ERR_ARG;
    if (!aligned16(proj[p].W) || !aligned16(proj[p].y)) return XQ_ERR_ALIGN;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (f.fused) {
    // 1. every input to Q8 (the last launch zeroes h's counters and the
    // layer's scheduling state, which follow one another)
    xq::QuantJob jobs[xq::kMaxProj];
    int n = 0, left = 0;
    for (int i = 0; i < n_inputs; ++i) left += f.in_k[i] ? 1 : 0;
    const int zero_words = static_cast<int>((f.ffn_bytes + sched_zero_bytes(f.sc_all)) / 4);
    for (int i = 0; i < n_inputs; ++i) {
      if (!f.in_k[i]) continue;
      xq::QuantJob& j = jobs[n++];
      j.x = inputs[i];
      j.xq = ws + f.off[i];
      j.M = M;
      j.K = f.in_k[i];
      --left;
      if (n == xq::kMaxProj || left == 0) {
        unsigned int* zero = left == 0 ? reinterpret_cast<unsigned int*>(ws + f.ffn_off) : nullptr;
        if (xq::launch_quantize_q8(jobs, n, s, true, zero, zero_words) != cudaSuccess) return XQ_ERR_CUDA;
        n = 0;
      }
    }
    // 2. the layer's matmuls, h written by the gate and up warps
    const uint8_t* q8[64];
    for (int p = 0; p < n_proj; ++p) q8[p] = p == down ? ws + f.h_off : ws + f.off[proj[p].input];
    const int F = proj[down].K;
    FfnSpec spec;
    spec.gate = gate;
    spec.up = up;
    spec.down = down;
    spec.arrive = reinterpret_cast<unsigned int*>(ws + f.ffn_off);
    spec.ready = spec.arrive + F / 32;
    spec.hq = ws + f.h_off;
    spec.F = F;
    spec.stall = stall;
    return layer_matmuls(f.all, n_proj, q8, M, f.sc_all, ws + f.sched_all, s, &spec);
  }
  // 1. every input to Q8 (the last launch zeroes A's scheduling state)
  {
    xq::QuantJob jobs[xq::kMaxProj];
    int n = 0, left = 0;
    for (int i = 0; i < n_inputs; ++i) left += f.in_k[i] ? 1 : 0;
    for (int i = 0; i < n_inputs; ++i) {
      if (!f.in_k[i]) continue;
      xq::QuantJob& j = jobs[n++];
      j.x = inputs[i];
      j.xq = ws + f.off[i];
      j.M = M;
      j.K = f.in_k[i];
      --left;
      if (n == xq::kMaxProj || left == 0) {
        unsigned int* zero = left == 0 ? reinterpret_cast<unsigned int*>(ws + f.sched_a) : nullptr;
        if (xq::launch_quantize_q8(jobs, n, s, true, zero, static_cast<int>(sched_zero_bytes(f.sc_a) / 4)) !=
            cudaSuccess)
          return XQ_ERR_CUDA;
        n = 0;
      }
    }
  }
  // 2. gate and up
  const uint8_t* q8a[2] = {ws + f.off[f.a[0].input], ws + f.off[f.a[1].input]};
  st = layer_matmuls(f.a, 2, q8a, M, f.sc_a, ws + f.sched_a, s);
  if (st != XQ_OK) return st;
  // 3. h = silu(y_gate) * y_up -> Q8 (zeroing C's scheduling state)
  xq::QuantJob job;
  job.x = f.a[0].y;
  job.up = f.a[1].y;
  job.xq = ws + f.h_off;
  job.M = M;
  job.K = proj[down].K;
  if (xq::launch_quantize_q8(&job, 1, s, true, reinterpret_cast<unsigned int*>(ws + f.sched_c),
                             static_cast<int>(sched_zero_bytes(f.sc_c) / 4)) != cudaSuccess)
    return XQ_ERR_CUDA;
  // 4. the other projections and down
  const uint8_t* q8c[64];
  for (int k = 0; k < f.n_c; ++k) q8c[k] = f.c_input[k] < 0 ? ws + f.h_off : ws + f.off[f.c_input[k]];
  return layer_matmuls(f.c, f.n_c, q8c, M, f.sc_c, ws + f.sched_c, s);
}

}  // namespace

extern "C" {

size_t xq_layer_ffn_workspace_bytes(const xq_proj* proj, int n_proj, int n_inputs, int M, int gate, int up,
                                    int down) {
  FfnPlan f;
  if (ffn_plan(proj, n_proj, n_inputs, M, gate, up, down, &f) != XQ_OK) return 0;
  return f.total;
}

xq_status xq_layer_mixed_ffn(const xq_proj* proj, int n_proj, int gate, int up, int down,
                             const float* const* inputs, int n_inputs, int M, void* workspace, size_t ws_bytes,
                             xq_stream stream) {
  return layer_ffn(proj, n_proj, gate, up, down, inputs, n_inputs, M, workspace, ws_bytes, stream, false);
}

xq_status xq_debug_stalled_ffn_layer(const xq_proj* proj, int n_proj, int gate, int up, int down,
                                     const float* const* inputs, int n_inputs, int M, void* workspace,
                                     size_t ws_bytes, xq_stream stream) {
  return layer_ffn(proj, n_proj, gate, up, down, inputs, n_inputs, M, workspace, ws_bytes, stream, true);
}

}  // extern "C"
