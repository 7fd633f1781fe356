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
  return type == XQ_TYPE_Q4_K ? xq::kQ4kBytes : (type == XQ_TYPE_Q6_K ? xq::kQ6kBytes : 0);
}

xq_status check_shape(int M, int N, int K) {
  if (M < 0 || N < 0 || K <= 0 || (K % 256) != 0) return XQ_ERR_SHAPE;
  return XQ_OK;
}

// Enqueue y = x W^T. M > 8: the tensor-memory tile kernel (both types).
// M <= 8: Q4_K on the warp-level MMA GEMV, Q6_K on the dp4a GEMV.
xq_status run_matmul(int type, const void* W, const void* xq, int M, int N, int K, float* y,
                     int32_t* isum, cudaStream_t s) {
  const xq::Q8Layout L = xq::q8_layout(M, K);
  const uint8_t* base = static_cast<const uint8_t*>(xq);
  if (M > kMaxGemvM) {
    const cudaError_t e = xq::launch_tile_mma(type, static_cast<const uint8_t*>(W), base, M, N, K, y, s, true);
    return e == cudaSuccess ? XQ_OK : XQ_ERR_CUDA;
  }
  if (type == XQ_TYPE_Q4_K) {
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
      if (n == xq::kMaxProj || c + 1 == L.chunks) {
        if (xq::launch_gemv_q4k_mma(items, n, s, true) != cudaSuccess) return XQ_ERR_CUDA;
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

// The layer workspace ends with the grouped matmul's scheduling state: a
// 256-byte task counter, the arrival counts of split projections, and their
// partial sums (sizes from the same helpers the launcher uses).
constexpr size_t kCounterBytes = 256;

struct SchedBytes {
  size_t arrive, partial;
};

SchedBytes sched_bytes(const xq_proj* proj, int n_proj, int M) {
  SchedBytes b = {0, 0};
  for (int p = 0; p < n_proj; ++p) {
    if (proj[p].type != XQ_TYPE_Q4_K || proj[p].N == 0) continue;
    const int nch = xq::q4k_split_chunks(proj[p].K, M);
    if (nch > 1) {
      b.arrive += xq::q4k_split_arrive_bytes(proj[p].N);
      b.partial += xq::q4k_split_partial_bytes(proj[p].N, nch);
    }
  }
  return b;
}

// Validate a layer description and find each input's K (0 = unused).
xq_status layer_inputs(const xq_proj* proj, int n_proj, int n_inputs, int M, int* in_k) {
  if (!proj || n_proj < 0 || n_inputs < 0 || n_inputs > 64) return XQ_ERR_ARG;
  if (M < 0) return XQ_ERR_SHAPE;
  for (int i = 0; i < n_inputs; ++i) in_k[i] = 0;
  for (int p = 0; p < n_proj; ++p) {
    const xq_proj& q = proj[p];
    if (block_bytes(q.type) == 0) return XQ_ERR_ARG;
    if (q.input < 0 || q.input >= n_inputs) return XQ_ERR_ARG;
    const xq_status st = check_shape(M, q.N, q.K);
    if (st != XQ_OK) return st;
    if (in_k[q.input] == 0) in_k[q.input] = q.K;
    if (in_k[q.input] != q.K) return XQ_ERR_SHAPE;
  }
  return XQ_OK;
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
  if (M > kMaxGemvM && (K % 256) != 0) return 0;  // the tile image is per super-block
  return xq::q8_layout(M, K).total;
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
  const SchedBytes sb = sched_bytes(proj, n_proj, M);
  return total + kCounterBytes + sb.arrive + sb.partial;
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
  const size_t counter_off = need;
  const SchedBytes sb = sched_bytes(proj, n_proj, M);
  need += kCounterBytes + sb.arrive + sb.partial;
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
  unsigned int* counter = reinterpret_cast<unsigned int*>(ws + counter_off);
  const int chunks = (M + 7) / 8;
  int q4_items = 0;
  for (int p = 0; p < n_proj; ++p)
    if (proj[p].N > 0 && proj[p].type == XQ_TYPE_Q4_K) q4_items += chunks;
  // Dynamic task fetch and K-split when every Q4_K chunk fits one launch:
  // the quantize launch just before it zeroes the counter and the arrival
  // counts (which the matmul also leaves at zero).
  const bool dynamic = q4_items > 0 && q4_items <= xq::kMaxProj;
  uint8_t* split_ws = dynamic ? ws + counter_off + kCounterBytes : nullptr;
  const int zero_words = static_cast<int>((kCounterBytes + sb.arrive) / 4);
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
        if (xq::launch_quantize_q8(jobs, n, s, true, (left == 0 && dynamic) ? counter : nullptr, zero_words) !=
            cudaSuccess)
          return XQ_ERR_CUDA;
        n = 0;
      }
    }
  }
  if (M > kMaxGemvM) {
    // every projection on the tile kernel, in the order given
    for (int p = 0; p < n_proj; ++p) {
      const xq_proj& q = proj[p];
      if (q.N == 0) continue;
      st = run_matmul(q.type, q.W, ws + off[q.input], M, q.N, q.K, q.y, nullptr, s);
      if (st != XQ_OK) return st;
    }
    return XQ_OK;
  }
  // One launch for the Q4_K projections (8-token chunks, kMaxProj items per launch).
  {
    xq::MmaProj items[xq::kMaxProj];
    int n = 0;
    for (int p = 0; p < n_proj; ++p) {
      const xq_proj& q = proj[p];
      if (q.N == 0 || q.type != XQ_TYPE_Q4_K) continue;
      for (int c = 0; c < chunks; ++c) {
        xq::MmaProj& it = items[n++];
        it.W = static_cast<const uint8_t*>(q.W);
        it.xq = ws + off[q.input];
        it.y = q.y;
        it.isum = nullptr;
        it.N = q.N;
        it.K = q.K;
        it.M_total = M;
        it.chunk = c;
        if (n == xq::kMaxProj) {
          if (xq::launch_gemv_q4k_mma(items, n, s, true, dynamic ? counter : nullptr, split_ws) != cudaSuccess)
            return XQ_ERR_CUDA;
          n = 0;
        }
      }
    }
    if (n && xq::launch_gemv_q4k_mma(items, n, s, true, dynamic ? counter : nullptr, split_ws) != cudaSuccess)
      return XQ_ERR_CUDA;
  }
  for (int p = 0; p < n_proj; ++p) {
    const xq_proj& q = proj[p];
    if (q.N == 0 || q.type != XQ_TYPE_Q6_K) continue;
    st = run_matmul(q.type, q.W, ws + off[q.input], M, q.N, q.K, q.y, nullptr, s);
    if (st != XQ_OK) return st;
  }
  return XQ_OK;
}

}  // extern "C"
