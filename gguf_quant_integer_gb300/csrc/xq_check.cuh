// Checked builds (compiled with -DXQ_CHECK; the build script makes one as
// _build_check/libxq_check.so). Before a global access whose index, range or
// alignment comes from nontrivial arithmetic, a kernel tests it against the
// extent of the buffer it addresses (from the shapes and the layouts the
// entry points document) and, for bulk and tensor copies, against the
// 16-byte rule. A failed check records a site number in this translation
// unit's check word and the access is skipped: nothing traps, and a skipped
// copy leaves its barrier short, so the bounded wait after it runs out and is
// recorded too. xq_device_error reports a recorded site as kernel 9, wait =
// site. Without XQ_CHECK every check is the constant true and no code is
// generated for it.
#pragma once

#include <cuda_runtime.h>

namespace xq {

#ifdef XQ_CHECK
namespace {
__device__ unsigned int g_check_word;  // one per translation unit

__device__ __forceinline__ bool check_at(bool ok, unsigned site) {
  if (!ok) atomicCAS(&g_check_word, 0u, site);
  return ok;
}

// Read and clear this translation unit's check word.
inline cudaError_t take_check_word(unsigned int* code) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_check_word, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_check_word, &z, sizeof(z));
  *code = v;
  return e;
}
}  // namespace
#define XQ_CHECKED(cond, site) (::xq::check_at((cond), (site)))
#else
namespace {
inline cudaError_t take_check_word(unsigned int* code) {
  *code = 0;
  return cudaSuccess;
}
}  // namespace
// the condition stays an unevaluated operand: no code, no unused variables
#define XQ_CHECKED(cond, site) ((void)sizeof(cond), true)
#endif
// index i inside an array of n elements (a negative i fails too)
#define XQ_IN(i, n, site) XQ_CHECKED(static_cast<size_t>(i) < static_cast<size_t>(n), (site))

// Check sites, by kernel file.
enum CheckSite : unsigned {
  // gemv_mma.cu
  kChkGemvY = 10,        // y store inside [M][N] of the chunk
  kChkGemvIsum = 11,     // isum store inside [M][N][K/32 or K/16]
  kChkGemvPartial = 12,  // split-K partial store or load inside the workspace slice
  kChkGemvArrive = 13,   // split-K arrival count inside the projection's counts
  kChkGemvAct = 14,      // activation bulk copy inside the Q8 buffer, 16-byte aligned
  kChkGemvBox = 15,      // weight box: x on a 16-byte boundary, y inside the map
  kChkGemvFfn = 16,      // fused SwiGLU feed: h reads and writes inside their buffers
  // tile_mma.cu
  kChkTileY = 20,
  kChkTileSums = 21,
  kChkTileQ6Window = 22,  // Q6_K row window: inside the weights, 16-byte aligned
  kChkTileItem = 23,      // token item copy inside the tile image
  kChkTileBox = 24,       // weight box x on a 16-byte boundary
  kChkTileQ6Cut = 25,     // Q6_K scales read from global memory inside the weights
  kChkTileSplit = 26,     // K-split arrival count inside the tile counts
  // quantize_q8.cu
  kChkQuantX = 30,     // input read inside [M][K]
  kChkQuantQ8 = 31,    // qs / d8 / s8 store inside the Q8 buffer
  kChkQuantImage = 32, // operand image store inside the Q8 buffer
  // gemv_q6k.cu
  kChkQ6W = 40,    // super-block read inside the weights
  kChkQ6Act = 41,  // quant / d8 read inside the Q8 buffer
  kChkQ6Y = 42,
  kChkQ6Isum = 43,
};

}  // namespace xq
