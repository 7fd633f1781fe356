/*
 * xq — GGUF Q4_K / Q6_K / Q8_0 / IQ4_XS x Q8 integer matmul on GB300 (sm_103a).
 *
 * The operation (xLLM v0.7 long-context article, Tencent Cloud, section 一
 * "背景"): weights stay in their GGUF k-quant super-blocks; activations are
 * quantized to 8-bit; each 32-weight (Q4_K) or 16-weight (Q6_K) sub-block is
 * reduced with an exact integer dot product; scales and mins are applied in
 * fp32 afterwards; the output is fp32. Weights are never dequantized.
 *
 *   y[m][n] = sum_k w[n][k] * (d8[m][k/32] * q8[m][k])
 *
 * with w from the block formulas (Q4_K: w = d*sc*q - dmin*m; Q6_K:
 * w = d*s*(q-32); Q8_0: w = d*q; IQ4_XS: w = d*(ls-32)*codebook[q]),
 * rearranged as sums of integer sub-block dot products.
 *
 * Conventions for every entry point:
 *  - Every pointer argument is a DEVICE pointer, owned by the caller. The
 *    library allocates nothing and keeps no state between calls.
 *  - Calls only enqueue work on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and return without synchronizing.
 *  - Argument, shape and alignment errors return before anything is enqueued.
 *    XQ_ERR_CUDA means a launch failed (the CUDA error is left for the caller
 *    to inspect with cudaGetLastError / cudaPeekAtLastError).
 *  - There is no fallback: nothing here dequantizes to a float matrix,
 *    calls cuBLAS, or computes on the CPU.
 *  - Shapes: K (input features) is a positive multiple of 256; N (output
 *    features) >= 0; M (tokens) >= 0. M == 0 or N == 0 is an empty product
 *    and returns XQ_OK without enqueuing anything.
 *  - Alignment: every pointer must be 16-byte aligned.
 *
 * Data layouts (all row-major):
 *  - x   : fp32 [M][K].
 *  - W   : GGUF blocks, row n is K/256 consecutive super-blocks (Q4_K 144 B,
 *          Q6_K 210 B, IQ4_XS 136 B) or K/32 Q8_0 blocks of 34 B (public
 *          GGUF layouts).
 *  - xq  : one buffer of xq_q8_bytes(M, K) bytes holding
 *            qs   int8 [M][K]          at byte 0
 *            d8   fp32 [M][K/32]       at byte M*K
 *            s8   fp32 [M][K/32]       at byte M*K + 4*M*(K/32)
 *          and, at F = round_up(1.25*M*K, 256), the operand image of the
 *          matmul that serves this M. d8 = amax/127 of the 32-block,
 *          q = round-half-away(x * (1/d8)) clamped to +-127, s8 = d8*sum(q)
 *          (q8_1 kind: scale and sum).
 *          M <= 64: frag fp16 [C][K/32][32][8] at F and fsc fp32 [C][K/32][4][4]
 *          at F + 16*C*K, C = ceil(M/8): the same numbers in the operand
 *          order of the warp-level tensor-core GEMV (8-token chunks:
 *          frag[c][j][4n+t][s] = qs[8c+n][32j+8t+p(s)], p = 0,2,1,3,4,6,5,7;
 *          fsc[c][j][t] = d8,d8,s8,s8 of tokens 8c+2t, 8c+2t+1).
 *          M > 64: T = ceil(M/128) tiles of 128 tokens; for tile t and
 *          super-block b a record of 77,824 bytes at F + (t*K/256 + b)*77824:
 *          for each 32-block 8b+i an 8,704-byte item (fp16 q of the 128
 *          tokens as a K-major tensor-core operand, 8x8 core matrices, then
 *          their 128 d8 values), then an 8,192-byte bf16 operand holding s8
 *          split into three bf16 pieces per 32-block.
 *          Tokens past M are zero. xq_quantize_q8 writes every region.
 *  - y   : fp32 [M][N].
 */
#ifndef XQ_H
#define XQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define XQ_API __attribute__((visibility("default")))
#else
#define XQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; the same type, spelled without the CUDA headers. */
typedef struct CUstream_st *xq_stream;

typedef enum {
    XQ_OK = 0,
    XQ_ERR_ARG = 1,         /* null pointer or unknown type / input index */
    XQ_ERR_SHAPE = 2,       /* K not a positive multiple of 256, negative M or N,
                               mismatched K between projections sharing an input */
    XQ_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    XQ_ERR_WORKSPACE = 4,   /* workspace smaller than xq_layer_workspace_bytes() */
    XQ_ERR_CUDA = 5,        /* a kernel launch failed */
    XQ_ERR_UNSUPPORTED = 6  /* a shape or type this build does not handle */
} xq_status;

/* GGUF tensor type ids. */
#define XQ_TYPE_Q8_0 8
#define XQ_TYPE_Q4_K 12
#define XQ_TYPE_Q6_K 14
#define XQ_TYPE_IQ4_XS 23

/* Human-readable name of a status code (static string, never NULL). */
XQ_API const char *xq_status_str(xq_status s);

/* Bytes of the Q8 activation buffer for M tokens of K features:
 * round_up(1.25*M*K, 256) + 18*K*ceil(M/8) for M <= 64,
 * round_up(1.25*M*K, 256) + 77824*(K/256)*ceil(M/128) for M > 64.
 * Returns 0 when M < 0, when K is not a positive multiple of 32, or when
 * M > 64 and K is not a multiple of 256. */
XQ_API size_t xq_q8_bytes(int M, int K);

/* Bytes of an N x K weight of GGUF type `type` (N*(K/256)*144 for Q4_K,
 * N*(K/256)*210 for Q6_K, N*(K/256)*272 for Q8_0, N*(K/256)*136 for
 * IQ4_XS). Returns 0 for an unknown type or a bad shape. */
XQ_API size_t xq_weight_bytes(int type, int N, int K);

/* Q8 activation quantization (xLLM v0.7 article, sections B1.3 and C.1:
 * the activation is quantized once to 8-bit and shared by every projection
 * that reads it; Agent Telemetry log, "批次化 MMVQ": q8_1 blocks of 32 with
 * a scale and a sum).
 *   x  : fp32 [M][K], device, read-only.
 *   xq : device buffer of xq_q8_bytes(M, K) bytes, written (layout above).
 * K must be a positive multiple of 256 (the super-block width) so that the
 * result feeds the matmuls directly. Deterministic and bit-exact: fp32 IEEE
 * divide and reciprocal, round-half-away-from-zero, no contraction. */
XQ_API xq_status xq_quantize_q8(const float *x, int M, int K, void *xq, xq_stream stream);

/* y = x * W^T for a Q4_K weight (xLLM v0.7 article, section 一 and the M
 * template of section B2; batch M read once per weight byte, Agent Telemetry
 * log "批次化 MMVQ").
 *   W  : Q4_K bytes [N][K/256][144], device, read-only.
 *   xq : Q8 activations from xq_quantize_q8(.., M, K, ..), device, read-only.
 *   y  : fp32 [M][N], device, overwritten.
 * Any M >= 0. Dispatch: M <= 8 runs a GEMV that streams every weight byte
 * once for all M tokens; 8 < M <= 64 runs it on 8-token chunks, up to 8 in
 * one launch (they share each weight tile through L2); M > 64 runs the tile
 * kernel (128 weight rows x 128 tokens per CTA on the tcgen05 tensor cores,
 * tile MMQ of section B2), whose operand image xq_quantize_q8 writes for
 * that M. */
XQ_API xq_status xq_matmul_q4k_q8(const void *W, const void *xq, int M, int N, int K,
                           float *y, xq_stream stream);

/* Same for a Q6_K weight (xLLM v0.7 article, section A2: attn_v and ffn_down
 * of the mixed model are Q6_K).
 *   W  : Q6_K bytes [N][K/256][210], device, read-only. Individual blocks are
 *        2-byte aligned (210 is not a multiple of 4); only the base pointer
 *        must be 16-byte aligned.
 * Dispatch at M <= 64, by shape only (never by M): the tensor-core GEMV when
 * rows are 16-byte multiples (K a multiple of 2048); otherwise, with g = 8, 4
 * or 2 the smallest count of consecutive rows whose bytes are a multiple of
 * 16, the tensor-core GEMV over g rows per tensor-map row when N is a
 * multiple of 16g and N >= 8192, else a dp4a GEMV. (xq_layer_mixed, which
 * splits long rows over K in its workspace, takes the tensor-core GEMV
 * whenever N is a multiple of 16g.) M > 64: the tile kernel. */
XQ_API xq_status xq_matmul_q6k_q8(const void *W, const void *xq, int M, int N, int K,
                           float *y, xq_stream stream);

/* Same for a Q8_0 weight (xLLM v0.7 article, section B3 + B4: symmetric
 * int8, one fp16 scale per 32 weights, no min term).
 *   W  : Q8_0 bytes [N][K/32][34] (public GGUF block: fp16 d, then 32 int8
 *        quants), device, read-only. Blocks are 2-byte aligned; only the base
 *        pointer must be 16-byte aligned. K % 256 == 0 (rows of 8-block
 *        groups, 272 bytes each, are 16-byte multiples).
 * M <= 64 runs the tensor-core GEMV; M > 64 the tile kernel (each block's
 * int8 quants as an exact fp16 operand, its scale applied per row to the
 * block's accumulator). */
XQ_API xq_status xq_matmul_q8_0_q8(const void *W, const void *xq, int M, int N, int K,
                            float *y, xq_stream stream);

/* Same for an IQ4_XS weight (Agent Telemetry log, entries on the IQ4_XS
 * batch kernels: 4-bit indices into a 16-entry int8 codebook, a 6-bit scale
 * per 32 weights).
 *   W        : IQ4_XS bytes [N][K/256][136] (public GGUF block: fp16 d,
 *              uint16 scales_h, 4 bytes scales_l, 128 index bytes), device,
 *              read-only; only the base pointer must be 16-byte aligned.
 *              Sub-block j's scale is ls = (4 bits of scales_l at bit 4j) |
 *              (2 bits of scales_h at bit 2j) << 4; weight i of sub-block j
 *              is index byte 16j + i%16, low nibble for i < 16, else high;
 *              w = d * (ls - 32) * codebook[index].
 *   codebook : HOST pointer to the format's 16 int8 values in index order,
 *              read during the call (the launch carries a copy).
 * K must be a multiple of 512 (rows of 16-byte multiples for the tensor
 * map; other K return XQ_ERR_SHAPE). M <= 64 runs the tensor-core GEMV,
 * M > 64 the tile kernel (the codebook lookup done once per weight tile and
 * reused by its 128 tokens). xq_layer_mixed takes IQ4_XS projections with
 * their codebook in xq_proj; the batch-invariant entry points take no
 * codebook and return XQ_ERR_UNSUPPORTED for IQ4_XS. */
XQ_API xq_status xq_matmul_iq4xs_q8(const void *W, const int8_t *codebook, const void *xq, int M, int N,
                             int K, float *y, xq_stream stream);

/* Batch-invariant mode (speculative-decoding verification: the rows of y for
 * a batch of M tokens must equal those of decoding each token alone).
 * xq_matmul_q4k_q8 / _q6k_q8 are invariant for M <= 64 (every token of an
 * 8-token chunk goes through the same operations), but M > 64 switches to
 * the tile kernel, whose fp32 combine runs in another order. These entry
 * points keep the M <= 8 arithmetic for every M: the activations hold the
 * 8-token GEMV image for all ceil(M/8) chunks (xq_q8_bytes_invariant bytes:
 * the M <= 8 layout above with C = ceil(M/8)), and the matmul runs the GEMV
 * chunk by chunk, never split over K. Row m of y is then bit-identical for
 * every M >= m+1, and to xq_matmul_* at M <= 8 on the same activations.
 * Arguments and errors as for xq_quantize_q8 and xq_matmul_*; type is
 * XQ_TYPE_Q4_K, XQ_TYPE_Q6_K or XQ_TYPE_Q8_0. */
XQ_API size_t xq_q8_bytes_invariant(int M, int K);
XQ_API xq_status xq_quantize_q8_invariant(const float *x, int M, int K, void *xq, xq_stream stream);
XQ_API xq_status xq_matmul_invariant(int type, const void *W, const void *xq, int M, int N, int K,
                                     float *y, xq_stream stream);

/* One projection of a transformer layer for xq_layer_mixed. */
typedef struct {
    int type;        /* XQ_TYPE_Q4_K, XQ_TYPE_Q6_K, XQ_TYPE_Q8_0 or
                        XQ_TYPE_IQ4_XS (K a multiple of 512) */
    int N, K;        /* output and input features */
    const void *W;   /* weight bytes, device */
    float *y;        /* fp32 [M][N] output, device */
    int input;       /* index into the layer's inputs[] */
    const int8_t *codebook;  /* IQ4_XS: HOST pointer to its 16 int8 codebook
                                values, read during the call; ignored (may be
                                NULL) for the other types */
} xq_proj;

/* Workspace bytes xq_layer_mixed needs: the Q8 buffers of every input that
 * some projection reads, each rounded up to 256 bytes, then scheduling
 * state: one 256-byte task counter per weight type (Q4_K, Q6_K, Q8_0,
 * IQ4_XS) and, for
 * each projection with more than 24 super-blocks per row that the grouped
 * tensor-core GEMV splits over K across CTAs (M <= 64; above 8 tokens once
 * per 8-token chunk), its arrival counts and partial sums; above 64 tokens,
 * for each projection whose 128 x 128 tiles number fewer than the SMs and
 * whose tile launch is therefore split over K, one arrival count per tile
 * and the [ranges][M][N] fp32 partial sums. 0 on bad arguments. */
XQ_API size_t xq_layer_workspace_bytes(const xq_proj *proj, int n_proj, int n_inputs, int M);

/* One layer's projections with a quant type per tensor (xLLM v0.7 article,
 * section A1: Q/K/V/attn_o/gate/up/down dispatch points; section A2: mixed
 * Q4_K/Q6_K; section C.1: one Q8 quantization shared by every reader).
 *   proj     : host array of n_proj descriptors (read during the call only).
 *   inputs   : host array of n_inputs device pointers, fp32 [M][K_i].
 *              All projections that read input i must agree on K.
 *   workspace: device buffer of at least xq_layer_workspace_bytes() bytes;
 *              receives the Q8 activations, one region per input.
 * Enqueues one quantization per used input and the projections, in order,
 * on `stream`: at M <= 8 one grouped GEMV launch per weight type; at
 * 8 < M <= 64 grouped GEMV launches over (projection, 8-token chunk) pairs,
 * 8 per launch; above 64 tokens the tile kernel per projection, split over
 * K (ranges added in order by the last CTA of each tile: deterministic)
 * where its tiles number fewer than the SMs; only the first of these tile
 * launches waits for the quantizer, the later ones start as the earlier
 * ones drain. */
XQ_API xq_status xq_layer_mixed(const xq_proj *proj, int n_proj,
                         const float *const *inputs, int n_inputs, int M,
                         void *workspace, size_t ws_bytes, xq_stream stream);

/* The SwiGLU feed of a down projection: h = silu(gate) * up, then the Q8
 * quantization of h, in one launch (the step either side of the matmul
 * path in the Agent Telemetry log's dispatch; silu(g) = g / (1 + e^-g)).
 *   gate, up : fp32 [M][K], device (the gate and up projection outputs).
 *   xq       : device buffer of xq_q8_bytes(M, K) bytes, written as by
 *              xq_quantize_q8 from h.
 *   h_out    : optional fp32 [M][K], device: receives h.
 * Each step is one fp32 operation: e = expf(-g) (CUDA's expf, within its
 * documented error bound, not correctly rounded), g / (1 + e) and the
 * product with u rounded to nearest; h then goes through the Q8 rules of
 * xq_quantize_q8. Shape and alignment rules as for xq_quantize_q8. */
XQ_API xq_status xq_silu_mul_quantize_q8(const float *gate, const float *up, int M, int K, void *xq,
                                  float *h_out, xq_stream stream);

/* Workspace bytes of xq_layer_mixed_ffn (0 on bad arguments). */
XQ_API size_t xq_layer_ffn_workspace_bytes(const xq_proj *proj, int n_proj, int n_inputs, int M,
                                    int gate, int up, int down);

/* xq_layer_mixed for a layer whose down projection reads silu(y_gate) * y_up
 * of the same call (gate, up, down: indices into proj; proj[down].input is
 * ignored; N of gate and up must equal K of down). Enqueues, in order on
 * `stream`, first the Q8 quantization of every input, then:
 *  - at M <= 8, when gate and up fall in one grouped GEMV launch (the same
 *    weight type, at most 8 projections of that type in the GEMV group):
 *    the layer's grouped launches, gate and up's type first. The warps that
 *    finish a 32-row block of gate and up compute that block of
 *    h = silu(y_gate) * y_up and its Q8 bytes (the operations of
 *    xq_silu_mul_quantize_q8, bit for bit). A down projection in the same
 *    launch runs after every other task of it and waits for h per
 *    256-feature super-block (bounded; see xq_device_error); one in a later
 *    launch reads h after the grid completes.
 *  - otherwise: the gate and up projections; one xq_silu_mul_quantize_q8
 *    launch on their outputs; every other projection together with down
 *    (grouped GEMV launches as in xq_layer_mixed, split over K like the
 *    layer's; the tile kernel per projection above 64 tokens).
 * Either way the workspace begins with the Q8 buffers of the inputs that
 * are read (in input order, each padded to a multiple of 256 bytes),
 * followed by h's Q8 buffer (xq_q8_bytes(M, K of down) bytes in the layout
 * xq_quantize_q8 writes), which the call leaves there. */
XQ_API xq_status xq_layer_mixed_ffn(const xq_proj *proj, int n_proj, int gate, int up, int down,
                             const float *const *inputs, int n_inputs, int M,
                             void *workspace, size_t ws_bytes, xq_stream stream);

/* Fixed workspace size of xq_layer_mixed_static: 4 MiB per device. */
#define XQ_LAYER_STATIC_SCRATCH_BYTES (4u << 20)

/* xq_layer_mixed for callers that cannot allocate device memory. (The pages
 * have no counterpart: this is an interface convenience, not a step of the
 * method.) Engines that give all device memory to their own pool at
 * start-up, plugins whose host owns the allocator, and latency-critical
 * decode loops that must not call cudaMalloc (it can synchronize the device
 * and fail under memory pressure mid-request) have no way to provide the
 * workspace xq_layer_mixed asks for. This entry point takes the same
 * arguments minus the workspace and uses a fixed device array of
 * XQ_LAYER_STATIC_SCRATCH_BYTES that the library holds on every GPU that
 * loads it, until the process exits. It allocates nothing.
 *  - Requests whose xq_layer_workspace_bytes() exceeds the fixed size return
 *    XQ_ERR_WORKSPACE before anything is enqueued (one decode layer of an
 *    8B-class model at M <= 8 needs about 1.3 MB).
 *  - Every call looks up the array's device address in the current context
 *    (cudaGetSymbolAddress, with the caller's device current); the address
 *    is valid per context and is not cached, so a context created after
 *    cudaDeviceReset gets its own. The first call on a device may load the
 *    module: make it before any stream capture. A failed lookup returns
 *    XQ_ERR_CUDA.
 *  - All calls on a device share the array; the state that must start at
 *    zero is cleared by every call. Calls whose work overlaps on the GPU
 *    (other streams, or unordered host threads) race on it: order them on
 *    one stream or synchronize between them.
 * Results equal xq_layer_mixed's with a caller-provided workspace. */
XQ_API xq_status xq_layer_mixed_static(const xq_proj *proj, int n_proj,
                                const float *const *inputs, int n_inputs, int M,
                                xq_stream stream);

/* Failure detection. Every mbarrier wait of the TMA / tensor-core kernels is
 * bounded (about 2^32 clocks). A wait that runs out records an error code in
 * a device word (the first such wait of a kernel's launches since the last
 * read is the one kept); the kernel then leaves its loops, waits for its own copies
 * and tensor-core work, frees tensor memory and exits, leaving some outputs
 * unwritten although the call that launched it already returned XQ_OK.
 * xq_device_error waits until `stream` is idle, then reads and clears those
 * words. *code_out = 0 if no wait ran out since the last read, else
 * (kernel << 8) | wait: kernel 1 = the warp-level MMA GEMV (M <= 64), 2 =
 * the tile kernel (M > 64); wait = the kernel's number of the wait that gave
 * up (GEMV: 1 the producer waiting for a free stage, 2 a consumer waiting for
 * a full one, 3 a down projection's producer waiting for h in the fused
 * feed of xq_layer_mixed_ffn). Checked builds (the library compiled with
 * -DXQ_CHECK) also test the index, range or 16-byte alignment of each global
 * access whose address comes from nontrivial arithmetic, skip an access that
 * fails and record the site: kernel 9, wait = site (10-16 the GEMV, 20-26
 * the tile kernel, 30-32 the quantizer, 40-43 the dp4a Q6_K GEMV), reported
 * after any wait code. If several kernels recorded one,
 * the lowest kernel number is reported and all are cleared. The reads and
 * writes are synchronous. XQ_ERR_ARG for a null code_out, XQ_ERR_CUDA if the
 * stream or the reads fail. */
XQ_API xq_status xq_device_error(xq_stream stream, unsigned int *code_out);

/* Test hook for the failure detection above: the Q4_K warp-level MMA GEMV
 * (1 <= M <= 8) launched with its producer issuing no stage and every wait
 * limited to about 10^5 clocks, so that the consumers' first waits run out
 * and record their code; y is left unwritten and xq_device_error then
 * reports kernel 1, wait 2. Arguments and errors as xq_matmul_q4k_q8. */
XQ_API xq_status xq_debug_stalled_matmul_q4k(const void *W, const void *xq, int M, int N, int K, float *y,
                                             xq_stream stream);

/* Test hook for wait 3 above: xq_layer_mixed_ffn's fused form (gate and up
 * warps write h's Q8 themselves) with h written but its super-blocks never
 * counted ready. Down's producers wait about 10^5 clocks for each, record
 * kernel 1, wait 3 and leave; down's stage waits are given four times that,
 * so wait 3 is the record xq_device_error reads. Down's y is left unwritten,
 * the other projections are computed as usual. Arguments, workspace and
 * errors as xq_layer_mixed_ffn, plus XQ_ERR_UNSUPPORTED (nothing launched)
 * when the call would not take the fused form. */
XQ_API xq_status xq_debug_stalled_ffn_layer(const xq_proj *proj, int n_proj, int gate, int up, int down,
                                            const float *const *inputs, int n_inputs, int M, void *workspace,
                                            size_t ws_bytes, xq_stream stream);

/* Test hook of checked builds: the Q4_K GEMV (2 <= M <= 8, y [M][N] fully
 * allocated) launched with its y extent declared one token row short, so
 * that the stores of token M-1 fail their bounds check (site 10), are
 * skipped (that row of y is left as it was) and are recorded for
 * xq_device_error. Normal builds: XQ_ERR_UNSUPPORTED, nothing launched. */
XQ_API xq_status xq_debug_check_probe(const void *W, const void *xq, int M, int N, int K, float *y,
                                      xq_stream stream);

/* Test hooks: the same matmul kernels with their exact int32 sub-block sums
 * written out instead of only consumed.
 *   Q4_K: isum int32 [M][N][K/32], sub-block j of super-block b at 8b+j.
 *   Q6_K: isum int32 [M][N][K/16], 16-weight scale group g at 16b+g.
 * Also writes y like the matmul. M must be in 1..8. */
XQ_API xq_status xq_debug_isums_q4k(const void *W, const void *xq, int M, int N, int K,
                             float *y, int32_t *isum, xq_stream stream);
XQ_API xq_status xq_debug_isums_q6k(const void *W, const void *xq, int M, int N, int K,
                             float *y, int32_t *isum, xq_stream stream);
/* Q8_0: isum int32 [M][N][K/32], block j at index j. */
XQ_API xq_status xq_debug_isums_q8_0(const void *W, const void *xq, int M, int N, int K,
                              float *y, int32_t *isum, xq_stream stream);
/* IQ4_XS: isum int32 [M][N][K/32] (sums of codebook value x Q8 quant),
 * sub-block j of super-block b at 8b+j. */
XQ_API xq_status xq_debug_isums_iq4xs(const void *W, const int8_t *codebook, const void *xq, int M,
                               int N, int K, float *y, int32_t *isum, xq_stream stream);

/* Test hook of the tile kernel (M > 64): the same launch as the matmul of
 * `type` (8, 12, 14 or 23; IQ4_XS with its codebook, K a multiple of 512),
 * writing y and, into sums int32 [M][N][K/32], each 32-block's exact integer
 * as the kernel accumulates it before any scale is applied:
 *   Q4_K   sc_j * isum_j              (the 6-bit scale is folded into the operand)
 *   Q6_K   s_2p * isum_2p + s_2p+1 * isum_2p+1   (both 16-weight groups)
 *   Q8_0   isum_j
 *   IQ4_XS (ls_j - 32) * isum_j
 * with isum the integer sub-block sums of xq_debug_isums_*. XQ_ERR_UNSUPPORTED
 * for M <= 64 (those token counts run the GEMV, whose hooks are above). */
XQ_API xq_status xq_debug_tile_sums(int type, const void *W, const int8_t *codebook, const void *xq, int M,
                                    int N, int K, float *y, int32_t *sums, xq_stream stream);

/* Timing hook: the matmul launches of xq_layer_mixed alone, without its
 * quantize launch, reading the Q8 activations that the last xq_layer_mixed
 * call with the same proj, n_proj, n_inputs and M left in `workspace`. Each
 * launch leaves the workspace's scheduling state (task counters, split-K
 * arrival counts) at zero, as it found it, so the call can be repeated; it
 * rewrites every projection's y with the same values, bit for bit. Errors as
 * xq_layer_mixed (XQ_ERR_WORKSPACE if ws_bytes is below
 * xq_layer_workspace_bytes). The result is undefined if the workspace does
 * not hold the state of such a call. */
XQ_API xq_status xq_debug_layer_matmuls(const xq_proj *proj, int n_proj, int n_inputs, int M, void *workspace,
                                        size_t ws_bytes, xq_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* XQ_H */
