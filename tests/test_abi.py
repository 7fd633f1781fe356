"""Host-side checks of the C ABI (no GPU needed, no compute calls).

libxq.so must load and export every entry point include/xq.h declares; the
size helpers and the argument checks that return before any CUDA call are
exercised directly.
"""
import ctypes
import os
import re

import pytest

from gguf_quant_integer_gb300 import build as xqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    xqbuild.build()
    from gguf_quant_integer_gb300 import xq
    return xq.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "xq.h")).read()
    return sorted(set(re.findall(r"XQ_API\s+[\w\s\*]*?\b(xq_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    from gguf_quant_integer_gb300 import xq
    decl = declared_symbols()
    assert len(decl) >= 10
    assert sorted(xq.SYMBOLS) == decl
    for name in decl:
        assert hasattr(L, name), name


def test_sizes(L):
    from gguf_quant_integer_gb300 import xq
    def layout(M, K):
        base = -(-int(1.25 * M * K) // 256) * 256
        if M <= 64:  # GEMV operand image: 18 bytes per feature per 8-token chunk
            return base + 18 * K * (-(-M // 8))
        # tile image: one 77,824-byte record per 128-token tile and super-block
        return base + 77824 * (K // 256) * (-(-M // 128))
    for M, K in ((1, 2048), (8, 4096), (9, 256), (64, 512), (65, 512), (129, 1536), (512, 12288), (0, 256)):
        assert xq.q8_bytes(M, K) == layout(M, K)
    assert L.xq_q8_bytes(1, 100) == 0
    assert L.xq_q8_bytes(8, 288) == 3072 + 18 * 288  # the GEMV image needs K % 32 only (no tcb then)
    assert L.xq_q8_bytes(64, 288) > 0
    assert L.xq_q8_bytes(65, 288) == 0    # the tile image is per 256-feature super-block
    # batch-invariant layout: the GEMV image for every 8-token chunk, any M
    for M, K in ((1, 2048), (8, 4096), (9, 256), (129, 1536), (512, 12288), (0, 256)):
        base = -(-int(1.25 * M * K) // 256) * 256
        assert xq.q8_bytes_invariant(M, K) == base + 18 * K * (-(-M // 8))
    assert L.xq_q8_bytes_invariant(9, 288) > 0
    assert L.xq_q8_bytes_invariant(1, 100) == 0
    assert xq.weight_bytes(12, 256, 2048) == 256 * 8 * 144
    assert xq.weight_bytes(8, 256, 2048) == 256 * 64 * 34   # Q8_0: 34 bytes per 32 weights
    assert xq.weight_bytes(14, 1024, 4096) == 1024 * 16 * 210
    assert xq.weight_bytes(99, 1, 256) == 0
    assert xq.weight_bytes(12, 1, 300) == 0


def test_status_strings(L):
    for code in range(7):
        assert L.xq_status_str(code)
    assert L.xq_status_str(99) == b"unknown status"


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced


def test_shape_and_argument_errors_return_before_launch(L):
    P = ctypes.c_void_p
    # K not a multiple of 256, negative sizes
    assert L.xq_matmul_q4k_q8(P(FAKE), P(FAKE), 1, 4, 300, P(FAKE), None) == 2
    assert L.xq_matmul_q6k_q8(P(FAKE), P(FAKE), -1, 4, 256, P(FAKE), None) == 2
    assert L.xq_matmul_q4k_q8(P(FAKE), P(FAKE), 1, -4, 256, P(FAKE), None) == 2
    assert L.xq_quantize_q8(P(FAKE), 1, 0, P(FAKE), None) == 2
    # empty products are no-ops
    assert L.xq_matmul_q4k_q8(None, None, 0, 4, 256, None, None) == 0
    assert L.xq_matmul_q6k_q8(None, None, 2, 0, 256, None, None) == 0
    assert L.xq_quantize_q8(None, 0, 256, None, None) == 0
    # null pointers
    assert L.xq_matmul_q4k_q8(None, P(FAKE), 1, 4, 256, P(FAKE), None) == 1
    assert L.xq_quantize_q8(P(FAKE), 1, 256, None, None) == 1
    assert L.xq_debug_isums_q4k(P(FAKE), P(FAKE), 1, 4, 256, P(FAKE), None, None) == 1
    # misaligned pointers
    assert L.xq_matmul_q4k_q8(P(FAKE + 8), P(FAKE), 1, 4, 256, P(FAKE), None) == 3
    assert L.xq_matmul_q6k_q8(P(FAKE), P(FAKE + 4), 1, 4, 256, P(FAKE), None) == 3
    assert L.xq_quantize_q8(P(FAKE + 2), 1, 256, P(FAKE), None) == 3
    # the isum hook is limited to one launch of at most 8 tokens
    assert L.xq_debug_isums_q6k(P(FAKE), P(FAKE), 9, 4, 256, P(FAKE), P(FAKE), None) == 6


def test_layer_argument_errors(L):
    from gguf_quant_integer_gb300 import xq
    P = ctypes.c_void_p

    def projs(*specs):
        return xq._proj_array([(t, n, k, None, None, i) for (t, n, k, i) in specs]), len(specs)

    arr, n = projs((12, 16, 512, 0), (14, 8, 512, 0), (12, 16, 1024, 1))
    need = L.xq_layer_workspace_bytes(arr, n, 2, 4)
    # Q8 buffers, then one 256-byte task counter per weight type (Q4_K, Q6_K,
    # Q8_0, IQ4_XS; no split at these K)
    expect = sum(((xq.q8_bytes(4, k) + 255) // 256) * 256 for k in (512, 1024)) + 4 * 256
    assert need == expect
    # mismatched K on one input
    bad, nb = projs((12, 16, 512, 0), (12, 16, 768, 0))
    assert L.xq_layer_workspace_bytes(bad, nb, 1, 4) == 0
    ins = (ctypes.c_void_p * 2)(FAKE, FAKE)
    assert L.xq_layer_mixed(bad, nb, ins, 1, 4, P(FAKE), 1 << 20, None) == 2
    # unknown type, input index out of range
    bad, nb = projs((13, 16, 512, 0))
    assert L.xq_layer_mixed(bad, nb, ins, 1, 4, P(FAKE), 1 << 20, None) == 1
    bad, nb = projs((12, 16, 512, 3))
    assert L.xq_layer_mixed(bad, nb, ins, 2, 4, P(FAKE), 1 << 20, None) == 1
    # workspace too small (checked before the projections' pointers)
    assert L.xq_layer_mixed(arr, n, ins, 2, 4, P(FAKE), need - 1, None) == 4
    # missing weight pointer
    assert L.xq_layer_mixed(arr, n, ins, 2, 4, P(FAKE), need, None) == 1


def test_layer_matmuls_timing_hook_argument_errors(L):
    """xq_debug_layer_matmuls validates like xq_layer_mixed (it takes no
    inputs: the activations are the workspace's)."""
    from gguf_quant_integer_gb300 import xq
    P = ctypes.c_void_p
    specs = [(12, 16, 512, 0), (14, 8, 512, 0), (12, 16, 1024, 1)]
    arr = xq._proj_array([(t, n, k, None, None, i) for (t, n, k, i) in specs])
    need = L.xq_layer_workspace_bytes(arr, 3, 2, 4)
    assert L.xq_debug_layer_matmuls(arr, 3, 2, 4, P(FAKE), need - 1, None) == 4     # workspace too small
    assert L.xq_debug_layer_matmuls(arr, 3, 2, 4, None, need, None) == 1            # no workspace
    assert L.xq_debug_layer_matmuls(arr, 3, 2, 4, P(FAKE + 8), need, None) == 3     # misaligned
    assert L.xq_debug_layer_matmuls(arr, 3, 2, 4, P(FAKE), need, None) == 1         # no weight pointers
    assert L.xq_debug_layer_matmuls(arr, 3, 1, 4, P(FAKE), need, None) == 1         # input 1 out of range
    assert L.xq_debug_layer_matmuls(arr, 3, 2, 0, None, 0, None) == 0               # M = 0: nothing to do


def test_check_probe_needs_the_checked_build(L):
    """The normal library refuses the checked build's probe before any CUDA call."""
    P = ctypes.c_void_p
    assert L.xq_debug_check_probe(P(FAKE), P(FAKE), 4, 64, 512, P(FAKE), None) == 6


def test_q8_0_entry_points_reject_before_launch(L):
    """Q8_0 shape and argument errors are refused before anything is
    enqueued; the layer sizes Q8_0 at every M."""
    from gguf_quant_integer_gb300 import xq
    P = ctypes.c_void_p
    assert L.xq_matmul_q8_0_q8(P(FAKE), P(FAKE), 8, 16, 300, P(FAKE), None) == 2
    assert L.xq_debug_isums_q8_0(P(FAKE), P(FAKE), 2, 16, 256, P(FAKE), None, None) == 1
    assert L.xq_debug_isums_q8_0(P(FAKE), P(FAKE), 9, 16, 256, P(FAKE), P(FAKE), None) == 6  # hook: M <= 8
    arr = xq._proj_array([(8, 16, 512, None, None, 0)])
    for M in (8, 64, 65, 512):
        assert L.xq_layer_workspace_bytes(arr, 1, 1, M) > 0


def test_ffn_entry_points_reject_before_launch(L):
    from gguf_quant_integer_gb300 import xq
    P = ctypes.c_void_p
    # gate, up: N = 512; down: K = 512 -> N = 256
    specs = [(12, 512, 256, 0), (12, 512, 256, 0), (12, 256, 512, 1)]
    arr = xq._proj_array([(t, n, k, None, None, i) for (t, n, k, i) in specs])
    good = L.xq_layer_ffn_workspace_bytes(arr, 3, 1, 4, 0, 1, 2)
    assert good > L.xq_layer_workspace_bytes(arr, 2, 1, 4)   # + h's Q8 buffer and down's state
    assert L.xq_layer_ffn_workspace_bytes(arr, 3, 1, 4, 0, 0, 2) == 0   # gate == up
    assert L.xq_layer_ffn_workspace_bytes(arr, 3, 1, 4, 0, 1, 3) == 0   # index out of range
    bad = xq._proj_array([(t, n, k, None, None, i) for (t, n, k, i) in [(12, 512, 256, 0), (12, 384, 256, 0),
                                                                      (12, 256, 512, 1)]])
    assert L.xq_layer_ffn_workspace_bytes(bad, 3, 1, 4, 0, 1, 2) == 0   # gate and up N differ
    ins = (ctypes.c_void_p * 1)(FAKE)
    assert L.xq_layer_mixed_ffn(bad, 3, 0, 1, 2, ins, 1, 4, P(FAKE), 1 << 20, None) == 2
    assert L.xq_layer_mixed_ffn(arr, 3, 0, 1, 2, ins, 1, 4, P(FAKE), good - 1, None) == 4
    # the wait-3 hook: the same checks; the unfused form (M > 8) is not hooked
    stalled = L.xq_debug_stalled_ffn_layer
    assert stalled(bad, 3, 0, 1, 2, ins, 1, 4, P(FAKE), 1 << 20, None) == 2
    assert stalled(arr, 3, 0, 1, 2, ins, 1, 4, P(FAKE), good - 1, None) == 4
    assert stalled(arr, 3, 0, 1, 2, ins, 1, 20, P(FAKE), 1 << 30, None) == 6
    assert L.xq_silu_mul_quantize_q8(P(FAKE), P(FAKE), 2, 300, P(FAKE), None, None) == 2
    assert L.xq_silu_mul_quantize_q8(P(FAKE + 4), P(FAKE), 2, 256, P(FAKE), None, None) == 3
    assert L.xq_silu_mul_quantize_q8(None, P(FAKE), 2, 256, P(FAKE), None, None) == 1


def test_iq4xs_entry_points_reject_before_launch(L):
    from gguf_quant_integer_gb300 import xq
    P = ctypes.c_void_p
    cb = (ctypes.c_int8 * 16)(*range(-8, 8))
    assert xq.weight_bytes(23, 10, 1024) == 10 * 4 * 136
    assert L.xq_matmul_iq4xs_q8(P(FAKE), cb, P(FAKE), 2, 16, 768, P(FAKE), None) == 2   # K % 512
    assert L.xq_debug_isums_iq4xs(P(FAKE), cb, P(FAKE), 9, 16, 1024, P(FAKE), P(FAKE), None) == 6  # hook: M <= 8
    assert L.xq_matmul_iq4xs_q8(P(FAKE), None, P(FAKE), 2, 16, 1024, P(FAKE), None) == 1
    assert L.xq_matmul_iq4xs_q8(P(FAKE + 8), cb, P(FAKE), 2, 16, 1024, P(FAKE), None) == 3
    assert L.xq_matmul_iq4xs_q8(None, None, None, 0, 16, 1024, None, None) == 0         # empty
    assert L.xq_debug_isums_iq4xs(P(FAKE), cb, P(FAKE), 2, 16, 1024, P(FAKE), None, None) == 1
    # the layer takes the codebook through xq_proj; the batch-invariant matmul has none
    import numpy as np
    ins = (ctypes.c_void_p * 1)(FAKE)
    arr = xq._proj_array([(23, 16, 1024, None, None, 0)])
    assert L.xq_layer_mixed(arr, 1, ins, 1, 4, P(FAKE), 1 << 20, None) == 1      # no codebook
    arr = xq._proj_array([(23, 16, 768, None, None, 0, np.arange(-8, 8, dtype=np.int8))])
    assert L.xq_layer_mixed(arr, 1, ins, 1, 4, P(FAKE), 1 << 20, None) == 2      # K % 512
    arr = xq._proj_array([(23, 16, 1024, None, None, 0, np.arange(-8, 8, dtype=np.int8))])
    assert L.xq_layer_workspace_bytes(arr, 1, 1, 4) > 0
    assert L.xq_matmul_invariant(23, P(FAKE), P(FAKE), 2, 16, 1024, P(FAKE), None) == 6


def test_layer_workspace_for_chunked_split(L):
    """8 < M <= 64: every (projection, 8-token chunk) pair of a row longer
    than 24 super-blocks gets its own arrival counts and partial sums, sized
    as the launcher consumes them."""
    from gguf_quant_integer_gb300 import xq

    def r256(b):
        return -(-b // 256) * 256

    def split_bytes(N, nch):
        rb = -(-N // 64)
        return r256(rb * 4 * 4) + r256(nch * 8 * rb * 64 * 4)

    # q: 16 super-blocks (no split); down: 56 super-blocks (4 chunks of 14)
    specs = [(12, 300, 4096, 0), (12, 130, 14336, 1)]
    arr = xq._proj_array([(t, n, k, None, None, i) for (t, n, k, i) in specs])
    for M in (9, 20, 64):
        chunks = -(-M // 8)
        q8 = r256(xq.q8_bytes(M, 4096)) + r256(xq.q8_bytes(M, 14336))
        want = q8 + 4 * 256 + chunks * split_bytes(130, 4)
        assert L.xq_layer_workspace_bytes(arr, 2, 2, M) == want, M
    # above 64 tokens (the tile kernel): where a projection's 128 x 128 tiles
    # leave the 152 SMs idle, K ranges per tile (at most 8, at most one per
    # two super-blocks), with an arrival count per tile and [ranges][M][N]
    # partial sums
    def tile_split_bytes(N, K, M):
        tiles = -(-N // 128) * -(-M // 128)
        splits = 1 if tiles >= 152 else max(1, min(152 // tiles, (K // 256) // 2, 8))
        return 0 if splits == 1 else r256(tiles * 4) + r256(splits * M * N * 4)
    for M in (80, 200, 512):
        q8 = r256(xq.q8_bytes(M, 4096)) + r256(xq.q8_bytes(M, 14336))
        want = q8 + 4 * 256 + tile_split_bytes(300, 4096, M) + tile_split_bytes(130, 14336, M)
        assert L.xq_layer_workspace_bytes(arr, 2, 2, M) == want, M
    # 80 tokens: 8 ranges for both projections (3 and 2 tiles)
    assert tile_split_bytes(300, 4096, 80) == 256 + 8 * 80 * 300 * 4


def test_failure_detection_entry_points_reject_before_launch(L):
    P = ctypes.c_void_p
    assert L.xq_device_error(None, None) == 1
    assert L.xq_debug_stalled_matmul_q4k(P(FAKE), P(FAKE), 9, 16, 256, P(FAKE), None) == 2   # M <= 8
    assert L.xq_debug_stalled_matmul_q4k(P(FAKE), P(FAKE), 1, 16, 300, P(FAKE), None) == 2   # K % 256
    assert L.xq_debug_stalled_matmul_q4k(None, P(FAKE), 1, 16, 256, P(FAKE), None) == 1
    assert L.xq_debug_stalled_matmul_q4k(P(FAKE + 4), P(FAKE), 1, 16, 256, P(FAKE), None) == 3
