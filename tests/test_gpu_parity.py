"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Rules (from the method's statement and its correctness lessons):
- Q8 bytes, d8 and s8 are bit-exact;
- per-sub-block int32 sums are bit-exact;
- y satisfies |y_gpu - y_ref| <= 1e-5 * sum|scaled sub-block terms| + 1e-7
  (fp32 combine against the fp64 oracle);
- outputs are poisoned with NaN before every launch, and the error must be
  nonzero somewhere (an exact match against an fp64 oracle would mean the
  kernel did not run; Agent Telemetry log, "一顆什麼都沒算的 kernel").
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gguf_quant_integer_gb300 import synth
from tile_image import expected_tile_image

pytestmark = pytest.mark.gpu

TOL_REL = 1e-5
TOL_ABS = 1e-7


@pytest.fixture(scope="module")
def xq():
    from gguf_quant_integer_gb300 import build, xq as _xq
    build.build()
    _xq.lib()
    # the oracle shares output rows over the host's cores (results do not
    # depend on the count), so full-size layers are checked on every row
    oracle.set_threads(os.cpu_count() or 1)
    yield _xq
    oracle.set_threads(1)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def poisoned(M, N):
    return torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")


def gpu_q8(xq, x):
    M, K = x.shape
    buf = xq.quantize_q8(dev(x))
    torch.cuda.synchronize()
    qs, d8, s8 = (t.cpu().numpy() for t in xq.q8_views(buf, M, K))
    return buf, qs, d8, s8


def assert_q8_exact(xq, x):
    buf, qs, d8, s8 = gpu_q8(xq, x)
    rq, rd, rs = oracle.quantize_q8(x)
    assert np.array_equal(qs, rq)
    assert np.array_equal(d8.view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(s8.view(np.uint32), rs.view(np.uint32))
    return buf, rq, rd


def check_y(y_gpu, y_ref, absterm):
    y_gpu = y_gpu.astype(np.float64)
    assert np.all(np.isfinite(y_gpu)), "an output was not written"
    err = np.abs(y_gpu - y_ref)
    bound = TOL_REL * absterm + TOL_ABS
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} outputs out of tolerance; worst ratio {np.max(err / bound):.3g}"
    return float(err.max())


# ------------------------------------------------------------ Q8

def test_quantize_bitexact_workload_inputs(xq):
    for name in ("tiny-gemv", "qwen2.5-1.5b-layer", "qwen3-8b-mixed-layer"):
        wl = synth.WORKLOADS[name]
        for x in synth.gen_layer_inputs(wl, max(wl.ms)):
            assert_q8_exact(xq, x)
    wl = synth.WORKLOADS["qwen3-8b-ffn-prefill512"]
    for x in synth.gen_layer_inputs(wl, 512):
        assert_q8_exact(xq, x)


PERM = [0, 2, 1, 3, 4, 6, 5, 7]


def expected_operand_image(qs, d8, s8):
    """The frag / fsc regions restated from their definition in include/xq.h."""
    M, K = qs.shape
    C = -(-M // 8)
    nsub = K // 32
    qp = np.zeros((8 * C, K), np.int8)
    qp[:M] = qs
    dp = np.zeros((8 * C, nsub), np.float32)
    sp = np.zeros((8 * C, nsub), np.float32)
    dp[:M], sp[:M] = d8, s8
    frag = np.zeros((C, nsub, 32, 8), np.float16)
    fsc = np.zeros((C, nsub, 4, 4), np.float32)
    for c in range(C):
        for n in range(8):
            for t in range(4):
                pos = 8 * t + np.array(PERM)
                frag[c, :, 4 * n + t, :] = qp[8 * c + n].reshape(nsub, 32)[:, pos].astype(np.float16)
        for t in range(4):
            fsc[c, :, t, 0] = dp[8 * c + 2 * t]
            fsc[c, :, t, 1] = dp[8 * c + 2 * t + 1]
            fsc[c, :, t, 2] = sp[8 * c + 2 * t]
            fsc[c, :, t, 3] = sp[8 * c + 2 * t + 1]
    return frag, fsc


@pytest.mark.parametrize("M,K", [(1, 256), (3, 2048), (8, 4096), (20, 512), (64, 256)])
def test_quantize_operand_image(xq, M, K):
    x = synth.gen_x(300 + M, M, K)
    buf, rq, rd = assert_q8_exact(xq, x)
    rs = oracle.quantize_q8(x)[2]
    frag, fsc = expected_operand_image(rq, rd, rs)
    raw = buf.cpu().numpy()
    F = -(-int(1.25 * M * K) // 256) * 256
    C = -(-M // 8)
    got_f = raw[F:F + 16 * C * K].view(np.float16).reshape(frag.shape)
    got_s = raw[F + 16 * C * K:F + 18 * C * K].view(np.float32).reshape(fsc.shape)
    assert np.array_equal(got_f.view(np.uint16), frag.view(np.uint16))
    assert np.array_equal(got_s.view(np.uint32), fsc.view(np.uint32))
    assert raw.size == F + 18 * C * K


@pytest.mark.parametrize("M,K", [(65, 256), (100, 1536), (130, 512)])
def test_quantize_tile_image(xq, M, K):
    x = synth.gen_x(310 + M, M, K)
    buf, rq, rd = assert_q8_exact(xq, x)
    rs = oracle.quantize_q8(x)[2]
    want = expected_tile_image(rq, rd, rs)
    raw = buf.cpu().numpy()
    F = -(-int(1.25 * M * K) // 256) * 256
    got = raw[F:F + want.size].reshape(want.shape)
    assert raw.size == F + want.size
    assert np.array_equal(got, want)


def test_quantize_edge_blocks(xq):
    K = 512
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, K)).astype(np.float32)
    x[0, 0:32] = 0.0                                   # all-zero block
    x[0, 32:64] = -0.0
    x[1, 0:32] = 0.0
    x[1, 0], x[1, 1], x[1, 2], x[1, 3] = 127.0, 2.5, -2.5, 0.5   # exact ties (d8 = 1)
    x[1, 32:64] = np.float32(3e-41)                    # subnormal inputs
    x[2] *= np.float32(1e30)                           # huge scale
    x[3] *= np.float32(1e-30)                          # tiny scale
    x[4, :] = np.float32(0.3)                          # constant blocks
    x[5, ::2] *= -1
    x[5, 100] = np.float32(1e6)                        # one dominant value
    assert_q8_exact(xq, x)


# ------------------------------------------------------------ matmul

def run_and_check(xq, qtype, N, K, M, wseed, xseed, want_isum=True):
    W = synth.gen_weight(qtype, wseed, N, K)
    x = synth.gen_x(xseed, M, K)
    return check_matmul(xq, qtype, W, x, want_isum)


def check_matmul(xq, qtype, W, x, want_isum=True):
    """One xq_matmul (and, for M <= 8, the isum hook) against the oracle."""
    M, K = x.shape
    N = W.shape[0]
    buf, rq, rd = assert_q8_exact(xq, x)
    y_ref, ab, isum_ref = oracle.matmul(qtype, W, rq, rd, K, want_isum=want_isum and M <= 8)
    Wd = dev(W.reshape(-1))
    y = poisoned(M, N)
    if want_isum and M <= 8:
        per = K // 16 if qtype == synth.Q6_K else K // 32
        isum = torch.full((M, N, per), -(2 ** 31), dtype=torch.int32, device="cuda")
        xq.debug_isums(qtype, Wd, buf, M, N, K, y=y, isum=isum)
        torch.cuda.synchronize()
        assert np.array_equal(isum.cpu().numpy(), isum_ref)
        y_isum = y.cpu().numpy()
        y = poisoned(M, N)
        xq.matmul(qtype, Wd, buf, M, N, K, y=y)
        torch.cuda.synchronize()
        # the test hook is the same kernel: its y matches the plain launch bit for bit
        assert np.array_equal(y.cpu().numpy().view(np.uint32), y_isum.view(np.uint32))
    else:
        xq.matmul(qtype, Wd, buf, M, N, K, y=y)
        torch.cuda.synchronize()
    return check_y(y.cpu().numpy(), y_ref, ab)


def test_tiny_gemv(xq):
    wl = synth.WORKLOADS["tiny-gemv"]
    p = wl.projs[0]
    err = run_and_check(xq, synth.Q4_K, p.N, p.K, 1, wl.weight_seed(0, 0), wl.x_seed(1))
    assert err > 0.0


SHAPES = [(1, 256), (5, 512), (37, 1536), (64, 4096), (130, 8960), (257, 2304), (3, 12288)]


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("N,K", SHAPES)
def test_shapes_all_m(xq, qtype, N, K):
    errs = [run_and_check(xq, qtype, N, K, M, 31 * N + K + qtype, 7 * M + N) for M in range(1, 9)]
    assert max(errs) > 0.0


# Q6_K rows that are not 16-byte multiples on the tensor-core GEMV: the
# tensor map takes 2^gs consecutive rows per map row (g = 8 for an odd
# super-block count, 4 for 2 mod 4, 2 for 4 mod 8), N a multiple of 16g. A
# single matmul takes that path from 128 row blocks of 64 (N >= 8192); the
# narrower shapes above run on the dp4a kernel. The layer test below takes it
# at N = 256 and 1536 with split-K.
Q6K_GROUPED = [(8192, 2304), (8192, 1536), (8192, 1024), (8448, 4864)]


@pytest.mark.parametrize("N,K", Q6K_GROUPED)
def test_q6k_grouped_rows_all_m(xq, N, K):
    errs = [run_and_check(xq, synth.Q6_K, N, K, M, 61 * N + K, 13 * M + N) for M in range(1, 9)]
    assert max(errs) > 0.0


@pytest.mark.parametrize("M", [1, 2, 8, 20, 80])
def test_qwen25_q4km_layer(xq, M):
    # Q6_K attn_v (K = 1536) and ffn_down (K = 8960, split over K at M <= 8)
    # beside Q4_K, through every path by M
    assert layer_check(xq, synth.WORKLOADS["qwen2.5-1.5b-q4km-layer"], M) > 0


# Q8_0 above 64 tokens: the tile kernel with per-block row scales, ragged N
# and M, every int8 value as a quant against +-1000 activations.
@pytest.mark.parametrize("N,K,M", [(130, 1024, 65), (37, 256, 200), (300, 2048, 129)])
def test_q8_0_tile(xq, N, K, M):
    assert run_and_check(xq, synth.Q8_0, N, K, M, 51 * N + K, 5 * M + K, want_isum=False) > 0.0


def test_q8_0_tile_extremes(xq):
    N, K, M = 64, 1024, 96
    W = synth.gen_q8_0(5, N, K).reshape(N, K // 32, 34)
    W[:, :, 2:] = (np.arange(N * (K // 32) * 32) % 256).astype(np.uint8).reshape(N, K // 32, 32)
    W[:, :, 0:2] = np.frombuffer(np.float16(0.25).tobytes(), np.uint8)
    x = synth.gen_x(6, M, K)
    x[0] = 1000.0
    x[1, ::2] = -1000.0
    check_matmul(xq, synth.Q8_0, W.reshape(N, -1), x, want_isum=False)


# 8 < M <= 64: the GEMV over 8-token chunks (several chunks per launch).
@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K, synth.Q8_0])
@pytest.mark.parametrize("M", [9, 13, 40, 64])
def test_more_than_eight_tokens(xq, qtype, M):
    run_and_check(xq, qtype, 48, 2048, M, 900 + M, 901 + M, want_isum=False)
    run_and_check(xq, qtype, 130, 4096, M, 910 + M, 911 + M, want_isum=False)


# M > 64: the tcgen05 tile kernel. Ragged N and M, one-super-block rows, and
# Q6_K rows whose byte length is not a multiple of 16 (row windows start at
# varying offsets; for (37, 256) and (130, 1536) the last window is cut at
# the end of the weight buffer, and N not a multiple of 2^gs keeps the copy
# per row; (128, 2304), (48, 1024), (64, 1536), (64, 256) and (136, 8960)
# take the grouped tensor-map view with 8, 2, 4, 8 and 8 rows per map row,
# (64, 256) with its last windows running past the end of the buffer).
TILE_SHAPES = [(37, 256, 70), (130, 1536, 200), (300, 4096, 129), (128, 2304, 65), (48, 1024, 128), (64, 1536, 96),
               (64, 256, 80), (136, 8960, 100)]


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("N,K,M", TILE_SHAPES)
def test_tile_shapes(xq, qtype, N, K, M):
    assert run_and_check(xq, qtype, N, K, M, 41 * N + K + qtype, 3 * M + K, want_isum=False) > 0.0


@pytest.mark.parametrize("M,K", [(4, 1024), (4, 2048), (70, 1024)])
def test_q6k_full_range_scales(xq, M, K):
    # GGUF Q6_K scales span int8; |s| > 64 takes the two-operand form in the
    # tile kernel. Rows 0..63 keep |s| <= 64 so that a tile mixes both forms.
    # At M = 4, K = 1024 runs the dp4a GEMV and K = 2048 the tensor-core GEMV.
    N = 160
    W = synth.gen_q6k(77, N, K)
    blocks = W.reshape(N, K // 256, 210)
    rng = np.random.default_rng(78)
    sc = rng.integers(-128, 128, size=(N, K // 256, 16)).astype(np.int8)
    sc[:64] = np.clip(sc[:64], -64, 64)
    sc[64, 0, :6] = (-128, 127, -127, 65, -65, 64)
    blocks[:, :, 192:208] = sc.view(np.uint8)
    x = synth.gen_x(79, M, K)
    assert check_matmul(xq, synth.Q6_K, W, x) > 0.0


def test_empty_products_leave_outputs_untouched(xq):
    W = dev(synth.gen_q4k(1, 4, 256).reshape(-1))
    buf = xq.quantize_q8(dev(synth.gen_x(2, 1, 256)))
    y = poisoned(1, 4)
    xq.matmul(synth.Q4_K, W, buf, 0, 4, 256, y=y)
    xq.matmul(synth.Q6_K, W, buf, 1, 0, 256, y=y)
    torch.cuda.synchronize()
    assert torch.isnan(y).all()


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K])
def test_row_split_is_bit_identical(xq, qtype):
    # Output rows are independent: computing a row slice of W gives the same
    # bits as the full launch (the N-sharding a multi-GPU split would use).
    N, K, M = 300, 4096, 8
    W = synth.gen_weight(qtype, 55, N, K)
    buf = xq.quantize_q8(dev(synth.gen_x(56, M, K)))
    full = poisoned(M, N)
    xq.matmul(qtype, dev(W.reshape(-1)), buf, M, N, K, y=full)
    parts = []
    for lo, hi in ((0, 77), (77, 128), (128, 300)):
        yp = poisoned(M, hi - lo)
        xq.matmul(qtype, dev(W[lo:hi].reshape(-1)), buf, M, hi - lo, K, y=yp)
        parts.append(yp)
    torch.cuda.synchronize()
    cat = torch.cat(parts, dim=1)
    assert torch.equal(cat.view(torch.int32), full.view(torch.int32))


# ------------------------------------------------------------ layers

def layer_check(xq, wl, M, layer=0, rows=None, codebooks=None):
    """Run one layer through xq_layer_mixed and check every projection
    (all rows, or `rows` sampled rows per projection) against the oracle.
    codebooks: per projection, the IQ4_XS codebook (None for other types)."""
    weights = synth.gen_layer_weights(wl, layer)
    inputs = synth.gen_layer_inputs(wl, M, layer)
    codebooks = codebooks or [None] * len(wl.projs)
    L = xq.Layer(wl.projs, weights, M, codebooks=codebooks)
    for y in L.y:
        y.fill_(float("nan"))
    L.forward([dev(x) for x in inputs])
    torch.cuda.synchronize()
    # the workspace holds each input's Q8 buffer: bit-exact
    q8 = [oracle.quantize_q8(x) for x in inputs]
    errs = []
    rng = np.random.default_rng(layer * 1000 + M)
    for t, p in enumerate(wl.projs):
        rq, rd, _ = q8[p.input]
        W = weights[t]
        sel = np.arange(p.N) if rows is None else np.sort(rng.choice(p.N, size=min(rows, p.N), replace=False))
        y_ref, ab, _ = oracle.matmul(p.qtype, W[sel], rq, rd, p.K, codebook=codebooks[t])
        y = L.y[t].cpu().numpy()[:, sel]
        errs.append(check_y(y, y_ref, ab))
    return max(errs)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 33])
def test_qwen25_layer_full(xq, M):
    assert layer_check(xq, synth.WORKLOADS["qwen2.5-1.5b-layer"], M) > 0


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_qwen3_mixed_layer(xq, M):
    assert layer_check(xq, synth.WORKLOADS["qwen3-8b-mixed-layer"], M) > 0


# Ragged projections whose rows are long enough to be split over K: output
# counts that leave partial 16-row groups and empty warps in the last task,
# a Q6_K and a Q8_0 projection next to Q4_K, and few enough tasks that the
# chunk length drops to 8 super-blocks.
RAGGED_SPLIT = synth.Workload(
    key="ragged-split", title="ragged split-K layer",
    projs=(synth.Proj("a", synth.Q4_K, 8192, 100, 0), synth.Proj("b", synth.Q6_K, 8192, 40, 0),
           synth.Proj("c", synth.Q4_K, 6400, 1000, 1), synth.Proj("d", synth.Q4_K, 6400, 17, 1)),
    seed_base=900, x_seed_base=19000, input_dims=(8192, 6400))
RAGGED_SPLIT_Q80 = synth.Workload(
    key="ragged-split-q8_0", title="ragged split-K Q8_0 layer",
    projs=(synth.Proj("a", synth.Q8_0, 7168, 77, 0), synth.Proj("b", synth.Q8_0, 7168, 300, 0)),
    seed_base=950, x_seed_base=19500, input_dims=(7168,))


@pytest.mark.parametrize("M", [1, 5, 8, 20, 40, 64])
def test_ragged_split_layer(xq, M):
    # M > 8: (projection, 8-token chunk) pairs over several grouped launches,
    # each pair of a long row with its own split workspace
    assert layer_check(xq, RAGGED_SPLIT, M) > 0
    assert layer_check(xq, RAGGED_SPLIT_Q80, M) > 0


Q80_SHAPES = [(1, 256), (5, 512), (37, 1536), (130, 4096), (3, 12288)]


@pytest.mark.parametrize("N,K", Q80_SHAPES)
def test_q8_0_shapes_all_m(xq, N, K):
    # Q8_0 on the tensor-core GEMV: exact block sums (isum hook) and y for M = 1..8
    errs = [run_and_check(xq, synth.Q8_0, N, K, M, 41 * N + K, 11 * M + N) for M in range(1, 9)]
    assert max(errs) > 0.0


@pytest.mark.parametrize("M", [1, 3, 8, 20, 64, 80])
def test_q8_0_layer(xq, M):
    # a Qwen2.5-1.5B-shaped layer requantized to Q8_0, through xq_layer_mixed
    # (one grouped Q8_0 launch; the 8960-wide down projection is split over K)
    assert layer_check(xq, synth.WORKLOADS["qwen2.5-1.5b-q8_0-layer"], M) > 0


def test_q8_0_extreme_bytes(xq):
    # every int8 value as a weight, with large scales, against extreme activations
    N, K, M = 64, 1024, 8
    W = synth.gen_q8_0(5, N, K).reshape(N, K // 32, 34)
    W[:, :, 2:] = (np.arange(N * (K // 32) * 32) % 256).astype(np.uint8).reshape(N, K // 32, 32)
    W[:, :, 0:2] = np.frombuffer(np.float16(0.25).tobytes(), np.uint8)
    x = synth.gen_x(6, M, K)
    x[0] = 1000.0
    x[1, ::2] = -1000.0
    check_matmul(xq, synth.Q8_0, W.reshape(N, -1), x)


@pytest.mark.parametrize("M", [100, 128, 200, 300])
def test_tile_layer_k_split(xq, M):
    """M > 64 inside a layer: projections whose 128 x 128 tiles leave SMs
    idle are split into K ranges whose partial sums the last CTA of each tile
    adds in range order (ragged N, N not a multiple of 4, Q4_K and Q6_K), and
    later tile launches of the layer start without waiting for the earlier
    ones. Every row against the oracle; two calls give the same bits."""
    assert layer_check(xq, RAGGED_SPLIT, M) > 0
    wl = RAGGED_SPLIT
    weights = synth.gen_layer_weights(wl, 0)
    inputs = [dev(x) for x in synth.gen_layer_inputs(wl, M, 0)]
    L = xq.Layer(wl.projs, weights, M)
    L.forward(inputs)
    first = [y.clone() for y in L.y]
    L.forward(inputs)
    torch.cuda.synchronize()
    assert xq.device_error() == 0
    for a, b in zip(first, L.y):
        assert torch.equal(a, b)


def test_qwen3_mixed_layer_tiles_128(xq):
    # the mixed layer at 128 tokens: q/k/v/o and down split over K, gate and
    # up (96 tiles) not; sampled rows of every projection
    assert layer_check(xq, synth.WORKLOADS["qwen3-8b-mixed-layer"], 128, rows=96) > 0


def test_qwen3_mixed_layer_tiles(xq):
    # M > 64: every row of every projection of the mixed layer (Q4_K and
    # Q6_K) on the tile kernel
    assert layer_check(xq, synth.WORKLOADS["qwen3-8b-mixed-layer"], 80) > 0


def test_qwen3_mixed_layer_gemv_chunks(xq):
    # 8 < M <= 64: every row of every projection of the mixed layer as GEMV chunks
    assert layer_check(xq, synth.WORKLOADS["qwen3-8b-mixed-layer"], 40) > 0


def test_llama3_32layer_sweep(xq):
    # The decode sweep as the bench runs it: all 32 layers resident (3.93 GB),
    # xq_layer_mixed per layer at M=8; every row of every projection of every
    # layer checked.
    wl = synth.WORKLOADS["llama3-8b-32layer"]
    M = 8
    layers = [xq.Layer(wl.projs, synth.gen_layer_weights(wl, l), M) for l in range(wl.layers)]
    inputs = [synth.gen_layer_inputs(wl, M, l) for l in range(wl.layers)]
    dins = [[dev(x) for x in ins] for ins in inputs]
    for L in layers:
        for y in L.y:
            y.fill_(float("nan"))
    for L, di in zip(layers, dins):
        L.forward(di)
    torch.cuda.synchronize()
    for l in range(wl.layers):
        q8 = [oracle.quantize_q8(x) for x in inputs[l]]
        weights = synth.gen_layer_weights(wl, l)
        for t, p in enumerate(wl.projs):
            rq, rd, _ = q8[p.input]
            y_ref, ab, _ = oracle.matmul(p.qtype, weights[t], rq, rd, p.K)
            check_y(layers[l].y[t].cpu().numpy(), y_ref, ab)
    # every layer wrote every output
    for L in layers:
        for y in L.y:
            assert torch.isfinite(y).all()


def test_prefill512_all_rows(xq):
    # the M = 512 prefill projections on their own inputs, every output
    wl = synth.WORKLOADS["qwen3-8b-ffn-prefill512"]
    M = 512
    weights = synth.gen_layer_weights(wl, 0)
    inputs = synth.gen_layer_inputs(wl, M, 0)
    for t, p in enumerate(wl.projs):
        x = inputs[p.input]
        buf, rq, rd = assert_q8_exact(xq, x)
        y = poisoned(M, p.N)
        xq.matmul(p.qtype, dev(weights[t].reshape(-1)), buf, M, p.N, p.K, y=y)
        torch.cuda.synchronize()
        yc = y.cpu().numpy()
        assert np.all(np.isfinite(yc))
        y_ref, ab, _ = oracle.matmul(p.qtype, weights[t], rq, rd, p.K)
        check_y(yc, y_ref, ab)


def test_misaligned_device_pointer_rejected(xq):
    W = dev(synth.gen_q4k(1, 4, 256).reshape(-1))
    buf = xq.quantize_q8(dev(synth.gen_x(2, 1, 256)))
    y = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(xq.XQError) as e:
        xq.matmul(synth.Q4_K, W[8:], buf, 1, 4, 256, y=y[:4])
    assert e.value.code == 3


# ------------------------------------------------------------ batch invariance

@pytest.mark.parametrize("qtype,N,K", [(synth.Q4_K, 200, 1536), (synth.Q6_K, 130, 2048), (synth.Q6_K, 70, 1024),
                                       (synth.Q8_0, 90, 1024)])
def test_batch_invariant_rows(xq, qtype, N, K):
    """Row m of y from the batch-invariant entry points is bit-identical for
    every batch that contains token m, equal to decoding the token alone with
    xq_matmul_*, deterministic across runs, and within the oracle's bound."""
    Mmax = 21
    W = synth.gen_weight(qtype, 901 + K + qtype, N, K)
    x = synth.gen_x(902 + N, Mmax, K)
    Wd = dev(W.reshape(-1))
    xd = dev(x)

    def run(M):
        buf = xq.quantize_q8_invariant(xd[:M].contiguous())
        y = poisoned(M, N)
        xq.matmul_invariant(qtype, Wd, buf, M, N, K, y=y)
        torch.cuda.synchronize()
        return buf, y.cpu().numpy()

    buf_full, y_full = run(Mmax)
    # the Q8 bytes of the invariant layout are the oracle's (qs / d8 / s8 regions)
    rq, rd, rs = oracle.quantize_q8(x)
    qs, d8, s8 = (t.cpu().numpy() for t in xq.q8_views(buf_full, Mmax, K))
    assert np.array_equal(qs, rq)
    assert np.array_equal(d8.view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(s8.view(np.uint32), rs.view(np.uint32))
    y_ref, ab, _ = oracle.matmul(qtype, W, rq, rd, K, want_isum=False)
    check_y(y_full, y_ref, ab)
    for M in (1, 3, 8, 9, 16, 20):
        _, y = run(M)
        assert np.array_equal(y.view(np.uint32), y_full[:M].view(np.uint32)), M
    _, y_again = run(Mmax)
    assert np.array_equal(y_again.view(np.uint32), y_full.view(np.uint32))
    # the plain entry point at M <= 8 computes the same rows
    for m in (0, 7, 13):
        buf1 = xq.quantize_q8(xd[m:m + 1].contiguous())
        y1 = poisoned(1, N)
        xq.matmul(qtype, Wd, buf1, 1, N, K, y=y1)
        torch.cuda.synchronize()
        assert np.array_equal(y1.cpu().numpy().view(np.uint32), y_full[m:m + 1].view(np.uint32)), m


# ------------------------------------------------------------ SwiGLU feed

def check_h(h_gpu, g, u):
    # e = expf(-g) is within 2 ulp (CUDA's documented bound); 1 + e, the
    # divide and the product are each rounded once: together within 8 ulp of
    # the exact silu(g) * u (relative 2^-20), or tiny where h underflows.
    h_ref = oracle.silu_mul(g, u)
    err = np.abs(h_gpu.astype(np.float64) - h_ref)
    assert np.all(err <= 2.0 ** -20 * np.abs(h_ref) + 1e-37), float(np.max(err / (np.abs(h_ref) + 1e-37)))


@pytest.mark.parametrize("M,K", [(1, 256), (5, 2048), (20, 512)])
def test_silu_mul_quantize(xq, M, K):
    rng = np.random.default_rng(M * 1000 + K)
    g = (rng.standard_normal((M, K)) * 4).astype(np.float32)
    u = rng.standard_normal((M, K)).astype(np.float32)
    g[0, :32] = np.array([-100, -88, -87, 0, 88, 89, 100, -1e30, 1e30, -0.0] + [0.0] * 22, np.float32)
    g[0, 32:64] = 0.0                                   # h = 0 block
    h = torch.empty((M, K), dtype=torch.float32, device="cuda")
    buf = xq.silu_mul_quantize_q8(dev(g), dev(u), h_out=h)
    torch.cuda.synchronize()
    h_gpu = h.cpu().numpy()
    check_h(h_gpu, g, u)
    # the Q8 of h is the oracle's quantization of the same fp32 values, bit for bit
    qs, d8, s8 = (t.cpu().numpy() for t in xq.q8_views(buf, M, K))
    rq, rd, rs = oracle.quantize_q8(h_gpu)
    assert np.array_equal(qs, rq)
    assert np.array_equal(d8.view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(s8.view(np.uint32), rs.view(np.uint32))


# xq_layer_mixed_ffn. At M <= 8 the gate/up warps of the grouped launch write
# h's Q8 themselves: down in the same launch (all-Q4_K layers: Qwen2.5-1.5B,
# F = 8960, and Llama-3-8B, F = 14336 with down split over K) or in a later
# launch (the Q4_K_M mix, down in Q6_K). Above 8 tokens the feed is a
# separate launch.
FFN_CASES = [("qwen2.5-1.5b-layer", None), ("qwen2.5-1.5b-q4km-layer", None), ("llama3-8b-32layer", 384)]


@pytest.mark.parametrize("key,rows", FFN_CASES)
@pytest.mark.parametrize("M", [1, 2, 8, 20, 80])
def test_ffn_layer_down_fed_by_silu_gate_up(xq, key, rows, M):
    """Every projection but down checked as in xq_layer_mixed (all rows, or
    `rows` sampled rows); h recomputed from the call's gate and up outputs by
    xq_silu_mul_quantize_q8 checked against the oracle's silu_mul; the Q8 of
    h the call left in its workspace equal to that launch's Q8, bit for bit,
    and to the oracle's quantization of the same fp32 h; down checked against
    the oracle on that Q8."""
    wl = synth.WORKLOADS[key]
    if rows is not None and M == 80:
        pytest.skip("the Llama-3-8B layer is covered at M <= 20")
    weights = synth.gen_layer_weights(wl, 0)
    inputs = synth.gen_layer_inputs(wl, M, 0)[:3]   # attn-in, o-in, ffn-in; down reads h
    Wd = [dev(w.reshape(-1)) for w in weights]
    ys = [poisoned(M, p.N) for p in wl.projs]
    desc = [(p.qtype, p.N, p.K, Wd[t], ys[t], min(p.input, 2)) for t, p in enumerate(wl.projs)]
    names = [p.name for p in wl.projs]
    gi, ui, di = names.index("gate"), names.index("up"), names.index("down")
    ws = torch.zeros(xq.layer_ffn_workspace_bytes(desc, 3, M, gi, ui, di), dtype=torch.uint8, device="cuda")
    xq.layer_mixed_ffn(desc, gi, ui, di, [dev(x) for x in inputs], M, ws)
    torch.cuda.synchronize()
    assert xq.device_error() == 0
    q8 = [oracle.quantize_q8(x) for x in inputs]
    rng = np.random.default_rng(M)
    for t, p in enumerate(wl.projs):
        if t == di:
            continue
        rq, rd, _ = q8[p.input]
        sel = np.arange(p.N) if rows is None else np.sort(rng.choice(p.N, size=min(rows, p.N), replace=False))
        y_ref, ab, _ = oracle.matmul(p.qtype, weights[t][sel], rq, rd, p.K)
        check_y(ys[t].cpu().numpy()[:, sel], y_ref, ab)
    g, u = ys[gi], ys[ui]
    F = wl.projs[di].K
    h = torch.empty_like(g)
    # zero-filled, like the workspace: the layout's padding bytes stay zero on both
    hbuf = xq.silu_mul_quantize_q8(g, u, out=torch.zeros(xq.q8_bytes(M, F), dtype=torch.uint8, device="cuda"),
                                   h_out=h)
    torch.cuda.synchronize()
    h_gpu = h.cpu().numpy()
    check_h(h_gpu, g.cpu().numpy(), u.cpu().numpy())
    # the workspace: the read inputs' Q8 buffers (256-byte padded), then h's
    h_off = sum(-(-xq.q8_bytes(M, x.shape[1]) // 256) * 256 for x in inputs)
    nb = xq.q8_bytes(M, F)
    assert torch.equal(ws[h_off:h_off + nb], hbuf[:nb])
    rq, rd, rs = oracle.quantize_q8(h_gpu)
    qs, d8, s8 = (t.cpu().numpy() for t in xq.q8_views(ws[h_off:h_off + nb], M, F))
    assert np.array_equal(qs, rq)
    assert np.array_equal(d8.view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(s8.view(np.uint32), rs.view(np.uint32))
    sel = np.arange(wl.projs[di].N) if rows is None else np.sort(rng.choice(wl.projs[di].N, size=rows, replace=False))
    y_ref, ab, _ = oracle.matmul(wl.projs[di].qtype, weights[di][sel], rq, rd, F)
    check_y(ys[di].cpu().numpy()[:, sel], y_ref, ab)


# ------------------------------------------------------------ IQ4_XS

def check_iq4xs(xq, W, x, codebook):
    """xq_matmul_iq4xs_q8 and its isum hook against the oracle (M <= 8)."""
    M, K = x.shape
    N = W.shape[0]
    buf, rq, rd = assert_q8_exact(xq, x)
    y_ref, ab, isum_ref = oracle.matmul(synth.IQ4_XS, W, rq, rd, K, want_isum=True, codebook=codebook)
    Wd = dev(W.reshape(-1))
    y = poisoned(M, N)
    isum = torch.full((M, N, K // 32), -(2 ** 31), dtype=torch.int32, device="cuda")
    xq.debug_isums_iq4xs(Wd, codebook, buf, M, N, K, y=y, isum=isum)
    torch.cuda.synchronize()
    assert np.array_equal(isum.cpu().numpy(), isum_ref)
    y_isum = y.cpu().numpy()
    y = poisoned(M, N)
    xq.matmul_iq4xs_q8(Wd, codebook, buf, M, N, K, y=y)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_isum.view(np.uint32))
    return check_y(y.cpu().numpy(), y_ref, ab)


IQ4XS_SHAPES = [(1, 512), (5, 1024), (37, 1536), (130, 5120), (64, 4096)]


@pytest.mark.parametrize("N,K", IQ4XS_SHAPES)
def test_iq4xs_shapes_all_m(xq, N, K):
    # IQ4_XS on the tensor-core GEMV: exact codebook-value sums and y for M = 1..8,
    # a different synthetic codebook per M
    errs = []
    for M in range(1, 9):
        cb = synth.gen_codebook(100 * M + N)
        W = synth.gen_iq4xs(43 * N + K + M, N, K)
        errs.append(check_iq4xs(xq, W, synth.gen_x(13 * M + N, M, K), cb))
    assert max(errs) > 0.0


def test_iq4xs_extremes(xq):
    # codebook ends (-128, 127) on every index, scales 0 and 63, large d,
    # against +-1000 activations
    N, K, M = 64, 1024, 8
    W = synth.gen_iq4xs(7, N, K).reshape(N, K // 256, 136)
    W[:, :, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), np.uint8)
    W[: N // 2, :, 2:8] = 0x00                # ls = 0 -> -32
    W[N // 2:, :, 2:8] = 0xFF                 # ls = 63 -> 31
    cb = np.array([-128, 127] * 8, dtype=np.int8)
    x = synth.gen_x(8, M, K)
    x[0] = 1000.0
    x[1, ::2] = -1000.0
    check_iq4xs(xq, W.reshape(N, -1), x, cb)


def test_iq4xs_rows_of_a_ragged_tail(xq):
    # N not a multiple of 16, one super-block pair, a codebook with zero in it
    cb = synth.gen_codebook(4)
    cb[7] = 0
    W = synth.gen_iq4xs(9, 19, 512)
    assert check_iq4xs(xq, W, synth.gen_x(10, 3, 512), cb) > 0.0


def check_iq4xs_tile(xq, W, x, codebook, rows=None):
    """M > 8: xq_matmul_iq4xs_q8 on the tile kernel against the oracle (all
    rows, or `rows` sampled rows)."""
    M, K = x.shape
    N = W.shape[0]
    buf, rq, rd = assert_q8_exact(xq, x)
    sel = np.arange(N) if rows is None else np.sort(np.random.default_rng(N + M).choice(N, rows, replace=False))
    y_ref, ab, _ = oracle.matmul(synth.IQ4_XS, W[sel], rq, rd, K, codebook=codebook)
    y = poisoned(M, N)
    xq.matmul_iq4xs_q8(dev(W.reshape(-1)), codebook, buf, M, N, K, y=y)
    torch.cuda.synchronize()
    return check_y(y.cpu().numpy()[:, sel], y_ref, ab)


# 9 and 40 tokens run as GEMV chunks, 130 and 200 on the tile kernel
@pytest.mark.parametrize("N,K,M", [(130, 1024, 9), (64, 4096, 40), (17, 512, 200), (300, 5120, 130)])
def test_iq4xs_more_than_eight_tokens(xq, N, K, M):
    cb = synth.gen_codebook(N + M)
    W = synth.gen_iq4xs(57 * N + K, N, K)
    assert check_iq4xs_tile(xq, W, synth.gen_x(3 * M + N, M, K), cb, rows=None if N * M <= 20000 else 96) > 0.0


def test_iq4xs_tile_scale_forms(xq):
    # |s| <= 16 everywhere (one operand per tile) and the extremes s = -32, 31
    # (the two-operand form), with the codebook ends on every index
    N, K, M = 256, 1024, 80
    cb = np.array([-128, 127] * 8, dtype=np.int8)
    x = synth.gen_x(5, M, K)
    x[0] = 1000.0
    W = synth.gen_iq4xs(6, N, K).reshape(N, K // 256, 136)
    W[:, :, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), np.uint8)
    narrow = W.copy()
    narrow[:, :, 2:4] = 0x55                     # scales_h bits 01 -> ls in 16..31
    narrow[:, :, 4:8] = 0x00                     # ls = 16 -> s = -16
    check_iq4xs_tile(xq, narrow.reshape(N, -1), x, cb)
    wide = W.copy()
    wide[: N // 2, :, 2:8] = 0x00                # s = -32
    wide[N // 2:, :, 2:8] = 0xFF                 # s = 31
    check_iq4xs_tile(xq, wide.reshape(N, -1), x, cb)


# A layer mixing IQ4_XS (two codebooks) with Q4_K and Q6_K: ragged output
# counts, a long IQ4_XS row that splits over K, through every path by M.
IQ4XS_LAYER = synth.Workload(
    key="iq4xs-layer", title="IQ4_XS mixed layer",
    projs=(synth.Proj("q", synth.IQ4_XS, 2048, 300, 0), synth.Proj("k", synth.Q4_K, 2048, 70, 0),
           synth.Proj("v", synth.IQ4_XS, 2048, 64, 0), synth.Proj("up", synth.Q6_K, 2048, 200, 0),
           synth.Proj("down", synth.IQ4_XS, 8192, 130, 1)),
    seed_base=960, x_seed_base=19700, input_dims=(2048, 8192))


@pytest.mark.parametrize("M", [1, 8, 20, 80])
def test_iq4xs_layer(xq, M):
    cbs = [synth.gen_codebook(1), None, synth.gen_codebook(2), None, synth.gen_codebook(3)]
    assert layer_check(xq, IQ4XS_LAYER, M, codebooks=cbs) > 0
