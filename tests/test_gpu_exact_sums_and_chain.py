"""GPU parity, second part: exact integer sums on the tile path, long rows
without a K-split, and the prefill FFN chained up -> down on every row.

- The tile kernel (M > 64) accumulates each 32-block's exact integer before
  any scale (the scale of a 4/6-bit sub-block is folded into its fp16
  operand); the test hook writes those integers and they must equal, bit for
  bit, the ones derived from the oracle's sub-block sums and decoded scales.
- A single matmul never splits a row over K, so each output's fp32 sum runs
  over all K/256 super-blocks; the kernels bound the rounding by summing each
  super-block into a fresh accumulator and that into a running sum. K = 14336
  (the longest row of the workloads) at M = 1, 8 and 40 stays inside the
  stated tolerance.
- The prefill FFN workload passes 512 tokens through ffn_up and then
  ffn_down: down reads the Q8 of up's output. The oracle runs the same chain
  on its own (fp64 up, fp32 cast, its own Q8). The GPU's down is checked
  against it with the parity tolerance plus the propagated difference of the
  two Q8 inputs, sum_k |w[n][k]| * |xhat_gpu[k] - xhat_ref[k]|, after the two
  Q8 buffers are checked to differ only by rounding-boundary flips.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gguf_quant_integer_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_REL = 1e-5
TOL_ABS = 1e-7


@pytest.fixture(scope="module")
def xq():
    from gguf_quant_integer_gb300 import build, xq as _xq
    build.build()
    _xq.lib()
    oracle.set_threads(os.cpu_count() or 1)
    yield _xq
    oracle.set_threads(1)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_y(y_gpu, y_ref, absterm, extra=0.0):
    y_gpu = y_gpu.astype(np.float64)
    assert np.all(np.isfinite(y_gpu)), "an output was not written"
    err = np.abs(y_gpu - y_ref)
    bound = TOL_REL * (absterm + extra) + TOL_ABS + extra
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} outputs out of tolerance; worst ratio {np.max(err / bound):.3g}"
    return float(err.max())


def block_scales(qtype, W, K, codebook=None):
    """Per 32-block integer scale factors of each row from the oracle's field
    decoders: Q4_K sc_j [N][K/32]; Q6_K the 16-weight group scales [N][K/16];
    IQ4_XS ls_j - 32 [N][K/32]."""
    N = W.shape[0]
    nsb = K // 256
    if qtype == synth.Q4_K:
        out = np.zeros((N, K // 32), np.int64)
        for n in range(N):
            for b in range(nsb):
                _, _, sc, _, _ = oracle.q4k_fields(W[n, 144 * b:144 * (b + 1)])
                out[n, 8 * b:8 * b + 8] = sc
        return out
    if qtype == synth.Q6_K:
        out = np.zeros((N, K // 16), np.int64)
        for n in range(N):
            for b in range(nsb):
                _, s, _ = oracle.q6k_fields(W[n, 210 * b:210 * (b + 1)])
                out[n, 16 * b:16 * b + 16] = s
        return out
    if qtype == synth.IQ4_XS:
        out = np.zeros((N, K // 32), np.int64)
        for n in range(N):
            for b in range(nsb):
                _, ls, _ = oracle.iq4xs_fields(W[n, 136 * b:136 * (b + 1)], codebook)
                out[n, 8 * b:8 * b + 8] = np.asarray(ls) - 32
        return out
    return None


def expected_tile_sums(qtype, W, rq, rd, K, codebook=None):
    """Each 32-block's integer as the tile kernel accumulates it, from the
    oracle's exact sub-block sums: [M][N][K/32] int64."""
    _, _, isum = oracle.matmul(qtype, W, rq, rd, K, want_isum=True, codebook=codebook)
    isum = isum.astype(np.int64)
    if qtype == synth.Q8_0:
        return isum
    s = block_scales(qtype, W, K, codebook)
    if qtype == synth.Q6_K:
        prod = isum * s[None, :, :]          # [M][N][K/16]
        return prod[:, :, 0::2] + prod[:, :, 1::2]
    return isum * s[None, :, :]


TILE_SUM_CASES = [(synth.Q4_K, 256, 4096, 512), (synth.Q6_K, 256, 4096, 512), (synth.Q8_0, 256, 4096, 512),
                  (synth.IQ4_XS, 256, 4096, 512), (synth.Q4_K, 130, 1536, 200), (synth.Q6_K, 130, 1536, 200),
                  (synth.Q6_K, 37, 2304, 70)]


@pytest.mark.parametrize("qtype,N,K,M", TILE_SUM_CASES)
def test_tile_exact_sums(xq, qtype, N, K, M):
    cb = synth.gen_codebook(31) if qtype == synth.IQ4_XS else None
    W = synth.gen_iq4xs(71, N, K) if qtype == synth.IQ4_XS else synth.gen_weight(qtype, 71 + qtype, N, K)
    if qtype == synth.Q6_K:
        # full-range int8 scales in half the rows: those tiles take the
        # two-operand form
        blocks = W.reshape(N, K // 256, 210)
        rng = np.random.default_rng(72)
        sc = rng.integers(-128, 128, size=(N, K // 256, 16)).astype(np.int8)
        sc[: N // 2] = np.clip(sc[: N // 2], -64, 64)
        blocks[:, :, 192:208] = sc.view(np.uint8)
    x = synth.gen_x(73 + M, M, K)
    buf = xq.quantize_q8(dev(x))
    rq, rd, _ = oracle.quantize_q8(x)
    sums = torch.full((M, N, K // 32), -(2 ** 31), dtype=torch.int32, device="cuda")
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    xq.debug_tile_sums(qtype, dev(W.reshape(-1)), buf, M, N, K, codebook=cb, y=y, sums=sums)
    torch.cuda.synchronize()
    want = expected_tile_sums(qtype, W, rq, rd, K, cb)
    got = sums.cpu().numpy().astype(np.int64)
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} sums differ"
    y_ref, ab, _ = oracle.matmul(qtype, W, rq, rd, K, codebook=cb)
    assert check_y(y.cpu().numpy(), y_ref, ab) > 0.0


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("M", [1, 8, 40])
def test_long_rows_single_matmul(xq, qtype, M):
    # K = 14336 (56 super-blocks) with no K-split: one output's fp32 sum runs
    # over the whole row
    N, K = 200, 14336
    W = synth.gen_weight(qtype, 81 + M, N, K)
    x = synth.gen_x(82 + M, M, K)
    buf = xq.quantize_q8(dev(x))
    rq, rd, _ = oracle.quantize_q8(x)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    xq.matmul(qtype, dev(W.reshape(-1)), buf, M, N, K, y=y)
    torch.cuda.synchronize()
    y_ref, ab, _ = oracle.matmul(qtype, W, rq, rd, K)
    assert check_y(y.cpu().numpy(), y_ref, ab) > 0.0


def test_prefill512_chain_all_rows(xq):
    wl = synth.WORKLOADS["qwen3-8b-ffn-prefill512"]
    up, down = wl.projs
    M = 512
    Wu, Wd = synth.gen_layer_weights(wl, 0)
    x = synth.gen_layer_inputs(wl, M, 0)[up.input]
    # GPU: x -> Q8 -> up -> y_up -> Q8 -> down -> y_down
    bx = xq.quantize_q8(dev(x))
    y_up = torch.full((M, up.N), float("nan"), dtype=torch.float32, device="cuda")
    xq.matmul(up.qtype, dev(Wu.reshape(-1)), bx, M, up.N, up.K, y=y_up)
    bh = xq.quantize_q8(y_up)
    y_dn = torch.full((M, down.N), float("nan"), dtype=torch.float32, device="cuda")
    xq.matmul(down.qtype, dev(Wd.reshape(-1)), bh, M, down.N, down.K, y=y_dn)
    torch.cuda.synchronize()
    # oracle: the same chain on its own
    rq, rd, _ = oracle.quantize_q8(x)
    yu_ref, ab_up, _ = oracle.matmul(up.qtype, Wu, rq, rd, up.K)
    check_y(y_up.cpu().numpy(), yu_ref, ab_up)          # every row of up
    hq, hd, _ = oracle.quantize_q8(yu_ref.astype(np.float32))
    yd_ref, ab_dn, _ = oracle.matmul(down.qtype, Wd, hq, hd, down.K)
    # the two Q8 inputs of down differ only where up's fp32 outputs straddle a
    # rounding boundary: codes by at most one step, rarely, scales by rounding
    gq, gd, _ = (t.cpu().numpy() for t in xq.q8_views(bh, M, down.K))
    dq = np.abs(gq.astype(np.int32) - hq.astype(np.int32))
    assert dq.max() <= 1 and np.count_nonzero(dq) <= 1e-3 * dq.size, (dq.max(), np.count_nonzero(dq))
    rel_d = np.abs(gd.astype(np.float64) - hd) / np.maximum(hd, 1e-30)
    assert rel_d.max() <= 1e-5, rel_d.max()
    # propagated bound sum_k |w[n][k]| * |xhat_gpu - xhat_ref| (fp64)
    xh_g = np.repeat(gd.astype(np.float64), 32, axis=1) * gq
    xh_r = np.repeat(hd.astype(np.float64), 32, axis=1) * hq
    wabs = np.abs(oracle.dequant_q6k(Wd, down.K))     # [N][K]
    prop = np.abs(xh_g - xh_r) @ wabs.T                # [M][N]
    check_y(y_dn.cpu().numpy(), yd_ref, ab_dn, extra=prop)
