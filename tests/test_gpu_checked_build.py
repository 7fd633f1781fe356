"""GPU runs of the checked build (the library compiled with -DXQ_CHECK).

In that build every kernel tests the index, range or 16-byte alignment of
each global access whose address comes from nontrivial arithmetic before it
makes the access; a failed check skips the access and records its site,
which xq_device_error reports as kernel 9. Nothing traps. Here every kernel
family runs small parity cases (the oracle's results, as in the parity
tests) and no check may fail; then a probe declares a y extent one token row
short of what its launch writes and must see exactly that check fire, with
the row left unwritten and the other rows correct.
"""
import numpy as np
import pytest
import torch

import oracle
import test_gpu_parity as par
from gguf_quant_integer_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xq():
    from gguf_quant_integer_gb300 import build, xq as _xq
    path = build.build(check=True)
    saved = _xq._lib
    _xq._lib = None
    _xq._lib = _xq.lib(path)
    yield _xq
    _xq._lib = saved


def no_check_failed(xq):
    code = xq.device_error()
    assert code == 0, hex(code)


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K, synth.Q8_0])
@pytest.mark.parametrize("N,K", [(37, 1536), (130, 4096)])
def test_checked_gemv_shapes(xq, qtype, N, K):
    # M = 1, 2 (Q4_K's one- and two-token form), 5, 8 with the isum hook;
    # 20 (8-token chunks) and 80 (tile kernel) without
    for M in (1, 2, 5, 8, 20, 80):
        par.run_and_check(xq, qtype, N, K, M, 7 * N + K + qtype, 3 * M + N, want_isum=M <= 8)
    no_check_failed(xq)


@pytest.mark.parametrize("N,K,M", [(8192, 1536, 3), (130, 8960, 1), (130, 8960, 4), (64, 8960, 70)])
def test_checked_q6k_paths(xq, N, K, M):
    # grouped tensor map (8192 x 1536), the dp4a kernel (ragged N, 7350-byte
    # rows) and the tile kernel's row windows cut at the end of the weights
    par.run_and_check(xq, synth.Q6_K, N, K, M, 11 * N + K, 5 * M + K, want_isum=M <= 8)
    no_check_failed(xq)


@pytest.mark.parametrize("M", [1, 8, 80])
def test_checked_iq4xs(xq, M):
    N, K = 130, 5120
    cb = synth.gen_codebook(7)
    W = synth.gen_iq4xs(9, N, K)
    x = synth.gen_x(10 + M, M, K)
    buf, rq, rd = par.assert_q8_exact(xq, x)
    y = par.poisoned(M, N)
    xq.matmul_iq4xs_q8(par.dev(W.reshape(-1)), cb, buf, M, N, K, y=y)
    torch.cuda.synchronize()
    y_ref, ab, _ = oracle.matmul(synth.IQ4_XS, W, rq, rd, K, codebook=cb)
    par.check_y(y.cpu().numpy(), y_ref, ab)
    no_check_failed(xq)


@pytest.mark.parametrize("M", [1, 8, 40, 80, 200])
def test_checked_layers(xq, M):
    # split-K hand-offs, mixed weight types and the grouped Q6_K view; above
    # 64 tokens the tile launches' K ranges (two token tiles at 200)
    assert par.layer_check(xq, par.RAGGED_SPLIT, M) > 0
    assert par.layer_check(xq, synth.WORKLOADS["qwen2.5-1.5b-q4km-layer"], M, rows=128) > 0
    no_check_failed(xq)


@pytest.mark.parametrize("M", [1, 8, 20])
def test_checked_fused_ffn(xq, M):
    # the SwiGLU feed written by the gate/up warps (M <= 8) and as its own launch
    wl = synth.WORKLOADS["qwen2.5-1.5b-layer"]
    weights = synth.gen_layer_weights(wl, 0)
    inputs = synth.gen_layer_inputs(wl, M, 0)[:3]
    Wd = [par.dev(w.reshape(-1)) for w in weights]
    ys = [par.poisoned(M, p.N) for p in wl.projs]
    desc = [(p.qtype, p.N, p.K, Wd[t], ys[t], min(p.input, 2)) for t, p in enumerate(wl.projs)]
    names = [p.name for p in wl.projs]
    gi, ui, di = names.index("gate"), names.index("up"), names.index("down")
    ws = torch.zeros(xq.layer_ffn_workspace_bytes(desc, 3, M, gi, ui, di), dtype=torch.uint8, device="cuda")
    xq.layer_mixed_ffn(desc, gi, ui, di, [par.dev(x) for x in inputs], M, ws)
    torch.cuda.synchronize()
    no_check_failed(xq)
    g, u = ys[gi], ys[ui]
    h = torch.empty_like(g)
    xq.silu_mul_quantize_q8(g, u, h_out=h)
    torch.cuda.synchronize()
    rq, rd, _ = oracle.quantize_q8(h.cpu().numpy())
    y_ref, ab, _ = oracle.matmul(wl.projs[di].qtype, weights[di], rq, rd, wl.projs[di].K)
    par.check_y(ys[di].cpu().numpy(), y_ref, ab)
    no_check_failed(xq)


def test_checked_build_probe_fires(xq):
    """A check that fails is recorded and its access skipped: the probe's
    last token row stays NaN, the others equal the normal launch bit for bit."""
    M, N, K = 4, 64, 512
    W = par.dev(synth.gen_q4k(21, N, K).reshape(-1))
    buf = xq.quantize_q8(par.dev(synth.gen_x(22, M, K)))
    y_ref = par.poisoned(M, N)
    xq.matmul(synth.Q4_K, W, buf, M, N, K, y=y_ref)
    torch.cuda.synchronize()
    no_check_failed(xq)
    y = par.poisoned(M, N)
    rc = xq.lib().xq_debug_check_probe(W.data_ptr(), buf.data_ptr(), M, N, K, y.data_ptr(), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert xq.device_error() == (9 << 8) | 10
    assert xq.device_error() == 0
    yc = y.cpu().numpy()
    assert np.isnan(yc[M - 1]).all()
    assert np.array_equal(yc[:M - 1].view(np.uint32), y_ref.cpu().numpy()[:M - 1].view(np.uint32))
