"""Failure detection without a GPU fault.

Every mbarrier wait of the TMA / tensor-core kernels is bounded; a wait that
runs out records an error code in a device word, and the kernel leaves its
loops, waits for its own copies and tensor-core work, frees tensor memory and
returns. xq_device_error reads and clears that record. Here a test hook
(xq_debug_stalled_matmul_q4k) launches the Q4_K GEMV with a producer that
issues nothing and waits cut to about 10^5 clocks: the consumers' first
waits run out (a flag nothing sets), the host reads the GEMV's code,
the outputs stay unwritten, and the context stays usable for the next call.
A second hook (xq_debug_stalled_ffn_layer) withholds the fused SwiGLU feed's
ready counts, so that down's producers give up waiting for h (wait 3).
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
    build.build()
    _xq.lib()
    return _xq


def test_stalled_wait_is_reported_and_context_stays_usable(xq):
    torch.cuda.synchronize()
    xq.device_error()  # clear any earlier record
    N, K, M = 256, 1024, 4
    W = synth.gen_q4k(3, N, K)
    x = synth.gen_x(4, M, K)
    Wd = torch.from_numpy(W.reshape(-1)).cuda()
    buf = xq.quantize_q8(torch.from_numpy(x).cuda())
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    xq.debug_stalled_matmul_q4k(Wd, buf, M, N, K, y)
    code = xq.device_error()
    # kernel 1 (the warp-level MMA GEMV), wait 2: a consumer waiting for the first stage
    assert code == (1 << 8) | 2, hex(code)
    assert torch.isnan(y).all()
    assert xq.device_error() == 0  # the read cleared it
    # the same launch without the hook is correct and records nothing
    xq.matmul(synth.Q4_K, Wd, buf, M, N, K, y=y)
    assert xq.device_error() == 0
    rq, rd, _ = oracle.quantize_q8(x)
    y_ref, ab, _ = oracle.matmul(synth.Q4_K, W, rq, rd, K)
    err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
    assert np.all(err <= 1e-5 * ab + 1e-7)


def test_parity_launches_record_no_timeout(xq):
    # a layer through every kernel family leaves no timed-out wait behind
    torch.cuda.synchronize()
    xq.device_error()
    wl = synth.WORKLOADS["qwen3-8b-mixed-layer"]
    for M in (1, 8, 80):
        L = xq.Layer(wl.projs, synth.gen_layer_weights(wl, 0), M)
        L.forward([torch.from_numpy(v).cuda() for v in synth.gen_layer_inputs(wl, M, 0)])
        assert xq.device_error() == 0, f"M={M}"


@pytest.mark.parametrize("M", [1, 4])
def test_withheld_ffn_feed_is_reported(xq, M):
    """Wait 3: down's producer waiting for h in the fused SwiGLU feed. The
    hook writes h but never counts it ready; down's waits run out, the host
    reads kernel 1 wait 3, down's y stays unwritten while gate and up are
    computed, and the same call without the hook, reusing the workspace, is
    correct and records nothing."""
    torch.cuda.synchronize()
    xq.device_error()
    wl = synth.WORKLOADS["qwen2.5-1.5b-layer"]
    weights = synth.gen_layer_weights(wl, 0)
    inputs = [torch.from_numpy(v).cuda() for v in synth.gen_layer_inputs(wl, M, 0)[:3]]
    Wd = [torch.from_numpy(w.reshape(-1)).cuda() for w in weights]
    names = [p.name for p in wl.projs]
    gi, ui, di = names.index("gate"), names.index("up"), names.index("down")

    def launch(fn):
        ys = [torch.full((M, p.N), float("nan"), dtype=torch.float32, device="cuda") for p in wl.projs]
        desc = [(p.qtype, p.N, p.K, Wd[t], ys[t], min(p.input, 2)) for t, p in enumerate(wl.projs)]
        fn(desc, gi, ui, di, inputs, M, ws)
        return ys

    desc0 = [(p.qtype, p.N, p.K, Wd[t], None, min(p.input, 2)) for t, p in enumerate(wl.projs)]
    ws = torch.zeros(xq.layer_ffn_workspace_bytes(desc0, 3, M, gi, ui, di), dtype=torch.uint8, device="cuda")
    stalled = launch(xq.debug_stalled_ffn_layer)
    code = xq.device_error()
    assert code == (1 << 8) | 3, hex(code)
    assert torch.isnan(stalled[di]).all()
    assert not torch.isnan(stalled[gi]).any() and not torch.isnan(stalled[ui]).any()
    assert xq.device_error() == 0
    ys = launch(xq.layer_mixed_ffn)
    assert xq.device_error() == 0
    # gate and up of the stalled call equal the normal call's bit for bit
    for t in (gi, ui):
        assert torch.equal(stalled[t], ys[t])
    # down against the oracle on h as the feed kernel computes it
    h = torch.empty_like(ys[gi])
    xq.silu_mul_quantize_q8(ys[gi], ys[ui], h_out=h)
    torch.cuda.synchronize()
    rq, rd, _ = oracle.quantize_q8(h.cpu().numpy())
    y_ref, ab, _ = oracle.matmul(wl.projs[di].qtype, weights[di], rq, rd, wl.projs[di].K)
    par.check_y(ys[di].cpu().numpy(), y_ref, ab)
