"""Failure detection without a GPU fault.

Every mbarrier wait of the TMA / tensor-core kernels is bounded; a wait that
runs out records an error code in a device word, and the kernel leaves its
loops, waits for its own copies and tensor-core work, frees tensor memory and
returns. xq_device_error reads and clears that record. Here a test hook
(xq_debug_stalled_matmul_q4k) launches the Q4_K GEMV with a producer that
issues nothing and waits cut to about 10^5 clocks: the consumers' first
waits run out (a flag nothing sets), the host reads the GEMV's code,
the outputs stay unwritten, and the context stays usable for the next call.
"""
import numpy as np
import pytest
import torch

import oracle
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
