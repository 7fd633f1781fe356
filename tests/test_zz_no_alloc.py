"""xq_layer_mixed_static: the layer entry point for callers that cannot allocate.

Some callers cannot hand the library a workspace: an engine that gives all
device memory to its own pool at start-up, a plugin whose host owns the
allocator, or a decode loop that must not call cudaMalloc mid-request. For
them xq_layer_mixed_static uses a fixed device array owned by the library.
This test calls it through the C ABI three times in a row (different inputs
and token counts: 8, 3 and 40, so each call runs on whatever the previous
one left in the shared array, and the last one takes the chunked path for 9
to 64 tokens with its own arrival counts and partial sums) and checks that
its outputs equal, bit for bit, those of xq_layer_mixed with a workspace of
its own: the two run the same kernels in the same order, and every split
sum is added in a fixed chunk order. The outputs are also checked against
the oracle within the parity tolerance of the other GPU tests. The layer has
a Q4_K projection long enough to be split across CTAs and a Q6_K one, so the
scratch holds Q8 buffers, scheduling state and partial sums.

The file sorts last so a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gguf_quant_integer_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_REL = 1e-5
TOL_ABS = 1e-7

PROJS = (synth.Proj("q", synth.Q4_K, 4096, 512, 0),
         synth.Proj("v", synth.Q6_K, 4096, 256, 0),
         synth.Proj("down", synth.Q4_K, 14336, 512, 1))


@pytest.fixture(scope="module")
def xq():
    from gguf_quant_integer_gb300 import build, xq as _xq
    build.build()
    _xq.lib()
    return _xq


def _run(xq, weights, xs, M, static):
    ys = [torch.full((M, p.N), float("nan"), dtype=torch.float32, device="cuda") for p in PROJS]
    desc = [(p.qtype, p.N, p.K, weights[t], ys[t], p.input) for t, p in enumerate(PROJS)]
    ins = [torch.from_numpy(x).cuda() for x in xs]
    if static:
        xq.layer_mixed_static(desc, ins, M)
    else:
        ws = torch.empty(xq.layer_workspace_bytes(desc, 2, M), dtype=torch.uint8, device="cuda")
        xq.layer_mixed(desc, ins, M, ws)
    torch.cuda.synchronize()
    return [y.cpu().numpy() for y in ys]


def test_static_scratch_matches_workspace_entry_point_three_calls(xq):
    weights = [torch.from_numpy(synth.gen_weight(p.qtype, 700 + t, p.N, p.K).reshape(-1)).cuda()
               for t, p in enumerate(PROJS)]
    host_w = [w.cpu().numpy() for w in weights]
    for call, M in enumerate((8, 3, 40)):
        xs = [synth.gen_x(800 + 10 * call + i, M, k) for i, k in enumerate((4096, 14336))]
        y_static = _run(xq, weights, xs, M, static=True)
        y_ws = _run(xq, weights, xs, M, static=False)
        q8 = [oracle.quantize_q8(x) for x in xs]
        for t, p in enumerate(PROJS):
            assert np.all(np.isfinite(y_static[t])), f"call {call}: {p.name} not written"
            assert np.array_equal(y_static[t].view(np.uint32), y_ws[t].view(np.uint32)), \
                f"call {call}: {p.name} differs from the workspace entry point"
            qs, d8, _ = q8[p.input]
            y_ref, ab, _ = oracle.matmul(p.qtype, host_w[t], qs, d8, p.K)
            err = np.abs(y_static[t].astype(np.float64) - y_ref)
            assert np.all(err <= TOL_REL * ab + TOL_ABS), f"call {call}: {p.name} out of tolerance"


def test_static_scratch_rejects_oversized_layer(xq):
    # A 512-token prefill input needs far more than the fixed array: refused
    # with XQ_ERR_WORKSPACE before anything is enqueued. The pointers are real
    # (small) device buffers, so nothing reads or writes a made-up address
    # even if the size check were skipped.
    W = torch.zeros(16 * (12288 // 256) * 144, dtype=torch.uint8, device="cuda")
    y = torch.full((512, 16), float("nan"), dtype=torch.float32, device="cuda")
    x = torch.zeros((512, 12288), dtype=torch.float32, device="cuda")
    P = xq.xq_proj
    arr = (P * 1)()
    arr[0].type, arr[0].N, arr[0].K, arr[0].W, arr[0].y, arr[0].input = 12, 16, 12288, W.data_ptr(), y.data_ptr(), 0
    ins = (ctypes.c_void_p * 1)(x.data_ptr())
    assert xq.lib().xq_layer_mixed_static(arr, 1, ins, 1, 512, None) == 4
    torch.cuda.synchronize()
    assert torch.isnan(y).all()
