"""GPU check of the matmul-only timing hook (xq_debug_layer_matmuls).

After a layer call, re-running only its matmul launches on the Q8 that the
call left in the workspace rewrites every output with the same bits, and
does so again on a second run: the launches leave the workspace's task
counters and split-K arrival counts at zero. Covered: the grouped GEMV with
the dynamic task counter and split-K (M <= 8, including the one- and
two-token form), GEMV chunks with per-chunk splits (8 < M <= 64) and the
tile kernel (M > 64).
"""
import numpy as np
import pytest
import torch

from gguf_quant_integer_gb300 import synth

pytestmark = pytest.mark.gpu

RAGGED = synth.Workload(
    key="hook-ragged", title="ragged split-K layer",
    projs=(synth.Proj("a", synth.Q4_K, 8192, 100, 0), synth.Proj("b", synth.Q6_K, 8192, 40, 0),
           synth.Proj("c", synth.Q4_K, 6400, 1000, 1), synth.Proj("d", synth.Q4_K, 6400, 17, 1)),
    seed_base=960, x_seed_base=19600, input_dims=(8192, 6400))


@pytest.fixture(scope="module")
def xq():
    from gguf_quant_integer_gb300 import build, xq as _xq
    build.build()
    _xq.lib()
    return _xq


@pytest.mark.parametrize("key", ["hook-ragged", "qwen3-8b-mixed-layer"])
@pytest.mark.parametrize("M", [1, 2, 8, 40, 80])
def test_matmuls_alone_rewrite_the_same_bits(xq, key, M):
    wl = RAGGED if key == "hook-ragged" else synth.WORKLOADS[key]
    L = xq.Layer(wl.projs, synth.gen_layer_weights(wl, 0), M)
    ins = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in synth.gen_layer_inputs(wl, M, 0)]
    L.forward(ins)
    torch.cuda.synchronize()
    ref = [y.clone() for y in L.y]
    for _ in range(2):
        for y in L.y:
            y.fill_(float("nan"))
        xq.debug_layer_matmuls(L.desc, L.n_inputs, M, L.workspace)
        torch.cuda.synchronize()
        for t, (y, r) in enumerate(zip(L.y, ref)):
            assert torch.equal(y.view(torch.int32), r.view(torch.int32)), (key, M, wl.projs[t].name)
    assert xq.device_error() == 0
