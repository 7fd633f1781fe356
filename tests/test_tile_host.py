"""Host-side checks of the M > 8 operand image definition (no GPU).

The tile kernel's min-term MMA is exact only if the three bf16 pieces of
every s8 add up to s8; the restated image must tile its 8,192-byte operands
without overlap.
"""
import numpy as np

import oracle
from gguf_quant_integer_gb300 import synth
from tile_image import bf16_pieces, tile_offsets


def test_bf16_split_is_exact():
    for seed, scale in ((17, 1.0), (18, 40.0), (19, 1e-30), (20, 3e30)):
        x = synth.gen_x(seed, 64, 2048) * np.float32(scale)
        _, _, s8 = oracle.quantize_q8(x)
        p0, p1, p2 = bf16_pieces(s8)
        for p in (p0, p1, p2):
            assert np.all((p.view(np.uint32) & np.uint32(0xFFFF)) == 0)
        assert np.array_equal(p0.astype(np.float64) + p1 + p2, s8.astype(np.float64))


def test_operand_layout_is_a_bijection():
    off = tile_offsets()
    assert off.shape == (128, 32)
    assert np.all(off % 2 == 0)
    assert np.array_equal(np.sort(off.ravel()), np.arange(0, 8192, 2))
