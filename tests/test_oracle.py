"""Pins for the CPU oracle, checked against things other than itself.

- hand-derived decode and Q8 fixtures (tests/golden/*.txt);
- an independent bit-offset reader for Q4_K / Q6_K / Q8_0 / IQ4_XS written
  from the format description, compared on every position of random blocks;
- one-hot blocks with closed-form weights;
- the integer route (exact sub-block sums + fp64 combine) against the plain
  dequantize-then-fp64-GEMV definition (they are one sum, rearranged);
- integer sub-block sums recomputed by brute force in numpy int64;
- the Q8 noise statistic (about 0.5% RMS, xLLM v0.7 article section B1.3)
  and its closed form, and arg-max preservation.
"""
import os

import numpy as np
import pytest

import oracle
from gguf_quant_integer_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ helpers

def _read_fixture(name):
    out = {}
    ws = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "w":
                ws.append((int(vals[0]), int(vals[1]), float(vals[2])))
            else:
                out[key] = vals
    out["w"] = ws
    return out


def _bits(buf: bytes, bit_off: int, nbits: int) -> int:
    """LSB-first bit reader over a byte string."""
    v = 0
    for i in range(nbits):
        b = bit_off + i
        v |= ((buf[b // 8] >> (b % 8)) & 1) << i
    return v


def _f16(buf: bytes, off: int) -> float:
    return float(np.frombuffer(buf[off:off + 2], np.float16)[0])


def ref_q4k_decode(blk: bytes):
    """Independent Q4_K field reader (bit offsets, not masks)."""
    d, dmin = _f16(blk, 0), _f16(blk, 2)
    S = 4 * 8  # bit offset of the 12 scale bytes
    sc, mn = [], []
    for j in range(8):
        if j < 4:
            sc.append(_bits(blk, S + 8 * j, 6))
            mn.append(_bits(blk, S + 8 * (j + 4), 6))
        else:
            sc.append(_bits(blk, S + 8 * (j + 4), 4) | (_bits(blk, S + 8 * (j - 4) + 6, 2) << 4))
            mn.append(_bits(blk, S + 8 * (j + 4) + 4, 4) | (_bits(blk, S + 8 * j + 6, 2) << 4))
    q = []
    for i in range(256):
        g, r = divmod(i, 64)
        byte = 16 + 32 * g + (r % 32)
        q.append(_bits(blk, 8 * byte + (0 if r < 32 else 4), 4))
    return d, dmin, sc, mn, q


def ref_q6k_decode(blk: bytes):
    """Independent Q6_K field reader (bit offsets, not masks)."""
    d = _f16(blk, 208)
    s = [int(np.int8(np.uint8(blk[192 + g]))) for g in range(16)]
    q = []
    for i in range(256):
        h, r = divmod(i, 128)
        quarter, l = divmod(r, 32)
        ql_byte = 64 * h + l + (32 if quarter in (1, 3) else 0)
        lo = _bits(blk, 8 * ql_byte + (4 if quarter >= 2 else 0), 4)
        hi = _bits(blk, 8 * (128 + 32 * h + l) + 2 * quarter, 2)
        q.append(lo | (hi << 4))
    return d, s, q


def pack_q4k(d_bits, dmin_bits, sc, mn, q):
    """Test-side packer (inverse of the reader above), for hand-built blocks."""
    blk = bytearray(144)
    blk[0:2] = int(d_bits).to_bytes(2, "little")
    blk[2:4] = int(dmin_bits).to_bytes(2, "little")
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    blk[4:16] = bytes(s)
    for i in range(256):
        g, r = divmod(i, 64)
        byte = 16 + 32 * g + (r % 32)
        if r < 32:
            blk[byte] = (blk[byte] & 0xF0) | q[i]
        else:
            blk[byte] = (blk[byte] & 0x0F) | (q[i] << 4)
    return bytes(blk)


# ------------------------------------------------------------ fp16

def test_half_to_double_matches_numpy_float16():
    for h in [0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0xC000, 0x3555, 0x7BFF, 0x1000, 0x0C00]:
        expect = float(np.array([h], np.uint16).view(np.float16)[0])
        assert oracle.half_to_double(h) == expect
    assert np.isinf(oracle.half_to_double(0x7C00))
    assert np.isnan(oracle.half_to_double(0x7E00))


# ------------------------------------------------------------ Q8

def _q8_block(spec):
    v = np.zeros(32, np.float64)
    for tok in spec:
        i, x = tok.split(":")
        v[int(i)] = float(x)
    return v


@pytest.mark.parametrize("blk", ["blockA", "blockB", "blockC"])
def test_q8_hand_blocks(blk):
    fx = _read_fixture("q8_hand_blocks.txt")
    x = _q8_block(fx[blk + "_x"]).astype(np.float32)[None, :]
    q_expect = _q8_block(fx[blk + "_q"]).astype(np.int8)
    qs, d8, s8 = oracle.quantize_q8(x)
    assert np.array_equal(qs[0], q_expect)
    assert d8[0, 0] == float(fx[blk + "_d8"][0])
    assert s8[0, 0] == float(fx[blk + "_s8"][0])


def test_q8_closed_form_cases():
    # one nonzero element: it maps to +-127, everything else to 0
    for pos in (0, 7, 31):
        for sgn in (1, -1):
            x = np.zeros((1, 32), np.float32)
            x[0, pos] = sgn * 3.7
            qs, d8, s8 = oracle.quantize_q8(x)
            expect = np.zeros(32, np.int8)
            expect[pos] = sgn * 127
            assert np.array_equal(qs[0], expect)
            assert d8[0, 0] == np.float32(3.7) / np.float32(127)
            assert np.isclose(s8[0, 0], sgn * 3.7, rtol=1e-6)
    # constant block: every element is the max, all 127, sum 4064
    x = np.full((1, 32), 0.3, np.float32)
    qs, d8, s8 = oracle.quantize_q8(x)
    assert np.all(qs == 127)
    assert np.isclose(s8[0, 0] / d8[0, 0], 4064, rtol=1e-6)
    # alternating sign: sum is 0
    x = np.array([[(-1) ** i * 2.0 for i in range(32)]], np.float32)
    qs, d8, s8 = oracle.quantize_q8(x)
    assert np.all(np.abs(qs) == 127) and s8[0, 0] == 0.0
    # blocks are independent: a big value in block 1 does not change block 0
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 64)).astype(np.float32)
    x2 = x.copy()
    x2[:, 40] = 1000.0
    a = oracle.quantize_q8(x)
    b = oracle.quantize_q8(x2)
    assert np.array_equal(a[0][:, :32], b[0][:, :32]) and np.array_equal(a[1][:, 0], b[1][:, 0])


def test_q8_bounds_and_reconstruction():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((8, 4096)) * rng.uniform(0.01, 100, (8, 1))).astype(np.float32)
    qs, d8, s8 = oracle.quantize_q8(x)
    assert np.abs(qs.astype(int)).max() == 127
    xh = oracle.dequant_q8(qs, d8)
    step = np.repeat(d8.astype(np.float64), 32, axis=1)
    # rounding to nearest: every reconstruction error is at most half a step
    assert np.all(np.abs(xh - x) <= 0.5 * step * (1 + 1e-6) + 1e-30)
    # s8 is the block sum times the scale (one fp32 rounding)
    sums = qs.reshape(8, -1, 32).astype(np.int64).sum(-1)
    assert np.allclose(s8, d8.astype(np.float64) * sums, rtol=1.2e-7, atol=0)


def test_q8_noise_is_about_half_a_percent():
    # xLLM v0.7 article, section B1.3: Q8 activation quantization adds about
    # 0.5% RMS noise. Closed form for a step d8 = amax/127: uniform rounding
    # error of variance d8^2/12, i.e. rel RMS = sqrt(E[amax^2])/(127*sqrt(12)).
    x = synth.gen_x(123, 64, 4096)
    qs, d8, _ = oracle.quantize_q8(x)
    xh = oracle.dequant_q8(qs, d8)
    rel = np.sqrt(np.mean((xh - x) ** 2) / np.mean(x.astype(np.float64) ** 2))
    amax = np.abs(x.reshape(-1, 32)).max(1).astype(np.float64)
    closed = np.sqrt(np.mean(amax ** 2)) / (127 * np.sqrt(12))
    assert 0.004 < rel < 0.006
    assert abs(rel - closed) / closed < 0.05


# ------------------------------------------------------------ Q4_K decode

def test_q4k_hand_fixture():
    fx = _read_fixture("q4k_block_hand.txt")
    blk = bytearray(144)
    blk[0:2] = int(fx["d_hex"][0], 16).to_bytes(2, "little")
    blk[2:4] = int(fx["dmin_hex"][0], 16).to_bytes(2, "little")
    blk[4:16] = bytes(int(v, 16) for v in fx["scales_hex"])
    blk[16:144] = bytes(range(128))
    d, dmin, sc, mn, q = oracle.q4k_fields(np.frombuffer(bytes(blk), np.uint8))
    assert d == 2.0 ** -11 and dmin == 2.0 ** -12
    assert list(sc) == [int(v) for v in fx["sc"]]
    assert list(mn) == [int(v) for v in fx["m"]]
    w = oracle.dequant_q4k(np.frombuffer(bytes(blk), np.uint8), 256)[0]
    for pos, qv, wv in fx["w"]:
        assert q[pos] == qv, pos
        assert w[pos] == wv, pos


def test_q4k_decode_matches_independent_reader():
    W = synth.gen_q4k(5, 3, 512)  # 6 random blocks
    for blk in W.reshape(-1, 144):
        b = bytes(blk)
        d, dmin, sc, mn, q = oracle.q4k_fields(blk)
        rd, rdmin, rsc, rmn, rq = ref_q4k_decode(b)
        assert (d, dmin) == (rd, rdmin)
        assert list(sc) == rsc and list(mn) == rmn and list(q) == rq
    w = oracle.dequant_q4k(W, 512)
    for n in range(3):
        for b in range(2):
            blk = bytes(W[n, b * 144:(b + 1) * 144])
            rd, rdmin, rsc, rmn, rq = ref_q4k_decode(blk)
            for i in range(256):
                expect = rd * rsc[i // 32] * rq[i] - rdmin * rmn[i // 32]
                assert w[n, b * 256 + i] == expect


def test_q4k_one_hot_blocks():
    # all scales and mins 63 (top bits set in every packed field), one
    # nonzero quant (15) at position p: w[p] = 63*15*d - 63*dmin, else -63*dmin.
    d_bits, dmin_bits = 0x1000, 0x0C00
    d, dmin = 2.0 ** -11, 2.0 ** -12
    for p in (0, 31, 32, 63, 64, 100, 191, 192, 255):
        q = [0] * 256
        q[p] = 15
        blk = pack_q4k(d_bits, dmin_bits, [63] * 8, [63] * 8, q)
        w = oracle.dequant_q4k(np.frombuffer(blk, np.uint8), 256)[0]
        expect = np.full(256, -63 * dmin)
        expect[p] = 63 * 15 * d - 63 * dmin
        assert np.array_equal(w, expect), p
    # one field at a time: sc_j = 48 (only the two top bits) for a single j
    for j in range(8):
        sc = [0] * 8
        sc[j] = 48
        blk = pack_q4k(d_bits, dmin_bits, sc, [0] * 8, [1] * 256)
        _, _, osc, omn, _ = oracle.q4k_fields(np.frombuffer(blk, np.uint8))
        assert list(osc) == sc and list(omn) == [0] * 8
        mn = [0] * 8
        mn[j] = 48
        blk = pack_q4k(d_bits, dmin_bits, [0] * 8, mn, [1] * 256)
        _, _, osc, omn, _ = oracle.q4k_fields(np.frombuffer(blk, np.uint8))
        assert list(omn) == mn and list(osc) == [0] * 8


# ------------------------------------------------------------ Q6_K decode

def test_q6k_hand_fixture():
    blk = bytearray(210)
    blk[0:128] = bytes(range(128))
    blk[128:192] = bytes([0xE4] * 64)
    blk[192:208] = np.arange(-8, 8, dtype=np.int8).view(np.uint8).tobytes()
    blk[208:210] = (0x1000).to_bytes(2, "little")
    fx = _read_fixture("q6k_block_hand.txt")
    d, s, q = oracle.q6k_fields(np.frombuffer(bytes(blk), np.uint8))
    assert d == 2.0 ** -11 and list(s) == list(range(-8, 8))
    w = oracle.dequant_q6k(np.frombuffer(bytes(blk), np.uint8), 256)[0]
    for pos, qv, wv in fx["w"]:
        assert q[pos] == qv, pos
        assert w[pos] == wv, pos


def test_q6k_decode_matches_independent_reader():
    W = synth.gen_q6k(7, 3, 512)
    for blk in W.reshape(-1, 210):
        d, s, q = oracle.q6k_fields(blk)
        rd, rs, rq = ref_q6k_decode(bytes(blk))
        assert d == rd and list(s) == rs and list(q) == rq
    w = oracle.dequant_q6k(W, 512)
    for n in range(3):
        for b in range(2):
            rd, rs, rq = ref_q6k_decode(bytes(W[n, b * 210:(b + 1) * 210]))
            for i in range(256):
                assert w[n, b * 256 + i] == rd * rs[i // 16] * (rq[i] - 32)


def test_q6k_extremes():
    # q = 0 -> w = -32*d*s ; q = 63 -> w = 31*d*s ; s in {-32, 31}
    for qv, s in ((0, -32), (63, 31), (0, 31), (63, -32)):
        blk = bytearray(210)
        lo, hi = qv & 15, qv >> 4
        blk[0:128] = bytes([lo | (lo << 4)] * 128)
        blk[128:192] = bytes([hi | (hi << 2) | (hi << 4) | (hi << 6)] * 64)
        blk[192:208] = np.full(16, s, np.int8).view(np.uint8).tobytes()
        blk[208:210] = (0x1000).to_bytes(2, "little")
        w = oracle.dequant_q6k(np.frombuffer(bytes(blk), np.uint8), 256)[0]
        assert np.all(w == 2.0 ** -11 * s * (qv - 32))


# ------------------------------------------------------------ matmul routes

@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_integer_route_equals_dequant_gemv(qtype, M):
    # The integer route is the dequantize-then-GEMV sum rearranged; in fp64
    # both agree to rounding: |diff| <= 1e-12 * sum|terms|.
    N, K = 40, 1024
    W = synth.gen_weight(qtype, 77 + M, N, K)
    x = synth.gen_x(500 + M, M, K)
    qs, d8, _ = oracle.quantize_q8(x)
    y, ab, _ = oracle.matmul(qtype, W, qs, d8, K)
    w = oracle.dequant_q4k(W, K) if qtype == synth.Q4_K else oracle.dequant_q6k(W, K)
    yd = oracle.gemv_f64(w, oracle.dequant_q8(qs, d8))
    assert np.all(np.abs(y - yd) <= 1e-12 * ab + 1e-300)
    assert np.all(ab > 0)


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K])
def test_isums_brute_force(qtype):
    N, K, M = 3, 512, 2
    W = synth.gen_weight(qtype, 9, N, K)
    x = synth.gen_x(19, M, K)
    qs, d8, _ = oracle.quantize_q8(x)
    _, _, isum = oracle.matmul(qtype, W, qs, d8, K, want_isum=True)
    nb = 144 if qtype == synth.Q4_K else 210
    for n in range(N):
        qrow = []
        for b in range(K // 256):
            blk = bytes(W[n, b * nb:(b + 1) * nb])
            if qtype == synth.Q4_K:
                qrow += ref_q4k_decode(blk)[4]
            else:
                qrow += [v - 32 for v in ref_q6k_decode(blk)[2]]
        qrow = np.array(qrow, np.int64)
        G = 32 if qtype == synth.Q4_K else 16
        for m in range(M):
            prod = (qrow * qs[m].astype(np.int64)).reshape(-1, G).sum(1)
            assert np.array_equal(isum[m, n], prod)


def test_min_term_sign_and_scale_association():
    # A Q4_K block with q = 0 everywhere computes -dmin * sum_j m_j * d8_j * isum8_j:
    # only the min term survives, with its minus sign.
    blk = pack_q4k(0x1000, 0x0C00, [5] * 8, list(range(1, 9)), [0] * 256)
    x = np.ones((1, 256), np.float32)
    qs, d8, _ = oracle.quantize_q8(x)          # all 127, d8 = 1/127
    y, _, _ = oracle.matmul_q4k_q8(np.frombuffer(blk, np.uint8), qs, d8, 256)
    expect = -(2.0 ** -12) * sum(m * float(d8[0, j]) * 127 * 32 for j, m in enumerate(range(1, 9)))
    assert y[0, 0] == pytest.approx(expect, rel=1e-12)


def test_q8_output_noise_and_argmax():
    # y from the Q8 route vs y from the unquantized fp32 activations: about
    # 0.5% RMS relative noise, and the arg-max over each row survives where
    # the top-2 gap is well above that noise (xLLM v0.7 article, B1.3).
    wl = synth.WORKLOADS["tiny-gemv"]
    p = wl.projs[0]
    W = synth.gen_q4k(wl.weight_seed(0, 0), p.N, p.K)
    x = synth.gen_x(4242, 8, p.K)
    qs, d8, _ = oracle.quantize_q8(x)
    y, _, _ = oracle.matmul_q4k_q8(W, qs, d8, p.K)
    w = oracle.dequant_q4k(W, p.K)
    yf = oracle.gemv_f64(w, x.astype(np.float64))
    rel = np.sqrt(np.mean((y - yf) ** 2) / np.mean(yf ** 2))
    assert 0.003 < rel < 0.007
    noise = np.sqrt(np.mean((y - yf) ** 2))
    checked = 0
    for m in range(8):
        top = np.sort(yf[m])[::-1]
        if top[0] - top[1] > 6 * noise:
            assert np.argmax(y[m]) == np.argmax(yf[m])
            checked += 1
    assert checked >= 1


def test_q8_overflowing_reciprocal_saturates():
    # amax so small that 1/d8 overflows to inf: x*id is +-inf for x != 0
    # (saturates to +-127) and NaN for x == 0 (maps to 0).
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = np.float32(3e-41)
    x[0, 1] = np.float32(-1e-41)
    qs, d8, s8 = oracle.quantize_q8(x)
    assert np.isinf(np.float32(1.0) / d8[0, 0])
    expect = np.zeros(32, np.int8)
    expect[0], expect[1] = 127, -127
    assert np.array_equal(qs[0], expect) and s8[0, 0] == 0.0


# ------------------------------------------------------------ Q8_0

def ref_q8_0_decode(blk: bytes):
    """Independent Q8_0 reader: d from the first two bytes as binary16, then
    each quant from its 8 bits as a two's-complement number."""
    d = _f16(blk, 0)
    q = []
    for i in range(32):
        u = _bits(blk, 8 * (2 + i), 8)
        q.append(u - 256 if u >= 128 else u)
    return d, q


def test_q8_0_decode_matches_independent_reader():
    W = synth.gen_q8_0(11, 3, 512)
    assert W.shape == (3, 16 * 34)
    for blk in W.reshape(-1, 34):
        d, q = oracle.q8_0_fields(blk)
        rd, rq = ref_q8_0_decode(bytes(blk))
        assert d == rd and list(q) == rq
    w = oracle.dequant_q8_0(W, 512)
    for n in range(3):
        for b in range(16):
            rd, rq = ref_q8_0_decode(bytes(W[n, 34 * b:34 * (b + 1)]))
            for i in range(32):
                assert w[n, 32 * b + i] == rd * rq[i]


def test_q8_0_extremes_and_hand_block():
    # every byte value as a quant: w = d * (int8) byte, with d = 2^-11 exactly
    blk = bytearray(34 * 8)
    vals = np.arange(256, dtype=np.uint8)
    for b in range(8):
        blk[34 * b:34 * b + 2] = (0x1000).to_bytes(2, "little")   # binary16 2^-11
        blk[34 * b + 2:34 * b + 34] = vals[32 * b:32 * (b + 1)].tobytes()
    w = oracle.dequant_q8_0(np.frombuffer(bytes(blk), np.uint8), 256)[0]
    assert np.array_equal(w, 2.0 ** -11 * vals.view(np.int8).astype(np.float64))
    # the product route on one-hot activations picks single weights back out
    qs = np.zeros((1, 256), np.int8)
    qs[0, 200] = 1
    d8 = np.ones((1, 8), np.float32)
    y, ab, isum = oracle.matmul_q8_0_q8(np.frombuffer(bytes(blk), np.uint8), qs, d8, 256, want_isum=True)
    assert y[0, 0] == 2.0 ** -11 * np.int8(200 - 256) and ab[0, 0] == abs(y[0, 0])
    assert isum[0, 0, 6] == 200 - 256 and np.count_nonzero(isum) == 1


def test_q8_0_integer_route_equals_dequant_gemv():
    for M in (1, 3, 8):
        N, K = 40, 1024
        W = synth.gen_weight(synth.Q8_0, 88 + M, N, K)
        x = synth.gen_x(600 + M, M, K)
        qs, d8, _ = oracle.quantize_q8(x)
        y, ab, _ = oracle.matmul(synth.Q8_0, W, qs, d8, K)
        yd = oracle.gemv_f64(oracle.dequant_q8_0(W, K), oracle.dequant_q8(qs, d8))
        assert np.all(np.abs(y - yd) <= 1e-12 * ab + 1e-300)
        assert np.all(ab > 0)


def test_q8_0_isums_brute_force():
    N, K, M = 3, 512, 2
    W = synth.gen_weight(synth.Q8_0, 12, N, K)
    x = synth.gen_x(21, M, K)
    qs, d8, _ = oracle.quantize_q8(x)
    _, _, isum = oracle.matmul(synth.Q8_0, W, qs, d8, K, want_isum=True)
    for n in range(N):
        qrow = []
        for b in range(K // 32):
            qrow += ref_q8_0_decode(bytes(W[n, 34 * b:34 * (b + 1)]))[1]
        qrow = np.array(qrow, np.int64)
        for m in range(M):
            assert np.array_equal(isum[m, n], (qrow * qs[m].astype(np.int64)).reshape(-1, 32).sum(1))


# ------------------------------------------------------------ IQ4_XS

def ref_iq4xs_decode(blk: bytes, codebook):
    """Independent IQ4_XS reader (bit offsets, not masks), from the block
    description: d fp16 at 0, scales_h (16 bits) at 2, scales_l (4 bytes) at
    4, 128 index bytes at 8; sub-block j's 6-bit scale takes 4 bits from
    scales_l at bit 4j and 2 bits from scales_h at bit 2j; weight i of
    sub-block j is the low (i < 16) or high nibble of index byte 16j + i%16."""
    d = _f16(blk, 0)
    ls = [_bits(blk, 32 + 4 * j, 4) | (_bits(blk, 16 + 2 * j, 2) << 4) for j in range(8)]
    v = []
    for i in range(256):
        j, r = divmod(i, 32)
        byte = 8 + 16 * j + (r % 16)
        v.append(int(codebook[_bits(blk, 8 * byte + (4 if r >= 16 else 0), 4)]))
    return d, ls, v


def test_iq4xs_decode_matches_independent_reader():
    cb = synth.gen_codebook(3)
    W = synth.gen_iq4xs(31, 3, 512)
    assert W.shape == (3, 2 * 136)
    for blk in W.reshape(-1, 136):
        d, ls, v = oracle.iq4xs_fields(blk, cb)
        rd, rls, rv = ref_iq4xs_decode(bytes(blk), cb)
        assert d == rd and list(ls) == rls and list(v) == rv
    w = oracle.dequant_iq4xs(W, 512, cb)
    for n in range(3):
        for b in range(2):
            rd, rls, rv = ref_iq4xs_decode(bytes(W[n, 136 * b:136 * (b + 1)]), cb)
            for i in range(256):
                assert w[n, 256 * b + i] == rd * (rls[i // 32] - 32) * rv[i]


def test_iq4xs_one_hot_and_scale_extremes():
    cb = np.arange(-8, 8, dtype=np.int8) * 3 + 1      # index k -> 3k - 23, all distinct
    blk = bytearray(136)
    blk[0:2] = (0x3C00).to_bytes(2, "little")         # d = 1
    # sub-block scales: ls = 0, 63, 33, 32, 1, 62, 17, 48 through both bit fields
    ls = [0, 63, 33, 32, 1, 62, 17, 48]
    sh = 0
    for j, l in enumerate(ls):
        blk[4 + j // 2] |= (l & 15) << (4 * (j % 2))
        sh |= (l >> 4) << (2 * j)
    blk[2:4] = sh.to_bytes(2, "little")
    # every index 8 (value 1) except one high and one low nibble per sub-block
    for k in range(128):
        blk[8 + k] = 0x88
    for j in range(8):
        blk[8 + 16 * j + j] = (blk[8 + 16 * j + j] & 0xF0) | j          # weight 32j + j: index j
        blk[8 + 16 * j + 15 - j] = (blk[8 + 16 * j + 15 - j] & 0x0F) | ((15 - j) << 4)  # weight 32j + 31 - j
    w = oracle.dequant_iq4xs(np.frombuffer(bytes(blk), np.uint8), 256, cb)[0]
    for j in range(8):
        s = ls[j] - 32
        for i in range(32):
            idx = j if i == j else (15 - j if i == 31 - j else 8)
            assert w[32 * j + i] == s * (3 * idx - 23), (j, i)
    assert w[0] == -32 * -23 and w[32 + 30] == 31 * (3 * 14 - 23)


@pytest.mark.parametrize("M", [1, 3, 8])
def test_iq4xs_integer_route_equals_dequant_gemv(M):
    cb = synth.gen_codebook(M)
    N, K = 40, 1024
    W = synth.gen_iq4xs(90 + M, N, K)
    x = synth.gen_x(700 + M, M, K)
    qs, d8, _ = oracle.quantize_q8(x)
    y, ab, _ = oracle.matmul(synth.IQ4_XS, W, qs, d8, K, codebook=cb)
    yd = oracle.gemv_f64(oracle.dequant_iq4xs(W, K, cb), oracle.dequant_q8(qs, d8))
    assert np.all(np.abs(y - yd) <= 1e-12 * ab + 1e-300)
    assert np.all(ab > 0)


def test_iq4xs_isums_brute_force():
    cb = synth.gen_codebook(9)
    N, K, M = 3, 512, 2
    W = synth.gen_iq4xs(13, N, K)
    x = synth.gen_x(22, M, K)
    qs, d8, _ = oracle.quantize_q8(x)
    _, _, isum = oracle.matmul(synth.IQ4_XS, W, qs, d8, K, want_isum=True, codebook=cb)
    for n in range(N):
        vrow = []
        for b in range(K // 256):
            vrow += ref_iq4xs_decode(bytes(W[n, 136 * b:136 * (b + 1)]), cb)[2]
        vrow = np.array(vrow, np.int64)
        for m in range(M):
            assert np.array_equal(isum[m, n], (vrow * qs[m].astype(np.int64)).reshape(-1, 32).sum(1))


def test_gen_codebook_is_sixteen_increasing_int8():
    for seed in range(5):
        cb = synth.gen_codebook(seed)
        assert cb.dtype == np.int8 and cb.shape == (16,)
        assert np.all(np.diff(cb.astype(np.int64)) > 0) and cb[0] == -128 and cb[-1] == 127


# ------------------------------------------------------------ sum|terms| pins

def _absterm_fixture():
    """tests/golden/absterm_hand.txt: key -> list of value strings."""
    out = {}
    with open(os.path.join(GOLD, "absterm_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *vals = line.split()
                out[key] = vals
    return out


def _hand_activation(fx):
    """The fixture's token: 32 copies of a_j per 32-block, d8_j = 2^e."""
    a = [int(v) for v in fx["a"]]
    qs = np.repeat(np.array(a, np.int8), 32).reshape(1, 256)
    d8 = np.full((1, 8), np.float32(2.0 ** int(fx["d8_log2"][0])), np.float32)
    return qs, d8


def _hex_bytes(vals):
    return [int(v, 16) for v in vals]


def test_absterm_q4k_hand_block():
    # Both the d-term and the dmin-term enter sum|terms| with their absolute
    # values: the fixture's terms alternate in sign, so a missing fabs, a
    # doubled or dropped min term changes the value.
    fx = _absterm_fixture()
    qs, d8 = _hand_activation(fx)
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.frombuffer(int(fx["q4k_d_hex"][0], 16).to_bytes(2, "little"), np.uint8)
    blk[2:4] = np.frombuffer(int(fx["q4k_dmin_hex"][0], 16).to_bytes(2, "little"), np.uint8)
    blk[4:16] = _hex_bytes(fx["q4k_scales_hex"])
    blk[16:] = int(fx["q4k_quant_byte"][0], 16)
    y, ab, _ = oracle.matmul(synth.Q4_K, blk.reshape(1, 144), qs, d8, 256)
    scale = 2.0 ** int(fx["q4k_log2"][0])
    assert y[0, 0] == int(fx["q4k_y_num"][0]) * scale
    assert ab[0, 0] == int(fx["q4k_abs_num"][0]) * scale


def test_absterm_q6k_hand_block():
    # y cancels to a small value while sum|terms| stays large: the pin of the
    # tolerance denominator is independent of y.
    fx = _absterm_fixture()
    qs, d8 = _hand_activation(fx)
    blk = np.zeros(210, np.uint8)
    blk[0:128] = int(fx["q6k_ql_byte"][0], 16)
    blk[128:192] = int(fx["q6k_qh_byte"][0], 16)
    blk[192:208] = np.array([int(v) for v in fx["q6k_scales"]], np.int8).view(np.uint8)
    blk[208:210] = np.frombuffer(int(fx["q6k_d_hex"][0], 16).to_bytes(2, "little"), np.uint8)
    y, ab, _ = oracle.matmul(synth.Q6_K, blk.reshape(1, 210), qs, d8, 256)
    scale = 2.0 ** int(fx["q6k_log2"][0])
    assert y[0, 0] == int(fx["q6k_y_num"][0]) * scale
    assert ab[0, 0] == int(fx["q6k_abs_num"][0]) * scale


def test_absterm_iq4xs_hand_block():
    fx = _absterm_fixture()
    qs, d8 = _hand_activation(fx)
    cb = np.array([int(v) for v in fx["iq4xs_codebook"]], np.int8)
    blk = np.zeros(136, np.uint8)
    blk[0:2] = np.frombuffer(int(fx["iq4xs_d_hex"][0], 16).to_bytes(2, "little"), np.uint8)
    blk[2:4] = np.frombuffer(int(fx["iq4xs_scales_h_hex"][0], 16).to_bytes(2, "little"), np.uint8)
    blk[4:8] = _hex_bytes(fx["iq4xs_scales_l_hex"])
    blk[8:] = int(fx["iq4xs_index_byte"][0], 16)
    y, ab, _ = oracle.matmul(synth.IQ4_XS, blk.reshape(1, 136), qs, d8, 256, codebook=cb)
    scale = 2.0 ** int(fx["iq4xs_log2"][0])
    assert y[0, 0] == int(fx["iq4xs_y_num"][0]) * scale
    assert ab[0, 0] == int(fx["iq4xs_abs_num"][0]) * scale


def test_threads_do_not_change_results():
    # output rows shared out among threads: every output is still computed by
    # one thread in the same order, so the results are bit-identical
    N, K, M = 37, 1024, 3
    x = synth.gen_x(61, M, K)
    qs, d8, _ = oracle.quantize_q8(x)
    cb = synth.gen_codebook(2)
    for qtype in (synth.Q4_K, synth.Q6_K, synth.Q8_0, synth.IQ4_XS):
        W = synth.gen_weight(qtype, 62, N, K) if qtype != synth.IQ4_XS else synth.gen_iq4xs(62, N, K)
        oracle.set_threads(1)
        one = oracle.matmul(qtype, W, qs, d8, K, want_isum=True, codebook=cb)
        used = oracle.set_threads(4)
        many = oracle.matmul(qtype, W, qs, d8, K, want_isum=True, codebook=cb)
        oracle.set_threads(1)
        assert used >= 1
        for a, b in zip(one, many):
            assert np.array_equal(a, b)


# ------------------------------------------------------------ SwiGLU feed

def test_silu_mul_pins():
    """oracle.silu_mul against what the definition silu(g) = g * sigma(g)
    fixes without retyping it:
    - sigma(ln 3) = 3/4 and sigma(-ln 3) = 1/4, so at the fp32 values nearest
      +-ln 3, h = 0.75 g u and 0.25 g u up to sigma's slope times the fp32
      rounding of ln 3 (relative 1e-7); this tells sigma(g) from sigma(-g);
    - silu(g) - silu(-g) = g for every g (sigma(g) + sigma(-g) = 1);
    - the limits: h = g u once e^-g is below fp64 resolution (g = 40, 100),
      h = +-0 once e^-g overflows (g = -800, -1e30), h = 0 at g = 0;
    - h is linear in u (u used once, as a factor)."""
    ln3 = np.float32(np.log(3.0))
    g = np.array([ln3, -ln3], np.float32)
    u = np.array([1.0, 1.0], np.float32)
    h = oracle.silu_mul(g, u)
    assert abs(h[0] - 0.75 * float(g[0])) <= 1e-7 * abs(float(g[0]))
    assert abs(h[1] - 0.25 * float(g[1])) <= 1e-7 * abs(float(g[1]))
    rng = np.random.default_rng(5)
    gs = (rng.standard_normal(2000) * 6).astype(np.float32)
    one = np.ones_like(gs)
    diff = oracle.silu_mul(gs, one) - oracle.silu_mul(-gs, one)
    assert np.all(np.abs(diff - gs.astype(np.float64)) <= 4e-16 * np.abs(gs) + 1e-300)
    lim = np.array([40.0, 100.0, -800.0, -1e30, 0.0], np.float32)
    ul = np.array([3.0, -2.0, 5.0, 7.0, 9.0], np.float32)
    hl = oracle.silu_mul(lim, ul)
    assert hl[0] == 120.0 and hl[1] == -200.0
    assert hl[2] == 0.0 and hl[3] == 0.0 and hl[4] == 0.0
    # u on a 2^-10 grid, so that u1 + u2 is exact in fp32
    u1 = (rng.integers(-4096, 4096, 2000) / 1024.0).astype(np.float32)
    u2 = (rng.integers(-4096, 4096, 2000) / 1024.0).astype(np.float32)
    h12 = oracle.silu_mul(gs, u1 + u2)
    lin = oracle.silu_mul(gs, u1) + oracle.silu_mul(gs, u2)
    assert np.all(np.abs(h12 - lin) <= 1e-15 * (np.abs(oracle.silu_mul(gs, u1)) + np.abs(oracle.silu_mul(gs, u2))))
