"""Seeded synthetic inputs: GGUF Q4_K / Q6_K / Q8_0 weight bytes and fp32 activations.

This module holds no arithmetic of the method: it only draws bytes and
numbers. It is the one module that both the CUDA path's tests/bench and the
CPU oracle's tests use, so that both sides see identical inputs.

Distributions (the workload specification):
  Q4_K super-block (144 B): fp16 d and dmin drawn uniform in [1e-4, 1e-3]
  (fp32 draw, then round-to-nearest-even to fp16; the fp16 value is the
  truth); eight 6-bit scales and eight 6-bit mins uniform in 0..63; 256
  4-bit quants uniform in 0..15.
  Q6_K super-block (210 B): 256 6-bit quants uniform in 0..63; 16 int8
  scales uniform in [-32, 31]; fp16 d uniform in [1e-4, 1e-3].
  Q8_0 block (34 B per 32 weights): fp16 d uniform in [1e-4, 1e-3]; 32
  int8 quants uniform over all 256 byte values.
  Activations: fp32 N(0, 1).

The 12 packed scale/min bytes of Q4_K, its 128 nibble bytes, and the 192
ql/qh bytes of Q6_K use every bit of the fields they pack, one bit per bit,
so drawing those bytes uniformly is the same as drawing each packed field
uniformly and independently; the generator therefore draws the bytes and
never packs anything. Byte offsets: Q4_K d at 0, dmin at 2, scales 4..15,
quants 16..143; Q6_K ql 0..127, qh 128..191, scales 192..207, d at 208;
Q8_0 d at 0, quants 2..33.

RNG: numpy PCG64 via ``numpy.random.default_rng(seed)``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

Q8_0 = 8  # GGUF type ids
Q4_K = 12
Q6_K = 14
IQ4_XS = 23
BLOCK_BYTES = {Q4_K: 144, Q6_K: 210, Q8_0: 8 * 34, IQ4_XS: 136}  # bytes per 256 weights
TYPE_NAME = {Q4_K: "Q4_K", Q6_K: "Q6_K", Q8_0: "Q8_0", IQ4_XS: "IQ4_XS"}


def weight_bytes(qtype: int, N: int, K: int) -> int:
    return N * (K // 256) * BLOCK_BYTES[qtype]


def _fp16_uniform(rng, n, lo=1e-4, hi=1e-3) -> np.ndarray:
    return rng.uniform(lo, hi, size=n).astype(np.float32).astype(np.float16)


def gen_q4k(seed: int, N: int, K: int) -> np.ndarray:
    """Q4_K weight bytes, shape [N, K/256*144], uint8."""
    assert K % 256 == 0 and N >= 0
    rng = np.random.default_rng(seed)
    nblk = N * (K // 256)
    raw = np.frombuffer(rng.bytes(nblk * 144), np.uint8).reshape(nblk, 144).copy()
    raw[:, 0:2] = _fp16_uniform(rng, nblk).view(np.uint8).reshape(nblk, 2)
    raw[:, 2:4] = _fp16_uniform(rng, nblk).view(np.uint8).reshape(nblk, 2)
    return raw.reshape(N, (K // 256) * 144)


def gen_q6k(seed: int, N: int, K: int) -> np.ndarray:
    """Q6_K weight bytes, shape [N, K/256*210], uint8."""
    assert K % 256 == 0 and N >= 0
    rng = np.random.default_rng(seed)
    nblk = N * (K // 256)
    raw = np.frombuffer(rng.bytes(nblk * 210), np.uint8).reshape(nblk, 210).copy()
    raw[:, 192:208] = rng.integers(-32, 32, size=(nblk, 16), dtype=np.int8).view(np.uint8)
    raw[:, 208:210] = _fp16_uniform(rng, nblk).view(np.uint8).reshape(nblk, 2)
    return raw.reshape(N, (K // 256) * 210)


def gen_q8_0(seed: int, N: int, K: int) -> np.ndarray:
    """Q8_0 weight bytes, shape [N, K/32*34], uint8."""
    assert K % 256 == 0 and N >= 0
    rng = np.random.default_rng(seed)
    nblk = N * (K // 32)
    raw = np.frombuffer(rng.bytes(nblk * 34), np.uint8).reshape(nblk, 34).copy()
    raw[:, 0:2] = _fp16_uniform(rng, nblk).view(np.uint8).reshape(nblk, 2)
    return raw.reshape(N, (K // 32) * 34)


def gen_iq4xs(seed: int, N: int, K: int) -> np.ndarray:
    """IQ4_XS weight bytes, shape [N, K/256*136], uint8: d fp16 uniform in
    [1e-4, 1e-3], every other byte (scale bits, 4-bit indices) uniform."""
    assert K % 256 == 0 and N >= 0
    rng = np.random.default_rng(seed)
    nblk = N * (K // 256)
    raw = np.frombuffer(rng.bytes(nblk * 136), np.uint8).reshape(nblk, 136).copy()
    raw[:, 0:2] = _fp16_uniform(rng, nblk).view(np.uint8).reshape(nblk, 2)
    return raw.reshape(N, (K // 256) * 136)


def gen_codebook(seed: int) -> np.ndarray:
    """A synthetic IQ4_XS codebook: 16 distinct int8 values in increasing
    order, spread over the whole int8 range and denser near zero (a signed
    cube of evenly spaced points, jittered). It stands in for the format's
    table, which the pages name but do not print."""
    rng = np.random.default_rng(seed)
    t = np.linspace(-1.0, 1.0, 16) + rng.uniform(-0.02, 0.02, 16)
    v = np.clip(np.round(127.0 * np.sign(t) * np.abs(t) ** 1.6), -128, 127).astype(np.int64)
    v[0], v[-1] = -128, 127
    for i in range(1, 16):  # strictly increasing
        v[i] = max(v[i], v[i - 1] + 1)
    return v.astype(np.int8)


def gen_weight(qtype: int, seed: int, N: int, K: int) -> np.ndarray:
    if qtype == IQ4_XS:
        return gen_iq4xs(seed, N, K)
    if qtype == Q8_0:
        return gen_q8_0(seed, N, K)
    if qtype == Q4_K:
        return gen_q4k(seed, N, K)
    if qtype == Q6_K:
        return gen_q6k(seed, N, K)
    raise ValueError(qtype)


def gen_x(seed: int, M: int, K: int) -> np.ndarray:
    """fp32 N(0,1) activations [M, K]."""
    return np.random.default_rng(seed).standard_normal((M, K), dtype=np.float32)


# ------------------------------------------------------------ workloads

@dataclass(frozen=True)
class Proj:
    name: str
    qtype: int
    K: int          # input features
    N: int          # output features
    input: int      # which layer input feeds it (0 attn-in, 1 o-in, 2 ffn-in, 3 down-in)


@dataclass(frozen=True)
class Workload:
    key: str
    title: str
    projs: tuple
    layers: int = 1
    ms: tuple = (1,)
    seed_base: int = 0
    seed_stride: int = 7
    x_seed_base: int = 10000
    input_dims: tuple = field(default=())

    def weight_seed(self, layer: int, t: int) -> int:
        return self.seed_base + self.seed_stride * layer + t

    def x_seed(self, M: int) -> int:
        return self.x_seed_base + M

    def layer_weight_bytes(self) -> int:
        return sum(weight_bytes(p.qtype, p.N, p.K) for p in self.projs)

    def total_weight_bytes(self) -> int:
        return self.layers * self.layer_weight_bytes()


def _layer(h: int, f: int, kv: int, types: dict) -> tuple:
    t = lambda n: types.get(n, Q4_K)  # noqa: E731
    return (Proj("q", t("q"), h, h, 0), Proj("k", t("k"), h, kv, 0), Proj("v", t("v"), h, kv, 0),
            Proj("o", t("o"), h, h, 1), Proj("gate", t("gate"), h, f, 2),
            Proj("up", t("up"), h, f, 2), Proj("down", t("down"), f, h, 3))


WORKLOADS = {
    # Tiny Q4_K x Q8 GEMV: N=256 rows x K=2048, M=1, weight seed 0.
    "tiny-gemv": Workload("tiny-gemv", "Tiny Q4_K x Q8 GEMV 256x2048",
                          (Proj("w", Q4_K, 2048, 256, 0),), 1, (1,), 0, 7, 10000, (2048,)),
    # Qwen2.5-1.5B-shaped layer, all Q4_K: hidden 1536, ffn 8960, kv 256.
    "qwen2.5-1.5b-layer": Workload("qwen2.5-1.5b-layer", "Qwen2.5-1.5B-shaped layer, all Q4_K",
                                   _layer(1536, 8960, 256, {}), 1, (1, 2, 4, 8), 100, 7, 10100,
                                   (1536, 1536, 1536, 8960)),
    # Qwen2.5-1.5B-shaped layer in the Q4_K_M mix: attn_v and ffn_down Q6_K
    # (rows of 6 and 35 super-blocks: 1260 and 7350 bytes, not 16-byte
    # multiples), the rest Q4_K.
    "qwen2.5-1.5b-q4km-layer": Workload("qwen2.5-1.5b-q4km-layer", "Qwen2.5-1.5B-shaped layer, Q4_K with Q6_K v/down",
                                        _layer(1536, 8960, 256, {"v": Q6_K, "down": Q6_K}), 1, (1, 2, 4, 8),
                                        600, 7, 10600, (1536, 1536, 1536, 8960)),
    # Qwen2.5-1.5B-shaped layer requantized to Q8_0 (the Q8_0 model of the
    # xLLM v0.7 article, section B3 + B4).
    "qwen2.5-1.5b-q8_0-layer": Workload("qwen2.5-1.5b-q8_0-layer", "Qwen2.5-1.5B-shaped layer, all Q8_0",
                                        _layer(1536, 8960, 256, {n: Q8_0 for n in
                                                                 ("q", "k", "v", "o", "gate", "up", "down")}),
                                        1, (1, 2, 4, 8), 500, 7, 10500, (1536, 1536, 1536, 8960)),
    # Qwen3-8B-shaped mixed layer: attn_v and ffn_down Q6_K, the rest Q4_K.
    "qwen3-8b-mixed-layer": Workload("qwen3-8b-mixed-layer", "Qwen3-8B-shaped mixed Q4_K/Q6_K layer",
                                     _layer(4096, 12288, 1024, {"v": Q6_K, "down": Q6_K}), 1,
                                     (1, 2, 4, 8), 200, 7, 10200, (4096, 4096, 4096, 12288)),
    # Llama-3-8B-shaped 32-layer decode sweep, all Q4_K, 3.93 GB of weights.
    "llama3-8b-32layer": Workload("llama3-8b-32layer", "Llama-3-8B-shaped 32-layer Q4_K decode sweep",
                                  _layer(4096, 14336, 1024, {}), 32, (8,), 1000, 7, 10300,
                                  (4096, 4096, 4096, 14336)),
    # Qwen3-8B FFN prefill tile: M=512, up 4096->12288 Q4_K then down 12288->4096 Q6_K.
    "qwen3-8b-ffn-prefill512": Workload("qwen3-8b-ffn-prefill512", "Qwen3-8B FFN prefill tile, M=512",
                                        (Proj("up", Q4_K, 4096, 12288, 0), Proj("down", Q6_K, 12288, 4096, 1)),
                                        1, (512,), 400, 1, 10400, (4096, 12288)),
}


def gen_layer_weights(wl: Workload, layer: int):
    """List of weight byte arrays, one per projection of the layer."""
    return [gen_weight(p.qtype, wl.weight_seed(layer, t), p.N, p.K) for t, p in enumerate(wl.projs)]


def gen_layer_inputs(wl: Workload, M: int, layer: int = 0):
    """fp32 activations for each layer input, drawn in input order from one stream.

    The stream for layer L at batch M is seeded with x_seed(M) + 1_000_000 * L.
    """
    rng = np.random.default_rng(wl.x_seed(M) + 1_000_000 * layer)
    return [rng.standard_normal((M, k), dtype=np.float32) for k in wl.input_dims]
