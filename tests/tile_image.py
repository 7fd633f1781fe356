"""The M > 8 operand image of the Q8 buffer, restated from its definition in
include/xq.h (test helper shared by the CPU and GPU tests)."""
import numpy as np

PR4 = [0, 2, 1, 3]


def tile_offsets():
    """Byte offset of (token r, k-slot s) in a 128 x 32 operand (include/xq.h)."""
    r = np.arange(128)[:, None]
    s = np.arange(32)[None, :]
    return (r // 8) * 512 + (s // 8) * 128 + (r % 8) * 16 + (s % 8) * 2


def bf16_pieces(v):
    """s8 split into three bf16 numbers by truncation, as fp32 values."""
    v = np.asarray(v, np.float32)
    p0 = (v.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    r1 = (v - p0).astype(np.float32)
    p1 = (r1.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    p2 = (r1 - p1).astype(np.float32)
    return p0, p1, p2


def expected_tile_image(qs, d8, s8):
    """The M > 8 operand image restated from its definition in include/xq.h."""
    M, K = qs.shape
    T, NB = -(-M // 128), K // 256
    qp = np.zeros((128 * T, K), np.int8)
    qp[:M] = qs
    dp = np.zeros((128 * T, K // 32), np.float32)
    dp[:M] = d8
    sp = np.zeros((128 * T, K // 32), np.float32)
    sp[:M] = s8
    off = tile_offsets() // 2
    slot_feat = np.array([4 * (s // 4) + PR4[s % 4] for s in range(32)])
    rec = np.zeros((T, NB, 77824), np.uint8)
    for t in range(T):
        rows = slice(128 * t, 128 * t + 128)
        for b in range(NB):
            for i in range(8):
                j = 8 * b + i
                op = np.zeros(4096, np.uint16)
                op[off] = qp[rows, 32 * j + slot_feat].astype(np.float16).view(np.uint16)
                item = rec[t, b, i * 8704:(i + 1) * 8704]
                item[:8192] = op.view(np.uint8)
                item[8192:] = np.ascontiguousarray(dp[rows, j]).view(np.uint8)
            beta = np.zeros(4096, np.uint16)
            for i in range(8):
                for p, pc in enumerate(bf16_pieces(sp[rows, 8 * b + i])):
                    beta[off[:, 3 * i + p]] = (pc.view(np.uint32) >> 16).astype(np.uint16)
            rec[t, b, 8 * 8704:] = beta.view(np.uint8)
    return rec
