"""Python binding of the xq C ABI (include/xq.h): argument marshalling only.

Every computation happens in libxq.so's CUDA kernels. Tensors are torch CUDA
tensors (torch supplies device memory and streams); the binding passes their
device pointers and the current stream to the C entry points of the same
name. A missing library is an error: there is no CPU or library fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libxq.so")

XQ_TYPE_Q8_0 = 8
XQ_TYPE_Q4_K = 12
XQ_TYPE_Q6_K = 14
XQ_TYPE_IQ4_XS = 23

STATUS = {0: "XQ_OK", 1: "XQ_ERR_ARG", 2: "XQ_ERR_SHAPE", 3: "XQ_ERR_ALIGN",
          4: "XQ_ERR_WORKSPACE", 5: "XQ_ERR_CUDA", 6: "XQ_ERR_UNSUPPORTED"}

# Every symbol include/xq.h declares.
SYMBOLS = ("xq_status_str", "xq_q8_bytes", "xq_weight_bytes", "xq_quantize_q8",
           "xq_matmul_q4k_q8", "xq_matmul_q6k_q8", "xq_layer_workspace_bytes",
           "xq_layer_mixed", "xq_debug_isums_q4k", "xq_debug_isums_q6k", "xq_layer_mixed_static",
           "xq_q8_bytes_invariant", "xq_quantize_q8_invariant", "xq_matmul_invariant",
           "xq_matmul_q8_0_q8", "xq_debug_isums_q8_0", "xq_silu_mul_quantize_q8",
           "xq_layer_ffn_workspace_bytes", "xq_layer_mixed_ffn", "xq_matmul_iq4xs_q8",
           "xq_debug_isums_iq4xs", "xq_device_error", "xq_debug_stalled_matmul_q4k", "xq_debug_tile_sums",
           "xq_debug_layer_matmuls", "xq_debug_check_probe", "xq_debug_stalled_ffn_layer")


class XQError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({lib().xq_status_str(code).decode()})")
        self.code = code


class xq_proj(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("W", ctypes.c_void_p), ("y", ctypes.c_void_p), ("input", ctypes.c_int),
                ("codebook", ctypes.c_void_p)]


_lib = None


def lib(path: str | None = None):
    """Open libxq.so (built in-tree by gguf_quant_integer_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libxq.so not found at {p}; build it with "
                           f"`python -m gguf_quant_integer_gb300.build` (no fallback exists)")
    L = ctypes.CDLL(p)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.xq_status_str.argtypes = [I]
    L.xq_status_str.restype = ctypes.c_char_p
    L.xq_q8_bytes.argtypes = [I, I]
    L.xq_q8_bytes.restype = S
    L.xq_weight_bytes.argtypes = [I, I, I]
    L.xq_weight_bytes.restype = S
    L.xq_quantize_q8.argtypes = [P, I, I, P, P]
    L.xq_silu_mul_quantize_q8.argtypes = [P, P, I, I, P, P, P]
    L.xq_silu_mul_quantize_q8.restype = I
    L.xq_layer_ffn_workspace_bytes.argtypes = [ctypes.POINTER(xq_proj), I, I, I, I, I, I]
    L.xq_layer_ffn_workspace_bytes.restype = S
    L.xq_layer_mixed_ffn.argtypes = [ctypes.POINTER(xq_proj), I, I, I, I, ctypes.POINTER(ctypes.c_void_p), I, I,
                                     P, S, P]
    L.xq_layer_mixed_ffn.restype = I
    L.xq_debug_stalled_ffn_layer.argtypes = L.xq_layer_mixed_ffn.argtypes
    L.xq_debug_stalled_ffn_layer.restype = I
    L.xq_q8_bytes_invariant.argtypes = [I, I]
    L.xq_q8_bytes_invariant.restype = S
    L.xq_quantize_q8_invariant.argtypes = [P, I, I, P, P]
    L.xq_quantize_q8_invariant.restype = I
    L.xq_matmul_invariant.argtypes = [I, P, P, I, I, I, P, P]
    L.xq_matmul_invariant.restype = I
    for fn in ("xq_matmul_q4k_q8", "xq_matmul_q6k_q8", "xq_matmul_q8_0_q8"):
        getattr(L, fn).argtypes = [P, P, I, I, I, P, P]
    for fn in ("xq_debug_isums_q4k", "xq_debug_isums_q6k", "xq_debug_isums_q8_0"):
        getattr(L, fn).argtypes = [P, P, I, I, I, P, P, P]
    L.xq_matmul_iq4xs_q8.argtypes = [P, P, P, I, I, I, P, P]
    L.xq_matmul_iq4xs_q8.restype = I
    L.xq_debug_isums_iq4xs.argtypes = [P, P, P, I, I, I, P, P, P]
    L.xq_debug_isums_iq4xs.restype = I
    L.xq_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
    L.xq_device_error.restype = I
    L.xq_debug_stalled_matmul_q4k.argtypes = [P, P, I, I, I, P, P]
    L.xq_debug_stalled_matmul_q4k.restype = I
    L.xq_debug_tile_sums.argtypes = [I, P, P, P, I, I, I, P, P, P]
    L.xq_debug_tile_sums.restype = I
    L.xq_layer_workspace_bytes.argtypes = [ctypes.POINTER(xq_proj), I, I, I]
    L.xq_layer_workspace_bytes.restype = S
    L.xq_layer_mixed.argtypes = [ctypes.POINTER(xq_proj), I, ctypes.POINTER(ctypes.c_void_p), I, I, P, S, P]
    L.xq_layer_mixed_static.argtypes = [ctypes.POINTER(xq_proj), I, ctypes.POINTER(ctypes.c_void_p), I, I, P]
    L.xq_debug_layer_matmuls.argtypes = [ctypes.POINTER(xq_proj), I, I, I, P, S, P]
    L.xq_debug_check_probe.argtypes = [P, P, I, I, I, P, P]
    for fn in ("xq_quantize_q8", "xq_matmul_q4k_q8", "xq_matmul_q6k_q8", "xq_debug_isums_q4k",
               "xq_debug_isums_q6k", "xq_layer_mixed", "xq_layer_mixed_static", "xq_matmul_q8_0_q8",
               "xq_debug_isums_q8_0", "xq_debug_layer_matmuls", "xq_debug_check_probe"):
        getattr(L, fn).restype = I
    if path is None:
        _lib = L
    return L


def _check(fn: str, rc: int):
    if rc != 0:
        raise XQError(fn, rc)


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def q8_bytes(M: int, K: int) -> int:
    return lib().xq_q8_bytes(M, K)


def weight_bytes(qtype: int, N: int, K: int) -> int:
    return lib().xq_weight_bytes(qtype, N, K)


def quantize_q8(x, out=None, stream=None):
    """Q8-quantize fp32 x [M, K] (CUDA) into a uint8 buffer of q8_bytes(M, K)."""
    import torch
    M, K = x.shape
    if out is None:
        out = torch.empty(q8_bytes(M, K), dtype=torch.uint8, device=x.device)
    _check("xq_quantize_q8", lib().xq_quantize_q8(_ptr(x), M, K, _ptr(out), _stream(stream)))
    return out


def q8_views(xq, M: int, K: int):
    """(qs int8 [M,K], d8 fp32 [M,K/32], s8 fp32 [M,K/32]) views into an xq buffer."""
    import torch
    mk = M * K
    qs = xq[:mk].view(torch.int8).view(M, K)
    d8 = xq[mk:mk + 4 * (mk // 32)].view(torch.float32).view(M, K // 32)
    s8 = xq[mk + 4 * (mk // 32):mk + 8 * (mk // 32)].view(torch.float32).view(M, K // 32)
    return qs, d8, s8


def matmul(qtype: int, W, xq, M: int, N: int, K: int, y=None, stream=None):
    """y [M, N] fp32 = x W^T from Q8 activations xq and GGUF weight bytes W (CUDA)."""
    import torch
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    fn = {XQ_TYPE_Q4_K: "xq_matmul_q4k_q8", XQ_TYPE_Q6_K: "xq_matmul_q6k_q8", XQ_TYPE_Q8_0: "xq_matmul_q8_0_q8"}[qtype]
    _check(fn, getattr(lib(), fn)(_ptr(W), _ptr(xq), M, N, K, _ptr(y), _stream(stream)))
    return y


def matmul_q4k_q8(W, xq, M, N, K, y=None, stream=None):
    return matmul(XQ_TYPE_Q4_K, W, xq, M, N, K, y, stream)


def matmul_q6k_q8(W, xq, M, N, K, y=None, stream=None):
    return matmul(XQ_TYPE_Q6_K, W, xq, M, N, K, y, stream)


def _codebook(codebook):
    """16 int8 codebook values as a host buffer (read by the C call)."""
    import numpy as np
    cb = np.ascontiguousarray(codebook, dtype=np.int8)
    if cb.shape != (16,):
        raise ValueError("an IQ4_XS codebook is 16 int8 values")
    return cb


def matmul_iq4xs_q8(W, codebook, xq, M: int, N: int, K: int, y=None, stream=None):
    """y [M, N] fp32 = x W^T for IQ4_XS weight bytes W and its 16-value int8
    codebook (host array), M <= 8."""
    import torch
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    cb = _codebook(codebook)
    _check("xq_matmul_iq4xs_q8", lib().xq_matmul_iq4xs_q8(_ptr(W), cb.ctypes.data, _ptr(xq), M, N, K, _ptr(y),
                                                         _stream(stream)))
    return y


def debug_isums_iq4xs(W, codebook, xq, M: int, N: int, K: int, y=None, isum=None, stream=None):
    """IQ4_XS matmul that also writes the exact int32 sub-block sums [M, N, K/32]."""
    import torch
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    if isum is None:
        isum = torch.empty((M, N, K // 32), dtype=torch.int32, device=W.device)
    cb = _codebook(codebook)
    _check("xq_debug_isums_iq4xs", lib().xq_debug_isums_iq4xs(_ptr(W), cb.ctypes.data, _ptr(xq), M, N, K, _ptr(y),
                                                             _ptr(isum), _stream(stream)))
    return y, isum


def q8_bytes_invariant(M: int, K: int) -> int:
    return lib().xq_q8_bytes_invariant(M, K)


def quantize_q8_invariant(x, out=None, stream=None):
    """Q8-quantize fp32 x [M, K] into the 8-token GEMV image for any M (the
    batch-invariant layout)."""
    import torch
    M, K = x.shape
    if out is None:
        out = torch.empty(q8_bytes_invariant(M, K), dtype=torch.uint8, device=x.device)
    _check("xq_quantize_q8_invariant", lib().xq_quantize_q8_invariant(_ptr(x), M, K, _ptr(out), _stream(stream)))
    return out


def matmul_invariant(qtype: int, W, xq, M: int, N: int, K: int, y=None, stream=None):
    """y [M, N] = x W^T with row m independent of M (batch-invariant mode)."""
    import torch
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    _check("xq_matmul_invariant",
           lib().xq_matmul_invariant(qtype, _ptr(W), _ptr(xq), M, N, K, _ptr(y), _stream(stream)))
    return y


def debug_isums(qtype: int, W, xq, M: int, N: int, K: int, y=None, isum=None, stream=None):
    """Matmul that also writes the exact int32 sub-block sums (test hook)."""
    import torch
    per = K // 16 if qtype == XQ_TYPE_Q6_K else K // 32
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    if isum is None:
        isum = torch.empty((M, N, per), dtype=torch.int32, device=W.device)
    fn = {XQ_TYPE_Q4_K: "xq_debug_isums_q4k", XQ_TYPE_Q6_K: "xq_debug_isums_q6k",
          XQ_TYPE_Q8_0: "xq_debug_isums_q8_0"}[qtype]
    _check(fn, getattr(lib(), fn)(_ptr(W), _ptr(xq), M, N, K, _ptr(y), _ptr(isum), _stream(stream)))
    return y, isum


def device_error(stream=None) -> int:
    """Read and clear the kernels' timed-out-wait record (xq_device_error):
    0 if no bounded device wait ran out since the last read, else
    (kernel << 8) | wait."""
    code = ctypes.c_uint(0)
    _check("xq_device_error", lib().xq_device_error(_stream(stream), ctypes.byref(code)))
    return code.value


def debug_stalled_matmul_q4k(W, xq, M: int, N: int, K: int, y, stream=None):
    """Test hook: the Q4_K warp-level MMA GEMV with no stage issued and short
    waits, so that its waits run out (y stays unwritten)."""
    _check("xq_debug_stalled_matmul_q4k",
           lib().xq_debug_stalled_matmul_q4k(_ptr(W), _ptr(xq), M, N, K, _ptr(y), _stream(stream)))


def debug_tile_sums(qtype: int, W, xq, M: int, N: int, K: int, codebook=None, y=None, sums=None, stream=None):
    """Tile-kernel matmul (M > 64) that also writes each 32-block's exact
    integer as the kernel accumulates it, int32 [M, N, K/32] (test hook)."""
    import torch
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    if sums is None:
        sums = torch.empty((M, N, K // 32), dtype=torch.int32, device=W.device)
    cb = _codebook(codebook) if codebook is not None else None
    _check("xq_debug_tile_sums", lib().xq_debug_tile_sums(qtype, _ptr(W), cb.ctypes.data if cb is not None else None,
                                                         _ptr(xq), M, N, K, _ptr(y), _ptr(sums), _stream(stream)))
    return y, sums


def _proj_array(projs):
    """projs: (type, N, K, W, y, input[, codebook]) tuples; an IQ4_XS entry
    carries its 16-value int8 codebook (host array) as the 7th element."""
    arr = (xq_proj * max(1, len(projs)))()
    keep = []
    for i, p in enumerate(projs):
        arr[i].type, arr[i].N, arr[i].K = int(p[0]), int(p[1]), int(p[2])
        arr[i].W = p[3].data_ptr() if p[3] is not None else None
        arr[i].y = p[4].data_ptr() if p[4] is not None else None
        arr[i].input = int(p[5])
        cb = p[6] if len(p) > 6 else None
        if cb is not None:
            cb = _codebook(cb)
            keep.append(cb)
            arr[i].codebook = cb.ctypes.data
    arr._codebooks = keep  # host codebooks live as long as the array
    return arr


def layer_workspace_bytes(projs, n_inputs: int, M: int) -> int:
    """projs: sequence of (type, N, K, W, y, input)."""
    return lib().xq_layer_workspace_bytes(_proj_array(projs), len(projs), n_inputs, M)


def layer_mixed(projs, inputs, M: int, workspace, stream=None):
    """Run one layer's projections. projs: (type, N, K, W, y, input) tuples;
    inputs: fp32 CUDA tensors [M, K_i]; workspace: uint8 CUDA tensor."""
    arr = _proj_array(projs)
    ins = (ctypes.c_void_p * max(1, len(inputs)))(*[t.data_ptr() for t in inputs])
    rc = lib().xq_layer_mixed(arr, len(projs), ins, len(inputs), M, _ptr(workspace),
                              workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("xq_layer_mixed", rc)


def debug_layer_matmuls(projs, n_inputs: int, M: int, workspace, stream=None):
    """The matmul launches of layer_mixed alone, on the Q8 activations the last
    layer_mixed call with the same projs, input count and M left in workspace."""
    arr = _proj_array(projs)
    rc = lib().xq_debug_layer_matmuls(arr, len(projs), n_inputs, M, _ptr(workspace),
                                      workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("xq_debug_layer_matmuls", rc)


def silu_mul_quantize_q8(gate, up, out=None, h_out=None, stream=None):
    """Q8 of h = silu(gate) * up (fp32 CUDA tensors [M, K]); h_out optional."""
    import torch
    M, K = gate.shape
    if out is None:
        out = torch.empty(q8_bytes(M, K), dtype=torch.uint8, device=gate.device)
    _check("xq_silu_mul_quantize_q8",
           lib().xq_silu_mul_quantize_q8(_ptr(gate), _ptr(up), M, K, _ptr(out), _ptr(h_out), _stream(stream)))
    return out


def layer_ffn_workspace_bytes(projs, n_inputs: int, M: int, gate: int, up: int, down: int) -> int:
    return lib().xq_layer_ffn_workspace_bytes(_proj_array(projs), len(projs), n_inputs, M, gate, up, down)


def layer_mixed_ffn(projs, gate: int, up: int, down: int, inputs, M: int, workspace, stream=None, _fn="xq_layer_mixed_ffn"):
    """layer_mixed with projs[down] fed by silu(y_gate) * y_up of the same call."""
    arr = _proj_array(projs)
    ins = (ctypes.c_void_p * max(1, len(inputs)))(*[t.data_ptr() for t in inputs])
    rc = getattr(lib(), _fn)(arr, len(projs), gate, up, down, ins, len(inputs), M, _ptr(workspace),
                             workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(_fn, rc)


def debug_stalled_ffn_layer(projs, gate: int, up: int, down: int, inputs, M: int, workspace, stream=None):
    """Test hook: layer_mixed_ffn's fused form with h never counted ready."""
    layer_mixed_ffn(projs, gate, up, down, inputs, M, workspace, stream, _fn="xq_debug_stalled_ffn_layer")


def layer_mixed_static(projs, inputs, M: int, stream=None):
    """layer_mixed without a workspace: the library's fixed per-device array
    (XQ_LAYER_STATIC_SCRATCH_BYTES) stands in for it; nothing is allocated."""
    arr = _proj_array(projs)
    ins = (ctypes.c_void_p * max(1, len(inputs)))(*[t.data_ptr() for t in inputs])
    _check("xq_layer_mixed_static", lib().xq_layer_mixed_static(arr, len(projs), ins, len(inputs), M, _stream(stream)))


class Layer:
    """Device-resident weights of one layer plus its outputs and workspace.

    Weights are uploaded once (the raw GGUF bytes stay resident; nothing is
    dequantized) and `forward` runs xq_layer_mixed on the current stream.
    """

    def __init__(self, projs, weights, M: int, device="cuda", codebooks=None):
        import torch
        self.projs = projs
        self.M = M
        self.W = [torch.from_numpy(w.reshape(-1)).to(device) for w in weights]
        self.y = [torch.empty((M, p.N), dtype=torch.float32, device=device) for p in projs]
        n_in = 1 + max(p.input for p in projs)
        self.n_inputs = n_in
        cbs = codebooks or [None] * len(projs)  # per projection; IQ4_XS needs one
        self.desc = [(p.qtype, p.N, p.K, self.W[i], self.y[i], p.input, cbs[i]) for i, p in enumerate(projs)]
        nb = layer_workspace_bytes(self.desc, n_in, M)
        self.workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=device)

    def forward(self, inputs, stream=None):
        layer_mixed(self.desc, inputs, self.M, self.workspace, stream)
        return self.y

    def weight_bytes(self) -> int:
        return sum(synth.weight_bytes(p.qtype, p.N, p.K) for p in self.projs)
