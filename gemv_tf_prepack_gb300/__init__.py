"""Python binding of libtf, the GB300 fused INT4/INT8-weight linear layer.

Argument marshalling only: every step of the computation runs in libtf's
CUDA kernels, reached through its C ABI (``include/tf.h``) with ctypes.
PyTorch supplies device memory and streams.  There is no fallback: if
``libtf.so`` has not been built, importing the device calls raises.

    from gemv_tf_prepack_gb300 import prepack, Weights, gemv, gemm
    blob = prepack(qweight, scales, zeros, N, K, bits=4, group=128)   # host, offline
    W = Weights.upload(blob)                                          # device copy
    y = gemv(W, x)     # x: torch.bfloat16 [M<=8, K] on the GPU -> y [M, N]
    y = gemm(W, x)     # any M
"""

from __future__ import annotations

import ctypes
import os
import re

import numpy as np

__all__ = [
    "TFError", "lib", "lib_path", "version", "prepack_size", "prepack", "prepack_awq", "unprepack",
    "blob_info", "Weights", "dequant", "gemv", "gemv_workspace_size", "gemv_noalloc", "gemm",
    "gemm_workspace_size", "device_error", "test_stall_copies",
    "header_declarations",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
lib_path = os.path.join(_HERE, "libtf.so")
HEADER = os.path.join(_ROOT, "include", "tf.h")

TF_OK = 0


class TFError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        msg = _lib().tf_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{call}: {msg} ({status})")


_LIB = None

_i = ctypes.c_int
_sz = ctypes.c_size_t
_p = ctypes.c_void_p

_SIGNATURES = {
    "tf_version": (_i, []),
    "tf_status_string": (ctypes.c_char_p, [_i]),
    "tf_prepack_size": (_i, [_i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "tf_prepack": (_i, [_p, _p, _p, _i, _i, _i, _i, _p, _sz]),
    "tf_prepack_awq": (_i, [_p, _p, _p, _i, _i, _i, _p, _sz]),
    "tf_unprepack": (_i, [_p, _sz, _p, _p, _p]),
    "tf_blob_info": (_i, [_p, _sz] + [ctypes.POINTER(_i)] * 4),
    "tf_dequant": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p]),
    "tf_gemv_workspace_size": (_i, [_i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "tf_gemv": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _i, _p, _sz, _p]),
    "tf_gemv_bias": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _p, _i, _p, _sz, _p]),
    "tf_gemm_workspace_size": (_i, [_i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "tf_gemm": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _i, _p, _sz, _p]),
    "tf_gemm_bias": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _p, _i, _p, _sz, _p]),
    "tf_gemv_noalloc": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _i, _p]),
    "tf_prepack_gate_up": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _p, _sz]),
    "tf_gemv_silu_gate": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _p, _i, _p, _sz, _p]),
    "tf_gemm_silu_gate": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _p, _i, _p, _sz, _p]),
    "tf_gemv_qkv": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _p, _p, _p, _i, _i, _i, _p, _sz, _p]),
    "tf_gemm_qkv": (_i, [_p, _sz, _i, _i, _i, _i, _p, _p, _p, _p, _p, _i, _i, _i, _p, _sz, _p]),
    "tf_device_error": (_i, [ctypes.POINTER(ctypes.c_uint)]),
    "tf_test_stall_copies": (_i, [_i, ctypes.c_uint]),
}


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(lib_path):
            raise RuntimeError(f"{lib_path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(lib_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def lib():
    """The loaded ctypes library (loads it on first use)."""
    return _lib()


def _check(status: int, call: str):
    if status != TF_OK:
        raise TFError(status, call)


def header_declarations():
    """Names of the functions declared in include/tf.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(tf_\w+)\s*\(", text, re.M)))


def version() -> int:
    return _lib().tf_version()


# ---------------------------------------------------------------------------
# host: pre-tiling


def prepack_size(N: int, K: int, bits: int, group: int) -> int:
    out = _sz()
    _check(_lib().tf_prepack_size(N, K, bits, group, ctypes.byref(out)), "tf_prepack_size")
    return out.value


def prepack(qweight: np.ndarray, scales: np.ndarray, zeros: np.ndarray, N: int, K: int,
            bits: int, group: int) -> np.ndarray:
    """Offline interleaved pre-tiling of natural-order inputs; returns the blob (uint8)."""
    qw = np.ascontiguousarray(qweight, dtype=np.uint32 if bits == 4 else np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint16)
    z = np.ascontiguousarray(zeros, dtype=np.uint8)
    g = K if group == 0 else group
    want_qw = (N, (K + 7) // 8) if bits == 4 else (N, K)
    if qw.shape != want_qw or s.shape != (N, K // g) or z.shape != (N, K // g):
        raise ValueError("qweight/scales/zeros shapes do not match N, K, bits, group")
    out = np.empty(prepack_size(N, K, bits, group), dtype=np.uint8)
    _check(_lib().tf_prepack(qw.ctypes.data, s.ctypes.data, z.ctypes.data, N, K, bits, group,
                             out.ctypes.data, out.size), "tf_prepack")
    return out


def _natural(qweight, scales, zeros, N: int, K: int, bits: int, group: int):
    qw = np.ascontiguousarray(qweight, dtype=np.uint32 if bits == 4 else np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint16)
    z = np.ascontiguousarray(zeros, dtype=np.uint8)
    g = K if group == 0 else group
    want_qw = (N, (K + 7) // 8) if bits == 4 else (N, K)
    if qw.shape != want_qw or s.shape != (N, K // g) or z.shape != (N, K // g):
        raise ValueError("qweight/scales/zeros shapes do not match N, K, bits, group")
    return qw, s, z


def prepack_gate_up(gate, up, F: int, K: int, bits: int, group: int) -> np.ndarray:
    """One blob of N = 2F rows from the gate and up projections of a gated MLP.

    gate and up are (qweight, scales, zeros) in natural order, each F x K;
    rows are interleaved in blocks of 8 (``tf_prepack_gate_up`` in include/tf.h).
    """
    gq, gs, gz = _natural(*gate, F, K, bits, group)
    uq, us, uz = _natural(*up, F, K, bits, group)
    out = np.empty(prepack_size(2 * F, K, bits, group), dtype=np.uint8)
    _check(_lib().tf_prepack_gate_up(gq.ctypes.data, gs.ctypes.data, gz.ctypes.data, uq.ctypes.data,
                                     us.ctypes.data, uz.ctypes.data, F, K, bits, group, out.ctypes.data,
                                     out.size), "tf_prepack_gate_up")
    return out


def prepack_awq(qweight: np.ndarray, qzeros: np.ndarray, scales: np.ndarray, N: int, K: int,
                group: int) -> np.ndarray:
    """Pre-tiling of an INT4 layer in AWQ's checkpoint layout; returns the blob (uint8).

    qweight int32 [K, N/8] and qzeros int32 [K/g, N/8] (eight output columns per word),
    scales float16 (or their uint16 bits) [K/g, N]; the layout is described at
    ``tf_prepack_awq`` in include/tf.h.
    """
    g = K if group == 0 else group
    qw, qz, sc = np.ascontiguousarray(qweight), np.ascontiguousarray(qzeros), np.ascontiguousarray(scales)
    if qw.dtype not in (np.int32, np.uint32) or qz.dtype not in (np.int32, np.uint32):
        raise ValueError("qweight and qzeros must be int32 (or uint32) arrays of packed nibbles")
    if sc.dtype not in (np.float16, np.uint16, np.int16):
        raise ValueError("scales must be float16 (or their 16-bit patterns)")
    qw, qz, sc = qw.view(np.int32), qz.view(np.int32), sc.view(np.uint16)
    if N % 8 or qw.shape != (K, N // 8) or qz.shape != (K // g, N // 8) or sc.shape != (K // g, N):
        raise ValueError("qweight/qzeros/scales shapes do not match N, K, group")
    out = np.empty(prepack_size(N, K, 4, group), dtype=np.uint8)
    _check(_lib().tf_prepack_awq(qw.ctypes.data, qz.ctypes.data, sc.ctypes.data, N, K, group,
                                 out.ctypes.data, out.size), "tf_prepack_awq")
    return out


def blob_info(blob: np.ndarray):
    b = np.ascontiguousarray(blob, dtype=np.uint8)
    v = [_i() for _ in range(4)]
    _check(_lib().tf_blob_info(b.ctypes.data, b.size, *[ctypes.byref(x) for x in v]), "tf_blob_info")
    return tuple(x.value for x in v)


def unprepack(blob: np.ndarray):
    """Exact inverse of prepack: (qweight, scales, zeros, N, K, bits, group)."""
    b = np.ascontiguousarray(blob, dtype=np.uint8)
    N, K, bits, group = blob_info(b)
    g = K if group == 0 else group
    qw = np.zeros((N, (K + 7) // 8), np.uint32) if bits == 4 else np.zeros((N, K), np.uint8)
    s = np.zeros((N, K // g), np.uint16)
    z = np.zeros((N, K // g), np.uint8)
    _check(_lib().tf_unprepack(b.ctypes.data, b.size, qw.ctypes.data, s.ctypes.data, z.ctypes.data),
           "tf_unprepack")
    return qw, s, z, N, K, bits, group


# ---------------------------------------------------------------------------
# device


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


_RAW_STREAM = None


def _stream_handle(stream) -> int:
    """cudaStream_t of the given torch stream, else of the current one (without building a Stream object)."""
    global _RAW_STREAM
    if stream is not None:
        return stream.cuda_stream
    torch = _torch()
    if _RAW_STREAM is None:
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None) or (
            lambda dev: torch.cuda.current_stream(dev).cuda_stream)
    return _RAW_STREAM(torch.cuda.current_device())


def _workspace_args(W, M: int, kind: str, workspace):
    """(device address, bytes) of the given workspace, else of the layer's cached one."""
    if workspace is not None:
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()
    args = W._ws_args.get((kind, M))
    if args is None:
        ws = W.workspace(M, kind)
        args = W._ws_args[(kind, M)] = (ws.data_ptr(), ws.numel() * ws.element_size())
    return args


class Weights:
    """A device-resident blob plus its layer description.

    The blob tensor is fixed at construction: its device address is kept for
    the calls, so replace the Weights object rather than its `blob`.
    """

    def __init__(self, blob_dev, N: int, K: int, bits: int, group: int):
        self.blob = blob_dev
        self.N, self.K, self.bits, self.group = N, K, bits, group
        self._ws = {}
        self._ws_args = {}  # (kind, M) -> (device address, bytes) of the cached workspace
        self._blob_ptr = blob_dev.data_ptr()
        self._blob_bytes = blob_dev.numel()

    @classmethod
    def upload(cls, blob: np.ndarray, device=None) -> "Weights":
        torch = _torch()
        N, K, bits, group = blob_info(blob)
        dev = torch.device("cuda") if device is None else torch.device(device)
        t = torch.from_numpy(np.ascontiguousarray(blob, dtype=np.uint8)).to(dev)
        return cls(t, N, K, bits, group)

    @property
    def nbytes(self) -> int:
        return self.blob.numel()

    def workspace(self, M: int, kind: str = "gemv"):
        """A zero-filled GEMV or GEMM workspace for this layer and M (cached)."""
        torch = _torch()
        key = (kind, M, self.blob.device)
        if key not in self._ws:
            size = gemv_workspace_size if kind == "gemv" else gemm_workspace_size
            n = size(self.N, self.K, self.bits, self.group, M)
            self._ws[key] = torch.zeros(max(n, 16), dtype=torch.uint8, device=self.blob.device)
        return self._ws[key]


def gemv_workspace_size(N: int, K: int, bits: int, group: int, M: int) -> int:
    out = _sz()
    _check(_lib().tf_gemv_workspace_size(N, K, bits, group, M, ctypes.byref(out)),
           "tf_gemv_workspace_size")
    return out.value


def _check_x(W: Weights, x):
    torch = _torch()
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != W.K or not x.is_cuda:
        raise ValueError(f"x must be a CUDA bfloat16 tensor [M, {W.K}]")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")


def _out(W: Weights, M: int, y):
    torch = _torch()
    if y is None:
        return torch.empty((M, W.N), dtype=torch.bfloat16, device=W.blob.device)
    if y.dtype != torch.bfloat16 or tuple(y.shape) != (M, W.N) or not y.is_contiguous():
        raise ValueError(f"y must be a contiguous bfloat16 tensor [{M}, {W.N}]")
    return y


def dequant(W: Weights, out=None, stream=None):
    """Dense BF16 W [N, K] from the blob, with the kernels' exact dequant arithmetic."""
    torch = _torch()
    if out is None:
        out = torch.empty((W.N, W.K), dtype=torch.bfloat16, device=W.blob.device)
    _check(_lib().tf_dequant(_ptr(W.blob), W.nbytes, W.N, W.K, W.bits, W.group, _ptr(out),
                             _stream(stream)), "tf_dequant")
    return out


def _check_bias(W: Weights, bias):
    torch = _torch()
    if bias.dtype != torch.bfloat16 or tuple(bias.shape) != (W.N,) or not bias.is_cuda or not bias.is_contiguous():
        raise ValueError(f"bias must be a contiguous CUDA bfloat16 tensor [{W.N}]")


def gemv(W: Weights, x, y=None, workspace=None, stream=None, bias=None):
    """y[M, N] = x[M, K] W^T (+ bias[N]) for 1 <= M <= 8 (fused unpack + dequant + mma.sync)."""
    _check_x(W, x)
    M = x.shape[0]
    y = _out(W, M, y)
    wp, wn = _workspace_args(W, M, "gemv", workspace)
    if bias is None:
        _check(_lib().tf_gemv(W._blob_ptr, W._blob_bytes, W.N, W.K, W.bits, W.group, x.data_ptr(), y.data_ptr(),
                              M, wp, wn, _stream_handle(stream)), "tf_gemv")
    else:
        _check_bias(W, bias)
        _check(_lib().tf_gemv_bias(W._blob_ptr, W._blob_bytes, W.N, W.K, W.bits, W.group, x.data_ptr(),
                                   bias.data_ptr(), y.data_ptr(), M, wp, wn, _stream_handle(stream)), "tf_gemv_bias")
    return y


def gemv_noalloc(W: Weights, x, y=None, stream=None):
    """tf_gemv without a workspace argument (scratch is a fixed array inside libtf).

    For callers that cannot allocate device memory; calls that overlap on the
    GPU share that scratch and must be ordered on one stream.
    """
    _check_x(W, x)
    M = x.shape[0]
    y = _out(W, M, y)
    _check(_lib().tf_gemv_noalloc(_ptr(W.blob), W.nbytes, W.N, W.K, W.bits, W.group, _ptr(x), _ptr(y), M,
                                  _stream(stream)), "tf_gemv_noalloc")
    return y


def gemm_workspace_size(N: int, K: int, bits: int, group: int, M: int) -> int:
    out = _sz()
    _check(_lib().tf_gemm_workspace_size(N, K, bits, group, M, ctypes.byref(out)), "tf_gemm_workspace_size")
    return out.value


def gemm(W: Weights, x, y=None, workspace=None, stream=None, stream_k=True, bias=None):
    """y[M, N] = x[M, K] W^T (+ bias[N]) for any M (fused dequant to SMEM + tcgen05 MMAs).

    With stream_k (default) the layer's cached workspace lets the last,
    partial wave of output tiles be split along K across all SMs; with
    stream_k False every tile is computed whole by one SM.  M <= 8 (K a
    multiple of 8) runs on the slab or tile GEMV instead, with the same
    per-weight BF16 rounding; stream_k False there passes no workspace, so
    a layer whose GEMV needs one falls back to whole tensor-core tiles.
    """
    _check_x(W, x)
    M = x.shape[0]
    y = _out(W, M, y)
    if stream_k:
        wp, wn = _workspace_args(W, M, "gemm", workspace)
    else:
        wp, wn = None, 0
    if bias is None:
        _check(_lib().tf_gemm(W._blob_ptr, W._blob_bytes, W.N, W.K, W.bits, W.group, x.data_ptr(), y.data_ptr(),
                              M, wp, wn, _stream_handle(stream)), "tf_gemm")
    else:
        _check_bias(W, bias)
        _check(_lib().tf_gemm_bias(W._blob_ptr, W._blob_bytes, W.N, W.K, W.bits, W.group, x.data_ptr(),
                                   bias.data_ptr(), y.data_ptr(), M, wp, wn, _stream_handle(stream)), "tf_gemm_bias")
    return y


def _bf16_out(t, shape, name: str):
    torch = _torch()
    if t.dtype != torch.bfloat16 or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor {list(shape)}")
    return t


def _epi_call(W: Weights, x, kind: str, workspace, stream, stream_k: bool):
    _check_x(W, x)
    M = x.shape[0]
    if kind == "gemm" and not stream_k:
        return M, None, 0
    wp, wn = _workspace_args(W, M, kind, workspace)
    return M, wp, wn


def _silu_gate(W: Weights, x, h, bias, workspace, stream, kind: str, stream_k: bool):
    """h[M, N/2] = silu(gate) * up of a layer packed by prepack_gate_up.

    kind "gemv" (1 <= M <= 8) calls tf_gemv_silu_gate, "gemm" (any M)
    tf_gemm_silu_gate; bias is in the layer's (interleaved) row order.
    """
    torch = _torch()
    if kind not in ("gemv", "gemm"):
        raise ValueError("kind must be 'gemv' or 'gemm'")
    M, wp, wn = _epi_call(W, x, kind, workspace, stream, stream_k)
    shape = (M, W.N // 2)
    h = torch.empty(shape, dtype=torch.bfloat16, device=W.blob.device) if h is None else _bf16_out(h, shape, "h")
    if bias is not None:
        _check_bias(W, bias)
    fn = "tf_gemv_silu_gate" if kind == "gemv" else "tf_gemm_silu_gate"
    _check(getattr(_lib(), fn)(W._blob_ptr, W._blob_bytes, W.N, W.K, W.bits, W.group, x.data_ptr(),
                               None if bias is None else bias.data_ptr(), h.data_ptr(), M, wp, wn,
                               _stream_handle(stream)), fn)
    return h


def _qkv(W: Weights, x, nq: int, nk: int, out, bias, workspace, stream, kind: str, stream_k: bool):
    """(q [M, nq], k [M, nk], v [M, N - nq - nk]) of a stacked QKV layer, written by the epilogue.

    kind "gemv" (1 <= M <= 8) calls tf_gemv_qkv, "gemm" (any M) tf_gemm_qkv;
    out, when given, is the (q, k, v) triple to write.
    """
    torch = _torch()
    if kind not in ("gemv", "gemm"):
        raise ValueError("kind must be 'gemv' or 'gemm'")
    M, wp, wn = _epi_call(W, x, kind, workspace, stream, stream_k)
    nv = W.N - nq - nk
    shapes = ((M, nq), (M, nk), (M, nv))
    if out is None:
        out = tuple(torch.empty(sh, dtype=torch.bfloat16, device=W.blob.device) for sh in shapes)
    else:
        out = tuple(_bf16_out(t, sh, nm) for t, sh, nm in zip(out, shapes, ("q", "k", "v")))
    if bias is not None:
        _check_bias(W, bias)
    ptrs = [t.data_ptr() if t.numel() else None for t in out]
    fn = "tf_gemv_qkv" if kind == "gemv" else "tf_gemm_qkv"
    _check(getattr(_lib(), fn)(W._blob_ptr, W._blob_bytes, W.N, W.K, W.bits, W.group, x.data_ptr(),
                               None if bias is None else bias.data_ptr(), ptrs[0], ptrs[1], ptrs[2], nq, nk, M,
                               wp, wn, _stream_handle(stream)), fn)
    return out


def gemv_silu_gate(W: Weights, x, h=None, bias=None, workspace=None, stream=None):
    """tf_gemv_silu_gate: h[M, N/2] = silu(gate) * up for 1 <= M <= 8."""
    return _silu_gate(W, x, h, bias, workspace, stream, "gemv", True)


def gemm_silu_gate(W: Weights, x, h=None, bias=None, workspace=None, stream=None, stream_k=True):
    """tf_gemm_silu_gate: h[M, N/2] = silu(gate) * up for any M."""
    return _silu_gate(W, x, h, bias, workspace, stream, "gemm", stream_k)


def gemv_qkv(W: Weights, x, nq: int, nk: int, out=None, bias=None, workspace=None, stream=None):
    """tf_gemv_qkv: (q, k, v) of a stacked QKV layer for 1 <= M <= 8."""
    return _qkv(W, x, nq, nk, out, bias, workspace, stream, "gemv", True)


def gemm_qkv(W: Weights, x, nq: int, nk: int, out=None, bias=None, workspace=None, stream=None, stream_k=True):
    """tf_gemm_qkv: (q, k, v) of a stacked QKV layer for any M."""
    return _qkv(W, x, nq, nk, out, bias, workspace, stream, "gemm", stream_k)


def device_error() -> int:
    """Read and clear the current device's error word (synchronous)."""
    v = ctypes.c_uint()
    _check(_lib().tf_device_error(ctypes.byref(v)), "tf_device_error")
    return v.value


def test_stall_copies(stall: bool, timeout_us: int = 0) -> None:
    """Failure-detection test hook (see tf_test_stall_copies in include/tf.h)."""
    _check(_lib().tf_test_stall_copies(1 if stall else 0, timeout_us), "tf_test_stall_copies")
