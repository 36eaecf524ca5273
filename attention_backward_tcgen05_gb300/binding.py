"""ctypes binding for libfab (declared in include/fab.h).

Argument marshalling only: each ``fab_*`` function takes torch CUDA tensors,
checks that they match the layouts the C ABI documents, and passes raw device
pointers, sizes and the current CUDA stream.  Every step of the computation
runs in libfab's kernels; there is no fallback of any kind, and a missing or
unloadable ``libfab.so`` raises.

Tensor shapes (torch, C order; the reverse of ggml's ne order):
    q (B, H, N, DK)  k (B, Hkv, M, DK)  v (B, Hkv, M, DV)
    d, o (B, N, H, DV)  lse (B, H, N) float32  mask (N, M) float16 or None
    packed: float32 of fab_packed_bytes(dims) / 4 elements
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfab.so")

FAB_OK, FAB_ERR_INVALID, FAB_ERR_UNSUPPORTED, FAB_ERR_WORKSPACE, FAB_ERR_CUDA, FAB_ERR_TIMEOUT = range(6)
FAB_F32, FAB_BF16, FAB_F16 = 0, 1, 2

EXPORTS = ("fab_version", "fab_status_string", "fab_packed_offsets", "fab_packed_bytes",
           "fab_backward_workspace_bytes", "fab_backward_recompute_workspace_bytes", "fab_forward_lse",
           "fab_backward", "fab_backward_preprocess",
           "fab_backward_main", "fab_backward_query_pass", "fab_backward_key_pass", "fab_backward_noalloc",
           "fab_last_device_error")
NOALLOC_MAX_ROWS = 1048576  # FAB_NOALLOC_MAX_ROWS


class fab_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "H", "Hkv", "N", "M", "DK", "DV")]

    def tuple(self):
        return tuple(getattr(self, n) for n in ("B", "H", "Hkv", "N", "M", "DK", "DV"))


class FabError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libfab.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: build it with attention_backward_tcgen05_gb300.build")
                L = ctypes.CDLL(LIB_PATH)
                vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
                dp = ctypes.POINTER(fab_dims)
                szp = ctypes.POINTER(ctypes.c_size_t)
                sig = {
                    "fab_version": ([], i32),
                    "fab_status_string": ([i32], ctypes.c_char_p),
                    "fab_packed_offsets": ([dp, szp, szp, szp], i32),
                    "fab_packed_bytes": ([dp], sz),
                    "fab_backward_workspace_bytes": ([dp, i32], sz),
                    "fab_backward_recompute_workspace_bytes": ([dp, i32], sz),
                    "fab_forward_lse": ([vp, vp, vp, vp, i32, f32, i32, dp, vp, vp, vp], i32),
                    "fab_backward": ([vp, vp, vp, vp, vp, vp, vp, i32, f32, i32, dp, vp, sz, vp, vp], i32),
                    "fab_backward_preprocess": ([vp, vp, i32, dp, vp, sz, vp, vp], i32),
                    "fab_backward_main": ([vp, vp, vp, vp, vp, vp, i32, f32, i32, dp, vp, sz, vp, vp], i32),
                    "fab_backward_query_pass": ([vp, vp, vp, vp, vp, vp, vp, i32, f32, i32, dp, vp, sz, vp, vp], i32),
                    "fab_backward_key_pass": ([vp, vp, vp, vp, vp, vp, i32, f32, i32, dp, vp, sz, vp, vp], i32),
                    "fab_backward_noalloc": ([vp, vp, vp, vp, vp, vp, vp, i32, f32, i32, dp, vp, vp], i32),
                    "fab_last_device_error": ([vp], i32),
                }
                for name, (args, res) in sig.items():
                    f = getattr(L, name)
                    f.argtypes = args
                    f.restype = res
                _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fab_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != FAB_OK:
        raise FabError(status, where)


def make_dims(B, H, Hkv, N, M, DK, DV) -> fab_dims:
    return fab_dims(int(B), int(H), int(Hkv), int(N), int(M), int(DK), int(DV))


def dims_of(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> fab_dims:
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D: (B,H,N,DK), (B,Hkv,M,DK), (B,Hkv,M,DV)")
    B, H, N, DK = q.shape
    Bk, Hkv, M, DKk = k.shape
    Bv, Hv, Mv, DV = v.shape
    if (Bk, DKk) != (B, DK) or (Bv, Hv, Mv) != (B, Hkv, M):
        raise ValueError("inconsistent q/k/v shapes")
    return make_dims(B, H, Hkv, N, M, DK, DV)


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return FAB_F32
    if t.dtype == torch.bfloat16:
        return FAB_BF16
    if t.dtype == torch.float16:
        return FAB_F16
    raise ValueError(f"unsupported dtype {t.dtype}: float32, bfloat16 or float16")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _mask(mask, dims: fab_dims):
    if mask is None:
        return None
    return _dev(mask, "mask", torch.float16, (dims.N, dims.M))


# ------------------------------------------------------------------ C ABI, one to one


def fab_version() -> int:
    return lib().fab_version()


def fab_packed_offsets(dims: fab_dims):
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().fab_packed_offsets(ctypes.byref(dims), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
           "fab_packed_offsets")
    return a.value, b.value, c.value


def fab_packed_bytes(dims: fab_dims) -> int:
    return lib().fab_packed_bytes(ctypes.byref(dims))


def fab_backward_workspace_bytes(dims: fab_dims, dtype: int) -> int:
    return lib().fab_backward_workspace_bytes(ctypes.byref(dims), int(dtype))


def fab_backward_recompute_workspace_bytes(dims: fab_dims, dtype: int) -> int:
    return lib().fab_backward_recompute_workspace_bytes(ctypes.byref(dims), int(dtype))


def fab_forward_lse(q, k, v, mask, causal, scale, o, lse, stream=None):
    dims = dims_of(q, k, v)
    t = dtype_code(q)
    args = (_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), _mask(mask, dims), int(bool(causal)),
            float(scale), t, ctypes.byref(dims),
            _dev(o, "o", q.dtype, (dims.B, dims.N, dims.H, dims.DV)),
            _dev(lse, "lse", torch.float32, (dims.B, dims.H, dims.N)), _stream(stream))
    _check(lib().fab_forward_lse(*args), "fab_forward_lse")


def fab_backward(q, k, v, d, o, lse, mask, causal, scale, workspace, packed_out, stream=None):
    """o and lse may both be None: the library then recomputes them into the
    workspace (sized by fab_backward_recompute_workspace_bytes)."""
    dims = dims_of(q, k, v)
    t = dtype_code(q)
    oshape = (dims.B, dims.N, dims.H, dims.DV)
    args = (_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), _dev(d, "d", q.dtype, oshape),
            None if o is None else _dev(o, "o", q.dtype, oshape),
            None if lse is None else _dev(lse, "lse", torch.float32, (dims.B, dims.H, dims.N)),
            _mask(mask, dims), int(bool(causal)), float(scale), t, ctypes.byref(dims),
            _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
            _dev(packed_out, "packed_out", torch.float32, (fab_packed_bytes(dims) // 4,)), _stream(stream))
    _check(lib().fab_backward(*args), "fab_backward")


def fab_backward_preprocess(d, o, dims: fab_dims, workspace, packed_out, stream=None):
    oshape = (dims.B, dims.N, dims.H, dims.DV)
    t = dtype_code(d)
    args = (_dev(d, "d", None, oshape), _dev(o, "o", d.dtype, oshape), t, ctypes.byref(dims),
            _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
            _dev(packed_out, "packed_out", torch.float32, (fab_packed_bytes(dims) // 4,)), _stream(stream))
    _check(lib().fab_backward_preprocess(*args), "fab_backward_preprocess")


def fab_backward_main(q, k, v, d, lse, mask, causal, scale, workspace, packed_out, stream=None):
    dims = dims_of(q, k, v)
    t = dtype_code(q)
    args = (_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype),
            _dev(d, "d", q.dtype, (dims.B, dims.N, dims.H, dims.DV)),
            _dev(lse, "lse", torch.float32, (dims.B, dims.H, dims.N)), _mask(mask, dims), int(bool(causal)),
            float(scale), t, ctypes.byref(dims), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(),
            _dev(packed_out, "packed_out", torch.float32, (fab_packed_bytes(dims) // 4,)), _stream(stream))
    _check(lib().fab_backward_main(*args), "fab_backward_main")


def fab_backward_query_pass(q, k, v, d, o, lse, mask, causal, scale, workspace, packed_out, stream=None):
    """Tensor-core query pass: D_i into the workspace, the dQ slice and the padding."""
    dims = dims_of(q, k, v)
    t = dtype_code(q)
    oshape = (dims.B, dims.N, dims.H, dims.DV)
    args = (_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), _dev(d, "d", q.dtype, oshape),
            _dev(o, "o", q.dtype, oshape), _dev(lse, "lse", torch.float32, (dims.B, dims.H, dims.N)),
            _mask(mask, dims), int(bool(causal)), float(scale), t, ctypes.byref(dims),
            _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
            _dev(packed_out, "packed_out", torch.float32, (fab_packed_bytes(dims) // 4,)), _stream(stream))
    _check(lib().fab_backward_query_pass(*args), "fab_backward_query_pass")


def fab_backward_key_pass(q, k, v, d, lse, mask, causal, scale, workspace, packed_out, stream=None):
    """Tensor-core key/value pass: the dK and dV slices (D_i read from the workspace)."""
    dims = dims_of(q, k, v)
    t = dtype_code(q)
    args = (_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype),
            _dev(d, "d", q.dtype, (dims.B, dims.N, dims.H, dims.DV)),
            _dev(lse, "lse", torch.float32, (dims.B, dims.H, dims.N)), _mask(mask, dims), int(bool(causal)),
            float(scale), t, ctypes.byref(dims), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(),
            _dev(packed_out, "packed_out", torch.float32, (fab_packed_bytes(dims) // 4,)), _stream(stream))
    _check(lib().fab_backward_key_pass(*args), "fab_backward_key_pass")


def fab_backward_noalloc(q, k, v, d, o, lse, mask, causal, scale, packed_out, stream=None):
    """fab_backward without a workspace: for callers that cannot allocate
    device memory.  The scratch is a fixed array inside libfab (B*H*N up to
    NOALLOC_MAX_ROWS); calls that may overlap on the GPU must be ordered."""
    dims = dims_of(q, k, v)
    t = dtype_code(q)
    oshape = (dims.B, dims.N, dims.H, dims.DV)
    args = (_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), _dev(d, "d", q.dtype, oshape),
            _dev(o, "o", q.dtype, oshape), _dev(lse, "lse", torch.float32, (dims.B, dims.H, dims.N)),
            _mask(mask, dims), int(bool(causal)), float(scale), t, ctypes.byref(dims),
            _dev(packed_out, "packed_out", torch.float32, (fab_packed_bytes(dims) // 4,)), _stream(stream))
    _check(lib().fab_backward_noalloc(*args), "fab_backward_noalloc")


def fab_last_device_error(stream=None) -> int:
    return lib().fab_last_device_error(_stream(stream))


# ------------------------------------------------------------------ conveniences (torch allocates, libfab computes)


def forward(q, k, v, mask=None, causal=False, scale=None, stream=None):
    """Returns (o (B,N,H,DV) in q's dtype, lse (B,H,N) float32)."""
    dims = dims_of(q, k, v)
    scale = dims.DK ** -0.5 if scale is None else scale
    o = torch.empty((dims.B, dims.N, dims.H, dims.DV), dtype=q.dtype, device=q.device)
    lse = torch.empty((dims.B, dims.H, dims.N), dtype=torch.float32, device=q.device)
    fab_forward_lse(q, k, v, mask, causal, scale, o, lse, stream)
    return o, lse


def alloc_backward(dims: fab_dims, dtype: int, device, recompute: bool = False):
    """(workspace uint8 tensor, packed float32 tensor) sized for fab_backward
    (recompute: for a call without o and lse)."""
    wsb = fab_backward_recompute_workspace_bytes(dims, dtype) if recompute else fab_backward_workspace_bytes(dims, dtype)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=device)
    packed = torch.empty(fab_packed_bytes(dims) // 4, dtype=torch.float32, device=device)
    return ws, packed


def backward(q, k, v, d, o=None, lse=None, mask=None, causal=False, scale=None, stream=None):
    """Returns the packed f32 [dQ | dK | dV] buffer (o, lse None: recomputed)."""
    dims = dims_of(q, k, v)
    scale = dims.DK ** -0.5 if scale is None else scale
    ws, packed = alloc_backward(dims, dtype_code(q), q.device, recompute=o is None and lse is None)
    fab_backward(q, k, v, d, o, lse, mask, causal, scale, ws, packed, stream)
    return packed


def unpack(packed: torch.Tensor, dims: fab_dims):
    """Views (dq (B,H,N,DK), dk (B,Hkv,M,DK), dv (B,Hkv,M,DV)) into a packed buffer."""
    off_k, off_v, end = fab_packed_offsets(dims)
    B, H, Hkv, N, M, DK, DV = dims.tuple()
    nq, nk, nv = B * H * N * DK, B * Hkv * M * DK, B * Hkv * M * DV
    dq = packed[:nq].view(B, H, N, DK)
    dk = packed[off_k // 4:off_k // 4 + nk].view(B, Hkv, M, DK)
    dv = packed[off_v // 4:off_v // 4 + nv].view(B, Hkv, M, DV)
    return dq, dk, dv
