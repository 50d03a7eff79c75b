"""Thin Python binding of libfa.so (argument marshalling only).

Every step of the attention path runs inside the CUDA library; this module
only turns torch tensors into pointers, strides and sizes, passes the current
CUDA stream and converts status codes into exceptions.  There is no fallback:
if libfa.so is missing or the tensors are not on a CUDA device, the call
fails loudly.

Entry points mirror include/fa.h:

* ``fa_fwd(q, k, v, o, lse, sm_scale, causal)``
* ``fa_bwd(q, k, v, o, do, lse, dq, dk, dv, sm_scale, causal, workspace)``
* ``fa_bwd_workspace_bytes(B, H, Nq, Nk, d)``
* ``fa_last_device_error()``, ``fa_status_string(code)``, ``fa_version()``

Tensors are either 4-D ``[B, H, seq, d]`` or 3-D ``[seq, heads, d]`` (the
layout of "BUG in flash attention kernel", batch 1), with the head dimension
contiguous; other strides are passed through to the ``*_strided`` entry
points.  ``lse`` is float32 ``[B, H, Nq]`` (``[1, H, Nq]`` for 3-D inputs).
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_WORKSPACE = 5

FA_FP16 = 0
FA_BF16 = 1
FA_FP32 = 2

FA_BWD_PREPROCESS = 1
FA_BWD_DKDV = 2
FA_BWD_DQ = 3

FA_FP8V_PAGE_STEPS = 0
FA_FP8V_LAZY_MAX = 1

FA_BWD_PATH_AUTO = 0
FA_BWD_PATH_TWO_PASS = 1
FA_BWD_PATH_FUSED = 2

EXPORTED_SYMBOLS = (
    "fa_fwd",
    "fa_fwd_strided",
    "fa_fwd_split_workspace_bytes",
    "fa_fwd_split_count",
    "fa_fwd_split",
    "fa_fwd_fp8v",
    "fa_fwd_fp8v_ex",
    "fa_bwd_workspace_bytes",
    "fa_bwd",
    "fa_bwd_strided",
    "fa_bwd_phase",
    "fa_bwd_workspace_bytes_path",
    "fa_bwd_ex",
    "fa_bwd_noalloc",
    "fa_softmax_rows",
    "fa_status_string",
    "fa_last_device_error",
    "fa_inject_device_error",
    "fa_version",
)


class FaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {fa_status_string(code)} (code {code})")


class Strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("s", ctypes.c_int64)]


class Layout(ctypes.Structure):
    _fields_ = [(n, Strides) for n in ("q", "k", "v", "o", "dout", "dq", "dk", "dv")]


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load libfa.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m tiled_attention_07_gb300.build` "
                               "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
        L.fa_fwd.restype = i
        L.fa_fwd_strided.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, ctypes.POINTER(Layout), vp]
        L.fa_fwd_strided.restype = i
        L.fa_fwd_split_workspace_bytes.argtypes = [i, i, i, i, i]
        L.fa_fwd_split_workspace_bytes.restype = ctypes.c_size_t
        L.fa_fwd_split_count.argtypes = [i, i, i, i, i, i]
        L.fa_fwd_split_count.restype = i
        L.fa_fwd_split.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, ctypes.POINTER(Layout), i, vp,
                                   ctypes.c_size_t, vp]
        L.fa_fwd_split.restype = i
        L.fa_fwd_fp8v.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_int64, f, i, i, vp]
        L.fa_fwd_fp8v.restype = i
        L.fa_fwd_fp8v_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_int64, f, i, i, i, vp]
        L.fa_fwd_fp8v_ex.restype = i
        L.fa_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
        L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, ctypes.c_size_t, vp]
        L.fa_bwd.restype = i
        L.fa_bwd_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i,
                                     ctypes.POINTER(Layout), vp, ctypes.c_size_t, vp]
        L.fa_bwd_strided.restype = i
        L.fa_bwd_phase.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i,
                                   ctypes.POINTER(Layout), vp, ctypes.c_size_t, vp]
        L.fa_bwd_phase.restype = i
        L.fa_bwd_workspace_bytes_path.argtypes = [i, i, i, i, i, i]
        L.fa_bwd_workspace_bytes_path.restype = ctypes.c_size_t
        L.fa_bwd_ex.argtypes = [i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i,
                                ctypes.POINTER(Layout), vp, ctypes.c_size_t, vp]
        L.fa_bwd_ex.restype = i
        L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
        L.fa_bwd_noalloc.restype = i
        L.fa_softmax_rows.argtypes = [vp, vp, vp, i, i, ctypes.c_int64, ctypes.c_int64, i, vp]
        L.fa_softmax_rows.restype = i
        L.fa_status_string.argtypes = [i]
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        L.fa_last_device_error.restype = i
        L.fa_inject_device_error.argtypes = [i]
        L.fa_inject_device_error.restype = i
        L.fa_version.argtypes = []
        L.fa_version.restype = ctypes.c_char_p
        _lib = L
        return L


def fa_status_string(code: int) -> str:
    return lib().fa_status_string(int(code)).decode()


def fa_version() -> str:
    return lib().fa_version().decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (fp16 or bf16)")


def _dims(t: torch.Tensor) -> Tuple[int, int, int, int]:
    """(B, H, seq, d) of a [B, H, seq, d] or [seq, heads, d] tensor."""
    if t.dim() == 4:
        return tuple(t.shape)  # type: ignore[return-value]
    if t.dim() == 3:
        return 1, t.shape[1], t.shape[0], t.shape[2]
    raise ValueError(f"expected a 3-D [seq, heads, d] or 4-D [B, H, seq, d] tensor, got shape {tuple(t.shape)}")


def _strides(t: torch.Tensor) -> Strides:
    if t.stride(-1) != 1:
        raise ValueError("the head dimension must be contiguous (stride 1)")
    if t.dim() == 4:
        return Strides(t.stride(0), t.stride(1), t.stride(2))
    # [seq, heads, d]: a single batch; its batch stride only has to be a valid
    # multiple of 16 bytes.
    return Strides(max(t.shape[0], 1) * t.stride(0), t.stride(1), t.stride(0))


def _is_bhsd_contiguous(t: torch.Tensor) -> bool:
    return t.dim() == 4 and t.is_contiguous()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream, device=None) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("fa_* entry points take CUDA tensors only (no CPU path)")


def _check_same_device(*ts):
    dev = next(t.device for t in ts if t is not None)
    for t in ts:
        if t is not None and t.device != dev:
            raise ValueError(f"all tensors of one call must be on one device ({dev}), got one on {t.device}")


def _check_attention(q, k, v=None, o=None, lse=None, q_like=None, k_like=None):
    """The library sees only pointers and sizes, so every tensor's shape and
    dtype is checked against q (queries) and k (keys) here: a mismatch would
    make a kernel read or write past a buffer.  ``v`` and the named tensors
    of ``k_like`` are [B, H, Nk, d] like k; ``o`` and those of ``q_like``
    [B, H, Nq, d] like q; ``lse``
    float32 with B*H*Nq contiguous elements.  Shapes are checked first, then
    that every tensor is on one CUDA device."""
    B, H, Nq, d = _dims(q)
    _, _, Nk, _ = _dims(k)
    if k.dim() != q.dim() or tuple(_dims(k)) != (B, H, Nk, d):
        raise ValueError(f"k has shape {tuple(k.shape)}; q {tuple(q.shape)} wants [B={B}, H={H}, Nk, d={d}]")
    if k.dtype != q.dtype:
        raise TypeError(f"k is {k.dtype}, q is {q.dtype}: one dtype per call")
    q_like, k_like = dict(q_like or {}), dict(k_like or {})
    for name, t, want in ([("v", v, (B, H, Nk, d))] + [(n, t, (B, H, Nk, d)) for n, t in k_like.items()] +
                          [("o", o, (B, H, Nq, d))] + [(n, t, (B, H, Nq, d)) for n, t in q_like.items()]):
        if t is None:
            continue
        if t.dim() != q.dim() or tuple(_dims(t)) != want:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {want} in the layout of q")
        if t.dtype != q.dtype:
            raise TypeError(f"{name} is {t.dtype}, q is {q.dtype}: one dtype per call")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * Nq):
        raise ValueError(f"lse must be a contiguous float32 tensor of B*H*Nq = {B * H * Nq} elements")
    ts = (q, k, v, o, lse, *q_like.values(), *k_like.values())
    _check_cuda(*ts)
    _check_same_device(*ts)


def fa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
           sm_scale: float, causal: bool, stream=None) -> None:
    """O and LSE of exact attention into the caller's ``o`` and ``lse``."""
    dt = _dtype_code(q)
    _check_attention(q, k, v, o, lse)
    B, H, Nq, d = _dims(q)
    _, _, Nk, _ = _dims(k)
    L = lib()
    with torch.cuda.device(q.device):
        if all(_is_bhsd_contiguous(t) for t in (q, k, v, o)):
            rc = L.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, float(sm_scale),
                          int(bool(causal)), dt, _stream(stream, q.device))
        else:
            lay = Layout()
            lay.q, lay.k, lay.v, lay.o = _strides(q), _strides(k), _strides(v), _strides(o)
            rc = L.fa_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                  float(sm_scale), int(bool(causal)), dt, ctypes.byref(lay),
                                  _stream(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")


def fa_fwd_fp8v(q: torch.Tensor, k: torch.Tensor, vt: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
                sm_scale: float, causal: bool, stream=None, mode: int = FA_FP8V_PAGE_STEPS) -> None:
    """The forward with V in float8 e5m2, transposed: ``vt`` is [B, H, d, ld]
    (torch.float8_e5m2 or its raw uint8 codes) with unit stride along keys,
    ld = vt.stride(2) >= Nk and a multiple of 16; q, k, o contiguous
    [B, H, seq, d] fp16/bf16.  ``mode``: FA_FP8V_PAGE_STEPS (the page's
    running max, moved at every block) or FA_FP8V_LAZY_MAX (fa_fwd_fp8v_ex)."""
    B, H, Nq, d = _dims(q)
    _, _, Nk, _ = _dims(k)
    dt = _dtype_code(q)
    if vt.dtype not in (torch.float8_e5m2, torch.uint8):
        raise TypeError(f"vt must be float8_e5m2 (or its uint8 codes), got {vt.dtype}")
    if vt.dim() != 4 or tuple(vt.shape[:3]) != (B, H, d) or vt.shape[3] < Nk or vt.stride(3) != 1:
        raise ValueError(f"vt must be [B, H, d, >= Nk] with unit key stride, got {tuple(vt.shape)}")
    ld = vt.stride(2)
    if vt.stride(1) != d * ld or vt.stride(0) != H * d * ld:
        raise ValueError("vt rows must be packed: strides (H*d*ld, d*ld, ld, 1)")
    _check_attention(q, k, None, o, lse)
    _check_cuda(vt)
    _check_same_device(q, vt)
    for t in (q, k, o):
        if not _is_bhsd_contiguous(t):
            raise ValueError("q, k and o must be contiguous [B, H, seq, d]")
    with torch.cuda.device(q.device):
        rc = lib().fa_fwd_fp8v_ex(_ptr(q), _ptr(k), _ptr(vt), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, int(ld),
                                  float(sm_scale), int(bool(causal)), dt, int(mode), _stream(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_fp8v")


def fa_fwd_split_workspace_bytes(B: int, H: int, Nq: int, d: int, n_splits: int) -> int:
    return int(lib().fa_fwd_split_workspace_bytes(B, H, Nq, d, n_splits))


def fa_fwd_split_count(B: int, H: int, Nq: int, Nk: int, d: int, causal: bool) -> int:
    return int(lib().fa_fwd_split_count(B, H, Nq, Nk, d, int(bool(causal))))


def fa_fwd_split(q, k, v, o, lse, sm_scale: float, causal: bool, n_splits: int,
                 workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """fa_fwd over ``n_splits`` key ranges merged by their log-sum-exps.

    ``workspace`` is a CUDA byte tensor of at least
    ``fa_fwd_split_workspace_bytes`` (unused when ``n_splits == 1``)."""
    dt = _dtype_code(q)
    _check_attention(q, k, v, o, lse)
    B, H, Nq, d = _dims(q)
    _, _, Nk, _ = _dims(k)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _check_cuda(workspace)
        _check_same_device(q, workspace)
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    lay = Layout()
    lay.q, lay.k, lay.v, lay.o = _strides(q), _strides(k), _strides(v), _strides(o)
    with torch.cuda.device(q.device):
        rc = lib().fa_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, float(sm_scale),
                                int(bool(causal)), dt, ctypes.byref(lay), int(n_splits), ws_ptr, ws_bytes,
                                _stream(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_split")


def fa_bwd_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, Nq, Nk, d))


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, sm_scale: float, causal: bool,
           workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """dQ, dK, dV of sum(O * dO) into the caller's ``dq``, ``dk``, ``dv``.

    ``workspace`` is a CUDA byte tensor of at least ``fa_bwd_workspace_bytes``;
    if omitted, one is allocated here with torch (the library itself never
    allocates).
    """
    dt = _dtype_code(q)
    _check_attention(q, k, v, o, lse, q_like={"do": do, "dq": dq}, k_like={"dk": dk, "dv": dv})
    if workspace is not None:
        _check_cuda(workspace)
        _check_same_device(q, workspace)
    B, H, Nq, d = _dims(q)
    _, _, Nk, _ = _dims(k)
    need = fa_bwd_workspace_bytes(B, H, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    L = lib()
    ts = (q, k, v, o, do, dq, dk, dv)
    with torch.cuda.device(q.device):
        if all(_is_bhsd_contiguous(t) for t in ts):
            rc = L.fa_bwd(*[_ptr(t) for t in (q, k, v, o, do, lse, dq, dk, dv)], B, H, Nq, Nk, d,
                          float(sm_scale), int(bool(causal)), dt, _ptr(workspace), ws_bytes,
                          _stream(stream, q.device))
        else:
            lay = Layout()
            lay.q, lay.k, lay.v, lay.o = _strides(q), _strides(k), _strides(v), _strides(o)
            lay.dout, lay.dq, lay.dk, lay.dv = _strides(do), _strides(dq), _strides(dk), _strides(dv)
            rc = L.fa_bwd_strided(*[_ptr(t) for t in (q, k, v, o, do, lse, dq, dk, dv)], B, H, Nq, Nk, d,
                                  float(sm_scale), int(bool(causal)), dt, ctypes.byref(lay), _ptr(workspace),
                                  ws_bytes, _stream(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")


def fa_bwd_phase(phase: int, q, k, v, o, do, lse, dq, dk, dv, sm_scale: float, causal: bool,
                 workspace: torch.Tensor, stream=None) -> None:
    """One of the three launches of fa_bwd (FA_BWD_PREPROCESS, FA_BWD_DKDV,
    FA_BWD_DQ); calling the three in order with one workspace equals fa_bwd."""
    dt = _dtype_code(q)
    _check_attention(q, k, v, o, lse, q_like={"do": do, "dq": dq}, k_like={"dk": dk, "dv": dv})
    _check_cuda(workspace)
    _check_same_device(q, workspace)
    B, H, Nq, d = _dims(q)
    _, _, Nk, _ = _dims(k)
    ts = (q, k, v, o, do, dq, dk, dv)
    lay = None
    if not all(_is_bhsd_contiguous(t) for t in ts):
        lay = Layout()
        lay.q, lay.k, lay.v, lay.o = _strides(q), _strides(k), _strides(v), _strides(o)
        lay.dout, lay.dq, lay.dk, lay.dv = _strides(do), _strides(dq), _strides(dk), _strides(dv)
    with torch.cuda.device(q.device):
        rc = lib().fa_bwd_phase(int(phase), *[_ptr(t) for t in (q, k, v, o, do, lse, dq, dk, dv)], B, H, Nq, Nk,
                                d, float(sm_scale), int(bool(causal)), dt,
                                None if lay is None else ctypes.byref(lay), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, f"fa_bwd_phase({phase})")


def fa_bwd_workspace_bytes_path(B: int, H: int, Nq: int, Nk: int, d: int, path: int) -> int:
    return int(lib().fa_bwd_workspace_bytes_path(B, H, Nq, Nk, d, int(path)))


def fa_bwd_ex(path: int, phase: int, q, k, v, o, do, lse, dq, dk, dv, sm_scale: float, causal: bool,
              workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """The backward on a chosen path (FA_BWD_PATH_*), whole (phase 0) or one
    launch at a time; ``workspace`` defaults to a torch buffer of the path's
    size (fa_bwd_workspace_bytes_path)."""
    dt = _dtype_code(q)
    _check_attention(q, k, v, o, lse, q_like={"do": do, "dq": dq}, k_like={"dk": dk, "dv": dv})
    B, H, Nq, d = _dims(q)
    _, _, Nk, _ = _dims(k)
    if workspace is None:
        need = fa_bwd_workspace_bytes_path(B, H, Nq, Nk, d, path)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda(workspace)
    _check_same_device(q, workspace)
    ts = (q, k, v, o, do, dq, dk, dv)
    lay = None
    if not all(_is_bhsd_contiguous(t) for t in ts):
        lay = Layout()
        lay.q, lay.k, lay.v, lay.o = _strides(q), _strides(k), _strides(v), _strides(o)
        lay.dout, lay.dq, lay.dk, lay.dv = _strides(do), _strides(dq), _strides(dk), _strides(dv)
    with torch.cuda.device(q.device):
        rc = lib().fa_bwd_ex(int(path), int(phase), *[_ptr(t) for t in (q, k, v, o, do, lse, dq, dk, dv)], B, H,
                             Nq, Nk, d, float(sm_scale), int(bool(causal)), dt,
                             None if lay is None else ctypes.byref(lay), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, f"fa_bwd_ex(path {path}, phase {phase})")


NOALLOC_SCRATCH_BYTES = 16 << 20


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, sm_scale: float, causal: bool, stream=None) -> None:
    """fa_bwd without a workspace, for callers that cannot allocate device
    memory (they are given only input and output buffers, e.g. plugins of an
    engine that plans all buffers in advance).  The library's own fixed
    16 MiB scratch array is used instead; problems needing more than that
    (B*H*ceil(Nq/128)*128 > 2,097,152 rows) raise FaError(FA_ERR_WORKSPACE).
    Calls that can overlap on the GPU share that array and race: serialise
    them.  Contiguous [B, H, seq, d] tensors only."""
    dt = _dtype_code(q)
    _check_attention(q, k, v, o, lse, q_like={"do": do, "dq": dq}, k_like={"dk": dk, "dv": dv})
    ts = (q, k, v, o, do, dq, dk, dv)
    if not all(_is_bhsd_contiguous(t) for t in ts):
        raise ValueError("fa_bwd_noalloc takes contiguous [B, H, seq, d] tensors")
    B, H, Nq, d = _dims(q)
    _, _, Nk, _ = _dims(k)
    with torch.cuda.device(q.device):
        rc = lib().fa_bwd_noalloc(*[_ptr(t) for t in (q, k, v, o, do, lse, dq, dk, dv)], B, H, Nq, Nk, d,
                                  float(sm_scale), int(bool(causal)), dt, _stream(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_noalloc")


def fa_last_device_error(stream=None, device=None) -> Tuple[int, int]:
    """(status, raw device code) of ``device`` (default: the current one);
    synchronises the stream."""
    detail = ctypes.c_int(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        rc = lib().fa_last_device_error(_stream(stream, device), ctypes.byref(detail))
    return rc, detail.value


def fa_inject_device_error(code: int) -> None:
    """Test hook: set the device error word as if a bounded wait had given up."""
    rc = lib().fa_inject_device_error(int(code))
    if rc != FA_OK:
        raise FaError(rc, "fa_inject_device_error")


# ---------------------------------------------------------------------------
# conveniences that allocate the outputs with torch (plumbing, no compute)
# ---------------------------------------------------------------------------

def lse_shape(q: torch.Tensor):
    B, H, Nq, _ = _dims(q)
    return (B, H, Nq)


def attention_forward(q, k, v, sm_scale: float, causal: bool, stream=None):
    o = torch.empty_like(q)
    lse = torch.empty(lse_shape(q), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, sm_scale, causal, stream)
    return o, lse


def attention_backward(q, k, v, o, do, lse, sm_scale: float, causal: bool, workspace=None, stream=None):
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    fa_bwd(q, k, v, o, do, lse, dq, dk, dv, sm_scale, causal, workspace, stream)
    return dq, dk, dv


_SOFTMAX_DTYPES = {torch.float32: FA_FP32, torch.float16: FA_FP16, torch.bfloat16: FA_BF16}


def fa_softmax_rows(x: torch.Tensor, z: torch.Tensor, lse: Optional[torch.Tensor] = None, stream=None) -> None:
    """Row softmax of the 2-D CUDA tensor ``x`` ([rows, T], unit column
    stride) into ``z`` (same shape and dtype; may be ``x`` itself), and the
    natural-log row log-sum-exp into the float32 [rows] ``lse`` if given."""
    if x.dim() != 2 or z.shape != x.shape or z.dtype != x.dtype:
        raise ValueError("x and z must be 2-D tensors of the same shape and dtype")
    _check_cuda(x, z, lse)
    _check_same_device(x, z, lse)
    if x.dtype not in _SOFTMAX_DTYPES:
        raise TypeError(f"unsupported dtype {x.dtype} (float32, float16 or bfloat16)")
    if x.stride(1) != 1 or z.stride(1) != 1:
        raise ValueError("rows must be contiguous (unit column stride)")
    rows, T = x.shape
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() != rows or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 tensor of `rows` elements")
    # a single row's stride is never used: give the smallest valid one
    one = -(-T * x.element_size() // 16) * 16 // x.element_size()
    with torch.cuda.device(x.device):
        rc = lib().fa_softmax_rows(_ptr(x), _ptr(z), _ptr(lse) if lse is not None else None, rows, T,
                                   x.stride(0) if rows > 1 else one, z.stride(0) if rows > 1 else one,
                                   _SOFTMAX_DTYPES[x.dtype], _stream(stream, x.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_softmax_rows")
