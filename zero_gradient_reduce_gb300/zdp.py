"""Thin ctypes binding of libzdp (include/zdp.h), with the same call names.

Argument marshalling only: torch CUDA tensors (or raw device addresses) go
in as pointers, the current torch CUDA stream is the default stream, and a
non-OK status raises ZdpError.  Every step of the computation runs in the
library's CUDA kernels; this module has no fallback, and it refuses to run
when the library cannot be loaded.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Union

from . import build as _build

ZDP_OK = 0
ZDP_ERR_INVALID = -1
ZDP_ERR_CUDA = -2
ZDP_MAX_P = 64
ZDP_BF16 = 0
ZDP_FP16 = 1
ZDP_F32 = 2
ZDP_MOMENTS_F32 = 0
ZDP_MOMENTS_BF16 = 1
ZDP_QBLOCK = 256
ZDP_NOALLOC_MAX_LEN = 16_777_216

EXPORTS = (
    "zdp_version", "zdp_shard_size", "zdp_reduce_scatter", "zdp_adamw_shard",
    "zdp_all_gather", "zdp_step_workspace_bytes", "zdp_step", "zdp_step_noalloc",
    "zdp_step_ring_workspace_bytes", "zdp_step_ring", "zdp_quantize_blocks",
    "zdp_dequantize_blocks", "zdp_step_zpp", "zdp_copy", "zdp_last_error",
)


class ZdpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"zdp status {status}: {message}")
        self.status = status


class zdp_step_args(ctypes.Structure):
    _fields_ = [
        ("grads", ctypes.c_void_p),
        ("gdt", ctypes.c_int),
        ("master", ctypes.c_void_p),
        ("m", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("replicas", ctypes.c_void_p),
        ("n", ctypes.c_int64),
        ("off", ctypes.c_int64),
        ("len", ctypes.c_int64),
        ("P", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("lr", ctypes.c_float),
        ("b1", ctypes.c_float),
        ("b2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("wd", ctypes.c_float),
        ("t", ctypes.c_int),
        ("bucket_elems", ctypes.c_int64),
        ("check_overflow", ctypes.c_int),
        ("d_overflow", ctypes.c_void_p),
        ("d_sumsq", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("moment_dtype", ctypes.c_int),
    ]


class zdp_zpp_args(ctypes.Structure):
    _fields_ = [
        ("grads", ctypes.c_void_p),
        ("grad_scales", ctypes.c_void_p),
        ("master", ctypes.c_void_p),
        ("m", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("moment_dtype", ctypes.c_int),
        ("replicas", ctypes.c_void_p),
        ("replica_scales", ctypes.c_void_p),
        ("n", ctypes.c_int64),
        ("off", ctypes.c_int64),
        ("len", ctypes.c_int64),
        ("P", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("lr", ctypes.c_float),
        ("b1", ctypes.c_float),
        ("b2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("wd", ctypes.c_float),
        ("t", ctypes.c_int),
        ("d_overflow", ctypes.c_void_p),
        ("d_sumsq", ctypes.c_void_p),
    ]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libzdp.so (compiling it first if it is missing or stale).

    ZDP_LIBRARY_PATH, when set, names another build of the library to load
    instead (it is not rebuilt).
    """
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("ZDP_LIBRARY_PATH") or _build.LIB
    if path == _build.LIB and build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise ZdpError(ZDP_ERR_CUDA, f"libzdp not built ({path}); run the package build")
    lib = ctypes.CDLL(path)
    i64, vp, f32, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    lib.zdp_version.restype = ci
    lib.zdp_version.argtypes = []
    lib.zdp_shard_size.restype = i64
    lib.zdp_shard_size.argtypes = [i64, ci]
    lib.zdp_reduce_scatter.restype = ci
    lib.zdp_reduce_scatter.argtypes = [vp, ci, vp, i64, ci, f32, vp, vp, vp]
    lib.zdp_adamw_shard.restype = ci
    lib.zdp_adamw_shard.argtypes = [vp, vp, vp, vp, i64, f32, f32, f32, f32, f32, ci, vp]
    lib.zdp_all_gather.restype = ci
    lib.zdp_all_gather.argtypes = [vp, vp, i64, ci, vp]
    lib.zdp_step_workspace_bytes.restype = ctypes.c_size_t
    lib.zdp_step_workspace_bytes.argtypes = [ctypes.POINTER(zdp_step_args)]
    lib.zdp_step.restype = ci
    lib.zdp_step.argtypes = [ctypes.POINTER(zdp_step_args), vp]
    lib.zdp_step_ring_workspace_bytes.restype = ctypes.c_size_t
    lib.zdp_step_ring_workspace_bytes.argtypes = [ctypes.POINTER(zdp_step_args)]
    lib.zdp_step_ring.restype = ci
    lib.zdp_step_ring.argtypes = [ctypes.POINTER(zdp_step_args), vp]
    lib.zdp_quantize_blocks.restype = ci
    lib.zdp_quantize_blocks.argtypes = [vp, ci, i64, vp, vp, vp]
    lib.zdp_dequantize_blocks.restype = ci
    lib.zdp_dequantize_blocks.argtypes = [vp, vp, i64, vp, vp]
    lib.zdp_step_zpp.restype = ci
    lib.zdp_step_zpp.argtypes = [ctypes.POINTER(zdp_zpp_args), vp]
    lib.zdp_step_noalloc.restype = ci
    lib.zdp_step_noalloc.argtypes = [ctypes.POINTER(zdp_step_args), vp]
    lib.zdp_copy.restype = ci
    lib.zdp_copy.argtypes = [vp, vp, ctypes.c_int64, vp]
    lib.zdp_last_error.restype = ctypes.c_char_p
    lib.zdp_last_error.argtypes = []
    _lib = lib
    return lib


Ptr = Union[int, None, "torch.Tensor"]  # noqa: F821


def _addr(x: Ptr) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptr_array(xs: Sequence[Ptr]):
    arr = (ctypes.c_void_p * len(xs))(*[_addr(x) for x in xs])
    return arr


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int):
    if status != ZDP_OK:
        msg = load().zdp_last_error()
        raise ZdpError(status, msg.decode() if msg else "")


def _gdt(x, gdt):
    """The gradient type: `gdt` when given, else from a tensor's dtype (bf16
    or fp16; any other dtype is an error), else bf16 for raw addresses."""
    if gdt is not None:
        return gdt
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.float16:
                return ZDP_FP16
            if x.dtype == torch.bfloat16:
                return ZDP_BF16
            raise ValueError(f"gradients must be bfloat16 or float16, not {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    return ZDP_BF16


def _same_lengths(**seqs):
    """The library reads P pointers from each array: every list must hold
    exactly P of them."""
    lens = {k: len(v) for k, v in seqs.items()}
    if len(set(lens.values())) != 1:
        raise ValueError("pointer lists of different lengths: " +
                         ", ".join(f"{k}={n}" for k, n in lens.items()))
    P = next(iter(lens.values()))
    if not 1 <= P <= ZDP_MAX_P:
        raise ValueError(f"{P} ranks, outside 1..{ZDP_MAX_P}")
    return P


def zdp_version() -> int:
    return int(load().zdp_version())


def zdp_shard_size(n: int, P: int) -> int:
    return int(load().zdp_shard_size(n, P))


def zdp_last_error() -> str:
    return load().zdp_last_error().decode()


def zdp_reduce_scatter(grads: Sequence[Ptr], shards: Ptr, n: int, P: int, scale: float,
                       d_overflow: Ptr = None, d_sumsq: Ptr = None, gdt: Optional[int] = None,
                       stream=None) -> None:
    if len(grads) != P:
        raise ValueError(f"{len(grads)} gradient pointers for P={P}")
    arr = _ptr_array(grads)
    _check(load().zdp_reduce_scatter(arr, _gdt(grads[0] if grads else None, gdt), _addr(shards),
                                     n, P, scale,
                                     _addr(d_overflow), _addr(d_sumsq), _stream(stream)))


def zdp_adamw_shard(master: Ptr, m: Ptr, v: Ptr, grad_shard: Ptr, count: int, lr: float,
                    b1: float, b2: float, eps: float, wd: float, t: int, stream=None) -> None:
    _check(load().zdp_adamw_shard(_addr(master), _addr(m), _addr(v), _addr(grad_shard), count,
                                  lr, b1, b2, eps, wd, t, _stream(stream)))


def zdp_all_gather(master: Ptr, replicas: Sequence[Ptr], n: int, P: int, stream=None) -> None:
    if len(replicas) != P:
        raise ValueError(f"{len(replicas)} replica pointers for P={P}")
    arr = _ptr_array(replicas)
    _check(load().zdp_all_gather(_addr(master), arr, n, P, _stream(stream)))


def make_step_args(grads: Sequence[Ptr], master: Ptr, m: Ptr, v: Ptr, replicas: Sequence[Ptr],
                   n: int, scale: float, lr: float, b1: float, b2: float, eps: float, wd: float,
                   t: int, off: int = 0, length: Optional[int] = None, bucket_elems: int = 0,
                   check_overflow: bool = False, d_overflow: Ptr = None, d_sumsq: Ptr = None,
                   workspace: Ptr = None, workspace_bytes: int = 0,
                   gdt: Optional[int] = None, moments: str = "f32"):
    """Builds a zdp_step_args for the range [off, off+length) (default: to n).

    moments: "f32" (m and v fp32) or "bf16" (m and v bf16 buffers).

    Returns (args, keepalive).  `keepalive` holds the pointer arrays behind
    the struct's grads/replicas fields and every object passed in (so tensors
    made inline, e.g. clones in the argument list, are not freed while their
    addresses sit in `args`); it must outlive every use of `args`.
    """
    P = _same_lengths(grads=grads, replicas=replicas)
    len_ = (n - off) if length is None else length
    garr = _ptr_array(grads)
    rarr = _ptr_array(replicas)
    a = zdp_step_args()
    a.grads = ctypes.cast(garr, ctypes.c_void_p)
    a.gdt = _gdt(grads[0], gdt)
    a.master = _addr(master)
    a.m = _addr(m)
    a.v = _addr(v)
    a.replicas = ctypes.cast(rarr, ctypes.c_void_p)
    a.n = n
    a.off = off
    a.len = len_
    a.P = P
    a.scale = scale
    a.lr, a.b1, a.b2, a.eps, a.wd = lr, b1, b2, eps, wd
    a.t = t
    a.bucket_elems = bucket_elems
    a.check_overflow = int(bool(check_overflow))
    a.d_overflow = _addr(d_overflow)
    a.d_sumsq = _addr(d_sumsq)
    a.workspace = _addr(workspace)
    a.workspace_bytes = workspace_bytes
    a.moment_dtype = {"f32": ZDP_MOMENTS_F32, "bf16": ZDP_MOMENTS_BF16}[moments]
    return a, (garr, rarr, list(grads), list(replicas), master, m, v, d_overflow, d_sumsq,
               workspace)


def zdp_step_workspace_bytes(args: zdp_step_args) -> int:
    return int(load().zdp_step_workspace_bytes(ctypes.byref(args)))


def zdp_step(args: zdp_step_args, stream=None) -> None:
    _check(load().zdp_step(ctypes.byref(args), _stream(stream)))


def zdp_step_ring_workspace_bytes(args: zdp_step_args) -> int:
    return int(load().zdp_step_ring_workspace_bytes(ctypes.byref(args)))


def zdp_step_ring(args: zdp_step_args, stream=None) -> None:
    """The step as the literal ring schedule (2P-1 launches); args.workspace
    must hold zdp_step_ring_workspace_bytes(args) bytes."""
    _check(load().zdp_step_ring(ctypes.byref(args), _stream(stream)))


def zdp_step_noalloc(args: zdp_step_args, stream=None) -> None:
    """The overflow-checked step with the library's own static scratch (no
    workspace, no allocation); len must not exceed ZDP_NOALLOC_MAX_LEN."""
    _check(load().zdp_step_noalloc(ctypes.byref(args), _stream(stream)))


def zdp_quantize_blocks(x: Ptr, xdt: int, n: int, q: Ptr, scales: Ptr, stream=None) -> None:
    """Block int8 quantization (blocks of 256) of n bf16/fp16/fp32 values."""
    _check(load().zdp_quantize_blocks(_addr(x), xdt, n, _addr(q), _addr(scales), _stream(stream)))


def zdp_dequantize_blocks(q: Ptr, scales: Ptr, n: int, out: Ptr, stream=None) -> None:
    _check(load().zdp_dequantize_blocks(_addr(q), _addr(scales), n, _addr(out), _stream(stream)))


def zdp_copy(dst: Ptr, src: Ptr, nbytes: int, stream=None) -> None:
    """Plain 16-byte streaming device copy (the copy-ceiling probe)."""
    _check(load().zdp_copy(_addr(dst), _addr(src), nbytes, _stream(stream)))


def make_zpp_args(grads: Sequence[Ptr], grad_scales: Sequence[Ptr], master: Ptr, m: Ptr, v: Ptr,
                  replicas: Sequence[Ptr], replica_scales: Sequence[Ptr], n: int, scale: float,
                  lr: float, b1: float, b2: float, eps: float, wd: float, t: int, off: int = 0,
                  length: Optional[int] = None, d_overflow: Ptr = None, d_sumsq: Ptr = None,
                  moments: str = "f32"):
    """Builds a zdp_zpp_args; returns (args, keepalive) as make_step_args
    (keepalive also holds every object passed in)."""
    P = _same_lengths(grads=grads, grad_scales=grad_scales, replicas=replicas,
                      replica_scales=replica_scales)
    arrs = [_ptr_array(x) for x in (grads, grad_scales, replicas, replica_scales)]
    a = zdp_zpp_args()
    a.grads, a.grad_scales, a.replicas, a.replica_scales = [
        ctypes.cast(x, ctypes.c_void_p) for x in arrs]
    a.master, a.m, a.v = _addr(master), _addr(m), _addr(v)
    a.moment_dtype = {"f32": ZDP_MOMENTS_F32, "bf16": ZDP_MOMENTS_BF16}[moments]
    a.n, a.off = n, off
    a.len = (n - off) if length is None else length
    a.P = P
    a.scale, a.lr, a.b1, a.b2, a.eps, a.wd, a.t = scale, lr, b1, b2, eps, wd, t
    a.d_overflow, a.d_sumsq = _addr(d_overflow), _addr(d_sumsq)
    return a, (arrs, list(grads), list(grad_scales), list(replicas), list(replica_scales),
               master, m, v, d_overflow, d_sumsq)


def zdp_step_zpp(args: zdp_zpp_args, stream=None) -> None:
    """The ZeRO++ step: int8-block gradients in, int8-block replicas out."""
    _check(load().zdp_step_zpp(ctypes.byref(args), _stream(stream)))
