"""CPU oracle for the ZeRO synchronisation-and-update step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
loads it, and it never loads the CUDA library: the two share no code.

The arithmetic lives in ``zdp_oracle.cpp`` (plain single-threaded C++17,
compiled with ``-ffp-contract=off`` so that every operation rounds on its own).
This module only compiles it on demand and marshals numpy arrays into it.
The ZeRO memory and communication accounting is in ``accounting.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zdp_oracle.cpp")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP16 = 1

_CXXFLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (skipped when up to date)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["g++", *_CXXFLAGS, "-o", tmp, _SRC], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
        vp = ctypes.c_void_p
        sig = {
            "ora_bf16_to_f32": (f32, [ctypes.c_uint16]),
            "ora_f16_to_f32": (f32, [ctypes.c_uint16]),
            "ora_f32_to_bf16": (ctypes.c_uint16, [f32]),
            "ora_bf16_to_f32_array": (None, [vp, vp, i64]),
            "ora_f16_to_f32_array": (None, [vp, vp, i64]),
            "ora_f32_to_bf16_array": (None, [vp, vp, i64]),
            "ora_shard_size": (i64, [i64, ctypes.c_int]),
            "ora_ring_reduce_scatter_sim": (None, [vp, ctypes.c_int, i64, ctypes.c_int, vp]),
            "ora_ring_all_gather_sim": (None, [vp, ctypes.c_int, i64, ctypes.c_int, vp]),
            "ora_reduce_scatter": (None, [vp, i64, ctypes.c_int, vp, i64, ctypes.c_int, f32, vp, vp]),
            "ora_adamw": (None, [vp, vp, vp, vp, i64, f32, f32, f32, f32, f32, ctypes.c_int]),
            "ora_all_gather": (None, [vp, vp, i64, i64, ctypes.c_int]),
            "ora_step": (ctypes.c_int, [vp, i64, ctypes.c_int, vp, vp, vp, vp, i64, i64, i64, i64,
                                        i64, ctypes.c_int, f32, f32, f32, f32, f32, f32,
                                        ctypes.c_int, ctypes.c_int, vp, vp]),
            "ora_step_sampled": (ctypes.c_int, [vp, vp, i64, ctypes.c_int, vp, vp, vp, vp, vp, i64,
                                                ctypes.c_int, f32, f32, f32, f32, f32, f32,
                                                ctypes.c_int, ctypes.c_int, vp]),
            "ora_quantize_blocks": (None, [vp, i64, vp, vp]),
            "ora_dequantize_blocks": (None, [vp, vp, i64, vp]),
            "ora_step_zpp": (ctypes.c_int, [vp, i64, vp, i64, vp, vp, vp, ctypes.c_int, vp, i64,
                                            vp, i64, i64, i64, i64, i64, ctypes.c_int, f32, f32,
                                            f32, f32, f32, f32, ctypes.c_int, vp, vp]),
            "ora_step_mdt": (ctypes.c_int, [vp, i64, ctypes.c_int, vp, vp, vp, ctypes.c_int, vp,
                                            i64, i64, i64, i64, i64, ctypes.c_int, f32, f32, f32,
                                            f32, f32, f32, ctypes.c_int, ctypes.c_int, vp, vp]),
            "ora_step_sampled_mdt": (ctypes.c_int, [vp, vp, i64, ctypes.c_int, vp, vp, vp,
                                                    ctypes.c_int, vp, vp, i64, ctypes.c_int, f32,
                                                    f32, f32, f32, f32, f32, ctypes.c_int,
                                                    ctypes.c_int, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        del i32, f64
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    out = np.ascontiguousarray(a, dtype=dtype)
    return out


def _gbits(grads) -> np.ndarray:
    """Gradient rows as a contiguous uint16 bit array (bf16 or fp16 payload)."""
    g = np.asarray(grads)
    if g.dtype == np.float16:
        g = g.view(np.uint16)
    if g.dtype != np.uint16:
        raise TypeError("gradients must be given as uint16 bit patterns or float16")
    return np.ascontiguousarray(g)


# ---- number formats ---------------------------------------------------------

def bf16_to_f32(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float32)
    _load().ora_bf16_to_f32_array(_ptr(b), _ptr(out), b.size)
    return out


def f16_to_f32(bits) -> np.ndarray:
    b = _c(np.asarray(bits).view(np.uint16) if np.asarray(bits).dtype == np.float16 else bits,
           np.uint16)
    out = np.empty(b.shape, np.float32)
    _load().ora_f16_to_f32_array(_ptr(b), _ptr(out), b.size)
    return out


def f32_to_bf16(x) -> np.ndarray:
    a = _c(x, np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().ora_f32_to_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


def shard_size(n: int, P: int) -> int:
    return int(_load().ora_shard_size(n, P))


# ---- the ring, literally ----------------------------------------------------

def ring_reduce_scatter_sim(bufs: np.ndarray, shift: int = 1):
    """In place on bufs[P, P*S] (fp32).  Returns per-rank element send counts."""
    P = bufs.shape[0]
    assert bufs.dtype == np.float32 and bufs.flags.c_contiguous and bufs.shape[1] % P == 0
    sent = np.zeros(P, np.int64)
    _load().ora_ring_reduce_scatter_sim(_ptr(bufs), P, bufs.shape[1] // P, shift, _ptr(sent))
    return sent


def ring_all_gather_sim(bufs: np.ndarray, shift: int = 1):
    P = bufs.shape[0]
    assert bufs.dtype == np.float32 and bufs.flags.c_contiguous and bufs.shape[1] % P == 0
    sent = np.zeros(P, np.int64)
    _load().ora_ring_all_gather_sim(_ptr(bufs), P, bufs.shape[1] // P, shift, _ptr(sent))
    return sent


# ---- collectives and optimizer by definition -----------------------------------

def reduce_scatter(grads, gdt: int, n: int, scale: float, want_sumsq: bool = False):
    """grads: [P, >=n] uint16 bit rows.  Returns (shards[P*S] fp32, overflow, sumsq)."""
    g = _gbits(grads)
    P = g.shape[0]
    S = shard_size(n, P)
    shards = np.empty(P * S, np.float32)
    flag = np.zeros(1, np.int32)
    ss = np.zeros(1, np.float64)
    _load().ora_reduce_scatter(_ptr(g), g.shape[1], gdt, _ptr(shards), n, P, scale, _ptr(flag),
                               _ptr(ss) if want_sumsq else None)
    return shards, int(flag[0]), float(ss[0])


def adamw(w, m, v, g, lr, b1, b2, eps, wd, t):
    """Elementwise AdamW; returns updated copies (w, m, v)."""
    w = _c(w, np.float32).copy()
    m = _c(m, np.float32).copy()
    v = _c(v, np.float32).copy()
    g = _c(g, np.float32)
    assert w.size == m.size == v.size == g.size
    _load().ora_adamw(_ptr(w), _ptr(m), _ptr(v), _ptr(g), w.size, lr, b1, b2, eps, wd, t)
    return w, m, v


def all_gather(master, n: int, P: int) -> np.ndarray:
    w = _c(master, np.float32)
    rep = np.empty((P, n), np.uint16)
    _load().ora_all_gather(_ptr(w), _ptr(rep), n, n, P)
    return rep


MOMENTS = {"f32": (0, np.float32), "bf16": (1, np.uint16)}


def step(grads, gdt, master, m, v, replicas, n, off, len_, scale, lr, b1, b2, eps, wd, t,
         check_overflow=False, base=0, moments="f32"):
    """The fused step on host arrays, in place on master/m/v/replicas.

    grads: [P, >=len_] uint16 rows holding elements [off, off+len_).
    master: float32 array holding global elements [base, off+len_); m and v
    likewise, float32 (moments="f32") or bf16 bit patterns as uint16
    (moments="bf16").
    replicas: [P, >= off+len_-base] uint16, element i in column i - base.
    Returns (overflow, sumsq).
    """
    g = _gbits(grads)
    P = g.shape[0]
    mdt, mtype = MOMENTS[moments]
    assert 0 <= base <= off
    need = off + len_ - base
    assert master.dtype == np.float32 and master.flags.c_contiguous and master.size >= need
    for a in (m, v):
        assert a.dtype == mtype and a.flags.c_contiguous and a.size >= need
    assert replicas.dtype == np.uint16 and replicas.flags.c_contiguous
    assert replicas.shape[0] == P and replicas.shape[1] >= need
    flag = np.zeros(1, np.int32)
    ss = np.zeros(1, np.float64)
    rc = _load().ora_step_mdt(_ptr(g), g.shape[1], gdt, _ptr(master), _ptr(m), _ptr(v), mdt,
                              _ptr(replicas), replicas.shape[1], base, n, off, len_, P, scale, lr,
                              b1, b2, eps, wd, t, int(bool(check_overflow)), _ptr(flag), _ptr(ss))
    if rc != 0:
        raise ValueError("oracle step: bad arguments")
    return int(flag[0]), float(ss[0])


def step_sampled(gs, idx, gdt, w, m, v, n, scale, lr, b1, b2, eps, wd, t, skip=False,
                 moments="f32"):
    """The step on k sampled global indices.

    gs: [P, k] uint16 gradient values at idx; w: [k] float32, m/v: [k]
    float32 or bf16 bits (moments="bf16"), all updated in place.  Returns
    (g_reduced[k] fp32, replica_bits[k] uint16, overflow).
    """
    g = _gbits(gs)
    P, k = g.shape
    mdt, mtype = MOMENTS[moments]
    idx = _c(idx, np.int64)
    assert idx.size == k
    assert w.dtype == np.float32 and w.flags.c_contiguous and w.size == k
    for a in (m, v):
        assert a.dtype == mtype and a.flags.c_contiguous and a.size == k
    gout = np.empty(k, np.float32)
    rep = np.empty(k, np.uint16)
    flag = np.zeros(1, np.int32)
    rc = _load().ora_step_sampled_mdt(_ptr(g), _ptr(idx), k, gdt, _ptr(w), _ptr(m), _ptr(v), mdt,
                                      _ptr(gout), _ptr(rep), n, P, scale, lr, b1, b2, eps, wd, t,
                                      int(bool(skip)), _ptr(flag))
    if rc != 0:
        raise ValueError("oracle step_sampled: bad arguments")
    return gout, rep, int(flag[0])


# ---- ZeRO++ block quantization (blocks of 256 elements) -------------------------

QBLOCK = 256


def quantize_blocks(x):
    """fp32 values -> (int8 q, fp32 scale per block of 256)."""
    a = _c(x, np.float32)
    q = np.empty(a.size, np.int8)
    sc = np.empty(-(-a.size // QBLOCK), np.float32)
    _load().ora_quantize_blocks(_ptr(a), a.size, _ptr(q), _ptr(sc))
    return q, sc


def dequantize_blocks(q, scales):
    qq = _c(q, np.int8)
    sc = _c(scales, np.float32)
    out = np.empty(qq.size, np.float32)
    _load().ora_dequantize_blocks(_ptr(qq), _ptr(sc), qq.size, _ptr(out))
    return out


def step_zpp(gq, gs, master, m, v, rq, rs, n, off, len_, scale, lr, b1, b2, eps, wd, t,
             base=0, moments="f32"):
    """The ZeRO++ step: int8-block gradients in, int8-block replicas out.

    gq: [P, >=len_] int8 rows (elements off..off+len_); gs: [P, blocks] fp32
    scales of those rows (block (off+j)//256 - off//256).  master/m/v hold
    global elements from `base`; rq: [P, >= off+len_-base] int8 and rs: [P,
    blocks] fp32 replica scales, block i//256 - base//256.  In place.
    Returns (overflow, sumsq).
    """
    gq = np.ascontiguousarray(gq, np.int8)
    gs = np.ascontiguousarray(gs, np.float32)
    P = gq.shape[0]
    mdt, mtype = MOMENTS[moments]
    assert master.dtype == np.float32 and m.dtype == mtype and v.dtype == mtype
    assert rq.dtype == np.int8 and rq.flags.c_contiguous and rs.dtype == np.float32
    flag = np.zeros(1, np.int32)
    ss = np.zeros(1, np.float64)
    rc = _load().ora_step_zpp(_ptr(gq), gq.shape[1], _ptr(gs), gs.shape[1], _ptr(master),
                              _ptr(m), _ptr(v), mdt, _ptr(rq), rq.shape[1], _ptr(rs),
                              rs.shape[1], base, n, off, len_, P, scale, lr, b1, b2, eps, wd, t,
                              _ptr(flag), _ptr(ss))
    if rc != 0:
        raise ValueError("oracle step_zpp: bad arguments")
    return int(flag[0]), float(ss[0])
