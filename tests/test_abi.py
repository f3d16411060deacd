"""The C ABI without a GPU: the library builds and loads, exports every
function include/zdp.h declares, and rejects bad arguments on the host
before touching CUDA (no call here reaches a kernel launch)."""

import ctypes
import os
import re

import pytest

from zero_gradient_reduce_gb300 import build, zdp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "zdp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(zdp_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return zdp.load()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert set(declared) == set(zdp.EXPORTS)
    raw = ctypes.CDLL(build.LIB)
    for name in declared:
        assert hasattr(raw, name), name


def test_pure_host_functions(lib):
    assert zdp.zdp_version() == 100
    assert zdp.zdp_shard_size(10, 4) == 3
    assert zdp.zdp_shard_size(8, 8) == 1
    assert zdp.zdp_shard_size(1, 64) == 1
    assert zdp.zdp_shard_size(1_311_227_904, 8) == 163_903_488
    assert zdp.zdp_shard_size(0, 4) == -1
    assert zdp.zdp_shard_size(10, 0) == -1
    assert zdp.zdp_shard_size(10, 65) == -1


FAKE = 1 << 40  # an address that is never dereferenced: every call below fails its checks first


def _args(**kw):
    P = kw.pop("P", 2)
    base = dict(n=1000, scale=0.5, t=1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)
    base.update(kw)
    grads = [FAKE + q * (1 << 20) for q in range(P)]
    reps = [FAKE + (16 + q) * (1 << 20) for q in range(P)]
    return zdp.make_step_args(grads, FAKE + (100 << 20), FAKE + (104 << 20),
                              FAKE + (108 << 20), reps, **base)


@pytest.mark.parametrize("mutate,needle", [
    (lambda a: setattr(a, "P", 0), "P=0"),
    (lambda a: setattr(a, "P", 65), "P=65"),
    (lambda a: setattr(a, "n", 0), "n=0"),
    (lambda a: setattr(a, "t", 0), "t=0"),
    (lambda a: setattr(a, "off", 999), "outside"),
    (lambda a: setattr(a, "len", -1), "outside"),
    (lambda a: setattr(a, "gdt", 7), "gradient type"),
    (lambda a: setattr(a, "master", None), "NULL"),
    (lambda a: setattr(a, "master", FAKE + (16 << 20)), "overlap"),
    (lambda a: setattr(a, "m", FAKE + (100 << 20) + 400), "overlap"),
    (lambda a: setattr(a, "master", FAKE + (100 << 20) + 2), "aligned"),
    (lambda a: setattr(a, "check_overflow", 1), "workspace"),
    (lambda a: setattr(a, "bucket_elems", -5), "bucket"),
])
def test_step_rejects_bad_arguments(lib, mutate, needle):
    a, keep = _args()
    mutate(a)
    with pytest.raises(zdp.ZdpError) as e:
        zdp.zdp_step(a, stream=0)
    assert e.value.status == zdp.ZDP_ERR_INVALID
    assert needle in str(e.value)


def test_step_rejects_small_workspace(lib):
    a, keep = _args(check_overflow=True)
    need = zdp.zdp_step_workspace_bytes(a)
    assert need == 256 + ((1000 + 8) * 4 + 255) // 256 * 256
    a.workspace = FAKE + (200 << 20)
    a.workspace_bytes = need - 1
    with pytest.raises(zdp.ZdpError, match="workspace of"):
        zdp.zdp_step(a, stream=0)


def test_gradient_overlapping_a_replica_is_rejected(lib):
    a, keep = _args()
    g = (ctypes.c_void_p * 2)(FAKE, FAKE + (16 << 20) + 64)  # grads[1] inside replicas[0]
    a.grads = ctypes.cast(g, ctypes.c_void_p)
    with pytest.raises(zdp.ZdpError, match="overlap"):
        zdp.zdp_step(a, stream=0)


def test_unfused_calls_reject_bad_arguments(lib):
    with pytest.raises(zdp.ZdpError, match="P=0"):
        zdp.zdp_reduce_scatter([], FAKE, 10, 0, 1.0, stream=0)
    with pytest.raises(zdp.ZdpError, match="overlap"):
        zdp.zdp_reduce_scatter([FAKE, FAKE + 4096], FAKE + 8, 100, 2, 1.0, stream=0)
    with pytest.raises(zdp.ZdpError, match="t=0"):
        zdp.zdp_adamw_shard(FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288, 10, 1e-3, 0.9, 0.95,
                            1e-8, 0.0, 0, stream=0)
    with pytest.raises(zdp.ZdpError, match="overlap"):
        zdp.zdp_adamw_shard(FAKE, FAKE + 16, FAKE + 8192, FAKE + 12288, 10, 1e-3, 0.9, 0.95,
                            1e-8, 0.0, 1, stream=0)
    with pytest.raises(zdp.ZdpError, match="overlap"):
        zdp.zdp_all_gather(FAKE, [FAKE + 4096, FAKE + 4096 + 100], 100, 2, stream=0)
    # count 0 is a valid no-op that never reaches CUDA
    zdp.zdp_adamw_shard(FAKE, FAKE, FAKE, FAKE, 0, 1e-3, 0.9, 0.95, 1e-8, 0.0, 1, stream=0)


def test_zero_length_step_is_a_host_no_op(lib):
    a, keep = _args(off=10, length=0)
    zdp.zdp_step(a, stream=0)


@pytest.mark.parametrize("mutate,needle", [
    (lambda a: setattr(a, "off", 1), "whole model"),
    (lambda a: setattr(a, "len", 10), "whole model"),
    (lambda a: setattr(a, "check_overflow", 1), "overflow"),
    (lambda a: setattr(a, "bucket_elems", 64), "buckets"),
    (lambda a: None, "workspace"),  # no workspace given
])
def test_ring_rejects_bad_arguments(lib, mutate, needle):
    a, keep = _args()
    mutate(a)
    with pytest.raises(zdp.ZdpError, match=needle):
        zdp.zdp_step_ring(a, stream=0)


def test_ring_workspace_bytes(lib):
    a, keep = _args()  # n = 1000, P = 2: S = 500, two message sets of P*S fp32
    assert zdp.zdp_step_ring_workspace_bytes(a) == (2 * 2 * 500 * 4 + 255) // 256 * 256


def _zpp_args(**kw):
    P = 2
    base = dict(n=1000, scale=0.5, t=1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)
    base.update(kw)
    g = [FAKE + q * (1 << 20) for q in range(P)]
    gs = [FAKE + (4 + q) * (1 << 20) for q in range(P)]
    r = [FAKE + (8 + q) * (1 << 20) for q in range(P)]
    rs = [FAKE + (12 + q) * (1 << 20) for q in range(P)]
    return zdp.make_zpp_args(g, gs, FAKE + (100 << 20), FAKE + (104 << 20), FAKE + (108 << 20),
                             r, rs, **base)


@pytest.mark.parametrize("mutate,needle", [
    (lambda a: (setattr(a, "off", 100), setattr(a, "len", 256)), "block"),
    (lambda a: setattr(a, "len", 300), "block"),
    (lambda a: setattr(a, "P", 0), "P=0"),
    (lambda a: setattr(a, "t", 0), "t=0"),
    (lambda a: setattr(a, "master", FAKE + (100 << 20) + 4), "16-byte"),
    (lambda a: setattr(a, "m", FAKE + (8 << 20) + 512), "overlap"),
    (lambda a: setattr(a, "moment_dtype", 5), "moment"),
])
def test_zpp_rejects_bad_arguments(lib, mutate, needle):
    a, keep = _zpp_args()
    mutate(a)
    with pytest.raises(zdp.ZdpError, match=needle):
        zdp.zdp_step_zpp(a, stream=0)


def test_copy_rejects_bad_arguments(lib):
    with pytest.raises(zdp.ZdpError, match="multiple of 16"):
        zdp.zdp_copy(FAKE, FAKE + 4096, 100, stream=0)
    with pytest.raises(zdp.ZdpError, match="aligned"):
        zdp.zdp_copy(FAKE + 8, FAKE + 4096, 256, stream=0)
    with pytest.raises(zdp.ZdpError, match="overlap"):
        zdp.zdp_copy(FAKE, FAKE + 64, 256, stream=0)
    with pytest.raises(zdp.ZdpError, match="NULL"):
        zdp.zdp_copy(0, FAKE, 256, stream=0)
    zdp.zdp_copy(FAKE, FAKE, 0, stream=0)  # nothing to do: never reaches CUDA


def test_quantizer_rejects_bad_arguments(lib):
    with pytest.raises(zdp.ZdpError, match="input type"):
        zdp.zdp_quantize_blocks(FAKE, 7, 10, FAKE + 4096, FAKE + 8192, stream=0)
    with pytest.raises(zdp.ZdpError, match="overlap"):
        zdp.zdp_quantize_blocks(FAKE, zdp.ZDP_F32, 1000, FAKE + 16, FAKE + 8192, stream=0)
    with pytest.raises(zdp.ZdpError, match="overlap"):
        zdp.zdp_dequantize_blocks(FAKE, FAKE + 8192, 1000, FAKE + 500, stream=0)


def test_keepalive_holds_every_buffer_passed_in(lib):
    # The struct stores raw addresses; the keepalive must keep the objects
    # behind them alive, or a tensor made inline would be freed at once.
    import gc
    import weakref

    import torch
    grads = [torch.zeros(16, dtype=torch.bfloat16) for _ in range(2)]
    reps = [torch.zeros(16, dtype=torch.bfloat16) for _ in range(2)]
    state = [torch.zeros(16) for _ in range(3)]
    refs = [weakref.ref(x) for x in (*grads, *reps, *state)]
    a, keep = zdp.make_step_args(grads, *state, reps, n=16, scale=0.5, t=1, lr=1e-3, b1=0.9,
                                 b2=0.95, eps=1e-8, wd=0.0)
    del grads, reps, state
    gc.collect()
    assert all(r() is not None for r in refs)
    del keep
    gc.collect()
    assert all(r() is None for r in refs)



def test_binding_rejects_pointer_lists_of_the_wrong_length(lib):
    # The library reads P pointers from each host array; a short list would
    # be read past its end, so the binding refuses it before the call.
    hp = dict(scale=0.5, t=1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.0)
    g2, r1 = [FAKE, FAKE + 4096], [FAKE + 8192]
    with pytest.raises(ValueError, match="different lengths"):
        zdp.make_step_args(g2, FAKE + 16384, FAKE + 20480, FAKE + 24576, r1, n=16, **hp)
    with pytest.raises(ValueError, match="outside"):
        zdp.make_step_args([], FAKE + 16384, FAKE + 20480, FAKE + 24576, [], n=16, **hp)
    with pytest.raises(ValueError, match="different lengths"):
        zdp.make_zpp_args(g2, g2, FAKE + 16384, FAKE + 20480, FAKE + 24576, g2, r1, n=256, **hp)
    with pytest.raises(ValueError, match="for P=3"):
        zdp.zdp_reduce_scatter(g2, FAKE + 8192, 16, 3, 0.5, stream=0)
    with pytest.raises(ValueError, match="for P=2"):
        zdp.zdp_all_gather(FAKE, r1, 16, 2, stream=0)


def test_binding_rejects_gradients_of_another_dtype(lib):
    import torch
    g = [torch.zeros(16, dtype=torch.float32) for _ in range(2)]
    with pytest.raises(ValueError, match="bfloat16 or float16"):
        zdp.make_step_args(g, FAKE + 16384, FAKE + 20480, FAKE + 24576, [FAKE, FAKE + 4096],
                           n=16, scale=0.5, t=1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.0)
