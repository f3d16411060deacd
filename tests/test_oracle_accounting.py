"""Pins of the ZeRO memory accounting: 16 bytes per parameter (CS336 Lecture 7
notes, section 7; Fudan MLSys ch. 9, 9.4.2) and exercise 6 of the CS336
notes, and the HBM bytes per parameter of one fused step."""

import pytest

from conftest import golden
from oracle import accounting


def test_sixteen_bytes_per_parameter():
    assert accounting.bytes_per_param() == 16
    assert accounting.optimizer_bytes_per_param() == 12


def test_exercise6_zero_memory():
    rows = {r[0]: r[1:] for r in golden("exercise6_zero_memory.txt")}
    gpus, psi = int(rows["gpus"][0]), float(rows["params"][0])
    for stage in range(4):
        want, tol, fits = rows[f"stage{stage}"]
        got = accounting.zero_bytes_per_gpu(psi, gpus, stage)
        assert got == pytest.approx(float(want), rel=float(tol) + 1e-12)
        assert (got <= 80e9) == (fits == "yes")


def test_fused_step_bytes():
    # 2P gradient reads + 12 state reads + 12 state writes + 2P replica writes
    assert [accounting.fused_step_bytes_per_param(P) for P in (2, 4, 8, 16, 64)] == \
        [32, 40, 56, 88, 280]


def test_twelve_bytes_with_bf16_moments():
    # CS336 Lecture 7 notes, 8.4: all but the master weight in BF16
    assert accounting.bytes_per_param("bf16") == 12
    assert accounting.fused_step_bytes_per_param(8, moment_bytes=2) == 48
