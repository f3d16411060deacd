"""ZeRO memory and communication accounting, written out from the pages.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
  * Fudan MLSys ch. 9 "Distributed training and data parallelism", 9.4.2:
    16 bytes of model state per parameter and the per-GPU formulas
    ZeRO-1 4Y + 12Y/N, ZeRO-2 2Y + 14Y/N, ZeRO-3 16Y/N (Y = parameter count).
  * CS336 Lecture 7 notes, section 7: 16 bytes per parameter = bf16 parameter,
    bf16 gradient, fp32 master weight, fp32 m, fp32 v.
  * CS336 Lecture 7 notes, 4.3 and exercise 2; the interview guide 2.4:
    a ring all-reduce sends 2(p-1) messages of n/p elements per rank; ZeRO-3
    moves 3Y per step against 2Y for DDP / ZeRO-1 / ZeRO-2.
"""

from __future__ import annotations

# bytes per parameter of mixed-precision AdamW state, component by component
STATE_BYTES = {
    "param_bf16": 2,
    "grad_bf16": 2,
    "master_fp32": 4,
    "m_fp32": 4,
    "v_fp32": 4,
}


# CS336 Lecture 7 notes, 8.4: everything except the fp32 master weight in
# BF16 -- 12 bytes per parameter.
STATE_BYTES_BF16_MOMENTS = {
    "param_bf16": 2,
    "grad_bf16": 2,
    "master_fp32": 4,
    "m_bf16": 2,
    "v_bf16": 2,
}


def bytes_per_param(moments: str = "f32") -> int:
    return sum((STATE_BYTES if moments == "f32" else STATE_BYTES_BF16_MOMENTS).values())


def optimizer_bytes_per_param() -> int:
    return STATE_BYTES["master_fp32"] + STATE_BYTES["m_fp32"] + STATE_BYTES["v_fp32"]


def zero_bytes_per_gpu(psi: float, n_gpus: int, stage: int) -> float:
    """Model-state bytes per GPU; stage 0 = plain data parallelism."""
    p = STATE_BYTES["param_bf16"] * psi
    g = STATE_BYTES["grad_bf16"] * psi
    o = optimizer_bytes_per_param() * psi
    if stage == 0:
        return p + g + o
    if stage == 1:
        return p + g + o / n_gpus
    if stage == 2:
        return p + (g + o) / n_gpus
    if stage == 3:
        return (p + g + o) / n_gpus
    raise ValueError(stage)


def ring_sent_elements_per_rank(n: int, p: int) -> int:
    """Elements one rank sends in a ring all-reduce of n elements (padded to p)."""
    s = -(-n // p)
    return 2 * (p - 1) * s


def ring_allreduce_bytes_per_rank(n: int, p: int, elem_bytes: int) -> float:
    """2 (p-1)/p * n * elem_bytes, unpadded, as the pages state it."""
    return 2.0 * (p - 1) / p * n * elem_bytes


def zero3_bytes_per_rank(n: int, p: int, elem_bytes: int) -> float:
    """Two parameter all-gathers and one gradient reduce-scatter: 3 (p-1)/p * n."""
    return 3.0 * (p - 1) / p * n * elem_bytes


def fused_step_bytes_per_param(P: int, grad_bytes: int = 2, param_bytes: int = 2,
                               moment_bytes: int = 4) -> int:
    """HBM bytes one fused step moves per parameter when the P ranks share one HBM.

    Each rank's gradient is read once (P * grad_bytes), the fp32 master and
    the two moments are read and written once (2 * (4 + 2 * moment_bytes)),
    and each rank's replica is written once (P * param_bytes).
    """
    state = 4 + 2 * moment_bytes
    return P * grad_bytes + state + state + P * param_bytes
