"""Small CPU-side helpers shared by the oracle tests."""

import numpy as np
import torch

HP = dict(lr=1e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)


def bf16_bits(x) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def random_state(n, rng):
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = rng.uniform(0, 1e-6, n).astype(np.float32)
    return w, m, v
