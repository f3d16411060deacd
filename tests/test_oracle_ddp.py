"""The data-parallel identities the pages state, on a tiny linear model.

CS336 Lecture 7 notes, 6.1: with equal shard sizes the mean of the ranks'
gradients is the full-batch gradient, so data parallelism equals one large
batch; 6.2: after the all-reduce every rank applies the same update, so the
replicas stay bit-identical.  Model: y = W x, W 4 x 3, batch 16, mean-squared
error; the gradients are computed here in fp64.
"""

import numpy as np

P, B, OUT, IN = 4, 16, 4, 3


def _grad(W, X, Y):
    # d/dW of mean((X W^T - Y)^2) over the batch and outputs
    R = X @ W.T - Y
    return 2.0 * R.T @ X / (X.shape[0] * W.shape[0])


def _data(seed, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        W = rng.integers(-2, 3, (OUT, IN)).astype(np.float64)
        X = rng.integers(-2, 3, (B, IN)).astype(np.float64)
        Y = rng.integers(-2, 3, (B, OUT)).astype(np.float64)
    else:
        W = rng.standard_normal((OUT, IN))
        X = rng.standard_normal((B, IN))
        Y = rng.standard_normal((B, OUT))
    return W, X, Y


def _shards(X, Y):
    b = B // P
    return [(X[r * b:(r + 1) * b], Y[r * b:(r + 1) * b]) for r in range(P)]


def _bf16_bits(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_mean_of_shard_gradients_is_the_full_batch_gradient(ora):
    W, X, Y = _data(0)
    full = _grad(W, X, Y).ravel()
    per_rank = np.stack([_grad(W, xs, ys).ravel() for xs, ys in _shards(X, Y)])
    assert np.max(np.abs(per_rank.mean(0) - full)) < 1e-15
    # the oracle's literal ring all-reduce (fp32), then x 1/P
    n = full.size
    S = ora.shard_size(n, P)
    bufs = np.zeros((P, P * S), np.float32)
    bufs[:, :n] = per_rank
    ora.ring_reduce_scatter_sim(bufs, shift=1)
    ora.ring_all_gather_sim(bufs, shift=1)
    avg = bufs[:, :n] * np.float32(1.0 / P)
    assert np.max(np.abs(avg - full) / np.abs(full)) < 1e-6
    assert all(np.array_equal(avg[0], avg[r]) for r in range(P))


def test_exact_identity_with_representable_gradients(ora):
    # Integer data: every shard gradient is a small multiple of 1/8, exact in
    # bf16, and so are the fp32 sums; the reduce-scatter times 1/P must
    # reproduce the full-batch gradient exactly.
    W, X, Y = _data(3, integer=True)
    full = _grad(W, X, Y).ravel()
    per_rank = np.stack([_grad(W, xs, ys).ravel() for xs, ys in _shards(X, Y)])
    bits = _bf16_bits(per_rank)
    assert np.array_equal(ora.bf16_to_f32(bits).astype(np.float64), per_rank)
    shards, flag, _ = ora.reduce_scatter(bits, 0, full.size, 1.0 / P)
    assert flag == 0
    assert np.array_equal(shards[:full.size].astype(np.float64), full)


def test_zero_step_training_matches_large_batch(ora):
    # k steps of the ZeRO step over P ranks (per-rank bf16 gradients) against
    # k steps of the same optimizer on the full batch (P = 1).  Replicas stay
    # bit-identical; the weights agree up to the bf16 rounding of gradients,
    # which Adam's normalisation keeps at the order of lr per step.
    W, X, Y = _data(5)
    n = W.size
    lr = 1e-2
    hp = dict(lr=lr, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)

    def state():
        S = ora.shard_size(n, P)
        w = np.zeros(P * S, np.float32)
        w[:n] = W.ravel()
        return w, np.zeros(P * S, np.float32), np.zeros(P * S, np.float32)

    wz, mz, vz = state()
    repz = np.zeros((P, n), np.uint16)
    wb, mb, vb = wz[:n].copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    repb = np.zeros((1, n), np.uint16)
    for t in range(1, 11):
        Wz = ora.bf16_to_f32(repz[0]).reshape(OUT, IN).astype(np.float64) if t > 1 else W
        Wb = ora.bf16_to_f32(repb[0]).reshape(OUT, IN).astype(np.float64) if t > 1 else W
        gz = _bf16_bits(np.stack([_grad(Wz, xs, ys).ravel() for xs, ys in _shards(X, Y)]))
        gb = _bf16_bits(_grad(Wb, X, Y).ravel()[None, :])
        ora.step(gz, 0, wz, mz, vz, repz, n, 0, n, 1.0 / P, t=t, **hp)
        ora.step(gb, 0, wb, mb, vb, repb, n, 0, n, 1.0, t=t, **hp)
        for r in range(1, P):
            assert np.array_equal(repz[r], repz[0])
    moved = np.max(np.abs(wz[:n] - W.ravel()))
    assert moved > 5 * lr                          # training really moved the weights
    assert np.max(np.abs(wz[:n] - wb)) < 0.02 * moved
