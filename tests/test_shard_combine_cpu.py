"""The vocabulary-shard contract of include/flce.h, checked on the CPU in
float64: per-shard (m, s, zt) as the shard forward defines them, combined by
max, rescaled sum and sum, give the whole vocabulary's lse and loss; per-shard
gradient parts formed from the combined lse sum (dH) and concatenate (dW) to
the whole vocabulary's gradients. The GPU shard tests rely on this algebra."""
import numpy as np
import pytest

import oracle


def _shard_forward(H, W_s, v0, y, ignore=-100):
    Z = oracle.logits_rows(H, W_s)
    m = Z.max(axis=1)
    s = np.exp(Z - m[:, None]).sum(axis=1)
    inside = (y != ignore) & (y >= v0) & (y < v0 + W_s.shape[0])
    zt = np.where(inside, Z[np.arange(len(y)), np.clip(y - v0, 0, W_s.shape[0] - 1)], 0.0)
    return m, s, zt


def _shard_backward(H, W_s, v0, y, lse, scale, ignore=-100):
    Z = oracle.logits_rows(H, W_s)
    G = np.exp(Z - lse[:, None])
    rows = np.flatnonzero((y != ignore) & (y >= v0) & (y < v0 + W_s.shape[0]))
    G[rows, y[rows] - v0] -= 1.0
    G *= np.where(y != ignore, scale, 0.0)[:, None]
    return G @ W_s, G.T @ H


@pytest.mark.parametrize("bounds", [[0, 40, 97, 150], [0, 1, 150], [0, 149, 150]])
def test_shards_combine_to_the_whole_vocabulary(bounds):
    g = np.random.default_rng(5)
    N, D, V = 37, 24, 150
    H = g.standard_normal((N, D))
    W = g.standard_normal((V, D)) * 0.3
    y = g.integers(0, V, N)
    y[[3, 11]] = -100
    ref = oracle.flce(H, W, y)
    parts = [_shard_forward(H, W[a:b], a, y) for a, b in zip(bounds[:-1], bounds[1:])]
    m = np.stack([p[0] for p in parts])
    s = np.stack([p[1] for p in parts])
    zt = np.stack([p[2] for p in parts]).sum(axis=0)
    M = m.max(axis=0)
    lse = M + np.log((s * np.exp(m - M)).sum(axis=0))
    np.testing.assert_allclose(lse, ref["lse"], rtol=0, atol=1e-12)
    valid = y != -100
    loss = (lse - zt)[valid].sum() / valid.sum()
    assert abs(loss - ref["loss"]) <= 1e-12 * abs(ref["loss"])
    dH = np.zeros_like(H)
    dWs = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        dh, dw = _shard_backward(H, W[a:b], a, y, lse, 1.0 / valid.sum())
        dH += dh
        dWs.append(dw)
    np.testing.assert_allclose(dH, ref["dH"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(dWs), ref["dW"], rtol=0, atol=1e-12)
