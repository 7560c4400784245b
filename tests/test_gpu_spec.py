"""GPU parity of the speculative verification against the fp64 oracle.

The accepted run and the next token are integers decided by floating point: the kernel's fp32
softmax sums may settle a decision differently from fp64 only when the decision is a tie within
that rounding. So every accepted-run length and next token must equal the oracle's, except
where the oracle's own margin (|u * P_draft - P_target|, or the distance of the inverse-CDF
threshold to a bucket edge) is below 1e-5 of the quantities compared; those cases must still be
a valid choice.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_147_gb300 import pkv

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _softmax64(x):
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


@pytest.mark.parametrize("B,K,V,noise,masked", [(32, 4, 32000, 0.3, 0.0),
                                                 (64, 4, 151936, 0.1, 0.0),
                                                 (8, 1, 1000, 1.0, 0.0), (16, 0, 5000, 0.0, 0.0),
                                                 (16, 3, 40000, 0.3, 0.1), (4, 5, 9000, 0.5, 0.5)])
def test_spec_verify_matches_oracle(B, K, V, noise, masked):
    """masked: a fraction of the vocabulary is -inf in both models (banned tokens)."""
    rng = np.random.default_rng(B * 7 + K + V)
    t = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    d = (t[:, :K] + noise * rng.standard_normal((B, K, V))).astype(np.float32)
    if masked > 0:
        ban = rng.random(V) < masked
        t[:, :, ban] = -np.inf
        d[:, :, ban] = -np.inf
    pd = _softmax64(d)
    x = np.zeros((B, K), np.int32)
    for b in range(B):
        for k in range(K):
            x[b, k] = rng.choice(V, p=pd[b, k])
    ua = rng.random((B, K)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    n_g, nt_g = pkv.spec_verify(torch.from_numpy(t).to(DEV), torch.from_numpy(d).to(DEV),
                                torch.from_numpy(x).to(DEV), torch.from_numpy(ua).to(DEV),
                                torch.from_numpy(us).to(DEV))
    torch.cuda.synchronize()
    n_g, nt_g = n_g.cpu().numpy(), nt_g.cpu().numpy()
    n_o, nt_o = oracle.spec_verify(t, d, x, ua, us)
    pt = _softmax64(t)
    for b in range(B):
        k = min(n_o[b], n_g[b])
        if n_g[b] != n_o[b]:
            # only a tie within fp32 rounding may be decided the other way
            xb = x[b, k]
            margin = abs(float(ua[b, k]) * pd[b, k, xb] - pt[b, k, xb])
            assert margin <= 1e-5 * pt[b, k, xb], (b, k, margin)
            continue
        w = pt[b, K] if n_o[b] == K else np.maximum(0.0, pt[b, k] - pd[b, k])
        cdf = np.cumsum(w)
        thr = float(us[b]) * cdf[-1]
        if nt_g[b] != nt_o[b]:
            v = int(nt_g[b])
            lo = cdf[v - 1] if v > 0 else 0.0
            assert w[v] > 0 and lo - 1e-5 * cdf[-1] <= thr <= cdf[v] + 1e-5 * cdf[-1], (b, v)
    assert np.mean(nt_g == nt_o) > 0.95 and np.mean(n_g == n_o) > 0.95
    assert pkv.device_error(clear=True) == 0


def test_out_of_range_draft_is_rejected_and_flagged():
    """A draft token outside the vocabulary (a caller's bug) stops that sequence's accepted
    run there and sets the token bit, without a fault; the other sequences are unaffected."""
    rng = np.random.default_rng(5)
    B, K, V = 6, 3, 4000
    t = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    d = t[:, :K].copy()                       # identical models: every valid draft is accepted
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    x[2, 1] = V + 3
    x[4, 0] = -1
    ua = rng.random((B, K)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    n_g, nt_g = pkv.spec_verify(torch.from_numpy(t).to(DEV), torch.from_numpy(d).to(DEV),
                                torch.from_numpy(x).to(DEV), torch.from_numpy(ua).to(DEV),
                                torch.from_numpy(us).to(DEV))
    torch.cuda.synchronize()
    assert pkv.device_error(clear=True) & pkv.DEVERR_TOKEN
    n_g, nt_g = n_g.cpu().numpy(), nt_g.cpu().numpy()
    assert n_g[2] == 1 and n_g[4] == 0
    assert 0 <= nt_g[2] < V and 0 <= nt_g[4] < V
    good = [b for b in range(B) if b not in (2, 4)]
    n_o, nt_o = oracle.spec_verify(t[good], d[good], x[good], ua[good], us[good])
    assert np.array_equal(n_g[good], n_o)
    assert np.array_equal(nt_g[good], nt_o)
