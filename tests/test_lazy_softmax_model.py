"""The lazy running maximum of the decode and prefill kernels, as a host model (no GPU).

The kernels keep a row's running maximum m until a step's score exceeds it by more than 2^8
(log2 domain); only then is m raised and the row's sum l and output O rescaled. Softmax is
invariant to the reference m, so any m that bounds every score within 2^8 gives the same
result: the weights 2^(x - m) stay <= 256, exact to fp16's relative precision. This model runs
that update step by step (weights rounded to fp16 as the kernels' P operands are, l and O in
fp32), splits the keys into parts merged by their own (m, l, O) as the split-context merge
does, and compares with the exact fp64 softmax-weighted sum. It also counts the refreshes: on
random scores the first step takes almost all of them; on scores climbing in levels several
happen mid-sequence.
"""
import numpy as np
import pytest

LAZY = 8.0


def _exact(x, v):
    """softmax(x) . V in fp64 (x in the log2 domain)."""
    w = np.exp2(x - x.max())
    return (w[:, None] * v).sum(0) / w.sum()


def _lazy_part(x, v, step):
    """One part's (m, l, O) by the lazy update, `step` keys per update; returns the refresh
    count too. Asserts the weight bound at every step."""
    m, l = -np.inf, np.float32(0)
    o = np.zeros(v.shape[1], np.float32)
    refreshes = 0
    for s0 in range(0, len(x), step):
        xs = x[s0:s0 + step]
        if xs.max() > m + LAZY:                      # the warp-wide vote
            m_new = max(m, xs.max())
            alpha = np.float32(np.exp2(m - m_new)) if m != -np.inf else np.float32(0)
            l, o = l * alpha, o * alpha
            m = m_new
            refreshes += 1
        w = np.exp2(xs - m)
        assert w.max() <= 2.0 ** LAZY
        p = w.astype(np.float16)                     # P as the mma operand
        l = np.float32(l + p.astype(np.float32).sum())
        o = (o + (p.astype(np.float32)[:, None] * v[s0:s0 + step].astype(np.float32)).sum(0)).astype(np.float32)
    return m, l, o, refreshes


def _merge(parts):
    """Split-context merge of parts' (m, l, O): weights l_p 2^(m_p - M)."""
    M = max(p[0] for p in parts)
    num = sum(p[2].astype(np.float64) * np.exp2(p[0] - M) for p in parts)
    den = sum(np.float64(p[1]) * np.exp2(p[0] - M) for p in parts)
    return num / den


def _scores(rng, n, kind):
    if kind == "random":
        return rng.standard_normal(n) * 1.5
    level = np.array([0, 2, 1, 3], float)[(4 * np.arange(n)) // n] * 11.0
    x = level + rng.standard_normal(n)
    spikes = rng.choice(np.arange(n // 8, n), size=3, replace=False)
    x[spikes] = 4.5 * 11.0
    return x


@pytest.mark.parametrize("kind", ["random", "climbing"])
@pytest.mark.parametrize("n,step,parts", [(1000, 16, 1), (4096, 32, 3), (777, 16, 5), (64, 64, 1)])
def test_lazy_update_equals_the_exact_softmax(kind, n, step, parts):
    rng = np.random.default_rng(n + step + parts + (kind == "climbing"))
    x = _scores(rng, n, kind)
    v = rng.standard_normal((n, 16))
    cuts = np.linspace(0, n, parts + 1).astype(int)
    states = [_lazy_part(x[a:b], v[a:b], step) for a, b in zip(cuts[:-1], cuts[1:])]
    got = _merge(states)
    ref = _exact(x, v)
    # fp16 weights (relative 2^-11) and fp32 sums: far inside the kernels' 2e-3 parity bar
    assert np.abs(got - ref).max() <= 2e-3 * max(1.0, np.abs(ref).max())
    refreshes = sum(s[3] for s in states)
    if kind == "random":
        assert refreshes == parts                    # each part's first step only
    elif n >= 8 * step * parts:
        assert refreshes > parts                     # the climb refreshes mid-part


def test_a_stale_maximum_within_the_margin_changes_nothing_but_rounding():
    """The same keys with the reference maximum forced low by up to 2^8 give the same output as
    the true maximum (the invariance the lazy update rests on)."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal(500) * 3
    v = rng.standard_normal((500, 8))
    ref = _exact(x, v)
    for lag in (0.0, 3.0, 7.99):
        m = x.max() - lag
        w = np.exp2(x - m)
        assert w.max() <= 2.0 ** LAZY
        p = w.astype(np.float16).astype(np.float64)
        out = (p[:, None] * v).sum(0) / p.sum()
        assert np.abs(out - ref).max() < 1e-3
