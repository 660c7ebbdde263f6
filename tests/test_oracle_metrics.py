"""Acceptance statistics of the oracle, pinned to the tables of "Speculative
Decoding on AMD GPUs" (appendix: MAL, AR and per-position rates per proposal
length) and to closed forms."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "amd_acceptance_tables.txt")


def _rows():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v = line.split()
            n = int(v[0])
            out.append((n, float(v[1]), float(v[2]), [int(x) for x in v[3:3 + n]]))
    return out


def _rounds_with_rates(n, rates):
    """100 rounds of proposal length n whose per-position acceptance (the share
    of rounds that accepted position j) is rates[j] percent."""
    lens = []
    prev = 100
    for j, r in enumerate(rates):          # rounds that stop after j accepted drafts
        lens += [j] * (prev - r)
        prev = r
    lens += [n] * prev
    return np.array(lens, np.int32), np.full(len(lens), n, np.int32)


@pytest.mark.parametrize("row", _rows(), ids=lambda r: f"N{r[0]}_MAL{r[1]}")
def test_printed_tables(row):
    n, mal, ar, rates = row
    a, k = _rounds_with_rates(n, rates)
    s = oracle.summarize(*oracle.metrics(a, k, n))
    assert np.allclose(s["per_position"], np.array(rates) / 100.0, atol=1e-12)
    # printed MAL and AR agree with the counts up to the rounding of the printed rates
    assert abs(s["mal"] - mal) <= 0.011 + 1e-9, (s["mal"], mal)
    assert abs(100.0 * s["acceptance_rate"] - ar) <= 0.25 + 1e-9, (s["acceptance_rate"], ar)


def test_closed_forms():
    k = np.array([4, 4, 4], np.int32)
    s = oracle.summarize(*oracle.metrics(np.array([4, 4, 4], np.int32), k, 4))
    assert s["mal"] == 5.0 and s["acceptance_rate"] == 1.0
    s = oracle.summarize(*oracle.metrics(np.array([0, 0, 0], np.int32), k, 4))
    assert s["mal"] == 1.0 and s["acceptance_rate"] == 0.0
    h, p, a = oracle.metrics(np.array([-1, 2, -1], np.int32), np.array([3, 3, 3], np.int32), 3)
    assert h.tolist() == [0, 0, 1, 0, 2] and p.tolist() == [1, 1, 1] and a.tolist() == [1, 1, 0]


def test_against_numpy_and_accumulation():
    rng = np.random.default_rng(4)
    max_k = 7
    k = rng.integers(0, max_k + 1, size=500).astype(np.int32)
    a = np.minimum(rng.integers(-1, max_k + 1, size=500), k).astype(np.int32)
    h, p, acc = oracle.metrics(a[:200], k[:200], max_k)
    h, p, acc = oracle.metrics(a[200:], k[200:], max_k, h, p, acc)   # running counts
    ok = a >= 0
    assert h[-1] == (~ok).sum()
    assert (h[:-1] == np.bincount(a[ok], minlength=max_k + 1)).all()
    for j in range(max_k):
        assert p[j] == (k[ok] > j).sum() and acc[j] == (a[ok] > j).sum()
    s = oracle.summarize(h, p, acc)
    assert np.isclose(s["mal"], 1 + a[ok].mean())
    # MAL = 1 + sum of per-position rates when every round proposes the same length
    kk = np.full(300, 5, np.int32)
    aa = rng.integers(0, 6, size=300).astype(np.int32)
    s = oracle.summarize(*oracle.metrics(aa, kk, 5))
    assert np.isclose(s["mal"], 1 + s["per_position"].sum())
    assert np.isclose(s["acceptance_rate"], s["per_position"].mean())
