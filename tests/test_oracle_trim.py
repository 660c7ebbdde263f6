"""Confidence-based window trimming in the oracle ("Speculative Decoding:
Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark", section 5, DSpark: survival
s_j = prod_{i<=j} c_i, estimated progress 1 + sum_{j<=k} s_j), pinned to
closed forms, to a second formulation of the rule, and to the full-window
verify on the common prefix."""
import numpy as np
import pytest

import oracle
from tests import cases


def leading_count(c, lam):
    """Second formulation: s_j never increases, so the progress minus cost is
    concave in k and the best window keeps the leading positions with s_j > lam."""
    s, k = 1.0, 0
    for ci in c:
        s *= float(ci)
        if s > lam:
            k += 1
        else:
            break
    return k


def test_closed_forms():
    w = np.array([4, 4, 4, 3, 0], np.int32)
    c = np.array([1, 1, 1, 1] + [0.5] * 4 + [0.9, 0.9, 0.0, 0.9] + [0.5] * 3, np.float32)
    k, st = oracle.trim(w, c, np.array([0.99, 0.2, 0.5, 1.0, 0.1], np.float32))
    # s = 1 > 0.99 always; s = 0.5, 0.25, 0.125 against 0.2; s = 0.9, 0.81, 0 against 0.5;
    # s <= 1 never beats a cost of 1; an empty window stays empty
    assert st == 0 and k.tolist() == [4, 2, 2, 0, 0]
    k, _ = oracle.trim(np.array([5], np.int32), np.full(5, 0.5, np.float32),
                       np.array([0.25], np.float32))
    assert k.tolist() == [1]          # s_2 = 0.25 == cost: a tie keeps the shorter window
    k, _ = oracle.trim(np.array([3], np.int32), np.ones(3, np.float32), np.array([-1.0], np.float32))
    assert k.tolist() == [3]          # negative cost: every position pays


@pytest.mark.parametrize("seed", range(5))
def test_second_formulation_and_monotone_in_cost(seed):
    rng = np.random.default_rng(seed)
    B = 200
    w = rng.integers(0, 12, size=B).astype(np.int32)
    c = rng.uniform(0, 1, size=int(w.sum())).astype(np.float32)
    c[rng.random(c.size) < 0.1] = 1.0
    lam = rng.uniform(-0.1, 1.1, size=B).astype(np.float32)
    k, st = oracle.trim(w, c, lam)
    assert st == 0
    off = np.concatenate([[0], np.cumsum(w)])
    for r in range(B):
        assert k[r] == leading_count(c[off[r]:off[r + 1]], float(lam[r]))
    k2, _ = oracle.trim(w, c, lam + np.float32(0.05))
    assert (k2 <= k).all() and (k <= w).all()


def test_bad_confidences():
    k, st = oracle.trim(np.array([2, 2, 2], np.int32),
                        np.array([0.5, np.nan, 0.5, 1.5, 0.5, 0.5], np.float32),
                        np.array([0.1, 0.1, np.nan], np.float32))
    assert st == oracle.BAD_CONF and k.tolist() == [-1, -1, -1]


def test_trimmed_verify_agrees_with_full_window():
    """Decisions on the common prefix are the full window's: a request the full
    window rejects before the trim point gets the same A and tokens; otherwise
    A = k* and the last token is the bonus from p_{k*}."""
    rng = np.random.default_rng(7)
    B = 60
    k = rng.integers(0, 7, size=B)
    temp = rng.choice([0.0, 0.7, 1.0], size=B)
    inp = cases.random_batch(k, temp, vocab=500, sigma_t=2.0, sigma_d=0.7, dtype="f32", seed=11)
    w = inp["num_draft"]
    conf = rng.uniform(0.3, 1.0, size=int(w.sum())).astype(np.float32)
    cost = rng.uniform(0.0, 0.8, size=B).astype(np.float32)
    full = oracle.verify(inp["target"], inp["draft"], inp["tokens"], w, inp["temperature"], 3, 6)
    tr = oracle.verify_trimmed(inp["target"], inp["draft"], inp["tokens"], w, conf, cost,
                               inp["temperature"], 3, 6)
    kt = tr["verified_k"]
    assert (kt <= w).all()
    d_off = np.concatenate([[0], np.cumsum(w)])
    for r in range(B):
        A, At = full["accepted_len"][r], tr["accepted_len"][r]
        if A < kt[r]:
            assert At == A and (tr["committed"][r] == full["committed"][r]).all()
        else:
            assert At == kt[r]
            assert (tr["committed"][r, :At] == full["committed"][r, :At]).all()
        f = tr["flags"][d_off[r]:d_off[r + 1]]
        assert f.sum() == At and (f[kt[r]:] == 0).all()
    # confidences of 1 and a cost below 1 keep every window: the full verify
    same = oracle.verify_trimmed(inp["target"], inp["draft"], inp["tokens"], w,
                                 np.ones(int(w.sum()), np.float32), np.full(B, 0.5, np.float32),
                                 inp["temperature"], 3, 6)
    assert (same["committed"] == full["committed"]).all()
    assert (same["flags"] == full["flags"]).all()
