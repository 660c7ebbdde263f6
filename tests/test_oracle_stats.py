"""Distributional pins of the oracle (no GPU needed).

"Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
section 1: accepting y_i ~ q_i with probability min(1, p_i(y_i)/q_i(y_i)),
drawing the correction from the normalised [p_i - q_i]_+ and the bonus from
the target preserves the target distribution.  So, over many independent
requests with identical rows:
  * the first committed token c_0 follows p_0,
  * c_1 given A >= 1 follows p_1, and the bonus c_2 given A = 2 follows p_2,
  * c_0 given A = 0 follows the normalised residual [p_0 - q_0]_+,
  * P(accept at i | prefix accepted) = sum_v min(p_i(v), q_i(v)) = 1 - TV(p_i, q_i).
The expected distributions are computed here with numpy, independently of the
oracle, and compared with chi-square and binomial z-tests.
"""
import math

import numpy as np
import pytest

import oracle

scipy_stats = pytest.importorskip("scipy.stats")


def _softmax(x, t):
    z = np.asarray(x, np.float64) / t
    z = np.exp(z - z.max())
    return z / z.sum()


def _chi2_pvalue(counts, probs):
    counts = np.asarray(counts, np.float64)
    n = counts.sum()
    exp = np.asarray(probs, np.float64) * n
    keep = exp > 0
    assert counts[~keep].sum() == 0, "mass on zero-probability tokens"
    # merge cells with tiny expectation into one
    small = keep & (exp < 5)
    c = list(counts[keep & ~small]) + ([counts[small].sum()] if small.any() else [])
    e = list(exp[keep & ~small]) + ([exp[small].sum()] if small.any() else [])
    c, e = np.array(c), np.array(e)
    stat = ((c - e) ** 2 / e).sum()
    return scipy_stats.chi2.sf(stat, len(c) - 1)


def _identical_requests(n, tgt_rows, drf_rows, temperature, seed):
    """n requests that share their rows; draft tokens drawn independently ~ q_i."""
    rng = np.random.default_rng(seed)
    k = len(drf_rows)
    V = tgt_rows.shape[1]
    target = np.tile(tgt_rows.astype(np.float32), (n, 1))
    draft = np.tile(drf_rows.astype(np.float32), (n, 1)) if k else np.zeros((0, V), np.float32)
    toks = np.empty((n, k), np.int32)
    for i in range(k):
        q = _softmax(drf_rows[i], temperature)
        toks[:, i] = rng.choice(V, size=n, p=q)
    return dict(target=target, draft=draft, tokens=toks.reshape(-1),
                num_draft=np.full(n, k, np.int32),
                temperature=np.full(n, temperature, np.float32), max_k=k)


@pytest.fixture(scope="module")
def million_trials():
    rng = np.random.default_rng(2024)
    V, k, T, n = 8, 2, 1.0, 1_000_000
    tgt = (rng.normal(size=(k + 1, V)) * 1.5).astype(np.float32)
    drf = (tgt[:k] + rng.normal(size=(k, V))).astype(np.float32)
    inp = _identical_requests(n, tgt, drf, T, seed=7)
    out = oracle.verify(seed=123, **inp)
    p = [_softmax(tgt[i], T) for i in range(k + 1)]
    q = [_softmax(drf[i], T) for i in range(k)]
    return out, p, q


def test_first_token_follows_target(million_trials):
    out, p, q = million_trials
    c0 = out["committed"][:, 0]
    assert _chi2_pvalue(np.bincount(c0, minlength=8), p[0]) > 1e-3


def test_second_token_given_acceptance_follows_target(million_trials):
    out, p, q = million_trials
    sel = out["accepted_len"] >= 1
    c1 = out["committed"][sel, 1]
    assert _chi2_pvalue(np.bincount(c1, minlength=8), p[1]) > 1e-3


def test_bonus_follows_last_target_row(million_trials):
    out, p, q = million_trials
    sel = out["accepted_len"] == 2
    assert sel.sum() > 10_000
    c2 = out["committed"][sel, 2]
    assert (out["race_kind"][sel] == oracle.RACE_BONUS).all()
    assert _chi2_pvalue(np.bincount(c2, minlength=8), p[2]) > 1e-3


def test_correction_follows_positive_residual(million_trials):
    out, p, q = million_trials
    sel = out["accepted_len"] == 0
    resid = np.maximum(p[0] - q[0], 0.0)
    resid /= resid.sum()
    c0 = out["committed"][sel, 0]
    assert _chi2_pvalue(np.bincount(c0, minlength=8), resid) > 1e-3


def test_acceptance_rate_is_one_minus_tv(million_trials):
    out, p, q = million_trials
    A = out["accepted_len"]
    n = len(A)
    a0 = np.minimum(p[0], q[0]).sum()
    z0 = ((A >= 1).mean() - a0) / math.sqrt(a0 * (1 - a0) / n)
    assert abs(z0) < 4.5
    n1 = (A >= 1).sum()
    a1 = np.minimum(p[1], q[1]).sum()
    z1 = ((A[A >= 1] == 2).mean() - a1) / math.sqrt(a1 * (1 - a1) / n1)
    assert abs(z1) < 4.5


@pytest.mark.parametrize("temperature", [0.5, 1.0, 1.7])
def test_plain_sampling_at_k0_follows_tempered_target(temperature):
    # k = 0: no drafts, the committed token is the bonus draw from softmax(x/T)
    rng = np.random.default_rng(int(temperature * 10))
    V, n = 40, 200_000
    tgt = (rng.normal(size=(1, V)) * 2).astype(np.float32)
    inp = _identical_requests(n, tgt, np.zeros((0, V), np.float32), temperature, seed=1)
    out = oracle.verify(seed=5, **inp)
    c = out["committed"][:, 0]
    assert _chi2_pvalue(np.bincount(c, minlength=V), _softmax(tgt[0], temperature)) > 1e-3


def test_acceptance_rate_at_larger_vocab():
    # the closed form on a 1000-token vocabulary with the drafter's own tokens
    rng = np.random.default_rng(17)
    V, T, n = 1000, 0.8, 40_000
    tgt = (rng.normal(size=(2, V)) * 3).astype(np.float32)
    drf = (tgt[:1] + rng.normal(size=(1, V))).astype(np.float32)
    inp = _identical_requests(n, tgt, drf, T, seed=3)
    out = oracle.verify(seed=9, **inp)
    a = np.minimum(_softmax(tgt[0], T), _softmax(drf[0], T)).sum()
    rate = (out["accepted_len"] == 1).mean()
    assert abs(rate - a) < 4.5 * math.sqrt(a * (1 - a) / n)
    # and the committed token still follows p_0
    p0 = _softmax(tgt[0], T)
    assert _chi2_pvalue(np.bincount(out["committed"][:, 0], minlength=V), p0) > 1e-3


def test_planted_mistakes_fail_the_pins():
    """A mutated acceptance rule (u p < q instead of u q < p) is caught."""
    rng = np.random.default_rng(5)
    V, n = 8, 200_000
    tgt = (rng.normal(size=(2, V)) * 1.5).astype(np.float32)
    drf = (tgt[:1] + rng.normal(size=(1, V))).astype(np.float32)
    inp = _identical_requests(n, tgt, drf, 1.0, seed=2)
    out = oracle.verify(seed=4, **inp)
    p0, q0 = _softmax(tgt[0], 1.0), _softmax(drf[0], 1.0)
    y = inp["tokens"]
    u = np.array([oracle.uniform_accept(oracle.random_word(4, 0, r, 0, 0)) for r in range(2000)])
    # the oracle's decisions agree with u q < p and disagree with the mutation
    dec = out["accepted_len"][:2000] == 1
    assert (dec == (u * q0[y[:2000]] < p0[y[:2000]])).all()
    assert not (dec == (u * p0[y[:2000]] < q0[y[:2000]])).all()


def test_race_draws_from_the_weights():
    """The exponential race draws token v with probability w_v / sum w over the
    positive weights: checked with zero weights scattered through the row."""
    rng = np.random.default_rng(31)
    V = 700
    w = rng.gamma(0.7, size=V)
    w[128:256] = 0.0                              # a run of zero weights
    w[rng.choice(V, 50, replace=False)] = 0.0     # scattered zero weights
    n = 40_000
    draws = np.array([oracle.race_weights(w, seed=3, request=r, position=2)[0] for r in range(n)])
    assert not np.isin(draws, np.flatnonzero(w == 0)).any()
    assert _chi2_pvalue(np.bincount(draws, minlength=V), w / w.sum()) > 1e-3


def test_race_equal_weights_follow_the_words():
    """Two ids of equal weight: E = -ln((word + 1/2) 2^-32) falls as the word
    grows, so the id whose stream-1 word is larger has the smaller key and wins.
    The words come from the Philox known-answer-pinned generator, keyed by the
    vocab id itself; both orders occur over the requests."""
    V, a, b = 40, 9, 22
    w = np.zeros(V)
    w[a] = w[b] = 0.37
    seen = set()
    for r in range(64):
        wa = oracle.random_word(11, 1, r, 3, a)
        wb = oracle.random_word(11, 1, r, 3, b)
        winner, _ = oracle.race_weights(w, seed=11, request=r, position=3)
        assert winner == (a if wa > wb else b), (r, wa, wb, winner)
        seen.add(winner)
    assert seen == {a, b}


def test_race_tie_goes_to_the_lowest_index():
    """Weights equal to the ids' own exponentials make every key exactly 1
    (x / x is exact in IEEE arithmetic): the lowest of the tied ids wins,
    whatever the words."""
    V = 30
    ids = [4, 17, 25]
    for r in range(8):
        w = np.zeros(V)
        for v in ids:
            w[v] = oracle.exponential(oracle.random_word(5, 1, r, 0, v))
        winner, keys = oracle.race_weights(w, seed=5, request=r, position=0)
        assert winner == ids[0]
        assert (keys[ids] == 1.0).all()
        # without the lowest, the next one takes it
        w[ids[0]] = 0.0
        assert oracle.race_weights(w, seed=5, request=r, position=0)[0] == ids[1]


def test_race_is_invariant_to_scale_and_keyed_by_vocab_id():
    """Normalisation does not change the winner (power-of-two scales are exact),
    and the key of id v depends only on v, not on the other weights: zeroing
    every other id but the winner and one rival leaves the winner in place."""
    rng = np.random.default_rng(8)
    w = rng.gamma(0.5, size=500)
    winner, keys = oracle.race_weights(w, seed=9, request=77, position=1)
    assert oracle.race_weights(w * 2.0 ** -40, seed=9, request=77, position=1)[0] == winner
    assert oracle.race_weights(w * 2.0 ** 30, seed=9, request=77, position=1)[0] == winner
    rival = int(np.argsort(keys)[1])
    w2 = np.zeros_like(w)
    w2[[winner, rival]] = w[[winner, rival]]
    win2, keys2 = oracle.race_weights(w2, seed=9, request=77, position=1)
    assert win2 == winner
    assert keys2[winner] == keys[winner] and keys2[rival] == keys[rival]
    assert np.isinf(keys2[np.flatnonzero(w2 == 0)]).all()
