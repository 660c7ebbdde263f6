"""Pins of the CPU oracle to facts fixed outside it (no GPU needed).

Each test checks the oracle against something other than itself: published
known-answer vectors, the worked examples printed on the pages, closed forms,
library routines (numpy argmax) or invariants of the rule.
"""
import math

import numpy as np
import pytest

import oracle
from tests import cases


# --- Philox4x32-10 against the SC'11 / Random123 known-answer vectors ---------

def test_philox_known_answer_vectors():
    kat = cases.read_kat()
    assert len(kat) == 3
    for ctr, key, want in kat:
        got = oracle.philox4x32_10(ctr, key)
        assert [int(x) for x in got] == want


def test_random_word_counter_layout():
    # the stated keying: key = (seed lo, seed hi); counter = (v/4, position,
    # request lo, stream | request hi << 8); word v mod 4
    seed, stream, req, pos = 0x0123456789ABCDEF, 1, (5 << 32) | 77, 3
    for v in (0, 1, 2, 3, 4, 7, 1021):
        ctr = [v // 4, pos, req & 0xFFFFFFFF, stream | ((req >> 32) << 8)]
        key = [seed & 0xFFFFFFFF, seed >> 32]
        assert oracle.random_word(seed, stream, req, pos, v) == int(oracle.philox4x32_10(ctr, key)[v % 4])


def test_uniform_and_exponential_closed_forms():
    assert oracle.uniform_accept(0) == 0.0
    assert oracle.uniform_accept(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform_accept(0x80000000) == 0.5
    assert oracle.uniform_accept(0x000000FF) == 0.0          # low 8 bits dropped
    assert oracle.exponential(0) == pytest.approx(33 * math.log(2), rel=1e-15)
    assert oracle.exponential(0xFFFFFFFF) == pytest.approx(2.0 ** -33, rel=1e-9)
    assert oracle.exponential(0x7FFFFFFF) == pytest.approx(math.log(2), rel=1e-9)


def test_exponential_draws_have_unit_mean():
    words = [oracle.random_word(7, 1, r, 0, v) for r in range(40) for v in range(500)]
    e = np.array([oracle.exponential(w) for w in words])
    # Exp(1): mean 1, variance 1; 20000 draws
    assert abs(e.mean() - 1.0) < 4.5 / math.sqrt(len(e))
    assert abs((e > 1.0).mean() - math.exp(-1)) < 4.5 * math.sqrt(0.25 / len(e))


# --- softmax and argmax closed forms -------------------------------------------

def test_softmax_hand_computed_row():
    x = np.log(np.array([1, 2, 3, 4], dtype=np.float64)).astype(np.float32)
    p = oracle.softmax(x, 1.0)
    want = np.array([1, 2, 3, 4]) / 10.0
    assert np.allclose(p, want, rtol=1e-6)          # fp32 rounding of the logs
    assert abs(p.sum() - 1.0) < 1e-12


def test_softmax_temperature_and_infinities():
    x = np.array([0.0, 2 * math.log(2), -np.inf], dtype=np.float32)
    p = oracle.softmax(x, 2.0)                    # exp(x/2) = [1, 2, 0]
    assert np.allclose(p, [1 / 3, 2 / 3, 0.0], rtol=1e-6)
    assert p[2] == 0.0
    big = np.array([1000.0, 1000.0, 999.0], dtype=np.float32)
    p = oracle.softmax(big, 1.0)
    e = math.exp(-1.0)
    assert np.allclose(p, [1 / (2 + e), 1 / (2 + e), e / (2 + e)], rtol=1e-12)


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(3)
    for t in (0.3, 0.7, 1.0, 2.5):
        p = oracle.softmax((rng.normal(size=4096) * 3).astype(np.float32), t)
        assert abs(p.sum() - 1.0) < 1e-12 and (p >= 0).all()


def test_argmax_first_index_and_signed_zero():
    assert oracle.argmax(np.array([1, 5, 5, 2], np.float32)) == 1
    assert oracle.argmax(np.array([-1, -0.0, 0.0, -2], np.float32)) == 1
    bits = cases.to_bf16_bits(np.array([-3, 7, 7, -np.inf], np.float32))
    assert oracle.argmax(bits) == 1


# --- worked examples printed on the pages ----------------------------------------

@pytest.mark.parametrize("case", cases.read_worked_examples(), ids=lambda c: c["case"])
@pytest.mark.parametrize("temperature", [1.0, 0.7, 0.0])
def test_worked_examples(case, temperature):
    inp, expect = cases.worked_case_batch(case, vocab=16, copies=64, temperature=temperature)
    for seed in range(8):
        out = oracle.verify(seed=seed, **inp)
        assert out["status"] == 0
        assert (out["accepted_len"] == case["expect_accepted"]).all()
        A = case["expect_accepted"]
        k = inp["max_k"]
        for r in range(64):
            row = out["committed"][r]
            assert list(row[:A + 1]) == expect
            assert (row[A + 1:] == -1).all()        # later drafts (D / outside) are never kept
        flags = out["flags"].reshape(64, k)
        assert (flags[:, :A] == 1).all() and (flags[:, A:] == 0).all()


# --- greedy equivalence against numpy's argmax chain ------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_chain_matches_numpy_argmax(dtype):
    rng = np.random.default_rng(11)
    B, V = 40, 257
    k = rng.integers(0, 7, size=B).astype(np.int32)
    # integer-valued logits make ties frequent; the rule keeps the first index
    nt, nd = int((k + 1).sum()), int(k.sum())
    tgt = rng.integers(-3, 4, size=(nt, V)).astype(np.float32)
    t_off = np.concatenate([[0], np.cumsum(k + 1)])
    # draft tokens: copy the target argmax for a random prefix, then disagree
    tokens = np.zeros(nd, np.int32)
    d = 0
    for r in range(B):
        agree = rng.integers(0, k[r] + 1)
        for i in range(k[r]):
            a = int(np.argmax(tgt[t_off[r] + i]))
            tokens[d] = a if i < agree else (a + 1 + rng.integers(0, V - 1)) % V
            d += 1
    tgt_in = cases.to_bf16_bits(tgt) if dtype == "bf16" else tgt
    drf = np.zeros((nd, V), np.float32)
    drf_in = cases.to_bf16_bits(drf) if dtype == "bf16" else drf
    out = oracle.verify(tgt_in, drf_in, tokens, k, np.zeros(B, np.float32), seed=5, max_k=6)
    assert out["status"] == 0
    d = 0
    for r in range(B):
        A = 0
        while A < k[r] and tokens[d + A] == np.argmax(tgt[t_off[r] + A]):
            A += 1
        assert out["accepted_len"][r] == A
        assert out["committed"][r][A] == np.argmax(tgt[t_off[r] + A])
        assert list(out["committed"][r][:A]) == list(tokens[d:d + A])
        d += k[r]


# --- acceptance rule boundary: accept iff u < p(y)/q(y) ---------------------------

@pytest.mark.parametrize("ratio_logits", [(0.0, 0.0, 0.5), (np.log(1 / 3), 0.0, None)])
def test_acceptance_threshold_direction(ratio_logits):
    # V=2. Target logits [a, 0] and draft logits [0, -inf]: q(0) = 1 and
    # p(0) = e^a / (e^a + 1).  The rule accepts y=0 iff u < p(0)/q(0) = p(0).
    a = np.float32(ratio_logits[0])
    B = 3000
    tgt = np.tile(np.array([[a, 0.0], [0.0, 0.0]], np.float32), (B, 1))
    drf = np.tile(np.array([[0.0, -np.inf]], np.float32), (B, 1))
    out = oracle.verify(tgt, drf, np.zeros(B, np.int32), np.ones(B, np.int32),
                        np.ones(B, np.float32), seed=99, max_k=1)
    p0 = math.exp(float(a)) / (math.exp(float(a)) + 1.0)
    u = np.array([oracle.uniform_accept(oracle.random_word(99, 0, r, 0, 0)) for r in range(B)])
    assert ((u < p0) == (out["accepted_len"] == 1)).all()
    assert 0.1 < (u < p0).mean() < 0.9


def test_zero_probabilities():
    # q(y) = 0 < p(y): always accepted; p(y) = 0: always rejected
    B = 500
    tgt = np.tile(np.array([[0.0, 0.0, 0.0], [0.0, 0.0, 0.0]], np.float32), (B, 1))
    drf = np.tile(np.array([[-np.inf, 0.0, 0.0]], np.float32), (B, 1))
    out = oracle.verify(tgt, drf, np.zeros(B, np.int32), np.ones(B, np.int32),
                        np.ones(B, np.float32), seed=3, max_k=1)
    assert (out["accepted_len"] == 1).all()
    tgt2 = np.tile(np.array([[-np.inf, 0.0, 0.0], [0.0, 0.0, 0.0]], np.float32), (B, 1))
    drf2 = np.tile(np.array([[0.0, 0.0, 0.0]], np.float32), (B, 1))
    out = oracle.verify(tgt2, drf2, np.zeros(B, np.int32), np.ones(B, np.int32),
                        np.ones(B, np.float32), seed=3, max_k=1)
    assert (out["accepted_len"] == 0).all()
    # the residual [p - q]_+ is positive on ids 1 and 2 only
    assert set(out["committed"][:, 0]) == {1, 2}


def test_identical_rows_accept_everything():
    # q == p: u q(y) < p(y) for every u < 1, so A = k for every request
    inp = cases.random_batch([3] * 50, [0.8] * 50, vocab=64, seed=4)
    t_off = np.concatenate([[0], np.cumsum(inp["num_draft"] + 1)])
    src = np.concatenate([np.arange(t_off[r], t_off[r] + 3) for r in range(50)])
    inp["draft"] = inp["target"][src].copy()
    out = oracle.verify(seed=1, **inp)
    assert (out["accepted_len"] == 3).all()
    assert (out["race_kind"] == oracle.RACE_BONUS).all()


def test_disjoint_supports_reject_at_once():
    # p and q have disjoint supports: p(y) = 0 for every y ~ q, so A = 0 and the
    # residual is p itself
    V, B = 8, 200
    tgt = np.full((2 * B, V), -np.inf, np.float32)
    tgt[:, :4] = 0.0
    drf = np.full((B, V), -np.inf, np.float32)
    drf[:, 4:] = 0.0
    tokens = (4 + np.arange(B) % 4).astype(np.int32)
    out = oracle.verify(tgt, drf, tokens, np.ones(B, np.int32), np.ones(B, np.float32),
                        seed=8, max_k=1)
    assert (out["accepted_len"] == 0).all()
    assert (out["committed"][:, 0] < 4).all()
    assert (out["race_kind"] == oracle.RACE_RESIDUAL).all()


# --- ragged layout: a batch equals its requests verified one by one ---------------

def test_ragged_batch_equals_single_requests():
    k = [0, 4, 1, 6, 2, 0, 3]
    temp = [1.0, 0.0, 0.7, 1.3, 0.0, 0.9, 1.0]
    inp = cases.random_batch(k, temp, vocab=300, dtype="bf16", seed=21)
    full = oracle.verify(seed=77, **inp)
    t_off = np.concatenate([[0], np.cumsum(np.array(k) + 1)])
    d_off = np.concatenate([[0], np.cumsum(k)])
    for r in range(len(k)):
        one = oracle.verify(inp["target"][t_off[r]:t_off[r + 1]],
                            inp["draft"][d_off[r]:d_off[r + 1]],
                            inp["tokens"][d_off[r]:d_off[r + 1]],
                            np.array([k[r]], np.int32), np.array([temp[r]], np.float32),
                            seed=77, max_k=inp["max_k"], request_ids=np.array([r]))
        assert one["accepted_len"][0] == full["accepted_len"][r]
        assert (one["committed"][0] == full["committed"][r]).all()
        assert (one["flags"] == full["flags"][d_off[r]:d_off[r + 1]]).all()


def test_flags_are_the_accepted_prefix():
    inp = cases.random_batch([5] * 64, [1.0] * 64, vocab=50, sigma_d=1.5, seed=9)
    out = oracle.verify(seed=2, **inp)
    flags = out["flags"].reshape(64, 5)
    for r in range(64):
        A = out["accepted_len"][r]
        assert (flags[r, :A] == 1).all() and (flags[r, A:] == 0).all()
        assert out["committed"][r][A] >= 0 and (out["committed"][r][A + 1:] == -1).all()
    # the debug values cover exactly the decided positions 0..A
    py = out["p_y"].reshape(64, 5)
    for r in range(64):
        A = out["accepted_len"][r]
        assert np.isfinite(py[r, :min(A + 1, 5)]).all() and np.isnan(py[r, A + 1:]).all()


# --- invalid inputs -----------------------------------------------------------------

def test_invalid_inputs_are_skipped_with_status():
    inp = cases.random_batch([2, 2, 2, 2], [1.0, 1.0, 1.0, 1.0], vocab=32, seed=5)
    bad = dict(inp)
    bad["tokens"] = inp["tokens"].copy()
    bad["tokens"][2] = 32                       # request 1: token out of range
    bad["temperature"] = inp["temperature"].copy()
    bad["temperature"][2] = -1.0                # request 2: negative temperature
    bad["target"] = inp["target"].copy()
    bad["target"][3 * 3 + 0, 5] = np.nan        # request 3: NaN in its first target row
    out = oracle.verify(seed=1, **bad)
    assert out["status"] == oracle.BAD_TOKEN | oracle.BAD_TEMP | oracle.NONFINITE
    assert out["accepted_len"][0] >= 0
    assert (out["accepted_len"][1:] == -1).all()
    assert (out["committed"][1:] == -1).all()
    assert list(out["req_status"]) == [0, oracle.BAD_TOKEN, oracle.BAD_TEMP, oracle.NONFINITE]

    wrong_k = dict(inp)
    wrong_k["num_draft"] = np.array([2, 2, 2, 3], np.int32)
    out = oracle.verify(seed=1, **wrong_k)     # max_k is 2
    assert out["status"] & oracle.BAD_K and (out["accepted_len"] == -1).all()
    out = oracle.verify(seed=1, total_draft=7, **inp)
    assert out["status"] == oracle.BAD_TOTAL and (out["accepted_len"] == -1).all()


def test_rows_after_the_first_rejection_are_never_read():
    """A round reads positions 0..A only: bad rows beyond A do not matter, bad rows
    the left-to-right procedure reaches do."""
    inp = cases.random_batch([4] * 40, [1.0] * 40, vocab=64, sigma_d=2.0, seed=12)
    base = oracle.verify(seed=3, **inp)
    A = base["accepted_len"]
    t_off = np.concatenate([[0], np.cumsum(inp["num_draft"] + 1)])
    d_off = np.concatenate([[0], np.cumsum(inp["num_draft"])])
    early = [r for r in range(40) if A[r] < 3]
    assert early
    late = dict(inp)
    late["target"], late["draft"] = inp["target"].copy(), inp["draft"].copy()
    for r in early:
        late["target"][t_off[r] + A[r] + 1:t_off[r + 1], 0] = np.nan   # beyond A
        late["draft"][d_off[r] + A[r] + 1:d_off[r + 1], 0] = np.inf
    out = oracle.verify(seed=3, **late)
    assert out["status"] == 0
    assert (out["committed"] == base["committed"]).all()
    reached = dict(inp)
    reached["target"] = inp["target"].copy()
    r = early[0]
    reached["target"][t_off[r] + A[r], 3] = np.nan                     # the rejected position
    out = oracle.verify(seed=3, **reached)
    assert out["status"] == oracle.NONFINITE and out["accepted_len"][r] == -1


def test_greedy_request_ignores_draft_rows_and_accepts_null_draft():
    inp = cases.random_batch([3, 2], [0.0, 0.0], vocab=40, seed=6)
    a = oracle.verify(seed=1, **inp)
    inp2 = dict(inp)
    inp2["draft"] = None
    b = oracle.verify(seed=1, **inp2)
    assert b["status"] == 0
    assert (a["committed"] == b["committed"]).all()
    inp3 = dict(inp)
    inp3["draft"] = np.full_like(inp["draft"], np.nan)
    c = oracle.verify(seed=1, **inp3)
    assert c["status"] == 0 and (c["committed"] == a["committed"]).all()
