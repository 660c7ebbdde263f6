"""Top-k / top-p truncation in the oracle ("Speculative Decoding: Medusa, MTP,
EAGLE, DFlash, DDTree, and DSpark", section 1: temperature and truncation must
enter the target and draft distributions consistently), pinned to a counting
formulation of top-k, the nucleus property of top-p, the closed form of the
renormalised distribution, and the greedy chain (top-1 truncation turns
sampling into greedy decoding)."""
import numpy as np
import pytest

import oracle
from tests import cases


def as_f32(a):
    return a if a.dtype == np.float32 else (a.astype(np.uint32) << 16).view(np.float32)


def one_row(x, t, k, p):
    out, _, m, _, st = oracle.truncate(x[None, :], None, [0], [t], [k], [p])
    return as_f32(out)[0], m[0], st


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_top_k_counts(dtype):
    rng = np.random.default_rng(1)
    for trial in range(40):
        V = int(rng.integers(2, 300))
        x = np.round(rng.normal(size=V) * 2, 1).astype(np.float32)   # repeated values
        if dtype == "bf16":
            x = (x.view(np.uint32) >> 16).astype(np.uint16)
        xf = as_f32(x)
        K = int(rng.integers(1, V + 2))
        out, _, st = one_row(x, 1.0, K, 1.0)
        assert st == 0
        keep = np.isfinite(out)
        for v in range(V):
            # kept iff fewer than K logits are strictly larger
            assert keep[v] == ((xf > xf[v]).sum() < K)
        assert (out[keep] == xf[keep]).all()


@pytest.mark.parametrize("T", [0.5, 1.0, 1.7])
def test_top_p_nucleus_property(T):
    rng = np.random.default_rng(2)
    for trial in range(60):
        V = int(rng.integers(2, 400))
        x = np.round(rng.normal(size=V) * 3, 1).astype(np.float32)
        K = int(rng.integers(0, V + 1))
        P = float(rng.uniform(0.05, 0.999))
        out, margin, st = one_row(x, T, K, P)
        assert st == 0
        keep = np.isfinite(out)
        # the top-k survivors (K = 0 or >= V: all)
        surv = np.ones(V, bool) if K <= 0 or K >= V else np.array(
            [(x > x[v]).sum() < K for v in range(V)])
        assert (keep <= surv).all()
        w = np.where(surv, np.exp((x.astype(np.float64) - x.max()) / T), 0.0)
        w /= w.sum()
        lowest = x[keep].min()
        if margin > 1e-9:
            # the kept set reaches P, and without its lowest logit value it would not
            assert w[keep].sum() >= P - 1e-12
            assert w[keep & (x > lowest)].sum() < P + 1e-12
        # kept = all survivors with a logit >= the lowest kept one
        assert (keep == (surv & (x >= lowest))).all()
        # softmax of the output row: the truncated, renormalised distribution
        z = np.exp((np.where(keep, x, -np.inf).astype(np.float64) - x.max()) / T)
        assert np.allclose(z / z.sum(), np.where(keep, w, 0) / w[keep].sum(), atol=1e-12)


def test_identity_and_invalid():
    x = np.array([0.5, 2.0, -1.0, 2.0], np.float32)
    for t, k, p in ((1.0, 0, 1.0), (1.0, 4, 1.0), (0.0, 1, 0.1), (1.0, 9, 1.5)):
        out, _, st = one_row(x, t, k, p)
        assert st == 0 and (out == x).all()
    out, _, st = one_row(x, 1.0, 2, float("nan"))
    assert st == oracle.BAD_TRUNC and (out == x).all()
    out, _, st = one_row(x, 1.0, 2, 0.0)
    assert st == oracle.BAD_TRUNC
    nanrow = x.copy()
    nanrow[2] = np.nan
    out, _, st = one_row(nanrow, 1.0, 1, 0.5)
    assert st == 0 and np.isnan(out[2]) and (out[[0, 1, 3]] == nanrow[[0, 1, 3]]).all()


def test_top_1_sampling_is_greedy():
    """Truncating both rows to their top-1 makes p' and q' point masses: the
    verify at T = 1 on the truncated rows commits exactly the greedy chain."""
    rng = np.random.default_rng(5)
    B = 50
    k = rng.integers(0, 6, size=B)
    inp = cases.random_batch(k, np.ones(B), vocab=300, sigma_t=2.0, sigma_d=1.0, dtype="f32",
                             seed=3)
    nd = inp["num_draft"]
    # draft tokens = the draft argmax (what sampling from q' gives)
    toks = np.array([int(np.argmax(r)) for r in inp["draft"]], np.int32)
    t_out, d_out, _, _, st = oracle.truncate(inp["target"], inp["draft"], nd, inp["temperature"],
                                             np.ones(B, np.int32), np.ones(B, np.float32))
    assert st == 0
    samp = oracle.verify(t_out, d_out, toks, nd, np.ones(B, np.float32), 9, 5)
    greedy = oracle.verify(inp["target"], None, toks, nd, np.zeros(B, np.float32), 9, 5)
    assert (samp["accepted_len"] == greedy["accepted_len"]).all()
    assert (samp["committed"] == greedy["committed"]).all()
