"""Truncated verify rounds (specverify_run_truncated): thresholds per row and a
mask applied as the waves load the rows, with no truncated copy.

Two chains of checks:
- against the two-step GPU path (specverify_truncate writes the truncated rows,
  specverify_run verifies them): both take the same thresholds, and a logit
  masked on load reads the -inf the copy holds, so every output is identical;
- against the oracle (truncate, then verify, both in fp64): for the requests
  none of whose rows has a top-p decision within 1e-5 of its threshold, the GPU
  thresholds are the oracle's, so the masked rows are the oracle's truncated
  rows and the round is checked by the parity rules on them.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_10_gb300 import Verifier, _lib, build
from tests import parity
from tests.test_gpu_trunc import MARGIN, batch, gpu_truncate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _dev(a, dt):
    return torch.as_tensor(np.ascontiguousarray(a, dt)).cuda()


def run_truncated(v, inp, top_k, top_p, seed):
    t = parity.to_torch(inp, "cuda")
    res = v.run_truncated(t["target"], t["draft"], t["tokens"], t["num_draft"],
                          t["temperature"], _dev(top_k, np.int32), _dev(top_p, np.float32), seed)
    torch.cuda.synchronize()
    return {"accepted_len": res.accepted_len.cpu().numpy(),
            "committed": res.committed.cpu().numpy(), "flags": res.flags.cpu().numpy(),
            "status": v.status()}


def sample_tokens(inp, od, rng):
    """Draft tokens drawn from the (oracle-)truncated draft rows, as a drafter
    sampling from its truncated distribution would."""
    V = inp["target"].shape[1]
    bf16 = od.dtype == np.uint16
    df = ((od.astype(np.uint32) << 16).view(np.float32) if bf16 else od).astype(np.float64)
    d_off = np.concatenate([[0], np.cumsum(inp["num_draft"])])
    toks = []
    for r in range(len(inp["num_draft"])):
        T = inp["temperature"][r]
        for i in range(inp["num_draft"][r]):
            row = df[d_off[r] + i]
            if T == 0 or not np.isfinite(row).any():
                toks.append(int(np.nanargmax(np.where(np.isnan(row), -np.inf, row))))
            else:
                w = np.exp((row - np.max(row[np.isfinite(row)])) / T)
                w = np.where(np.isfinite(w), w, 0.0)
                toks.append(int(rng.choice(V, p=w / w.sum())))
    return np.array(toks, np.int32)


def two_step(v, inp, top_k, top_p, seed):
    gt, gd, st = gpu_truncate(inp, top_k, top_p)
    g = parity.run_gpu(v, dict(inp, target=gt, draft=gd), seed, debug=False)
    g["status"] |= st
    return g


@pytest.mark.parametrize("dtype,vocab,B", [("bf16", 4096, 40), ("f32", 3000, 40),
                                           ("bf16", 1001, 24), ("f32", 777, 24),
                                           ("bf16", 262144, 12)])
def test_truncated_round_equals_truncate_then_run(dtype, vocab, B):
    """Bit-identical to truncating into a copy and verifying the copy; draft
    tokens drawn at random over the whole vocabulary, so some lie outside the
    truncated draft support (q(y) = 0)."""
    inp, top_k, top_p = batch(B, vocab, dtype, vocab + 7)
    rng = np.random.default_rng(vocab)
    inp["tokens"] = rng.integers(0, vocab, size=len(inp["tokens"])).astype(np.int32)
    with Verifier(B, inp["max_k"], vocab, dtype) as v:
        for seed in (1, 2):
            f = run_truncated(v, inp, top_k, top_p, seed)
            g = two_step(v, inp, top_k, top_p, seed)
            for key in ("accepted_len", "committed", "flags", "status"):
                assert np.array_equal(np.asarray(f[key]), np.asarray(g[key])), (key, seed)


@pytest.mark.parametrize("dtype,vocab,B", [("bf16", 4096, 48), ("f32", 2000, 32),
                                           ("bf16", 262144, 16)])
def test_truncated_round_matches_oracle(dtype, vocab, B):
    inp, top_k, top_p = batch(B, vocab, dtype, 2 * vocab + 1)
    ot, od, mt, md, _ = oracle.truncate(inp["target"], inp["draft"], inp["num_draft"],
                                        inp["temperature"], top_k, top_p)
    inp["tokens"] = sample_tokens(inp, od, np.random.default_rng(5))
    k = inp["num_draft"]
    d_off = np.concatenate([[0], np.cumsum(k)])
    t_off = np.concatenate([[0], np.cumsum(k + 1)])
    clean = np.array([not ((mt[t_off[r]:t_off[r + 1]] <= MARGIN).any()
                           or (md[d_off[r]:d_off[r + 1]] <= MARGIN).any()) for r in range(B)])
    assert clean.sum() >= B // 2
    same = dict(inp, target=ot, draft=od)
    with Verifier(B, inp["max_k"], vocab, dtype) as v:
        for seed in (3, 4):
            f = run_truncated(v, inp, top_k, top_p, seed)
            plain = parity.run_gpu(v, same, seed)
            o = parity.run_oracle(same, seed)
            rep = parity.compare(plain, o, same, seed)        # the round on the oracle's rows
            assert rep["exempt_accept"] + rep["exempt_race"] <= max(1, B // 20), rep
            for r in np.flatnonzero(clean):                   # the masked rows are those rows
                assert f["accepted_len"][r] == plain["accepted_len"][r], (r, seed)
                assert (f["committed"][r] == plain["committed"][r]).all(), (r, seed)
                assert (f["flags"][d_off[r]:d_off[r + 1]]
                        == plain["flags"][d_off[r]:d_off[r + 1]]).all(), (r, seed)


def test_truncated_round_bad_top_p_and_nan_rows():
    """A top_p NaN or <= 0 keeps its request's rows whole and sets BAD_TRUNC;
    a row with a NaN is kept whole by the threshold pass and then skips its
    request as in an untruncated round; the others verify as usual."""
    B, V = 16, 1024
    inp, top_k, _ = batch(B, V, "f32", 21)
    top_p = np.full(B, 0.8, np.float32)
    top_p[3] = np.nan
    top_p[6] = 0.0
    inp["target"][0, 5] = np.nan
    with Verifier(B, inp["max_k"], V, "f32") as v:
        f = run_truncated(v, inp, top_k, top_p, 9)
        g = two_step(v, inp, top_k, top_p, 9)
    assert f["status"] & _lib.STATUS_BAD_TRUNC
    assert f["status"] == g["status"]
    for key in ("accepted_len", "committed", "flags"):
        assert np.array_equal(f[key], g[key]), key


def test_truncated_round_all_greedy_and_no_truncation():
    """Greedy requests are never truncated, and top_k = 0 with top_p = 1 is the
    plain round: both give specverify_run's outputs."""
    B, V = 24, 2048
    inp, _, _ = batch(B, V, "bf16", 31)
    top_k = np.zeros(B, np.int32)
    top_p = np.ones(B, np.float32)
    with Verifier(B, inp["max_k"], V, "bf16") as v:
        f = run_truncated(v, inp, top_k, top_p, 4)
        g = parity.run_gpu(v, inp, 4, debug=False)
        for key in ("accepted_len", "committed", "flags", "status"):
            assert np.array_equal(np.asarray(f[key]), np.asarray(g[key])), key
        greedy = dict(inp, temperature=np.zeros(B, np.float32))
        tk = np.full(B, 3, np.int32)
        f = run_truncated(v, greedy, tk, np.full(B, 0.5, np.float32), 4)
        g = parity.run_gpu(v, greedy, 4, debug=False)
        for key in ("accepted_len", "committed", "flags", "status"):
            assert np.array_equal(np.asarray(f[key]), np.asarray(g[key])), key


def test_truncated_round_without_draft_logits():
    """An all-greedy batch may pass no draft logits: the threshold passes then
    see target rows only, and the round is specverify_run's."""
    B, V = 20, 4096
    inp, _, _ = batch(B, V, "bf16", 41)
    inp = dict(inp, temperature=np.zeros(B, np.float32))
    t = parity.to_torch(inp, "cuda")
    tk, tp = _dev(np.full(B, 7, np.int32), np.int32), _dev(np.full(B, 0.5, np.float32), np.float32)
    with Verifier(B, inp["max_k"], V, "bf16") as v:
        f = v.run_truncated(t["target"], None, t["tokens"], t["num_draft"], t["temperature"],
                            tk, tp, 3)
        g = v.run(t["target"], None, t["tokens"], t["num_draft"], t["temperature"], 3)
        torch.cuda.synchronize()
        assert v.status() == 0
        for a, b in ((f.accepted_len, g.accepted_len), (f.committed, g.committed),
                     (f.flags, g.flags)):
            assert torch.equal(a, b)
