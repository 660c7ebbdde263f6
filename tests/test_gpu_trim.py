"""Trimmed verify rounds (specverify_run_trimmed) against the oracle's trimmed
verify, element by element, at the chosen and the one-position wave depths."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_10_gb300 import Verifier, build
from speculative_decoding_verification_10_gb300 import workloads as W
from tests import cases, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def run_trimmed_gpu(v, inp, conf, cost, seed):
    t = parity.to_torch(inp, "cuda")
    res = v.run_trimmed(t["target"], t["draft"], t["tokens"], t["num_draft"],
                        torch.from_numpy(np.ascontiguousarray(conf, np.float32)).cuda(),
                        torch.from_numpy(np.ascontiguousarray(cost, np.float32)).cuda(),
                        t["temperature"], seed, debug=True)
    torch.cuda.synchronize()
    return {"accepted_len": res.accepted_len.cpu().numpy(), "committed": res.committed.cpu().numpy(),
            "flags": res.flags.cpu().numpy(), "p_y": res.p_y.cpu().numpy(),
            "q_y": res.q_y.cpu().numpy(), "u": res.u.cpu().numpy(),
            "req_status": res.req_status.cpu().numpy(), "status": v.status(),
            "verified_k": res.verified_k.cpu().numpy()}


def check(inp, conf, cost, seeds, depth=0, dtype=None):
    dtype = dtype or ("bf16" if inp["target"].dtype == np.uint16 else "f32")
    B = len(inp["num_draft"])
    reps = []
    with Verifier(max(B, 1), inp["max_k"], inp["target"].shape[1], dtype) as v:
        v.set_depth(depth)
        for seed in seeds:
            g = run_trimmed_gpu(v, inp, conf, cost, seed)
            o = oracle.verify_trimmed(inp["target"], inp.get("draft"), inp["tokens"],
                                      inp["num_draft"], conf, cost, inp["temperature"], seed,
                                      inp["max_k"])
            assert (g["verified_k"] == o["verified_k"]).all()
            reps.append(parity.compare(g, o, inp, seed))
    return reps


def batch(B, vocab, dtype, seed, max_k=6):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, max_k + 1, size=B)
    temp = rng.choice([0.0, 0.6, 1.0], size=B)
    inp = cases.random_batch(k, temp, vocab=vocab, sigma_t=2.0, sigma_d=0.8, dtype=dtype,
                             seed=seed)
    inp["max_k"] = max_k
    n = int(inp["num_draft"].sum())
    conf = rng.uniform(0.2, 1.0, size=n).astype(np.float32)
    conf[rng.random(n) < 0.1] = 1.0
    cost = rng.uniform(-0.1, 0.9, size=B).astype(np.float32)
    return inp, conf, cost


@pytest.mark.parametrize("depth", [0, 1])
@pytest.mark.parametrize("dtype,vocab", [("bf16", 4096), ("f32", 3000), ("bf16", 1001),
                                         ("bf16", 32000)])
def test_trimmed_rounds(depth, dtype, vocab):
    inp, conf, cost = batch(45, vocab, dtype, vocab + 3)
    reps = check(inp, conf, cost, (1, 4), depth=depth)
    assert sum(r["exempt_accept"] + r["exempt_race"] for r in reps) <= 2


def test_large_vocab_trimmed():
    b = W.make_batch("w4_v262144_bf16", device="cpu", batch=16)
    inp = b.numpy_inputs()
    rng = np.random.default_rng(5)
    conf = rng.uniform(0.5, 1.0, size=int(inp["num_draft"].sum())).astype(np.float32)
    cost = np.full(len(inp["num_draft"]), 0.4, np.float32)
    check(inp, conf, cost, (1,))


def test_extremes_and_bad_confidences():
    inp, conf, _ = batch(30, 777, "bf16", 9)
    B = 30
    # a cost of 1 or more: nothing is verified, every request draws one token from p_0
    g = check(inp, conf, np.full(B, 1.0, np.float32), (2,))
    # a negative cost keeps every window: the plain verify round
    check(inp, conf, np.full(B, -1.0, np.float32), (2,))
    with Verifier(B, inp["max_k"], 777, "bf16") as v:
        full = parity.run_gpu(v, inp, 2)
        g = run_trimmed_gpu(v, inp, conf, np.full(B, -1.0, np.float32), 2)
    assert (g["committed"] == full["committed"]).all() and (g["flags"] == full["flags"]).all()
    # invalid confidences and costs skip their requests
    bad_c, bad_cost = conf.copy(), np.full(B, 0.3, np.float32)
    d_off = np.concatenate([[0], np.cumsum(inp["num_draft"])])
    r1 = int(np.nonzero(inp["num_draft"] > 0)[0][0])
    bad_c[d_off[r1]] = 1.5
    r2 = int(np.nonzero(inp["num_draft"] > 0)[0][1])
    bad_c[d_off[r2]] = np.nan
    bad_cost[3] = np.nan
    check(inp, bad_c, bad_cost, (3,))


def test_rows_past_the_trimmed_window_are_never_read():
    inp, conf, cost = batch(40, 2048, "bf16", 17)
    k, _ = oracle.trim(inp["num_draft"], conf, cost)
    w = inp["num_draft"]
    t_off = np.concatenate([[0], np.cumsum(w + 1)])
    d_off = np.concatenate([[0], np.cumsum(w)])
    late = dict(inp)
    late["target"], late["draft"] = inp["target"].copy(), inp["draft"].copy()
    for r in range(len(w)):
        late["target"][t_off[r] + k[r] + 1:t_off[r + 1]] = 0x7fc0   # bf16 NaN
        late["draft"][d_off[r] + k[r]:d_off[r + 1]] = 0x7f80        # bf16 +inf
    with Verifier(40, 6, 2048, "bf16") as v:
        a = run_trimmed_gpu(v, inp, conf, cost, 6)
        b = run_trimmed_gpu(v, late, conf, cost, 6)
    assert b["status"] == 0
    assert (a["committed"] == b["committed"]).all() and (a["accepted_len"] == b["accepted_len"]).all()


def test_empty_windows():
    inp, _, _ = batch(12, 512, "bf16", 2, max_k=0)
    check(inp, np.zeros(0, np.float32), np.full(12, 0.1, np.float32), (1,))
