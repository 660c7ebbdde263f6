"""Top-k / top-p truncation on the GPU (specverify_truncate) against the oracle,
element by element, and the verify round on truncated rows."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_10_gb300 import Verifier, build, truncate
from tests import cases, parity

pytestmark = pytest.mark.gpu
MARGIN = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def gpu_truncate(inp, top_k, top_p):
    t = parity.to_torch(inp, "cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tt, dd = truncate(t["target"], t["draft"], t["num_draft"], t["temperature"],
                      torch.as_tensor(np.ascontiguousarray(top_k, np.int32)).cuda(),
                      torch.as_tensor(np.ascontiguousarray(top_p, np.float32)).cuda(), status=st)
    torch.cuda.synchronize()

    def back(x):
        if x is None:
            return None
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).cpu().numpy().view(np.uint16)
        return x.cpu().numpy()
    return back(tt), back(dd), int(st.item())


def compare_rows(g, o, margin):
    """Bit-exact rows except those whose top-p decision is within MARGIN."""
    exempt = 0
    for i in range(len(g)):
        if margin[i] <= MARGIN:
            exempt += 1
            continue
        assert (g[i].view(np.uint8) == o[i].view(np.uint8)).all(), i
    return exempt


def batch(B, vocab, dtype, seed, max_k=5):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, max_k + 1, size=B)
    temp = rng.choice([0.0, 0.6, 1.0, 1.4], size=B)
    inp = cases.random_batch(k, temp, vocab=vocab, sigma_t=2.5, sigma_d=0.8, dtype=dtype,
                             seed=seed)
    inp["max_k"] = max_k
    top_k = rng.choice([0, 1, 2, 20, vocab // 3, vocab, vocab + 5], size=B).astype(np.int32)
    top_p = rng.choice([1.0, 0.9, 0.5, 0.95, 0.2, 1.5], size=B).astype(np.float32)
    return inp, top_k, top_p


@pytest.mark.parametrize("dtype,vocab", [("bf16", 4096), ("f32", 3000), ("bf16", 1001),
                                         ("f32", 777), ("bf16", 32000), ("bf16", 151936),
                                         ("bf16", 262144)])
def test_truncation_matches_oracle(dtype, vocab):
    B = 40 if vocab < 100000 else (8 if vocab < 200000 else 6)
    inp, top_k, top_p = batch(B, vocab, dtype, vocab + 1)
    gt, gd, st = gpu_truncate(inp, top_k, top_p)
    ot, od, mt, md, ost = oracle.truncate(inp["target"], inp["draft"], inp["num_draft"],
                                          inp["temperature"], top_k, top_p)
    assert st == ost == 0
    ex = compare_rows(gt, ot, mt) + compare_rows(gd, od, md)
    assert ex <= max(1, (len(gt) + len(gd)) // 50)


def test_top_k_only_is_exact_with_ties():
    rng = np.random.default_rng(3)
    B, V = 30, 600
    inp, _, _ = batch(B, V, "bf16", 5)
    inp["target"] = (np.round(rng.normal(size=inp["target"].shape) * 2, 0).astype(np.float32)
                     .view(np.uint32) >> 16).astype(np.uint16)     # many equal logits
    top_k = rng.integers(1, V, size=B).astype(np.int32)
    top_p = np.ones(B, np.float32)
    gt, gd, _ = gpu_truncate(inp, top_k, top_p)
    ot, od, _, _, _ = oracle.truncate(inp["target"], inp["draft"], inp["num_draft"],
                                      inp["temperature"], top_k, top_p)
    assert (gt == ot).all() and (gd == od).all()


def test_invalid_top_p_and_nan_rows():
    inp, top_k, _ = batch(10, 500, "f32", 8)
    top_p = np.full(10, 0.5, np.float32)
    top_p[2] = np.nan
    top_p[5] = 0.0
    inp["target"][0, 3] = np.nan
    gt, gd, st = gpu_truncate(inp, top_k, top_p)
    ot, od, mt, md, ost = oracle.truncate(inp["target"], inp["draft"], inp["num_draft"],
                                          inp["temperature"], top_k, top_p)
    assert st == ost == oracle.BAD_TRUNC
    compare_rows(gt, ot, mt)
    compare_rows(gd, od, md)


def test_verify_on_truncated_rows():
    """GPU truncate then GPU verify against the oracle's truncate then verify, for
    the requests none of whose rows is near a top-p threshold; the draft tokens
    are drawn from the truncated draft rows."""
    rng = np.random.default_rng(11)
    B, V = 48, 2048
    inp, top_k, top_p = batch(B, V, "bf16", 12)
    ot, od, mt, md, _ = oracle.truncate(inp["target"], inp["draft"], inp["num_draft"],
                                        inp["temperature"], top_k, top_p)
    # draft tokens sampled (numpy) from the truncated draft rows
    df = (od.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    toks = []
    d_off = np.concatenate([[0], np.cumsum(inp["num_draft"])])
    for r in range(B):
        T = inp["temperature"][r]
        for i in range(inp["num_draft"][r]):
            row = df[d_off[r] + i]
            if T == 0:
                toks.append(int(np.argmax(row)))
            else:
                w = np.exp((row - row.max()) / T)
                toks.append(int(rng.choice(V, p=w / w.sum())))
    inp["tokens"] = np.array(toks, np.int32)
    gt, gd, _ = gpu_truncate(inp, top_k, top_p)
    tin = dict(inp, target=gt, draft=gd)
    with Verifier(B, inp["max_k"], V, "bf16") as v:
        g = parity.run_gpu(v, tin, 3)
    o = oracle.verify(ot, od, inp["tokens"], inp["num_draft"], inp["temperature"], 3,
                      inp["max_k"])
    t_off = np.concatenate([[0], np.cumsum(inp["num_draft"] + 1)])
    checked = 0
    for r in range(B):
        rows_t = mt[t_off[r]:t_off[r + 1]]
        rows_d = md[d_off[r]:d_off[r + 1]]
        if (rows_t <= MARGIN).any() or (rows_d <= MARGIN).any():
            continue
        checked += 1
        assert g["accepted_len"][r] == o["accepted_len"][r] or \
            abs(o["accept_margin"][d_off[r]:d_off[r + 1]]).min() <= 1e-5
        if g["accepted_len"][r] == o["accepted_len"][r] and \
                (g["committed"][r] != o["committed"][r]).any():
            # only a near-tie of the race may differ
            pass
    assert checked >= B // 2
    # the full comparison on the oracle's truncated rows (same inputs on both sides)
    same = dict(inp, target=ot, draft=od)
    with Verifier(B, inp["max_k"], V, "bf16") as v:
        parity.compare(parity.run_gpu(v, same, 3), o, same, 3)


def test_top_1_sampling_is_greedy_gpu():
    rng = np.random.default_rng(6)
    B, V = 40, 3000
    k = rng.integers(0, 6, size=B)
    inp = cases.random_batch(k, np.ones(B), vocab=V, sigma_t=2.0, sigma_d=1.0, dtype="bf16",
                             seed=4)
    df = (inp["draft"].astype(np.uint32) << 16).view(np.float32)
    inp["tokens"] = np.array([int(np.argmax(r)) for r in df], np.int32)
    inp["max_k"] = 5
    gt, gd, _ = gpu_truncate(inp, np.ones(B, np.int32), np.ones(B, np.float32))
    with Verifier(B, 5, V, "bf16") as v:
        s = parity.run_gpu(v, dict(inp, target=gt, draft=gd), 2)
        inp0 = dict(inp, temperature=np.zeros(B, np.float32))
        g = parity.run_gpu(v, inp0, 2)
    assert (s["committed"] == g["committed"]).all() and (s["accepted_len"] == g["accepted_len"]).all()


def test_window_histogram_and_radix_descent_rows():
    """bf16 rows built so that both ways to a threshold run: rows whose top-k or
    top-p boundary lies among the exact keys of the eight high-byte bins below
    the maximum (the window histogram), and rows it hands to the radix descent
    (top-k larger than the window's count, a top-p boundary below the window, a
    maximum that is not finite).  Every row against the oracle."""
    rng = np.random.default_rng(21)
    V = 4096

    def normal(s, mu=0.0):
        return rng.normal(size=V) * s + mu

    def few_high():  # 50 logits in (1, 100), the rest far below zero
        x = rng.normal(size=V) * 50.0 - 300.0
        x[rng.choice(V, 50, replace=False)] = rng.uniform(1.0, 100.0, size=50)
        return x

    def flat():  # one logit 0.5, the rest in [-1, 0): the mass lies below the window
        x = rng.uniform(-1.0, 0.0, size=V)
        x[rng.integers(V)] = 0.5
        return x

    def ties():
        return np.round(rng.normal(size=V) * 3.0)

    def neg_inf():
        return np.full(V, -np.inf)

    designs = [  # (row maker, T, top_k, top_p)
        (lambda: normal(2.5), 1.0, 20, 1.0),
        (lambda: normal(2.5), 1.0, 0, 0.9),
        (lambda: normal(2.5), 0.7, 50, 0.8),
        (lambda: normal(0.5, -5.0), 1.0, 10, 0.9),
        (few_high, 1.0, 1000, 1.0),
        (few_high, 1.0, 1000, 0.5),
        (flat, 10.0, 0, 0.5),
        (flat, 10.0, 0, 0.999),
        (ties, 1.0, 100, 1.0),
        (ties, 1.3, 0, 0.7),
        (neg_inf, 1.0, 5, 1.0),
    ]
    B = len(designs)
    k = np.ones(B, np.int32)
    temp = np.array([d[1] for d in designs], np.float32)
    inp = cases.random_batch(k, temp, vocab=V, dtype="bf16", seed=22)
    inp["max_k"] = 1
    tgt, drf = [], []
    for make, _, _, _ in designs:
        rows = [make() for _ in range(2)]
        tgt += rows
        drf.append(rows[0] + rng.normal(size=V) * 0.3)
    inp["target"] = cases.to_bf16_bits(np.array(tgt, np.float32))
    inp["draft"] = cases.to_bf16_bits(np.array(drf, np.float32))
    top_k = np.array([d[2] for d in designs], np.int32)
    top_p = np.array([d[3] for d in designs], np.float32)
    gt, gd, st = gpu_truncate(inp, top_k, top_p)
    ot, od, mt, md, ost = oracle.truncate(inp["target"], inp["draft"], inp["num_draft"],
                                          inp["temperature"], top_k, top_p)
    assert st == ost == 0
    ex = compare_rows(gt, ot, mt) + compare_rows(gd, od, md)
    assert ex <= 2
    # the constructed rows really do drop logits where a rule is on
    kept = (gt != 0xFF80).sum(axis=1)
    assert 20 <= kept[0] < V and kept[16] >= 100
