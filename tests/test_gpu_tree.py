"""Greedy tree verification on the GPU (through the C ABI) against the oracle,
element by element: accepted lengths, paths and committed tokens are integers
and must match exactly."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_10_gb300 import TreeVerifier, Verifier, build
from tests import parity
from tests.test_oracle_tree import read_tree_cases, tree_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def random_trees(B, max_nodes, V, dtype, seed, p_match=0.8, ties=0.1):
    rng = np.random.default_rng(seed)
    num = rng.integers(0, max_nodes + 1, size=B).astype(np.int32)
    rows, par_all, tok_all = [], [], []
    for r in range(B):
        n = int(num[r])
        par = [int(rng.integers(max(-1, i - 8), i)) if i > 0 else -1 for i in range(n)]
        tok = [int(rng.integers(0, V)) for _ in range(n)]
        arg = []
        for j in range(n + 1):
            kids = [tok[i] for i in range(n) if par[i] == j - 1]
            arg.append(int(rng.choice(kids)) if kids and rng.random() < p_match
                       else int(rng.integers(0, V)))
        x = rng.normal(size=(n + 1, V)).astype(np.float32) - 4.0
        for j, a in enumerate(arg):
            x[j, a] = 3.0
            if rng.random() < ties and a + 1 < V:
                x[j, a + 1] = 3.0                 # a tie on a later index
        rows.append(x)
        par_all += par
        tok_all += tok
    target = np.concatenate(rows) if rows else np.zeros((0, V), np.float32)
    if dtype == "bf16":
        target = (target.view(np.uint32) >> 16).astype(np.uint16)
    return (target, num, np.array(par_all, np.int32), np.array(tok_all, np.int32))


def run_gpu(tv, target, num, par, tok):
    t = torch.from_numpy(target.view(np.int16) if target.dtype == np.uint16 else target)
    t = t.view(torch.bfloat16) if target.dtype == np.uint16 else t
    dev = "cuda"
    res = tv.run(t.to(dev), torch.from_numpy(num).to(dev), torch.from_numpy(par).to(dev),
                 torch.from_numpy(tok).to(dev))
    torch.cuda.synchronize()
    return {"accepted_len": res.accepted_len.cpu().numpy(), "path": res.path.cpu().numpy(),
            "committed": res.committed.cpu().numpy(), "req_status": res.req_status.cpu().numpy(),
            "status": tv.status()}


def check(target, num, par, tok, max_nodes, dtype, max_batch=None):
    V = target.shape[1]
    o = oracle.tree_greedy(target, num, par, tok, max_nodes)
    with TreeVerifier(max_batch or max(1, len(num)), max_nodes, V, dtype) as tv:
        g = run_gpu(tv, target, num, par, tok)
    assert g["status"] == o["status"]
    assert (g["accepted_len"] == o["accepted_len"]).all()
    assert (g["committed"] == o["committed"]).all()
    if max_nodes:
        assert (g["path"] == o["path"]).all()
    assert (g["req_status"] == o["req_status"]).all()
    return g


@pytest.mark.parametrize("dtype,V", [("f32", 6), ("bf16", 6), ("bf16", 1001), ("f32", 1001),
                                     ("bf16", 4096), ("f32", 70000), ("bf16", 151936),
                                     ("bf16", 262144)])
def test_random_trees(dtype, V):
    B = 40 if V < 100000 else 12
    for seed in range(2):
        check(*random_trees(B, 24, V, dtype, seed * 13 + V), 24, dtype)


@pytest.mark.parametrize("max_nodes", [0, 1, 63, 1024])
def test_tree_sizes(max_nodes):
    B = 6 if max_nodes == 1024 else 50
    check(*random_trees(B, max_nodes, 512, "bf16", max_nodes + 5), max_nodes, "bf16")


@pytest.mark.parametrize("case", read_tree_cases(), ids=lambda c: c["name"])
def test_constructed_cases_gpu(case):
    rows = tree_rows(case["argmax"], case["V"], "bf16")
    n = len(case["parents"])
    g = check(rows, np.array([n], np.int32), np.array(case["parents"], np.int32),
              np.array(case["tokens"], np.int32), max(n, 1), "bf16")
    A = len(case["path"])
    assert g["committed"][0, :A + 1].tolist() == case["committed"]


def test_chain_tree_equals_verify_kernel():
    rng = np.random.default_rng(21)
    B, k, V = 64, 6, 32000
    num = rng.integers(0, k + 1, size=B).astype(np.int32)
    target = (rng.normal(size=(int((num + 1).sum()), V)) * 2).astype(np.float32)
    t_off = np.concatenate([[0], np.cumsum(num + 1)])
    toks = np.array([int(np.argmax(target[t_off[r] + i])) if rng.random() < 0.8
                     else int(rng.integers(0, V)) for r in range(B) for i in range(num[r])],
                    np.int32)
    par = np.concatenate([np.arange(-1, num[r] - 1) for r in range(B)]).astype(np.int32)
    g = check(target, num, par, toks, k, "f32")
    inp = dict(target=target, draft=None, tokens=toks, num_draft=num,
               temperature=np.zeros(B, np.float32), max_k=k)
    with Verifier(B, k, V, "f32") as v:
        c = parity.run_gpu(v, inp, 1)
    assert (g["accepted_len"] == c["accepted_len"]).all()
    assert (g["committed"] == c["committed"]).all()


def test_invalid_trees_gpu():
    V = 300
    target, num, par, tok = random_trees(8, 6, V, "f32", 3)
    n_off = np.concatenate([[0], np.cumsum(num)])
    t_off = np.concatenate([[0], np.cumsum(num + 1)])
    bad_par, bad_tok, bad_t = par.copy(), tok.copy(), target.copy()
    r = int(np.nonzero(num >= 2)[0][0])
    bad_par[n_off[r] + 1] = 1                # not an earlier node
    r2 = int(np.nonzero(num >= 1)[0][1])
    bad_tok[n_off[r2]] = V                   # token == V
    bad_t[t_off[0], 5] = np.nan              # the root row is always read
    check(target, num, bad_par, tok, 6, "f32")
    check(target, num, par, bad_tok, 6, "f32")
    check(bad_t, num, par, tok, 6, "f32")
    over = num.copy()
    over[0] = 7                              # above max_nodes: the batch is skipped
    o = oracle.tree_greedy(target, over, par, tok, 6, total_nodes=int(num.sum()))
    with TreeVerifier(8, 6, V, "f32") as tv:
        g = run_gpu(tv, target, over, par, tok)
    assert g["status"] == o["status"] == oracle.BAD_K
    assert (g["accepted_len"] == -1).all()


def test_empty_batch():
    with TreeVerifier(4, 3, 64, "bf16") as tv:
        res = tv.run(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"),
                     torch.empty(0, dtype=torch.int32, device="cuda"),
                     torch.empty(0, dtype=torch.int32, device="cuda"),
                     torch.empty(0, dtype=torch.int32, device="cuda"))
        assert res.accepted_len.numel() == 0 and tv.status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_rows_off_the_accepted_path_are_never_read(dtype):
    """The walk reads only the rows of its accepted path: filling every other
    row with NaN changes nothing and raises no status bit, while NaN in a row on
    the path does."""
    target, num, par, tok = random_trees(24, 16, 4096, dtype, seed=77)
    g = check(target, num, par, tok, 16, dtype)
    t_off = np.concatenate([[0], np.cumsum(num.astype(np.int64) + 1)])
    on_path = np.zeros(len(target), bool)
    for r in range(len(num)):
        if g["accepted_len"][r] < 0:
            continue
        on_path[t_off[r]] = True                                   # the root row
        for d in range(g["accepted_len"][r]):
            on_path[t_off[r] + 1 + g["path"][r][d]] = True         # the accepted nodes' rows
    poisoned = target.copy()
    nan = np.uint16(0x7fc0) if dtype == "bf16" else np.float32(np.nan)
    poisoned[~on_path] = nan
    with TreeVerifier(len(num), 16, 4096, dtype) as tv:
        h = run_gpu(tv, poisoned, num, par, tok)
        assert h["status"] == 0
        assert (h["accepted_len"] == g["accepted_len"]).all()
        assert (h["committed"] == g["committed"]).all() and (h["path"] == g["path"]).all()
        # NaN in the root row of the first request, which every walk reads
        poisoned[t_off[0]] = nan
        h = run_gpu(tv, poisoned, num, par, tok)
        assert h["status"] == oracle.NONFINITE and h["accepted_len"][0] == -1
