"""Greedy tree verification in the oracle, pinned to constructed cases of the
DDTree rule ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and
DSpark", section 5), to the greedy chain of the verify oracle (a chain is a
tree), and to a brute force that defines the accepted path node by node."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_examples.txt")


def read_tree_cases():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            elif key == "V":
                cur["V"] = int(vals[0])
            else:
                cur[key] = [int(v) for v in vals]
    return cases


def tree_rows(argmax, V, dtype="f32", rng=None):
    """Rows whose argmax is the given token (noise below the maximum)."""
    rng = rng or np.random.default_rng(0)
    rows = rng.uniform(-3.0, 0.0, size=(len(argmax), V)).astype(np.float32)
    for i, a in enumerate(argmax):
        rows[i, a] = 2.0
    if dtype == "bf16":
        rows = (rows.view(np.uint32) >> 16).astype(np.uint16)
    return rows


def brute_force(rows, parents, tokens):
    """Node by node: node i is accepted when its parent is accepted (or is the
    root), its token is the parent row's argmax, and no lower-index sibling has
    that token.  The accepted nodes form the path; the bonus is the argmax of
    the deepest accepted node's row (the root's when none is)."""
    x = rows if rows.dtype == np.float32 else (rows.astype(np.uint32) << 16).view(np.float32)
    arg = [int(np.argmax(x[j])) for j in range(len(x))]   # first maximum
    n = len(parents)
    ok = [False] * n
    for i in range(n):
        p = parents[i]
        parent_ok = p == -1 or ok[p]
        first = all(not (parents[s] == p and tokens[s] == tokens[i]) for s in range(i))
        ok[i] = parent_ok and first and tokens[i] == arg[p + 1]
    path = [i for i in range(n) if ok[i]]
    deepest = path[-1] if path else -1
    return path, [tokens[i] for i in path] + [arg[deepest + 1]]


def run_one(rows, parents, tokens, max_nodes=None):
    n = len(parents)
    mx = n if max_nodes is None else max_nodes
    return oracle.tree_greedy(rows, [n], np.array(parents, np.int32), np.array(tokens, np.int32), mx)


@pytest.mark.parametrize("case", read_tree_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_constructed_cases(case, dtype):
    rows = tree_rows(case["argmax"], case["V"], dtype)
    o = run_one(rows, case["parents"], case["tokens"])
    A = len(case["path"])
    assert o["status"] == 0
    assert o["accepted_len"][0] == A
    assert o["path"][0, :A].tolist() == case["path"] and (o["path"][0, A:] == -1).all()
    assert o["committed"][0, :A + 1].tolist() == case["committed"]
    assert (o["committed"][0, A + 1:] == -1).all()
    assert brute_force(rows, case["parents"], case["tokens"]) == (case["path"], case["committed"])


def test_chain_tree_equals_greedy_chain_verify():
    rng = np.random.default_rng(3)
    B, k, V = 40, 6, 50
    num = rng.integers(0, k + 1, size=B).astype(np.int32)
    t_rows = int((num + 1).sum())
    target = rng.normal(size=(t_rows, V)).astype(np.float32)
    # drafts that often follow the target argmax
    t_off = np.concatenate([[0], np.cumsum(num + 1)])
    toks = []
    for r in range(B):
        for i in range(num[r]):
            a = int(np.argmax(target[t_off[r] + i]))
            toks.append(a if rng.random() < 0.7 else int(rng.integers(0, V)))
    toks = np.array(toks, np.int32)
    parents = np.concatenate([np.arange(-1, num[r] - 1) for r in range(B)]).astype(np.int32)
    tr = oracle.tree_greedy(target, num, parents, toks, k)
    ch = oracle.verify(target, None, toks, num, np.zeros(B, np.float32), 1, k)
    assert tr["status"] == 0
    assert (tr["accepted_len"] == ch["accepted_len"]).all()
    assert (tr["committed"] == ch["committed"]).all()
    for r in range(B):
        A = tr["accepted_len"][r]
        assert tr["path"][r, :A].tolist() == list(range(A))


@pytest.mark.parametrize("seed", range(6))
def test_random_trees_against_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    V, B, max_nodes = 6, 25, 24
    num = rng.integers(0, max_nodes + 1, size=B).astype(np.int32)
    rows_all, par_all, tok_all = [], [], []
    for r in range(B):
        n = int(num[r])
        par = [int(rng.integers(-1, i)) if i > 0 else -1 for i in range(n)]
        tok = [int(rng.integers(0, V)) for _ in range(n)]
        # the target mostly selects a token one of the node's children carries
        arg = []
        for j in range(n + 1):
            kids = [tok[i] for i in range(n) if par[i] == j - 1]
            arg.append(int(rng.choice(kids)) if kids and rng.random() < 0.8 else int(rng.integers(0, V)))
        rows = tree_rows(arg, V, rng=rng)
        # ties: a second maximum on a later index sometimes
        for j in range(n + 1):
            if rng.random() < 0.2 and arg[j] + 1 < V:
                rows[j, arg[j] + 1] = rows[j, arg[j]]
        rows_all.append(rows)
        par_all += par
        tok_all += tok
    target = np.concatenate(rows_all)
    o = oracle.tree_greedy(target, num, np.array(par_all, np.int32), np.array(tok_all, np.int32),
                           max_nodes)
    assert o["status"] == 0
    n_off = 0
    for r in range(B):
        n = int(num[r])
        path, com = brute_force(rows_all[r], par_all[n_off:n_off + n], tok_all[n_off:n_off + n])
        A = o["accepted_len"][r]
        assert A == len(path) and o["path"][r, :A].tolist() == path
        assert o["committed"][r, :A + 1].tolist() == com
        n_off += n


def test_invalid_trees():
    rows = tree_rows([1, 2, 3, 0], 4)
    o = run_one(rows, [-1, 1, 0], [1, 2, 3])       # parent 1 of node 1 is not earlier
    assert o["status"] == oracle.BAD_PARENT and o["accepted_len"][0] == -1
    o = run_one(rows, [-1, 0, 0], [1, 4, 3])       # token == V
    assert o["status"] == oracle.BAD_TOKEN and (o["committed"][0] == -1).all()
    bad = rows.copy()
    bad[2, 0] = np.nan                              # row of node 1, on the walk
    o = run_one(bad, [-1, 0, 1], [1, 2, 3])
    assert o["status"] == oracle.NONFINITE
    bad = rows.copy()
    bad[3, 1] = np.nan                              # row of node 2, never read
    o = run_one(bad, [-1, -1, 1], [1, 2, 3])
    assert o["status"] == 0 and o["accepted_len"][0] == 1
    o = oracle.tree_greedy(rows, [3], np.array([-1, 0, 1], np.int32), np.array([1, 2, 3], np.int32), 2)
    assert o["status"] == oracle.BAD_K and o["accepted_len"][0] == -1
