"""GPU path (through the C ABI) against the CPU oracle, element by element.

Run on a CUDA device (``-m gpu``).  Tolerances are those stated in
tests/parity.py: exact tokens / lengths / flags, except decisions within a
relative 1e-5 of their threshold, which are counted.
"""
import math

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


def _verifier(inp, dtype, max_batch=None, max_k=None, depth=0):
    B = len(inp["num_draft"])
    V = inp["target"].shape[1]
    v = Verifier(max(1, max_batch or B), inp["max_k"] if max_k is None else max_k, V, dtype)
    v.set_depth(depth)
    return v


def _dtype_of(inp):
    return "bf16" if inp["target"].dtype == np.uint16 else "f32"


def _check(inp, seeds=(1,), max_batch=None, max_k=None, depth=0):
    dtype = _dtype_of(inp)
    reps = []
    with _verifier(inp, dtype, max_batch, max_k, depth) as v:
        for seed in seeds:
            g = parity.run_gpu(v, inp, seed)
            o = parity.run_oracle(inp, seed)
            reps.append(parity.compare(g, o, inp, seed))
    return reps


# --- the five synthetic workloads ------------------------------------------------

@pytest.mark.parametrize("name", ["w0_v1024_f32", "w1_v32000_bf16"])
def test_small_workloads_full_parity(name):
    b = W.make_batch(name, device="cpu")
    inp = b.numpy_inputs()
    reps = _check(inp, seeds=(1, 2, 3, 4))
    total = sum(r["sampling"] + r["greedy"] for r in reps)
    print(name, reps)
    assert _exempt(reps) <= max(1, total // 100)


def _exempt(reps):
    return sum(r["exempt_accept"] + r["exempt_race"] + r["exempt_residual_mass"] for r in reps)


@pytest.mark.parametrize("name", ["w2_v128256_bf16", "w3_v151936_bf16", "w4_v262144_bf16"])
def test_large_vocab_reduced_batch_parity(name):
    # full vocabulary, fewer requests: several vocab chunks per row and a ragged tail
    b = W.make_batch(name, device="cuda", batch=20)
    inp = b.numpy_inputs()
    reps = _check(inp, seeds=(1, 7))
    reps += _check(inp, seeds=(3,), depth=1)
    reps += _check(inp, seeds=(8,), depth=2)
    print(name, reps)
    assert _exempt(reps) <= max(1, sum(r["sampling"] + r["greedy"] for r in reps) // 100)


@pytest.mark.parametrize("name", ["w2_v128256_bf16", "w3_v151936_bf16", "w4_v262144_bf16"])
def test_full_size_workload_parity(name):
    """The full batch in the benchmark's launch configuration, every request
    compared with the oracle; near-threshold exemptions stay under 1 %."""
    b = W.make_batch(name, device="cuda")
    seed = 1
    nd = b.num_draft.cpu().numpy()
    with Verifier(b.batch, b.max_k, b.vocab, b.dtype) as v:
        res = v.run(b.target, b.draft, b.tokens, b.num_draft, b.temperature, seed, debug=True)
        torch.cuda.synchronize()
        gpu = {"accepted_len": res.accepted_len.cpu().numpy(),
               "committed": res.committed.cpu().numpy(), "flags": res.flags.cpu().numpy(),
               "p_y": res.p_y.cpu().numpy(), "q_y": res.q_y.cpu().numpy(),
               "u": res.u.cpu().numpy(), "req_status": res.req_status.cpu().numpy(),
               "status": v.status()}
    assert gpu["status"] == 0
    inp = b.numpy_inputs()
    o = parity.run_oracle(inp, seed)
    rep = parity.compare(gpu, o, inp, seed)
    print(name, rep)
    assert rep["sampling"] + rep["greedy"] == b.batch
    assert _exempt([rep]) <= max(1, b.batch // 100)
    # invariants over the whole batch
    A = gpu["accepted_len"]
    assert (A >= 0).all() and (A <= nd).all()
    d_off = np.concatenate([[0], np.cumsum(nd)])
    for r in range(b.batch):
        f = gpu["flags"][d_off[r]:d_off[r + 1]]
        assert f.sum() == A[r] and (f[:A[r]] == 1).all()
        c = gpu["committed"][r]
        assert (c[:A[r] + 1] >= 0).all() and (c[:A[r] + 1] < b.vocab).all()
        assert (c[A[r] + 1:] == -1).all()


# --- the worked examples on the GPU path ------------------------------------------

@pytest.mark.parametrize("case", cases.read_worked_examples(), ids=lambda c: c["case"])
@pytest.mark.parametrize("temperature", [1.0, 0.7, 0.0])
@pytest.mark.parametrize("dtype,vocab", [("f32", 16), ("bf16", 16), ("bf16", 1001), ("f32", 70000)])
def test_worked_examples_gpu(case, temperature, dtype, vocab):
    inp, expect = cases.worked_case_batch(case, vocab=vocab, copies=48, temperature=temperature,
                                          dtype=dtype)
    A = case["expect_accepted"]
    with _verifier(inp, dtype) as v:
        for seed in (0, 1, 12345, 2**63 + 5):
            g = parity.run_gpu(v, inp, seed)
            assert g["status"] == 0
            assert (g["accepted_len"] == A).all()
            assert (g["committed"][:, :A + 1] == np.array(expect)).all()
            assert (g["committed"][:, A + 1:] == -1).all()


# --- ragged batches, odd vocabularies, mixed modes ---------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vocab", [1, 5, 8, 1000, 1001, 4099, 33000])
def test_random_ragged_batches(dtype, vocab):
    rng = np.random.default_rng(vocab)
    B = 37
    k = rng.integers(0, 7, size=B)
    temp = rng.choice([0.0, 0.5, 0.7, 1.0, 1.6], size=B)
    inp = cases.random_batch(k, temp, vocab=vocab, sigma_t=2.5, sigma_d=1.0, dtype=dtype,
                             seed=vocab + 1)
    inp["max_k"] = 6
    _check(inp, seeds=(3, 99))


@pytest.mark.parametrize("depth", [1, 2, 3, 5, 7])
@pytest.mark.parametrize("dtype,vocab", [("bf16", 4096), ("bf16", 1001), ("f32", 3000)])
def test_wave_depths(depth, dtype, vocab):
    """Positions per wave launch change the launches, never the results: every
    depth is compared with the oracle (aligned and scalar paths, ragged k with
    k = 0, greedy and sampling requests mixed, groups cut mid-window)."""
    rng = np.random.default_rng(depth * 7 + vocab)
    B = 41
    k = rng.integers(0, 7, size=B)
    temp = rng.choice([0.0, 0.6, 1.0, 1.3], size=B)
    inp = cases.random_batch(k, temp, vocab=vocab, sigma_t=2.0, sigma_d=0.6, dtype=dtype,
                             seed=depth + vocab)
    inp["max_k"] = 6
    _check(inp, seeds=(2, 5), depth=depth)


@pytest.mark.parametrize("depth", [1, 4])
def test_small_workload_depths(depth):
    b = W.make_batch("w1_v32000_bf16", device="cpu")
    _check(b.numpy_inputs(), seeds=(1, 2), depth=depth)


@pytest.mark.parametrize("max_k", [15, 31])
def test_long_windows(max_k):
    B = 9
    k = np.array([max_k] * 4 + [0, 1, max_k // 2, max_k, 3])
    temp = np.array([1.0, 0.8, 0.0, 1.0, 1.0, 0.0, 0.9, 1.0, 0.7])
    inp = cases.random_batch(k, temp, vocab=2048, sigma_t=2.0, sigma_d=0.3, dtype="bf16", seed=5)
    inp["max_k"] = max_k
    _check(inp, seeds=(1, 2))


def test_identical_and_disjoint_rows():
    inp = cases.random_batch([4] * 16, [0.9] * 16, vocab=3000, dtype="bf16", seed=8)
    t_off = np.concatenate([[0], np.cumsum(inp["num_draft"] + 1)])
    src = np.concatenate([np.arange(t_off[r], t_off[r] + 4) for r in range(16)])
    inp["draft"] = inp["target"][src].copy()
    with _verifier(inp, "bf16") as v:
        g = parity.run_gpu(v, inp, 4)
    assert (g["accepted_len"] == 4).all()
    V, B = 64, 100
    tgt = np.full((2 * B, V), -np.inf, np.float32)
    tgt[:, :32] = 0.0
    drf = np.full((B, V), -np.inf, np.float32)
    drf[:, 32:] = 0.0
    inp = dict(target=tgt, draft=drf, tokens=(32 + np.arange(B) % 32).astype(np.int32),
               num_draft=np.ones(B, np.int32), temperature=np.ones(B, np.float32), max_k=1)
    reps = _check(inp, seeds=(1,))
    with _verifier(inp, "f32") as v:
        g = parity.run_gpu(v, inp, 1)
    assert (g["accepted_len"] == 0).all() and (g["committed"][:, 0] < 32).all()


def test_greedy_only_without_draft_logits():
    inp = cases.random_batch([3, 0, 5, 2], [0.0] * 4, vocab=5000, dtype="bf16", seed=2)
    inp["max_k"] = 5
    o = parity.run_oracle(inp, 1)
    inp2 = dict(inp)
    inp2["draft"] = None
    with _verifier(inp2, "bf16") as v:
        g = parity.run_gpu(v, inp2, 1)
    assert g["status"] == 0
    assert (g["committed"] == o["committed"]).all() and (g["accepted_len"] == o["accepted_len"]).all()


def test_all_zero_drafts_and_empty_batch():
    inp = cases.random_batch([0] * 10, [1.0] * 5 + [0.0] * 5, vocab=777, dtype="bf16", seed=3)
    inp["max_k"] = 2
    _check(inp, seeds=(1, 2))
    inp = cases.random_batch([0] * 10, [1.0] * 5 + [0.0] * 5, vocab=776, dtype="bf16", seed=3)
    inp["max_k"] = 2
    _check(inp, seeds=(1, 2))
    with Verifier(4, 2, 777, "bf16") as v:
        e = torch.empty(0, dtype=torch.int32, device="cuda")
        res = v.run(torch.empty(0, 777, dtype=torch.bfloat16, device="cuda"), None, e, e,
                    torch.empty(0, dtype=torch.float32, device="cuda"), 1)
        assert res.accepted_len.numel() == 0


@pytest.mark.parametrize("depth", [1, 2, 6])
def test_rows_after_the_first_rejection_do_not_matter(depth):
    """Garbage (NaN / +inf) in rows beyond the first rejection changes nothing:
    at depth 1 those rows are never read; at larger depths they may be read but
    their positions are never decided."""
    inp = cases.random_batch([5] * 48, [1.0] * 24 + [0.0] * 24, vocab=4096, sigma_d=2.5,
                             dtype="bf16", seed=13)
    with _verifier(inp, "bf16", depth=depth) as v:
        base = parity.run_gpu(v, inp, 5)
        A = base["accepted_len"]
        k = inp["num_draft"]
        t_off = np.concatenate([[0], np.cumsum(k + 1)])
        d_off = np.concatenate([[0], np.cumsum(k)])
        late = dict(inp)
        late["target"], late["draft"] = inp["target"].copy(), inp["draft"].copy()
        for r in range(48):
            if A[r] + 1 <= k[r]:
                late["target"][t_off[r] + A[r] + 1:t_off[r + 1]] = 0x7fc0   # bf16 NaN
                late["draft"][d_off[r] + A[r] + 1:d_off[r + 1]] = 0x7f80    # bf16 +inf
        g = parity.run_gpu(v, late, 5)
    assert g["status"] == 0
    assert (g["committed"] == base["committed"]).all()
    assert (g["accepted_len"] == A).all()


# --- invalid inputs: reported, skipped, never a fault --------------------------------

def test_invalid_inputs_status_and_skip():
    inp = cases.random_batch([2, 2, 2, 2, 2, 2, 2], [1.0, 1.0, 0.0, 1.0, 1.0, 1.0, 1.0],
                             vocab=300, dtype="f32", seed=6)
    bad = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
    bad["tokens"][2] = 300              # request 1: token == V
    bad["tokens"][4] = -1               # request 2 (greedy): negative token
    bad["temperature"][3] = np.nan      # request 3
    bad["target"][4 * 3 + 0, 7] = np.nan   # request 4: NaN in its first target row
    bad["draft"][5 * 2 + 0, 9] = np.inf    # request 5: +inf in its first draft row
    # request 6: draft rows equal to the target rows (so both drafts are accepted
    # and the bonus row is read), and a bonus row without a finite logit
    bad["draft"][6 * 2:6 * 2 + 2] = bad["target"][6 * 3:6 * 3 + 2]
    bad["target"][6 * 3 + 2, :] = -np.inf
    for depth in (0, 1):
        _check(bad, seeds=(1,), depth=depth)
        with _verifier(bad, "f32", depth=depth) as v:
            g = parity.run_gpu(v, bad, 1)
        assert g["status"] == (oracle.BAD_TOKEN | oracle.BAD_TEMP | oracle.NONFINITE)
        assert g["accepted_len"][0] >= 0 and (g["accepted_len"][1:] == -1).all()
    # layout errors skip the whole batch
    wrong = dict(inp)
    wrong["num_draft"] = np.array([2, 2, 2, 2, 2, 2, 3], np.int32)   # k > max_k
    _layout_errors(inp, wrong)
    nod = dict(inp)
    nod["draft"] = None
    with _verifier(inp, "f32") as v:
        g = parity.run_gpu(v, nod, 1)
    assert g["status"] == oracle.NO_DRAFT
    assert (g["accepted_len"][[0, 1, 3, 4, 5, 6]] == -1).all() and g["accepted_len"][2] >= 0


def _layout_errors(inp, wrong):
    with _verifier(inp, "f32") as v:
        t = parity.to_torch(wrong, "cuda")
        res = v.run(t["target"], t["draft"], t["tokens"], t["num_draft"], t["temperature"], 1,
                    total_draft=14)
        assert v.status() == oracle.BAD_K
        assert (res.accepted_len.cpu().numpy() == -1).all()
        t = parity.to_torch(inp, "cuda")
        res = v.run(t["target"], t["draft"], t["tokens"][:13], t["num_draft"], t["temperature"], 1,
                    total_draft=13)
        assert v.status() == oracle.BAD_TOTAL
        # a valid run right after clears the status
        v.run(t["target"], t["draft"], t["tokens"], t["num_draft"], t["temperature"], 1)
        assert v.status() == 0


# --- properties of the randomness ------------------------------------------------------

def test_request_ids_make_results_order_independent():
    b = W.make_batch("w1_v32000_bf16", device="cuda", batch=24)
    with Verifier(24, 3, b.vocab, "bf16") as v:
        r1 = v.run(b.target, b.draft, b.tokens, b.num_draft, b.temperature, 5)
        c1 = r1.committed.clone()
        r2 = v.run(b.target, b.draft, b.tokens, b.num_draft, b.temperature, 5)
        assert torch.equal(c1, r2.committed)            # deterministic
        perm = np.random.default_rng(1).permutation(24)
        sub = W.subset(b, perm)                           # request_ids = original index
        r3 = v.run(sub.target, sub.draft, sub.tokens, sub.num_draft, sub.temperature, 5,
                   request_ids=sub.request_ids)
        assert torch.equal(r3.committed, c1[torch.as_tensor(perm, device="cuda")])


def test_million_trials_distribution_and_bit_exactness():
    rng = np.random.default_rng(2024)
    V, k, T, n = 8, 2, 1.0, 1_000_000
    tgt = (rng.normal(size=(k + 1, V)) * 1.5).astype(np.float32)
    drf = (tgt[:k] + rng.normal(size=(k, V))).astype(np.float32)
    toks = np.stack([rng.choice(V, size=n, p=_softmax(drf[i], T)) for i in range(k)], 1)
    inp = dict(target=np.tile(tgt, (n, 1)), draft=np.tile(drf, (n, 1)),
               tokens=toks.reshape(-1).astype(np.int32), num_draft=np.full(n, k, np.int32),
               temperature=np.full(n, T, np.float32), max_k=k)
    # one handle serves at most 4096 requests: verify in slices keyed by request
    # id, which draws exactly what one large batch would
    S = 4096
    acc = np.empty(n, np.int32)
    com = np.empty((n, k + 1), np.int32)
    with Verifier(S, k, V, "f32") as v:
        for a in range(0, n, S):
            b = min(n, a + S)
            part = dict(target=inp["target"][a * (k + 1):b * (k + 1)],
                        draft=inp["draft"][a * k:b * k], tokens=inp["tokens"][a * k:b * k],
                        num_draft=inp["num_draft"][a:b], temperature=inp["temperature"][a:b],
                        request_ids=np.arange(a, b, dtype=np.int64), max_k=k)
            gp = parity.run_gpu(v, part, 123, debug=False)
            acc[a:b] = gp["accepted_len"]
            com[a:b] = gp["committed"]
    g = {"accepted_len": acc, "committed": com}
    o = parity.run_oracle(inp, 123)
    same = (g["committed"] == o["committed"]).all(1)
    # exact agreement except near-threshold draws
    assert same.mean() > 1 - 1e-4
    p = [_softmax(tgt[i], T) for i in range(k + 1)]
    scipy_stats = pytest.importorskip("scipy.stats")
    for col, sel, probs in ((0, np.ones(n, bool), p[0]),
                            (1, g["accepted_len"] >= 1, p[1]),
                            (2, g["accepted_len"] == 2, p[2])):
        cnt = np.bincount(g["committed"][sel, col], minlength=V).astype(np.float64)
        e = probs * cnt.sum()
        stat = ((cnt - e) ** 2 / e).sum()
        assert scipy_stats.chi2.sf(stat, V - 1) > 1e-3
    a0 = np.minimum(p[0], _softmax(drf[0], T)).sum()
    z = ((g["accepted_len"] >= 1).mean() - a0) / math.sqrt(a0 * (1 - a0) / n)
    assert abs(z) < 4.5


def _softmax(x, t):
    z = np.asarray(x, np.float64) / t
    z = np.exp(z - z.max())
    return z / z.sum()


# --- host-buffer entry point ----------------------------------------------------------

@pytest.mark.parametrize("mode,pinned,in_place", [("auto", True, 1), ("stage", True, 0),
                                                   ("auto", False, 0)])
def test_run_host_matches_device_run(mode, pinned, in_place):
    """Pinned host logits read in place ('auto'), staged ('stage'), and pageable
    ones (always staged): the same outputs as the device run."""
    b = W.make_batch("w3_v151936_bf16", device="cuda", batch=12)
    with Verifier(12, b.max_k, b.vocab, "bf16", host_staging=True) as v:
        v.set_host_reads(mode)
        assert v.last_host_reads() == -1
        dev = v.run(b.target, b.draft, b.tokens, b.num_draft, b.temperature, 9)
        torch.cuda.synchronize()
        h = b.to("cpu")
        acc = torch.empty(12, dtype=torch.int32).pin_memory()
        com = torch.empty(12, b.max_k + 1, dtype=torch.int32).pin_memory()
        flg = torch.empty(b.total_draft, dtype=torch.uint8).pin_memory()
        tgt = h.target.pin_memory() if pinned else h.target.clone()
        drf = h.draft.pin_memory() if pinned else h.draft.clone()
        v.run_host(tgt, drf, h.tokens, h.num_draft, h.temperature, 9, acc, com, flg)
        assert v.last_host_reads() == in_place
        assert torch.equal(acc, dev.accepted_len.cpu())
        assert torch.equal(com, dev.committed.cpu())
        assert torch.equal(flg, dev.flags.cpu())


# --- round tags ---------------------------------------------------------------------------

def test_rounds_across_the_round_tag_wrap():
    """Completion counters carry a 32-bit round tag; five rounds from 0xfffffffd
    cross the wrap (counters cleared, numbering restarted at 1), alternating
    one-wave-per-position and all-positions-in-one-wave rounds, and each
    matches the oracle."""
    b = W.make_batch("w1_v32000_bf16", device="cpu", batch=64)
    inp = b.numpy_inputs()
    with _verifier(inp, "bf16") as v:
        parity.run_gpu(v, inp, 1)
        v.debug_set_epoch(0xfffffffd)
        for i, seed in enumerate(range(1, 6)):
            v.set_depth(1 if i % 2 else 0)
            g = parity.run_gpu(v, inp, seed)
            rep = parity.compare(g, parity.run_oracle(inp, seed), inp, seed)
            assert _exempt([rep]) <= 1, (seed, rep)
