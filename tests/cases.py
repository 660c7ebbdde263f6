"""Constructed verify batches for tests (inputs only; no verify arithmetic).

Host numpy arrays in the library's ragged layout.  bf16 logits are carried as
their uint16 bit patterns (``to_bf16_bits``) so the oracle reads them exactly.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest even) and return the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    nan = np.isnan(x)
    rounded = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    rounded[nan] = 0x7FC0
    return rounded


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def read_worked_examples():
    """Parse tests/golden/worked_examples.txt into a list of dicts."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "worked_examples.txt")) as f:
        for line in f:
            line = line.rstrip("\n")
            if line.startswith("#"):
                continue
            if not line.strip():
                if cur:
                    cases.append(cur)
                cur = None
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"case": rest}
            elif key in ("source",):
                cur[key] = rest
            elif key in ("expect_accepted",):
                cur[key] = int(rest)
            else:
                cur[key] = rest.split()
    if cur:
        cases.append(cur)
    return cases


def read_kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            left, right = line.split("|")
            inp = [int(t, 16) for t in left.split()]
            out = [int(t, 16) for t in right.split()]
            rows.append((inp[:4], inp[4:6], out))
    return rows


def worked_case_batch(case, vocab, copies, temperature, dtype="f32", seed=0):
    """A batch of `copies` identical requests realising one worked example.

    Accepted positions: the target row is one-hot on the draft token (logit 0,
    -inf elsewhere), so p(y) = 1 >= q(y) and every sampling round accepts it;
    for a greedy round it is the argmax.  The rejected position: the target
    row is one-hot on the correction token, so p(y) = 0 (always rejected) and
    the positive residual [p - q]_+ lives on the correction token alone.
    Other rows hold N(0, 1) logits.
    """
    names = case["vocab"]
    ids = {n: i for i, n in enumerate(names)}
    assert vocab >= len(names)
    draft_ids = [ids[n] for n in case["draft"]]
    target_ids = [ids[n] for n in case["target"]]
    k = len(draft_ids)
    rng = np.random.default_rng(seed)
    tgt = rng.normal(size=(k + 1, vocab)).astype(np.float32)
    drf = rng.normal(size=(k, vocab)).astype(np.float32)
    for i, t in enumerate(target_ids):
        tgt[i, :] = -np.inf
        tgt[i, t] = 0.0
    if dtype == "bf16":
        tgt_b, drf_b = to_bf16_bits(tgt), to_bf16_bits(drf)
    else:
        tgt_b, drf_b = tgt, drf
    target = np.concatenate([tgt_b] * copies)
    draft = np.concatenate([drf_b] * copies)
    tokens = np.array(draft_ids * copies, dtype=np.int32)
    num_draft = np.full(copies, k, dtype=np.int32)
    temp = np.full(copies, temperature, dtype=np.float32)
    expect = [ids[n] for n in case["expect_commit"]]
    return dict(target=target, draft=draft, tokens=tokens, num_draft=num_draft,
                temperature=temp, max_k=k), expect


def random_batch(num_draft, temperature, vocab, sigma_t=2.0, sigma_d=1.0, dtype="f32",
                 seed=0, sample_tokens=True):
    """Gaussian target/draft logits; draft tokens drawn from softmax(draft/T) by numpy
    (the simulated drafter; greedy requests take the draft argmax)."""
    rng = np.random.default_rng(seed)
    num_draft = np.asarray(num_draft, dtype=np.int32)
    temperature = np.asarray(temperature, dtype=np.float32)
    nt = int((num_draft + 1).sum())
    nd = int(num_draft.sum())
    tgt = (rng.normal(size=(nt, vocab)) * sigma_t).astype(np.float32)
    t_off = np.concatenate([[0], np.cumsum(num_draft + 1)])
    src = np.concatenate([np.arange(t_off[r], t_off[r] + num_draft[r])
                          for r in range(len(num_draft))]) if nd else np.zeros(0, np.int64)
    drf = (tgt[src] + rng.normal(size=(nd, vocab)) * sigma_d).astype(np.float32)
    if dtype == "bf16":
        tgt_s, drf_s = to_bf16_bits(tgt), to_bf16_bits(drf)
        drf_f = bf16_bits_to_f32(drf_s)
    else:
        tgt_s, drf_s, drf_f = tgt, drf, drf
    tokens = np.zeros(nd, dtype=np.int32)
    req_of = np.repeat(np.arange(len(num_draft)), num_draft)
    for d in range(nd):
        t = temperature[req_of[d]]
        row = drf_f[d].astype(np.float64)
        if t > 0 and sample_tokens:
            z = row / t
            z = np.exp(z - z.max())
            tokens[d] = rng.choice(vocab, p=z / z.sum())
        else:
            tokens[d] = int(np.argmax(row))
    return dict(target=tgt_s, draft=drf_s, tokens=tokens, num_draft=num_draft,
                temperature=temperature, max_k=int(num_draft.max()) if len(num_draft) else 0)
