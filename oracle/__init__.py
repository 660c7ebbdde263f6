"""CPU oracle for the speculative-sampling verify step (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline / reference leg may import this module.  The CUDA
library and its Python binding never do.

The oracle itself is plain C (``specverify_oracle.c``), single-threaded and in
double precision; this module compiles it with gcc on first use and wraps it
with ctypes on numpy arrays.  bf16 logits are passed as their raw uint16 bit
patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specverify_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libspecverify_oracle.so")

DTYPE_F32 = 0
DTYPE_BF16 = 1

BAD_TOKEN = 1
BAD_K = 2
BAD_TEMP = 4
NONFINITE = 8
BAD_TOTAL = 16
NO_DRAFT = 64

RACE_NONE = 0
RACE_GREEDY = 1
RACE_BONUS = 2
RACE_RESIDUAL = 3
RACE_FALLBACK = 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build (IEEE double, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.orc_philox4x32_10.argtypes = [P, P, P]
        lib.orc_philox4x32_10.restype = None
        lib.orc_random_word.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                        ctypes.c_uint32, ctypes.c_uint32]
        lib.orc_random_word.restype = ctypes.c_uint32
        lib.orc_uniform_accept.argtypes = [ctypes.c_uint32]
        lib.orc_uniform_accept.restype = ctypes.c_double
        lib.orc_exponential.argtypes = [ctypes.c_uint32]
        lib.orc_exponential.restype = ctypes.c_double
        lib.orc_softmax.argtypes = [P, ctypes.c_int, ctypes.c_size_t, ctypes.c_int,
                                    ctypes.c_double, P]
        lib.orc_softmax.restype = None
        lib.orc_argmax.argtypes = [P, ctypes.c_int, ctypes.c_size_t, ctypes.c_int]
        lib.orc_argmax.restype = ctypes.c_int
        lib.orc_verify.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, P, P, P, P, P, P, ctypes.c_uint64,
                                   P, P, P, P, P, P, P, P, P, P, P]
        lib.orc_verify.restype = ctypes.c_uint32
        lib.orc_race_keys.argtypes = [ctypes.c_int, ctypes.c_int, P, P, ctypes.c_float,
                                      ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
                                      ctypes.c_int, P]
        lib.orc_race_keys.restype = ctypes.c_int
        lib.orc_race_weights.argtypes = [P, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                         ctypes.c_int, P]
        lib.orc_race_weights.restype = ctypes.c_int
        lib.orc_metrics.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P, P]
        lib.orc_metrics.restype = None
        lib.orc_tree_greedy.argtypes = [ctypes.c_int] * 5 + [P] * 8
        lib.orc_tree_greedy.restype = ctypes.c_uint32
        lib.orc_trim.argtypes = [ctypes.c_int, P, P, P, P]
        lib.orc_trim.restype = ctypes.c_uint32
        lib.orc_truncate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int] + [P] * 10
        lib.orc_truncate.restype = ctypes.c_uint32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """Return (contiguous array, dtype code) for fp32 or bf16-as-uint16 logits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, DTYPE_F32
    if a.dtype == np.uint16:
        return a, DTYPE_BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


def philox4x32_10(ctr, key):
    """Raw Philox4x32-10 block: ctr is 4 words, key is 2 words; returns 4 words."""
    lib = _load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib.orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def random_word(seed, stream, request, position, v):
    return int(_load().orc_random_word(seed, stream, request, position, v))


def uniform_accept(word):
    return float(_load().orc_uniform_accept(word))


def exponential(word):
    return float(_load().orc_exponential(word))


def softmax(row, temperature):
    """softmax(row / T) of one logit row (fp32 or bf16 bits), in float64."""
    row, dt = _logits(np.asarray(row).reshape(1, -1))
    vocab = row.shape[1]
    out = np.zeros(vocab, dtype=np.float64)
    _load().orc_softmax(_ptr(row), dt, 0, vocab, float(temperature), _ptr(out))
    return out


def argmax(row):
    row, dt = _logits(np.asarray(row).reshape(1, -1))
    return int(_load().orc_argmax(_ptr(row), dt, 0, row.shape[1]))


def verify(target, draft, tokens, num_draft, temperature, seed, max_k,
           request_ids=None, total_draft=None):
    """Run the oracle over a ragged batch.

    target: [sum(k_r+1), V] float32 or uint16 (bf16 bits); draft: [sum(k_r), V] or
    None; tokens: [sum(k_r)] int32; num_draft: [B] int32; temperature: [B] float32.
    Returns a dict of numpy arrays (see orc_verify in specverify_oracle.c).
    """
    lib = _load()
    target, dt = _logits(target)
    vocab = int(target.shape[1]) if target.ndim == 2 else 0
    if draft is not None:
        draft, dt2 = _logits(draft)
        if draft.size and dt2 != dt:
            raise TypeError("target and draft logits must share a dtype")
        if draft.size == 0:
            draft = np.zeros((0, vocab), dtype=target.dtype)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    num_draft = np.ascontiguousarray(num_draft, dtype=np.int32)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    batch = int(num_draft.shape[0])
    if total_draft is None:
        total_draft = int(tokens.shape[0])
    rid = None if request_ids is None else np.ascontiguousarray(request_ids, dtype=np.int64)
    width = max_k + 1
    out = {
        "accepted_len": np.zeros(batch, np.int32),
        "committed": np.zeros((batch, width), np.int32),
        "flags": np.zeros(total_draft, np.uint8),
        "p_y": np.zeros(total_draft, np.float64),
        "q_y": np.zeros(total_draft, np.float64),
        "u": np.zeros(total_draft, np.float64),
        "accept_margin": np.zeros(total_draft, np.float64),
        "race_kind": np.zeros(batch, np.int32),
        "race_pos": np.zeros(batch, np.int32),
        "race_margin": np.zeros(batch, np.float64),
        "req_status": np.zeros(batch, np.int32),
    }
    status = lib.orc_verify(
        dt, vocab, batch, max_k, int(total_draft), _ptr(target),
        None if draft is None else _ptr(draft), _ptr(tokens), _ptr(num_draft),
        _ptr(temperature), _ptr(rid), int(seed) & (2**64 - 1),
        _ptr(out["accepted_len"]), _ptr(out["committed"]), _ptr(out["flags"]),
        _ptr(out["p_y"]), _ptr(out["q_y"]), _ptr(out["u"]), _ptr(out["accept_margin"]),
        _ptr(out["race_kind"]), _ptr(out["race_pos"]), _ptr(out["race_margin"]),
        _ptr(out["req_status"]))
    out["status"] = int(status)
    return out


def race_keys(target_row, draft_row, temperature, seed, request, position, kind):
    """Keys E_v / w_v of one request's correction/bonus draw.

    Returns (winner, keys[V]); keys are +inf where the weight is not positive.
    """
    lib = _load()
    t, dt = _logits(np.asarray(target_row).reshape(1, -1))
    d = None
    if draft_row is not None:
        d, _ = _logits(np.asarray(draft_row).reshape(1, -1))
    vocab = t.shape[1]
    keys = np.zeros(vocab, dtype=np.float64)
    winner = lib.orc_race_keys(dt, vocab, _ptr(t), _ptr(d), float(temperature),
                               int(seed) & (2**64 - 1), int(request) & (2**64 - 1),
                               int(position), int(kind), _ptr(keys))
    return int(winner), keys


def race_weights(weights, seed, request, position):
    """The exponential race over explicit float64 weights: (winner, keys[V])."""
    lib = _load()
    w = np.ascontiguousarray(weights, dtype=np.float64)
    vocab = len(w)
    keys = np.zeros(vocab, dtype=np.float64)
    winner = lib.orc_race_weights(_ptr(w), vocab, int(seed) & (2**64 - 1),
                                  int(request) & (2**64 - 1), int(position), _ptr(keys))
    return int(winner), keys


def metrics(accepted_len, num_draft, max_k, hist=None, proposed=None, accepted=None):
    """Add a batch of round outputs to acceptance counts (see orc_metrics).

    Returns (hist [max_k + 2], proposed [max_k], accepted [max_k]) as uint64."""
    lib = _load()
    a = np.ascontiguousarray(accepted_len, dtype=np.int32)
    k = np.ascontiguousarray(num_draft, dtype=np.int32)
    hist = np.zeros(max_k + 2, np.uint64) if hist is None else hist
    proposed = np.zeros(max(max_k, 1), np.uint64) if proposed is None else proposed
    accepted = np.zeros(max(max_k, 1), np.uint64) if accepted is None else accepted
    lib.orc_metrics(len(a), max_k, _ptr(a), _ptr(k), _ptr(hist), _ptr(proposed), _ptr(accepted))
    return hist, proposed, accepted


def summarize(hist, proposed, accepted):
    """The [AMD] signals from acceptance counts: mean accepted length MAL (the
    round's committed tokens, the target's own token included), the overall
    acceptance rate and the per-position rates."""
    hist = np.asarray(hist, dtype=np.float64)
    proposed = np.asarray(proposed, dtype=np.float64)
    accepted = np.asarray(accepted, dtype=np.float64)
    rounds = hist[:-1].sum()
    mal = 1.0 + (np.arange(len(hist) - 1) * hist[:-1]).sum() / rounds if rounds else float("nan")
    with np.errstate(invalid="ignore", divide="ignore"):
        per_pos = accepted / proposed
    overall = accepted.sum() / proposed.sum() if proposed.sum() else float("nan")
    return {"mal": mal, "acceptance_rate": overall, "per_position": per_pos,
            "rounds": int(rounds), "skipped": int(hist[-1])}


BAD_PARENT = 32


def tree_greedy(target, num_nodes, parent, tokens, max_nodes, total_nodes=None):
    """Greedy tree verification (see orc_tree_greedy): returns a dict with
    accepted_len [B], path [B, max_nodes], committed [B, max_nodes + 1],
    req_status [B] and the status bits."""
    lib = _load()
    t, dt = _logits(target)
    n = np.ascontiguousarray(num_nodes, dtype=np.int32)
    par = np.ascontiguousarray(parent, dtype=np.int32)
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    B = len(n)
    total = int(n.astype(np.int64).sum()) if total_nodes is None else int(total_nodes)
    acc = np.empty(B, np.int32)
    path = np.empty((B, max(max_nodes, 0)), np.int32)
    com = np.empty((B, max_nodes + 1), np.int32)
    rs = np.empty(B, np.int32)
    st = lib.orc_tree_greedy(dt, t.shape[1], B, int(max_nodes), total, _ptr(t), _ptr(n),
                             _ptr(par if par.size else np.zeros(1, np.int32)),
                             _ptr(tok if tok.size else np.zeros(1, np.int32)),
                             _ptr(acc), _ptr(path if path.size else np.zeros(1, np.int32)),
                             _ptr(com), _ptr(rs))
    return {"accepted_len": acc, "path": path, "committed": com, "req_status": rs,
            "status": int(st)}


BAD_CONF = 512


def trim(window, confidence, cost):
    """Trimmed window per request (see orc_trim): returns (k [B] int32, status)."""
    lib = _load()
    w = np.ascontiguousarray(window, dtype=np.int32)
    c = np.ascontiguousarray(confidence, dtype=np.float32)
    lam = np.ascontiguousarray(cost, dtype=np.float32)
    k = np.empty(len(w), np.int32)
    st = lib.orc_trim(len(w), _ptr(w), _ptr(c if c.size else np.zeros(1, np.float32)),
                      _ptr(lam if lam.size else np.zeros(1, np.float32)), _ptr(k))
    return k, int(st)


def verify_trimmed(target, draft, tokens, window, confidence, cost, temperature, seed, max_k,
                   request_ids=None):
    """Verify the trimmed windows of a full-window layout ([SD] section 5: compact,
    variable-length verification of the selected per-request windows): trim, copy
    the rows of positions 0..k* of every request with valid confidences into a
    compact batch (keeping its request id, so it draws the same numbers), verify
    it, and put the results back in the full layout (flags 0, debug values NaN
    past k*).  A request with invalid confidences or cost is skipped with
    BAD_CONF alone (accepted_len -1)."""
    w = np.ascontiguousarray(window, dtype=np.int32)
    B = len(w)
    k, st = trim(w, confidence, cost)
    t_off = np.concatenate([[0], np.cumsum(w + 1)]).astype(np.int64)
    d_off = np.concatenate([[0], np.cumsum(w)]).astype(np.int64)
    good = np.nonzero(k >= 0)[0]
    kk = k[good].astype(np.int32)
    t_rows = np.concatenate([np.arange(t_off[r], t_off[r] + k[r] + 1) for r in good] +
                            [np.zeros(0, np.int64)]).astype(np.int64)
    d_rows = np.concatenate([np.arange(d_off[r], d_off[r] + k[r]) for r in good] +
                            [np.zeros(0, np.int64)]).astype(np.int64)
    sub_draft = None if draft is None else np.asarray(draft)[d_rows]
    ids = np.arange(B, dtype=np.int64) if request_ids is None else np.asarray(request_ids, np.int64)
    temp = np.asarray(temperature, np.float32)
    c = verify(np.asarray(target)[t_rows], sub_draft, np.asarray(tokens)[d_rows], kk,
               temp[good], seed, max_k, request_ids=ids[good])
    total = int(w.sum())
    out = {"accepted_len": np.full(B, -1, np.int32),
           "committed": np.full((B, max_k + 1), -1, np.int32),
           "race_kind": np.zeros(B, np.int32), "race_pos": np.zeros(B, np.int32),
           "race_margin": np.zeros(B, np.float64),
           "req_status": np.full(B, BAD_CONF, np.int32),
           "verified_k": k, "status": int(c["status"]) | st}
    for key in ("accepted_len", "committed", "race_kind", "race_pos", "race_margin",
                "req_status"):
        out[key][good] = c[key]
    # per-position values in the full layout: flags 0, debug values NaN and no
    # near-threshold margin (+inf) past the trimmed window
    c_off = np.concatenate([[0], np.cumsum(kk)]).astype(np.int64)
    for key, fill, dt in (("flags", 0, np.uint8), ("p_y", np.nan, np.float64),
                          ("q_y", np.nan, np.float64), ("u", np.nan, np.float64),
                          ("accept_margin", np.inf, np.float64)):
        full = np.full(total, fill, dt)
        for i, r in enumerate(good):
            full[d_off[r]:d_off[r] + k[r]] = c[key][c_off[i]:c_off[i + 1]]
        out[key] = full
    return out


BAD_TRUNC = 1024


def truncate(target, draft, num_draft, temperature, top_k, top_p):
    """Top-k / top-p truncation of every row (see orc_truncate).  Returns
    (target_out, draft_out, margin_t, margin_d, status); logits keep their dtype
    (float32, or bf16 bits as uint16) with -inf where truncated."""
    lib = _load()
    t, dt = _logits(target)
    d = None if draft is None else _logits(draft)[0]
    nd = np.ascontiguousarray(num_draft, dtype=np.int32)
    temp = np.ascontiguousarray(temperature, dtype=np.float32)
    k = np.ascontiguousarray(top_k, dtype=np.int32)
    p = np.ascontiguousarray(top_p, dtype=np.float32)
    t_out = np.empty_like(t)
    d_out = None if d is None else np.empty_like(d)
    m_t = np.empty(t.shape[0], np.float64)
    m_d = np.empty(0 if d is None else d.shape[0], np.float64)
    st = lib.orc_truncate(dt, t.shape[1], len(nd), _ptr(nd), _ptr(temp), _ptr(k), _ptr(p),
                          _ptr(t), None if d is None or d.size == 0 else _ptr(d), _ptr(t_out),
                          None if d is None or d.size == 0 else _ptr(d_out), _ptr(m_t),
                          _ptr(m_d) if m_d.size else None)
    return t_out, d_out, m_t, m_d, int(st)
