"""GPU-vs-oracle comparison for verify rounds (test infrastructure).

Tolerance (stated for this verify step): accepted lengths, committed tokens and
flags must match the oracle exactly, except where the oracle's own decision
sits within a relative 1e-5 of its threshold, because fp32 (GPU) and fp64
(oracle) arithmetic may then legitimately disagree:
  * acceptance: |u q(y) - p(y)| <= 1e-5 max(u q(y), p(y)) at a decided position
    (everything downstream in that request is exempt too);
  * race: the GPU's token has an oracle key E_v / w_v <= (1 + 1e-5) x the
    best key of the exponential race;
  * residual draws whose whole positive residual mass is below 1e-5 (the
    fp32 residual is then rounding noise).
Exemptions are counted and returned.  Debug p(y)/q(y) must agree within 1e-5
absolute and the acceptance uniforms exactly, on the decided positions
0..A (both sides report NaN after the first rejection, and for greedy requests).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL_TOL = 1e-5
ABS_PROB_TOL = 1e-5


def to_torch(inp: dict, device) -> dict:
    """numpy inputs (fp32 or bf16 bits) -> contiguous torch tensors on `device`."""
    def logits(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
    out = dict(target=logits(inp["target"]), draft=logits(inp.get("draft")),
               tokens=torch.from_numpy(np.ascontiguousarray(inp["tokens"], np.int32)).to(device),
               num_draft=torch.from_numpy(np.ascontiguousarray(inp["num_draft"], np.int32)).to(device),
               temperature=torch.from_numpy(np.ascontiguousarray(inp["temperature"], np.float32)).to(device))
    rid = inp.get("request_ids")
    out["request_ids"] = None if rid is None else torch.from_numpy(
        np.ascontiguousarray(rid, np.int64)).to(device)
    return out


def run_gpu(verifier, inp: dict, seed: int, device="cuda", debug=True):
    t = to_torch(inp, device)
    res = verifier.run(t["target"], t["draft"], t["tokens"], t["num_draft"], t["temperature"],
                       seed, request_ids=t["request_ids"], debug=debug)
    torch.cuda.synchronize()
    out = {"accepted_len": res.accepted_len.cpu().numpy(), "committed": res.committed.cpu().numpy(),
           "flags": res.flags.cpu().numpy(), "status": verifier.status()}
    if debug:
        out.update(p_y=res.p_y.cpu().numpy(), q_y=res.q_y.cpu().numpy(), u=res.u.cpu().numpy(),
                   req_status=res.req_status.cpu().numpy())
    return out


def run_oracle(inp: dict, seed: int):
    return oracle.verify(inp["target"], inp.get("draft"), inp["tokens"], inp["num_draft"],
                         inp["temperature"], seed, inp["max_k"],
                         request_ids=inp.get("request_ids"))


def compare(gpu: dict, orc: dict, inp: dict, seed: int) -> dict:
    """Element-by-element comparison; raises AssertionError on a real mismatch."""
    k = np.asarray(inp["num_draft"], np.int64)
    temp = np.asarray(inp["temperature"])
    B = len(k)
    d_off = np.concatenate([[0], np.cumsum(k)])
    t_off = np.concatenate([[0], np.cumsum(k + 1)])
    rid = inp.get("request_ids")
    rep = {"requests": B, "exempt_accept": 0, "exempt_race": 0, "exempt_residual_mass": 0,
           "greedy": 0, "sampling": 0, "skipped": 0}
    assert gpu["status"] == orc["status"], (gpu["status"], orc["status"])
    if "req_status" in gpu:
        assert (gpu["req_status"] == orc["req_status"]).all()
    for r in range(B):
        ga, oa = int(gpu["accepted_len"][r]), int(orc["accepted_len"][r])
        gc, oc = gpu["committed"][r], orc["committed"][r]
        fl = slice(d_off[r], d_off[r + 1])
        if oa < 0:
            rep["skipped"] += 1
            assert ga == -1 and (gc == -1).all() and (gpu["flags"][fl] == 0).all(), r
            continue
        if temp[r] == 0:
            rep["greedy"] += 1
            assert ga == oa and (gc == oc).all() and (gpu["flags"][fl] == orc["flags"][fl]).all(), \
                (r, ga, oa, gc, oc)
            if "p_y" in gpu:   # no acceptance test is made for greedy rows: NaN debug values
                assert np.isnan(gpu["p_y"][fl]).all() and np.isnan(gpu["q_y"][fl]).all(), r
                assert np.isnan(gpu["u"][fl]).all(), r
            continue
        rep["sampling"] += 1
        # debug values of the decided positions (NaN after the first rejection)
        if "p_y" in gpu:
            assert np.allclose(gpu["p_y"][fl], orc["p_y"][fl], rtol=0, atol=ABS_PROB_TOL,
                               equal_nan=True), r
            assert np.allclose(gpu["q_y"][fl], orc["q_y"][fl], rtol=0, atol=ABS_PROB_TOL,
                               equal_nan=True), r
            uo = orc["u"][fl].astype(np.float32)
            assert ((gpu["u"][fl] == uo) | (np.isnan(uo) & np.isnan(gpu["u"][fl]))).all(), r
        # decisions up to and including the first rejection
        decided = orc["accept_margin"][fl][:min(oa + 1, k[r])]
        if (np.abs(decided) <= REL_TOL).any():
            rep["exempt_accept"] += 1
            continue
        assert ga == oa, (r, ga, oa, orc["accept_margin"][fl])
        assert (gpu["flags"][fl] == orc["flags"][fl]).all(), r
        assert (gc[:oa] == oc[:oa]).all() and (gc[oa + 1:] == -1).all(), r
        if gc[oa] == oc[oa]:
            continue
        # different correction/bonus token: is the race itself within tolerance?
        kind = int(orc["race_kind"][r])
        j = oa
        trow = inp["target"][t_off[r] + j]
        drow = inp["draft"][d_off[r] + j] if kind == oracle.RACE_RESIDUAL else None
        req = r if rid is None else int(rid[r])
        if kind == oracle.RACE_RESIDUAL:
            p = oracle.softmax(trow, temp[r])
            q = oracle.softmax(inp["draft"][d_off[r] + j], temp[r])
            if np.maximum(p - q, 0).sum() <= REL_TOL:
                rep["exempt_residual_mass"] += 1
                continue
        winner, keys = oracle.race_keys(trow, drow, temp[r], seed, req, j, kind)
        assert winner == oc[oa]
        g = int(gc[oa])
        assert 0 <= g < len(keys), (r, g)
        assert keys[g] <= (1 + REL_TOL) * keys[winner], (r, kind, g, winner, keys[g], keys[winner])
        rep["exempt_race"] += 1
    return rep
