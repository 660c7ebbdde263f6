"""specverify_run_static (no handle, no allocation) against the oracle and the
handle entry point.

The static entry point serves callers that may not allocate device memory: a
server that reserves the GPU's memory for its own pool at start-up, where a
cudaMalloc would fail or eat into the pool, or a runtime that forbids
allocation while serving because it can block on device-wide synchronisation.
Its scratch is one static device array shared by every call.

Collected last on purpose: it must pass both alone in a fresh process and after
every other GPU test has used the library in the same process.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_10_gb300 import (SpecVerifyError, Verifier, build,
                                                        static_debug_set_epoch, verify_static)
from speculative_decoding_verification_10_gb300 import _lib
from speculative_decoding_verification_10_gb300 import workloads as W
from tests import cases, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _batch(B, seed, dtype, vocab=4096, max_k=_lib.STATIC_MAX_K):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, max_k + 1, size=B)
    temp = rng.choice([0.0, 0.7, 1.0], size=B)
    inp = cases.random_batch(k, temp, vocab=vocab, sigma_t=2.0, sigma_d=0.7, dtype=dtype,
                             seed=seed)
    inp["max_k"] = max_k
    return inp


def _outputs(B, total, max_k):
    return (torch.empty(B, dtype=torch.int32, device="cuda"),
            torch.empty(B, max_k + 1, dtype=torch.int32, device="cuda"),
            torch.empty(max(total, 1), dtype=torch.uint8, device="cuda"))


def _run_static(inp, seed):
    """One static round; returns the outputs as numpy arrays (parity's layout)."""
    t = parity.to_torch(inp, "cuda")
    B, total = len(inp["num_draft"]), int(inp["num_draft"].sum())
    acc, com, flg = _outputs(B, total, inp["max_k"])
    verify_static(t["target"], t["draft"], t["tokens"], t["num_draft"], t["temperature"],
                  seed, inp["max_k"], acc, com, flg)
    torch.cuda.synchronize()
    return {"accepted_len": acc.cpu().numpy(), "committed": com.cpu().numpy(),
            "flags": flg[:total].cpu().numpy(), "status": 0}


def _exempt(rep):
    return rep["exempt_accept"] + rep["exempt_race"] + rep["exempt_residual_mass"]


def test_static_entry_matches_oracle_and_handle_on_two_calls_in_a_row():
    max_k = _lib.STATIC_MAX_K
    calls = [(_lib.STATIC_MAX_BATCH, 11, "bf16"), (37, 12, "bf16"), (64, 13, "f32")]
    for B, seed, dtype in calls:
        inp = _batch(B, seed, dtype)
        g = _run_static(inp, seed)
        o = parity.run_oracle(inp, seed)
        rep = parity.compare(g, o, inp, seed)
        assert _exempt(rep) <= max(1, B // 100), rep
        assert (g["accepted_len"] >= 0).all()
        t = parity.to_torch(inp, "cuda")
        with Verifier(B, max_k, 4096, dtype) as v:
            ref = v.run(t["target"], t["draft"], t["tokens"], t["num_draft"],
                        t["temperature"], seed)
            torch.cuda.synchronize()
            assert v.status() == 0
        assert (g["accepted_len"] == ref.accepted_len.cpu().numpy()).all(), (B, seed)
        assert (g["committed"] == ref.committed.cpu().numpy()).all(), (B, seed)
        assert (g["flags"] == ref.flags.cpu().numpy()).all(), (B, seed)


@pytest.mark.parametrize("name,batch", [("w2_v128256_bf16", 256), ("w4_v262144_bf16", 256)])
def test_static_entry_multi_wave_windows(name, batch):
    """Windows above 192 MiB: the arena carries the two-position waves (w2, a
    722 MB window) and the one-position waves with their correction lists and
    the 1024-CTA grid cap (w4 at 256 requests, 1.21 GB), checked against the
    oracle request by request."""
    b = W.make_batch(name, device="cuda", batch=batch)
    inp = b.numpy_inputs()
    del b
    for seed in (2, 3):
        g = _run_static(inp, seed)
        o = parity.run_oracle(inp, seed)
        rep = parity.compare(g, o, inp, seed)
        assert rep["sampling"] + rep["greedy"] == batch
        assert _exempt(rep) <= max(1, batch // 100), rep


def test_static_entry_allocates_nothing():
    """Device free memory (cudaMemGetInfo, which sees every allocation of the
    process, the library's included) does not move across a second call of the
    same shape, and neither does torch's own count."""
    inp = _batch(200, 21, "bf16")
    t = parity.to_torch(inp, "cuda")
    B, total = 200, int(inp["num_draft"].sum())
    acc, com, flg = _outputs(B, total, inp["max_k"])
    args = (t["target"], t["draft"], t["tokens"], t["num_draft"], t["temperature"])
    verify_static(*args, 4, inp["max_k"], acc, com, flg)
    torch.cuda.synchronize()
    first = com.clone()
    free0, _ = torch.cuda.mem_get_info()
    torch_bytes = torch.cuda.memory_allocated()
    verify_static(*args, 4, inp["max_k"], acc, com, flg)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == torch_bytes
    assert torch.equal(com, first)


def test_static_entry_across_the_round_tag_wrap():
    """The arena's completion counters are tagged with a 32-bit round number;
    five rounds from 0xfffffffd cross the wrap (the counters are cleared and the
    numbering restarts) and each matches the oracle."""
    b = W.make_batch("w1_v32000_bf16", device="cpu", batch=64)
    inp = b.numpy_inputs()
    _run_static(inp, 1)                       # the arena's set-up on this device
    static_debug_set_epoch(torch.cuda.current_device(), 0xfffffffd)
    for seed in range(1, 6):
        g = _run_static(inp, seed)
        rep = parity.compare(g, parity.run_oracle(inp, seed), inp, seed)
        assert _exempt(rep) <= 1, (seed, rep)


def test_static_entry_rejects_a_batch_above_its_limit():
    big = _lib.STATIC_MAX_BATCH + 1
    acc, com, flg = _outputs(big, 8, _lib.STATIC_MAX_K)
    nd = torch.zeros(big, dtype=torch.int32, device="cuda")
    temp = torch.ones(big, dtype=torch.float32, device="cuda")
    tgt = torch.zeros(big, 4096, dtype=torch.bfloat16, device="cuda")
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    with pytest.raises(SpecVerifyError) as e:
        verify_static(tgt, None, empty, nd, temp, 1, _lib.STATIC_MAX_K, acc, com, flg)
    assert e.value.code == _lib.ERR_TOO_LARGE


def test_static_entry_checks_its_tensors():
    """Wrong dtypes, short outputs and foreign devices are refused before the
    library is called (an undersized output would otherwise be written past)."""
    inp = _batch(16, 4, "bf16")
    t = parity.to_torch(inp, "cuda")
    B, total = 16, int(inp["num_draft"].sum())
    args = (t["target"], t["draft"], t["tokens"], t["num_draft"], t["temperature"])
    acc, com, flg = _outputs(B, total, inp["max_k"])
    with pytest.raises(TypeError):
        verify_static(t["target"], t["draft"], t["tokens"].long(), t["num_draft"],
                      t["temperature"], 1, inp["max_k"], acc, com, flg)
    with pytest.raises(TypeError):
        verify_static(t["target"].half(), t["draft"], t["tokens"], t["num_draft"],
                      t["temperature"], 1, inp["max_k"], acc, com, flg)
    with pytest.raises(ValueError):
        verify_static(*args, 1, inp["max_k"], acc[:B - 1], com, flg)
    with pytest.raises(ValueError):
        verify_static(*args, 1, inp["max_k"], acc, com[:, :inp["max_k"]], flg)
    with pytest.raises(ValueError):
        verify_static(*args, 1, inp["max_k"], acc, com, flg[:total - 1])
    with pytest.raises(ValueError):
        verify_static(*args, 1, inp["max_k"], acc.cpu(), com, flg)
