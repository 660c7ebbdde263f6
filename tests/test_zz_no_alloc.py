"""specverify_run_static (no handle, no allocation) against the handle entry point.

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
                                                        verify_static)
from speculative_decoding_verification_10_gb300 import _lib
from tests import cases, parity

pytestmark = pytest.mark.gpu


def _batch(B, seed, dtype):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, _lib.STATIC_MAX_K + 1, size=B)
    temp = rng.choice([0.0, 0.7, 1.0], size=B)
    inp = cases.random_batch(k, temp, vocab=4096, sigma_t=2.0, sigma_d=0.7, dtype=dtype,
                             seed=seed)
    return parity.to_torch(inp, "cuda")


def _outputs(B, total, max_k):
    return (torch.empty(B, dtype=torch.int32, device="cuda"),
            torch.empty(B, max_k + 1, dtype=torch.int32, device="cuda"),
            torch.empty(max(total, 1), dtype=torch.uint8, device="cuda"))


def test_static_entry_matches_handle_entry_on_two_calls_in_a_row():
    build.build()
    max_k = _lib.STATIC_MAX_K
    calls = [(_lib.STATIC_MAX_BATCH, 11, "bf16"), (37, 12, "bf16"), (64, 13, "f32")]
    for B, seed, dtype in calls:
        t = _batch(B, seed, dtype)
        total = int(t["tokens"].shape[0])
        with Verifier(B, max_k, 4096, dtype) as v:
            ref = v.run(t["target"], t["draft"], t["tokens"], t["num_draft"],
                        t["temperature"], seed)
            torch.cuda.synchronize()
            assert v.status() == 0
        acc, com, flg = _outputs(B, total, max_k)
        before = torch.cuda.memory_allocated()
        verify_static(t["target"], t["draft"], t["tokens"], t["num_draft"], t["temperature"],
                      seed, max_k, acc, com, flg)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        assert torch.equal(acc, ref.accepted_len), (B, seed)
        assert torch.equal(com, ref.committed), (B, seed)
        assert torch.equal(flg[:total], ref.flags), (B, seed)
        assert (acc >= 0).all()


def test_static_entry_rejects_a_batch_above_its_limit():
    t = _batch(8, 3, "bf16")
    big = _lib.STATIC_MAX_BATCH + 1
    acc, com, flg = _outputs(big, 8, _lib.STATIC_MAX_K)
    nd = torch.zeros(big, dtype=torch.int32, device="cuda")
    temp = torch.ones(big, dtype=torch.float32, device="cuda")
    tgt = torch.zeros(big, 4096, dtype=torch.bfloat16, device="cuda")
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    with pytest.raises(SpecVerifyError) as e:
        verify_static(tgt, None, empty, nd, temp, 1, _lib.STATIC_MAX_K, acc, com, flg)
    assert e.value.code == _lib.ERR_TOO_LARGE
    del t
