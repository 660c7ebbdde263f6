"""Device acceptance statistics (specverify_metrics) against the oracle's
counts and summary, element by element."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_10_gb300 import (AcceptanceCounts, Verifier,
                                                        acceptance_metrics, build)
from speculative_decoding_verification_10_gb300 import workloads as W
from tests import parity
from tests.test_oracle_metrics import _rounds_with_rates, _rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _cuda(a):
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32), device="cuda")


def _compare(c, h, p, a, max_k):
    torch.cuda.synchronize()
    assert (c.hist.cpu().numpy().astype(np.uint64) == h).all()
    if max_k:
        assert (c.proposed.cpu().numpy()[:max_k].astype(np.uint64) == p[:max_k]).all()
        assert (c.accepted.cpu().numpy()[:max_k].astype(np.uint64) == a[:max_k]).all()
    want = oracle.summarize(h, p[:max_k] if max_k else np.zeros(0), a[:max_k] if max_k else np.zeros(0))
    got = c.as_dict()
    for key in ("mal", "acceptance_rate"):
        if np.isnan(want[key]):
            assert np.isnan(got[key])
        else:
            assert abs(got[key] - want[key]) <= 1e-12 * max(1.0, abs(want[key]))
    assert np.allclose(np.array(got["per_position"], np.float64), want["per_position"],
                       rtol=1e-12, atol=0, equal_nan=True)
    assert got["rounds"] == want["rounds"] and got["skipped"] == want["skipped"]


@pytest.mark.parametrize("max_k", [0, 1, 4, 7, 31])
@pytest.mark.parametrize("batch", [0, 1, 33, 1024, 5000])
def test_random_batches_and_running_counts(max_k, batch):
    rng = np.random.default_rng(batch * 37 + max_k)
    k = rng.integers(0, max_k + 3, size=batch)                 # some above max_k
    a = np.minimum(rng.integers(-1, max_k + 2, size=batch), k)  # -1 = skipped
    h, p, acc = oracle.metrics(a, k, max_k)
    c = acceptance_metrics(_cuda(a), _cuda(k), max_k)
    _compare(c, h, p, acc, max_k)
    # a second batch adds to the same counts
    k2 = rng.integers(0, max_k + 1, size=batch // 2 + 1)
    a2 = np.minimum(rng.integers(-1, max_k + 1, size=len(k2)), k2)
    h, p, acc = oracle.metrics(a2, k2, max_k, h, p, acc)
    acceptance_metrics(_cuda(a2), _cuda(k2), max_k, counts=c)
    _compare(c, h, p, acc, max_k)


@pytest.mark.parametrize("row", _rows(), ids=lambda r: f"N{r[0]}_MAL{r[1]}")
def test_printed_tables_on_the_device(row):
    n, mal, ar, rates = row
    a, k = _rounds_with_rates(n, rates)
    c = acceptance_metrics(_cuda(a), _cuda(k), n)
    got = c.as_dict()
    assert np.allclose(got["per_position"], np.array(rates) / 100.0, atol=1e-12)
    assert abs(got["mal"] - mal) <= 0.011 + 1e-9
    assert abs(100.0 * got["acceptance_rate"] - ar) <= 0.25 + 1e-9


def test_counts_of_verify_rounds():
    """Statistics of real verify rounds (w1, several seeds) through the device
    path equal the oracle's statistics of the oracle's own rounds."""
    b = W.make_batch("w1_v32000_bf16", device="cpu")
    inp = b.numpy_inputs()
    c = AcceptanceCounts.zeros(b.max_k, "cuda")
    h = p = a = None
    with Verifier(b.batch, b.max_k, b.vocab, b.dtype) as v:
        for seed in (1, 2, 3):
            g = parity.run_gpu(v, inp, seed)
            o = parity.run_oracle(inp, seed)
            assert (g["accepted_len"] == o["accepted_len"]).all()
            acceptance_metrics(_cuda(g["accepted_len"]), _cuda(inp["num_draft"]), b.max_k, counts=c)
            h, p, a = oracle.metrics(o["accepted_len"], inp["num_draft"], b.max_k, h, p, a)
    _compare(c, h, p, a, b.max_k)
    s = c.as_dict()
    assert 1.0 <= s["mal"] <= 1.0 + b.max_k and s["rounds"] == 3 * b.batch


def test_invalid_arguments():
    from speculative_decoding_verification_10_gb300 import SpecVerifyError
    with pytest.raises(SpecVerifyError):
        acceptance_metrics(_cuda([1]), _cuda([1]), 32)
    with pytest.raises(SpecVerifyError):
        acceptance_metrics(_cuda([1]), _cuda([1]), -1)
