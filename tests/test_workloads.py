"""The synthetic input recipe (CPU, reduced sizes): what the design notes state
about the seeded workloads holds for the generator."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_10_gb300 import workloads as W


def _small(name, batch=16, vocab=4096):
    return W.make_batch(name, device="cpu", batch=batch, vocab=vocab)


@pytest.mark.parametrize("name", list(W.SPECS))
def test_seeded_and_laid_out(name):
    a, b = _small(name), _small(name)
    for x, y in ((a.target, b.target), (a.draft, b.draft), (a.tokens, b.tokens),
                 (a.num_draft, b.num_draft), (a.temperature, b.temperature)):
        assert torch.equal(x, y)
    k = a.num_draft.numpy().astype(np.int64)
    assert a.target.shape == (int((k + 1).sum()), 4096)
    assert a.draft.shape == (int(k.sum()), 4096)
    assert a.tokens.shape == (int(k.sum()),)
    tok = a.tokens.numpy()
    assert (tok >= 0).all() and (tok < 4096).all()
    want = torch.bfloat16 if W.SPECS[name].dtype == "bf16" else torch.float32
    assert a.target.dtype == want and a.draft.dtype == want
    allowed = {np.float32(t) for t in W.SPECS[name].temps} | {np.float32(0.0)}
    assert set(np.unique(a.temperature.numpy()).tolist()) <= {float(t) for t in allowed}


def _draft_minus_target(b):
    k = b.num_draft.numpy().astype(np.int64)
    t_off = np.concatenate([[0], np.cumsum(k + 1)])
    src = np.concatenate([t_off[r] + np.arange(k[r]) for r in range(len(k))])
    return (b.draft.float() - b.target.float()[src]).numpy()


@pytest.mark.parametrize("name", list(W.SPECS))
def test_noise_levels(name):
    s = W.SPECS[name]
    b = _small(name)
    t = b.target.float().numpy()
    if not s.peaks:
        assert abs(t.std() - s.sigma_t) < 0.05 * s.sigma_t
    # the draft is the target plus N(0, sigma_d^2), both rounded to the dtype
    d = _draft_minus_target(b)
    assert abs(d.std() - s.sigma_d) < 0.05 * s.sigma_d + (0.02 if s.dtype == "bf16" else 0)
    assert abs(d.mean()) < 0.02


def test_w4_rows_carry_64_raised_ids():
    s = W.SPECS["w4_v262144_bf16"]
    b = _small("w4_v262144_bf16")
    t = b.target.float().numpy()
    # N(0, 4^2) alone puts about 3e-5 of the logits above 4 sigma = 16; with 64 ids
    # per row raised by +8 about 64 * 0.023 per row land there
    per_row = (t > 4 * s.sigma_t).sum(axis=1)
    expected = s.peaks * 0.0228
    assert abs(per_row.mean() - expected) < 0.35 * expected
    assert per_row.mean() > 10 * t.shape[1] * 3.2e-5


def test_w3_draft_counts_are_ragged_in_1_to_6():
    b = _small("w3_v151936_bf16", batch=400, vocab=64)
    k = b.num_draft.numpy()
    assert k.min() == 1 and k.max() == 6
    counts = np.bincount(k, minlength=7)[1:]
    assert (np.abs(counts - 400 / 6) < 4 * np.sqrt(400 / 6)).all()


def test_w2_temperatures_and_greedy_tokens():
    b = _small("w2_v128256_bf16", batch=300, vocab=256)
    temp = b.temperature.numpy()
    counts = {t: int((temp == np.float32(t)).sum()) for t in (0.0, 0.7, 1.0)}
    assert sum(counts.values()) == 300 and min(counts.values()) > 60
    k = b.num_draft.numpy().astype(np.int64)
    req = np.repeat(np.arange(300), k)
    greedy = temp[req] == 0
    arg = b.draft.float().numpy().argmax(axis=1)
    assert (b.tokens.numpy()[greedy] == arg[greedy]).all()


def test_w0_appends_greedy_copies():
    b = W.make_batch("w0_v1024_f32", device="cpu")
    B = b.batch // 2
    t = b.temperature.numpy()
    assert (t[:B] == 1.0).all() and (t[B:] == 0.0).all()
    half_t = b.target.shape[0] // 2
    half_d = b.draft.shape[0] // 2
    assert torch.equal(b.target[:half_t], b.target[half_t:])
    assert torch.equal(b.draft[:half_d], b.draft[half_d:])
    assert torch.equal(b.tokens[:half_d], b.tokens[half_d:])
