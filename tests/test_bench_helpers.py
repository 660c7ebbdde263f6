"""bench.py's host helpers on the CPU: the NVML clock sampler against a fake
library (read-only queries), and the draft-token redraw of truncated runs."""
import ctypes
import types

import numpy as np
import torch

import bench


class FakeNvml:
    """The few read-only NVML calls the sampler makes, with fixed answers."""

    def __init__(self, mhz, max_mhz, reasons):
        self.mhz, self.max_mhz, self.reasons = mhz, max_mhz, reasons
        self.calls = []

    def nvmlDeviceGetClockInfo(self, dev, which, out):
        self.calls.append(("clock", which))
        ctypes.cast(out, ctypes.POINTER(ctypes.c_uint))[0] = self.mhz
        return 0

    def nvmlDeviceGetMaxClockInfo(self, dev, which, out):
        ctypes.cast(out, ctypes.POINTER(ctypes.c_uint))[0] = self.max_mhz
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, dev, out):
        ctypes.cast(out, ctypes.POINTER(ctypes.c_ulonglong))[0] = self.reasons
        return 0


def fake_sampler(mhz, max_mhz, reasons):
    s = bench.NvmlClocks.__new__(bench.NvmlClocks)
    s.ct = ctypes
    s.lib = FakeNvml(mhz, max_mhz, reasons)
    s.dev = ctypes.c_void_p()
    s.reasons_fn = s.lib.nvmlDeviceGetCurrentClocksEventReasons
    s.samples = []
    s.running = False
    return s


def test_nvml_sampler_reports_median_clock_and_reasons():
    s = fake_sampler(1980, 2070, 0x4 | 0x40)   # sw power cap, hw thermal slowdown
    s.start()
    import time
    time.sleep(0.02)
    info = s.stop()
    assert info["samples"] >= 1
    assert info["sm_mhz"] == 1980 and info["sm_max_mhz"] == 2070
    assert info["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert all(c == ("clock", 1) for c in s.lib.calls)          # the SM clock only


def test_nvml_sampler_without_reasons_and_without_samples():
    s = fake_sampler(2070, 2070, 0x1)   # GPU idle: not a reason the bench reports
    s.samples = [s._one()]
    s.running = False
    s.thread = types.SimpleNamespace(join=lambda timeout=None: None)
    assert s.stop()["reasons"] == []
    s.samples = []
    assert s.stop() is None


def test_clock_sampler_falls_back_without_nvml():
    c = bench.ClockSampler(0)
    if c.nvml is None:                  # no GPU driver here: the nvidia-smi path
        c.mark("start")
        c.mark("stop")
        assert c.stop() is None


def _fake_batch(rows, V, num_draft, temps, seed=0):
    g = torch.Generator().manual_seed(seed)
    draft = (torch.randn(rows, V, generator=g) * 3).to(torch.bfloat16)
    return types.SimpleNamespace(draft=draft, num_draft=torch.tensor(num_draft, dtype=torch.int32),
                                 temperature=torch.tensor(temps, dtype=torch.float32),
                                 tokens=torch.full((rows,), -7, dtype=torch.int32),
                                 total_draft=rows)


def test_truncated_tokens_lie_in_the_truncated_support():
    b = _fake_batch(6, 500, [2, 3, 1], [1.0, 0.0, 0.7])
    bench.truncated_draft_tokens(b, 5, 1.0, seed=3, chunk=4)
    x = b.draft.float()
    row_t = np.repeat([1.0, 0.0, 0.7], [2, 3, 1])
    for i in range(6):
        if row_t[i] == 0:
            assert int(b.tokens[i]) == -7                   # greedy rows keep their tokens
        else:
            kth = torch.topk(x[i], 5).values[-1]
            assert x[i, int(b.tokens[i])] >= kth            # among the 5 largest logits


def test_truncated_tokens_top_p_keeps_the_nucleus():
    b = _fake_batch(8, 300, [8], [1.0])
    bench.truncated_draft_tokens(b, 0, 0.5, seed=4)
    for i in range(8):
        x = b.draft[i].float().double()
        p = torch.softmax(x, 0)
        tok = int(b.tokens[i])
        # the mass of the logits strictly larger than the token's is below 0.5
        assert p[x > x[tok]].sum() < 0.5
