"""GB300 verify step for speculative sampling -- Python binding of libspecverify.

Thin argument marshalling over the C ABI in include/specverify.h: every step
of the verify round runs in the library's CUDA kernels.  PyTorch supplies
device memory and streams only.

    v = Verifier(max_batch=512, max_k=4, vocab=262144, dtype="bf16")
    out = v.run(target, draft, tokens, num_draft, temperature, seed=1)
    out.accepted_len, out.committed, out.flags

Layout: request r has k_r = num_draft[r] draft positions; its k_r+1 target
rows start at row sum_{s<r}(k_s+1) of `target`, its k_r draft rows and draft
tokens at sum_{s<r} k_s.  T = 0 requests are greedy.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import (CREATE_HOST_STAGING, STATUS_BAD_K, STATUS_BAD_TEMP, STATUS_BAD_TOKEN,
                   STATUS_BAD_TOTAL, STATUS_NO_DRAFT, STATUS_NONFINITE)

__all__ = ["Verifier", "VerifyResult", "SpecVerifyError", "verify", "verify_static",
           "AcceptanceCounts", "acceptance_metrics", "TreeVerifier", "TreeResult", "truncate",
           "STATUS_BAD_TOKEN", "STATUS_BAD_K", "STATUS_BAD_TEMP", "STATUS_NONFINITE",
           "STATUS_BAD_TOTAL", "STATUS_NO_DRAFT"]

_DTYPES = {"f32": (_lib.DTYPE_F32, torch.float32), "bf16": (_lib.DTYPE_BF16, torch.bfloat16)}


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {_lib.error_string(code)} ({code})")
        self.code = code


def _check(code: int, what: str):
    if code != _lib.OK:
        raise SpecVerifyError(code, what)


@dataclass
class VerifyResult:
    accepted_len: torch.Tensor          # [B] int32, -1 = skipped
    committed: torch.Tensor             # [B, max_k+1] int32, -1 padded
    flags: torch.Tensor                 # [sum k] uint8
    p_y: torch.Tensor | None = None     # [sum k] float32 (debug)
    q_y: torch.Tensor | None = None
    u: torch.Tensor | None = None
    req_status: torch.Tensor | None = None
    verified_k: torch.Tensor | None = None  # trimmed runs: [B] int32 window verified


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_inputs(target, draft, tokens, num_draft, temperature, torch_dtype, device, vocab):
    """Dtypes, devices, contiguity and shapes of a round's inputs (raises before
    anything reaches the library)."""
    if not isinstance(target, torch.Tensor) or target.dtype != torch_dtype:
        raise TypeError(f"target logits must be a {torch_dtype} tensor")
    if draft is not None and draft.numel() and draft.dtype != torch_dtype:
        raise TypeError(f"draft logits must be {torch_dtype}")
    for name, t, dt in (("draft_tokens", tokens, torch.int32),
                        ("num_draft", num_draft, torch.int32),
                        ("temperature", temperature, torch.float32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}")
    for t in (target, draft, tokens, num_draft, temperature):
        if t is not None and t.numel() and (t.device != device or not t.is_contiguous()):
            raise ValueError("inputs must be contiguous tensors on the handle's device")
    if target.dim() != 2 or target.shape[1] != vocab:
        raise ValueError(f"target logits must be [rows, {vocab}]")
    if tokens.dim() != 1 or num_draft.dim() != 1 or temperature.dim() != 1:
        raise ValueError("draft_tokens, num_draft and temperature must be 1-D")
    batch, total = int(num_draft.shape[0]), int(tokens.shape[0])
    if temperature.shape[0] != batch:
        raise ValueError("temperature must have one entry per request")
    if batch and target.shape[0] < batch + total:
        raise ValueError("target logits need sum(k_r + 1) rows")
    if draft is not None and draft.numel() and (draft.dim() != 2 or draft.shape[1] != vocab
                                                or draft.shape[0] < total):
        raise ValueError(f"draft logits must be [sum(k_r), {vocab}]")


def _check_outputs(accepted_len, committed, flags, batch, total_draft, max_k, device):
    """Outputs must be contiguous int32 / int32 / uint8 tensors on the device,
    at least [batch], [batch, max_k + 1] and [total_draft] long: the kernels
    write that much."""
    for name, t, dt, n in (("accepted_len", accepted_len, torch.int32, batch),
                           ("committed", committed, torch.int32, batch * (max_k + 1)),
                           ("flags", flags, torch.uint8, total_draft)):
        if not isinstance(t, torch.Tensor) or t.dtype != dt:
            raise TypeError(f"{name} must be a {dt} tensor")
        if t.numel() and (t.device != device or not t.is_contiguous()):
            raise ValueError(f"{name} must be contiguous on the inputs' device")
        if t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements, the round writes {n}")
    if committed.dim() != 2 or committed.shape[1] != max_k + 1:
        raise ValueError(f"committed must be [batch, {max_k + 1}]")


def _stream_of(stream, device):
    s = torch.cuda.current_stream(device) if stream is None else stream
    if s.device != device:
        raise ValueError("the stream must belong to the inputs' device")
    return ctypes.c_void_p(s.cuda_stream)


class Verifier:
    """Owns one library handle (scratch memory sized at construction)."""

    def __init__(self, max_batch: int, max_k: int, vocab: int, dtype: str = "bf16",
                 device: int | torch.device | None = None, host_staging: bool = False):
        if dtype not in _DTYPES:
            raise ValueError(f"dtype must be one of {list(_DTYPES)}")
        self.lib = _lib.load()
        if device is None:
            device = torch.cuda.current_device()
        self.device = torch.device("cuda", device if isinstance(device, int) else device.index)
        self.max_batch, self.max_k, self.vocab, self.dtype = max_batch, max_k, vocab, dtype
        self.code, self.torch_dtype = _DTYPES[dtype]
        h = ctypes.c_void_p()
        flags = CREATE_HOST_STAGING if host_staging else 0
        _check(self.lib.specverify_create_ex(ctypes.byref(h), self.device.index, max_batch,
                                             max_k, vocab, self.code, flags),
               "specverify_create")
        self._h = h

    # -- helpers --------------------------------------------------------------
    def _stream(self, stream):
        return _stream_of(stream, self.device)

    def _check_inputs(self, target, draft, tokens, num_draft, temperature):
        _check_inputs(target, draft, tokens, num_draft, temperature, self.torch_dtype,
                      self.device, self.vocab)

    def outputs(self, batch: int, total_draft: int, debug: bool = False) -> VerifyResult:
        """Allocate output tensors for a batch (run() does this when none are given)."""
        dev = self.device
        res = VerifyResult(torch.empty(batch, dtype=torch.int32, device=dev),
                           torch.empty(batch, self.max_k + 1, dtype=torch.int32, device=dev),
                           torch.empty(total_draft, dtype=torch.uint8, device=dev))
        if debug:
            res.p_y = torch.empty(total_draft, dtype=torch.float32, device=dev)
            res.q_y = torch.empty(total_draft, dtype=torch.float32, device=dev)
            res.u = torch.empty(total_draft, dtype=torch.float32, device=dev)
            res.req_status = torch.empty(batch, dtype=torch.int32, device=dev)
        return res

    # -- entry points ------------------------------------------------------------
    def run(self, target, draft, tokens, num_draft, temperature, seed: int, *,
            total_draft: int | None = None, out: VerifyResult | None = None,
            request_ids=None, debug: bool = False, stream=None) -> VerifyResult:
        """One verify round on device tensors (asynchronous on the current stream)."""
        self._check_inputs(target, draft, tokens, num_draft, temperature)
        batch = int(num_draft.shape[0])
        if total_draft is None:
            total_draft = int(tokens.shape[0])
        if out is None:
            out = self.outputs(batch, total_draft, debug=debug)
        _check_outputs(out.accepted_len, out.committed, out.flags, batch, total_draft,
                       self.max_k, self.device)
        if request_ids is not None and (request_ids.dtype != torch.int64
                                        or request_ids.device != self.device):
            raise TypeError("request_ids must be int64 on the handle's device")
        d = draft if (draft is not None and draft.numel()) else None
        code = self.lib.specverify_run_ex(
            self._h, _ptr(target), _ptr(d), _ptr(tokens), _ptr(num_draft), _ptr(temperature),
            int(seed) & (2**64 - 1), batch, int(total_draft), _ptr(out.accepted_len),
            _ptr(out.committed), _ptr(out.flags), _ptr(request_ids), _ptr(out.p_y),
            _ptr(out.q_y), _ptr(out.u), _ptr(out.req_status), self._stream(stream))
        _check(code, "specverify_run")
        return out

    def run_truncated(self, target, draft, tokens, num_draft, temperature, top_k, top_p,
                      seed: int, *, total_draft: int | None = None,
                      out: VerifyResult | None = None, stream=None) -> VerifyResult:
        """One verify round on top-k / top-p truncated distributions
        (specverify_run_truncated): top_k [B] int32, top_p [B] float32 on the
        handle's device.  No truncated copy is made: the waves mask the rows
        as they load them."""
        self._check_inputs(target, draft, tokens, num_draft, temperature)
        batch = int(num_draft.shape[0])
        for t, dt, name in ((top_k, torch.int32, "top_k"), (top_p, torch.float32, "top_p")):
            if t.dtype != dt or t.device != self.device or t.numel() < batch:
                raise TypeError(f"{name} must be [batch] {dt} on the handle's device")
        if total_draft is None:
            total_draft = int(tokens.shape[0])
        if out is None:
            out = self.outputs(batch, total_draft)
        _check_outputs(out.accepted_len, out.committed, out.flags, batch, total_draft,
                       self.max_k, self.device)
        d = draft if (draft is not None and draft.numel()) else None
        code = self.lib.specverify_run_truncated(
            self._h, _ptr(target), _ptr(d), _ptr(tokens), _ptr(num_draft), _ptr(temperature),
            _ptr(top_k), _ptr(top_p), int(seed) & (2**64 - 1), batch, int(total_draft),
            _ptr(out.accepted_len), _ptr(out.committed), _ptr(out.flags), self._stream(stream))
        _check(code, "specverify_run_truncated")
        return out

    def run_trimmed(self, target, draft, tokens, window, confidence, cost, temperature,
                    seed: int, *, total_draft: int | None = None, debug: bool = False,
                    stream=None) -> VerifyResult:
        """Verify the windows trimmed from draft confidences (specverify_run_trimmed):
        `window` [B] is the layout of the inputs, `confidence` [sum window] float32
        the c_i, `cost` [B] float32 the cost of a verified position.  The result
        also carries verified_k [B] (the window each request verified)."""
        self._check_inputs(target, draft, tokens, window, temperature)
        batch = int(window.shape[0])
        if total_draft is None:
            total_draft = int(tokens.shape[0])
        out = self.outputs(batch, total_draft, debug=debug)
        out.verified_k = torch.empty(batch, dtype=torch.int32, device=self.device)
        d = draft if (draft is not None and draft.numel()) else None
        c = confidence if confidence.numel() else None
        code = self.lib.specverify_run_trimmed(
            self._h, _ptr(target), _ptr(d), _ptr(tokens), _ptr(window), _ptr(c), _ptr(cost),
            _ptr(temperature), int(seed) & (2**64 - 1), batch, int(total_draft),
            _ptr(out.verified_k), _ptr(out.accepted_len), _ptr(out.committed), _ptr(out.flags),
            _ptr(out.p_y), _ptr(out.q_y), _ptr(out.u), _ptr(out.req_status), self._stream(stream))
        _check(code, "specverify_run_trimmed")
        return out

    def run_host(self, target, draft, tokens, num_draft, temperature, seed: int,
                 accepted_len, committed, flags, *, stream=None) -> None:
        """One verify round on host (ideally pinned) CPU tensors; blocks until done."""
        batch = int(num_draft.shape[0])
        total_draft = int(tokens.shape[0])
        for t in (target, tokens, num_draft, temperature, accepted_len, committed, flags):
            if t.device.type != "cpu" or not t.is_contiguous():
                raise ValueError("run_host takes contiguous CPU tensors")
        d = draft if (draft is not None and draft.numel()) else None
        code = self.lib.specverify_run_host(
            self._h, _ptr(target), _ptr(d), _ptr(tokens), _ptr(num_draft), _ptr(temperature),
            int(seed) & (2**64 - 1), batch, total_draft, _ptr(accepted_len), _ptr(committed),
            _ptr(flags), self._stream(stream))
        _check(code, "specverify_run_host")

    def set_timing_events(self, starts, stops) -> None:
        """Record the given torch.cuda.Event pairs around the row-pass kernel of the
        following runs (run i uses pair i % n); pass empty lists to stop."""
        n = len(starts)
        arr_s = (ctypes.c_void_p * max(n, 1))(*[ctypes.c_void_p(e.cuda_event) for e in starts])
        arr_e = (ctypes.c_void_p * max(n, 1))(*[ctypes.c_void_p(e.cuda_event) for e in stops])
        _check(self.lib.specverify_set_timing_events(self._h, n, arr_s, arr_e),
               "specverify_set_timing_events")

    def launches_per_run(self, batch: int) -> int:
        """Kernel launches a run of `batch` requests makes (the plan and the waves)."""
        n = ctypes.c_int()
        _check(self.lib.specverify_launches_per_run(self._h, batch, ctypes.byref(n)),
               "specverify_launches_per_run")
        return int(n.value)

    def set_schedule(self, schedule: str):
        """'auto' or 'waves' (see specverify_set_schedule)."""
        code = {"auto": _lib.SCHEDULE_AUTO, "waves": _lib.SCHEDULE_WAVES}[schedule]
        _check(self.lib.specverify_set_schedule(self._h, code), "specverify_set_schedule")

    def set_host_reads(self, mode: str):
        """'auto' (read pinned, mapped host logits in place) or 'stage' (copy them
        in first): how run_host gets the logits to the GPU."""
        code = {"auto": _lib.HOST_READS_AUTO, "stage": _lib.HOST_READS_STAGE}[mode]
        _check(self.lib.specverify_set_host_reads(self._h, code), "specverify_set_host_reads")

    def wave_depth(self, batch: int) -> int:
        """Positions per wave launch a run of `batch` requests uses."""
        out = ctypes.c_int(0)
        _check(self.lib.specverify_wave_depth(self._h, batch, ctypes.byref(out)),
               "specverify_wave_depth")
        return out.value

    def last_host_reads(self) -> int:
        """1 if the last run_host read the logits in place, 0 if it staged them,
        -1 before the first."""
        out = ctypes.c_int(0)
        _check(self.lib.specverify_last_host_reads(self._h, ctypes.byref(out)),
               "specverify_last_host_reads")
        return out.value

    def debug_set_epoch(self, epoch: int) -> None:
        """Test aid: the round tag of the last round (see specverify_debug_set_epoch);
        the next round is tagged epoch + 1, wrapping to a cleared restart."""
        _check(self.lib.specverify_debug_set_epoch(self._h, int(epoch) & 0xffffffff),
               "specverify_debug_set_epoch")

    def set_depth(self, depth: int):
        """Positions per wave launch: 1 .. max_k + 1, or 0 to choose per run."""
        _check(self.lib.specverify_set_depth(self._h, depth), "specverify_set_depth")

    def status(self) -> int:
        """Status bits of the last run (waits for its stream)."""
        st = ctypes.c_int32()
        _check(self.lib.specverify_status(self._h, ctypes.byref(st)), "specverify_status")
        return int(st.value)

    def close(self):
        if getattr(self, "_h", None) is not None:
            _check(self.lib.specverify_destroy(self._h), "specverify_destroy")
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def verify_static(target, draft, tokens, num_draft, temperature, seed: int, max_k: int,
                  accepted_len, committed, flags, stream=None) -> None:
    """One verify round through specverify_run_static: no handle and no device
    allocation (scratch is the library's static arena; batch <= 256, max_k <= 7),
    for callers that may not allocate device memory, such as a server that has
    reserved the GPU's memory for its own pool.  Outputs go to the caller's
    tensors: accepted_len [B] int32, committed [B, max_k + 1] int32, flags
    [sum k] uint8.  The first call on a device sets the arena up (takes its
    address, clears it): make it before any stream capture begins.  Calls that
    overlap in time race on the arena: keep them on one stream."""
    lib = _lib.load()
    if not isinstance(target, torch.Tensor) or target.dtype not in (torch.bfloat16,
                                                                      torch.float32):
        raise TypeError("target logits must be a bfloat16 or float32 tensor")
    dtype = "bf16" if target.dtype == torch.bfloat16 else "f32"
    code_dtype, torch_dtype = _DTYPES[dtype]
    dev = target.device
    if dev.type != "cuda":
        raise ValueError("verify_static takes CUDA tensors")
    if target.dim() != 2:
        raise ValueError("target logits must be [rows, vocab]")
    _check_inputs(target, draft, tokens, num_draft, temperature, torch_dtype, dev,
                  int(target.shape[1]))
    _check_outputs(accepted_len, committed, flags, int(num_draft.shape[0]),
                   int(tokens.shape[0]), int(max_k), dev)
    s = _stream_of(stream, dev)
    d = draft if (draft is not None and draft.numel()) else None
    code = lib.specverify_run_static(
        dev.index, int(max_k), int(target.shape[1]), code_dtype, _ptr(target), _ptr(d),
        _ptr(tokens), _ptr(num_draft), _ptr(temperature), int(seed) & (2**64 - 1),
        int(num_draft.shape[0]), int(tokens.shape[0]), _ptr(accepted_len), _ptr(committed),
        _ptr(flags), s)
    _check(code, "specverify_run_static")


def static_debug_set_epoch(device: int, epoch: int) -> None:
    """Test aid: the round tag of the static arena on `device` (see
    specverify_static_debug_set_epoch); needs one verify_static call first."""
    _check(_lib.load().specverify_static_debug_set_epoch(int(device), int(epoch) & 0xffffffff),
           "specverify_static_debug_set_epoch")


def verify(target, draft, tokens, num_draft, temperature, seed: int, max_k: int | None = None,
           request_ids=None, debug: bool = False) -> VerifyResult:
    """One-shot verify round (makes a handle sized for this batch)."""
    batch = int(num_draft.shape[0])
    if max_k is None:
        max_k = int(num_draft.max().item()) if batch else 0
    dtype = "bf16" if target.dtype == torch.bfloat16 else "f32"
    with Verifier(max(batch, 1), max_k, int(target.shape[1]), dtype,
                  device=target.device.index) as v:
        out = v.run(target, draft, tokens, num_draft, temperature, seed,
                    request_ids=request_ids, debug=debug)
        torch.cuda.current_stream(v.device).synchronize()
        return out


@dataclass
class AcceptanceCounts:
    """Running acceptance counts on the device (see specverify_metrics):
    hist [max_k + 2], proposed [max_k], accepted [max_k] (uint64 as int64
    tensors), and the summary written by the last call: [MAL, acceptance rate,
    per-position rates (max_k), rounds, skipped] as float64."""
    max_k: int
    hist: torch.Tensor
    proposed: torch.Tensor
    accepted: torch.Tensor
    summary: torch.Tensor

    @classmethod
    def zeros(cls, max_k: int, device) -> "AcceptanceCounts":
        z = lambda n: torch.zeros(n, dtype=torch.int64, device=device)
        return cls(max_k, z(max_k + 2), z(max(max_k, 1)), z(max(max_k, 1)),
                   torch.full((max_k + 4,), float("nan"), dtype=torch.float64, device=device))

    def as_dict(self) -> dict:
        s = self.summary.cpu().tolist()
        k = self.max_k
        return {"mal": s[0], "acceptance_rate": s[1], "per_position": s[2:2 + k],
                "rounds": int(s[2 + k]), "skipped": int(s[3 + k])}


def acceptance_metrics(accepted_len, num_draft, max_k: int, counts: AcceptanceCounts | None = None,
                       stream=None) -> AcceptanceCounts:
    """Adds one batch of round outputs (device int32 tensors) to `counts` (new
    zero counts if None) and writes their summary, asynchronously on `stream`."""
    lib = _lib.load()
    dev = accepted_len.device
    if counts is None:
        counts = AcceptanceCounts.zeros(max_k, dev)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    code = lib.specverify_metrics(_ptr(accepted_len), _ptr(num_draft), int(accepted_len.shape[0]),
                                  int(max_k), _ptr(counts.hist), _ptr(counts.proposed),
                                  _ptr(counts.accepted), _ptr(counts.summary),
                                  ctypes.c_void_p(s.cuda_stream))
    _check(code, "specverify_metrics")
    return counts


@dataclass
class TreeResult:
    accepted_len: torch.Tensor   # [B] int32, -1 = skipped
    path: torch.Tensor           # [B, max_nodes] int32 accepted node indices, -1 after
    committed: torch.Tensor      # [B, max_nodes + 1] int32 accepted tokens then the bonus
    req_status: torch.Tensor     # [B] int32


class TreeVerifier:
    """Greedy verification of drafted token trees (one library tree handle)."""

    def __init__(self, max_batch: int, max_nodes: int, vocab: int, dtype: str = "bf16",
                 device: int | None = None):
        self.lib = _lib.load()
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.max_batch, self.max_nodes, self.vocab, self.dtype = max_batch, max_nodes, vocab, dtype
        h = ctypes.c_void_p()
        _check(self.lib.specverify_tree_create(ctypes.byref(h), self.device, max_batch, max_nodes,
                                               vocab, _DTYPES[dtype][0]), "specverify_tree_create")
        self._h = h

    def run(self, target, num_nodes, parent, tokens, total_nodes: int | None = None,
            stream=None) -> TreeResult:
        """One round on device tensors: target [B + sum n, V], num_nodes [B],
        parent and tokens [sum n] (int32).  Asynchronous on the current stream."""
        B = int(num_nodes.shape[0])
        dev = torch.device("cuda", self.device)
        if total_nodes is None:
            total_nodes = int(tokens.shape[0])
        out = TreeResult(torch.empty(B, dtype=torch.int32, device=dev),
                         torch.empty(B, max(self.max_nodes, 1), dtype=torch.int32, device=dev),
                         torch.empty(B, self.max_nodes + 1, dtype=torch.int32, device=dev),
                         torch.empty(B, dtype=torch.int32, device=dev))
        s = torch.cuda.current_stream(dev) if stream is None else stream
        p = parent if parent.numel() else None
        t = tokens if tokens.numel() else None
        _check(self.lib.specverify_tree_run(self._h, _ptr(target), _ptr(num_nodes), _ptr(p),
                                            _ptr(t), B, int(total_nodes), _ptr(out.accepted_len),
                                            _ptr(out.path), _ptr(out.committed),
                                            _ptr(out.req_status), ctypes.c_void_p(s.cuda_stream)),
               "specverify_tree_run")
        if self.max_nodes == 0:
            out.path = out.path[:, :0]
        return out

    def status(self) -> int:
        st = ctypes.c_int32()
        _check(self.lib.specverify_tree_status(self._h, ctypes.byref(st)), "specverify_tree_status")
        return int(st.value)

    def close(self):
        if getattr(self, "_h", None) is not None:
            _check(self.lib.specverify_tree_destroy(self._h), "specverify_tree_destroy")
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def truncate(target, draft, num_draft, temperature, top_k, top_p, *, out_target=None,
             out_draft=None, status=None, stream=None):
    """Top-k / top-p truncation of every target and draft row (specverify_truncate):
    returns (target_out, draft_out) with -inf where truncated.  top_k [B] int32,
    top_p [B] float32; status (optional [1] int32 device tensor) gets BAD_TRUNC OR-ed."""
    lib = _lib.load()
    dtype = "bf16" if target.dtype == torch.bfloat16 else "f32"
    dev = target.device
    B = int(num_draft.shape[0])
    d = draft if (draft is not None and draft.numel()) else None
    out_target = torch.empty_like(target) if out_target is None else out_target
    if d is not None and out_draft is None:
        out_draft = torch.empty_like(d)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    total = 0 if d is None else int(d.shape[0])
    code = lib.specverify_truncate(_DTYPES[dtype][0], int(target.shape[1]), _ptr(target), _ptr(d),
                                   _ptr(num_draft), _ptr(temperature), _ptr(top_k), _ptr(top_p),
                                   B, total if d is not None else int(target.shape[0]) - B,
                                   _ptr(out_target), _ptr(out_draft if d is not None else None),
                                   _ptr(status), ctypes.c_void_p(s.cuda_stream))
    _check(code, "specverify_truncate")
    return out_target, (out_draft if d is not None else draft)
