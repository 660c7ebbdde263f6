"""Seeded synthetic verify batches (inputs only).

This module makes the inputs that the CUDA path and the CPU oracle are both
fed: target logits, draft logits, draft tokens, per-request draft counts and
temperatures, in the ragged layout the library takes.  It holds none of the
verify arithmetic: the draft tokens are drawn by torch (``torch.multinomial``
on ``torch.softmax`` of the draft logits, i.e. a simulated drafter), and the
rest is Gaussian noise from a seeded ``torch.Generator``.

Layout (shared by the library and the oracle): request r has k_r draft
positions; its k_r+1 target rows start at row sum_{s<r}(k_s+1) of ``target``;
its k_r draft rows and draft tokens start at sum_{s<r} k_s.

The five named workloads are the synthetic verify batches the library is
measured on (vocabulary sizes of common LLM tokenizers; draft noise levels
spanning the high- and low-acceptance regimes of the per-position acceptance
tables on "Speculative Decoding on AMD GPUs"):

  w0_v1024_f32    : 4 requests at T=1 plus their 4 greedy copies, k=3, V=1024, fp32,
                    target N(0, 2^2), draft = target + N(0, 1^2)
  w1_v32000_bf16  : 64 requests, k=3, V=32000, bf16, N(0, 3^2), sigma_d=0.5, T=0.7
  w2_v128256_bf16 : 256 requests, k=5, V=128256, bf16, N(0, 3^2), sigma_d=1,
                    T uniform over {0 (greedy), 0.7, 1.0}
  w3_v151936_bf16 : 32 requests, ragged k uniform in [1, 6], V=151936, bf16,
                    N(0, 3^2), sigma_d=1.5, T=1
  w4_v262144_bf16 : 512 requests, k=4, V=262144, bf16, N(0, 4^2) with 64 distinct
                    ids per target row raised by +8, sigma_d=1, T=1
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Spec:
    name: str
    batch: int
    k: int                      # fixed draft count (or the upper bound when ragged)
    vocab: int
    dtype: str                  # "f32" or "bf16"
    sigma_t: float
    sigma_d: float
    temps: tuple                # temperatures drawn uniformly per request
    ragged: bool = False        # k_r uniform in [1, k]
    peaks: int = 0              # ids per target row raised by peak_boost
    peak_boost: float = 0.0
    greedy_copies: bool = False  # append a T=0 copy of every request
    gen_seed: int = 1000


SPECS = {
    "w0_v1024_f32": Spec("w0_v1024_f32", 4, 3, 1024, "f32", 2.0, 1.0, (1.0,),
                         greedy_copies=True, gen_seed=1000),
    "w1_v32000_bf16": Spec("w1_v32000_bf16", 64, 3, 32000, "bf16", 3.0, 0.5, (0.7,),
                           gen_seed=1001),
    "w2_v128256_bf16": Spec("w2_v128256_bf16", 256, 5, 128256, "bf16", 3.0, 1.0,
                            (0.0, 0.7, 1.0), gen_seed=1002),
    "w3_v151936_bf16": Spec("w3_v151936_bf16", 32, 6, 151936, "bf16", 3.0, 1.5, (1.0,),
                            ragged=True, gen_seed=1003),
    "w4_v262144_bf16": Spec("w4_v262144_bf16", 512, 4, 262144, "bf16", 4.0, 1.0, (1.0,),
                            peaks=64, peak_boost=8.0, gen_seed=1004),
}

WORKLOAD_ORDER = list(SPECS)


@dataclass
class Batch:
    """One verify batch.  Tensors live on one device; logits are fp32 or bf16."""
    name: str
    target: torch.Tensor        # [sum(k_r+1), V]
    draft: torch.Tensor         # [sum(k_r), V]
    tokens: torch.Tensor        # [sum(k_r)] int32
    num_draft: torch.Tensor     # [B] int32
    temperature: torch.Tensor   # [B] float32
    max_k: int
    vocab: int
    dtype: str
    request_ids: torch.Tensor | None = None   # [B] int64, None = batch index
    info: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.num_draft.shape[0])

    @property
    def total_draft(self) -> int:
        return int(self.tokens.shape[0])

    def to(self, device) -> "Batch":
        rid = None if self.request_ids is None else self.request_ids.to(device)
        return Batch(self.name, self.target.to(device), self.draft.to(device),
                     self.tokens.to(device), self.num_draft.to(device),
                     self.temperature.to(device), self.max_k, self.vocab, self.dtype,
                     rid, dict(self.info))

    def numpy_inputs(self):
        """Host copies for the oracle: logits as float32 or bf16 bit patterns."""
        def rows(t):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy().astype(np.float32, copy=False)
        rid = None if self.request_ids is None else self.request_ids.cpu().numpy()
        return dict(target=rows(self.target), draft=rows(self.draft),
                    tokens=self.tokens.cpu().numpy().astype(np.int32),
                    num_draft=self.num_draft.cpu().numpy().astype(np.int32),
                    temperature=self.temperature.cpu().numpy().astype(np.float32),
                    request_ids=rid, max_k=self.max_k)

    def offsets(self):
        """Host prefix sums (target offsets [B+1], draft offsets [B+1])."""
        k = self.num_draft.cpu().numpy().astype(np.int64)
        t = np.concatenate([[0], np.cumsum(k + 1)])
        d = np.concatenate([[0], np.cumsum(k)])
        return t, d

    def io_bytes(self) -> int:
        """Bytes of the small inputs and the outputs of one round."""
        k = self.num_draft.cpu().numpy().astype(np.int64)
        io_in = 4 * self.batch * 2 + 4 * int(k.sum())
        io_out = 4 * self.batch + 4 * self.batch * (self.max_k + 1) + int(k.sum())
        return io_in + io_out

    def full_window_bytes(self) -> int:
        """Logit bytes of every row of the batch a round could read: 2k+1 rows per
        sampling request, k+1 per greedy one."""
        k = self.num_draft.cpu().numpy().astype(np.int64)
        t = self.temperature.cpu().numpy()
        es = 4 if self.dtype == "f32" else 2
        return int(np.where(t > 0, 2 * k + 1, k + 1).sum()) * self.vocab * es

    def needed_bytes(self, accepted_len) -> int:
        """Logit bytes a round must read given its outcome: positions 0..A of each
        request (target and draft rows when sampling, target rows when greedy), plus
        the bonus row when A = k.  Rows after the first rejection are never needed."""
        k = self.num_draft.cpu().numpy().astype(np.int64)
        t = self.temperature.cpu().numpy()
        A = np.asarray(accepted_len, dtype=np.int64)
        es = 4 if self.dtype == "f32" else 2
        rows = np.where(t > 0, np.where(A < k, 2 * (A + 1), 2 * k + 1), A + 1)
        return int(rows.sum()) * self.vocab * es

    def verified_rows(self) -> int:
        """Target positions verified per batch: sum_r (k_r + 1)."""
        return int(self.num_draft.to(torch.int64).sum().item()) + self.batch


def _to_dtype(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def make_batch(name: str, device="cpu", batch: int | None = None, vocab: int | None = None,
               gen_seed: int | None = None) -> Batch:
    """Generate a named workload (optionally with fewer requests / a smaller vocab)."""
    s = SPECS[name]
    B = s.batch if batch is None else batch
    V = s.vocab if vocab is None else vocab
    g = torch.Generator(device=device)
    g.manual_seed(s.gen_seed if gen_seed is None else gen_seed)

    if s.ragged:
        k = torch.randint(1, s.k + 1, (B,), generator=g, device=device, dtype=torch.int64)
    else:
        k = torch.full((B,), s.k, dtype=torch.int64, device=device)
    temps = torch.tensor(s.temps, dtype=torch.float32, device=device)
    if len(s.temps) > 1:
        temp = temps[torch.randint(0, len(s.temps), (B,), generator=g, device=device)]
    else:
        temp = temps[0].repeat(B)

    nt = int((k + 1).sum().item())
    nd = int(k.sum().item())
    tgt = torch.randn(nt, V, generator=g, device=device, dtype=torch.float32) * s.sigma_t
    if s.peaks:
        keys = torch.rand(nt, V, generator=g, device=device)
        ids = keys.topk(s.peaks, dim=1).indices
        del keys
        tgt.scatter_add_(1, ids, torch.full(ids.shape, s.peak_boost, device=device))
    # draft row (r, i) perturbs target row (r, i)
    t_off = torch.cumsum(k + 1, 0) - (k + 1)
    req_of_draft = torch.repeat_interleave(torch.arange(B, device=device), k)
    d_off = torch.cumsum(k, 0) - k
    pos = torch.arange(nd, device=device) - d_off[req_of_draft]
    src = t_off[req_of_draft] + pos
    drf = tgt[src] + torch.randn(nd, V, generator=g, device=device) * s.sigma_d

    tgt = _to_dtype(tgt, s.dtype)
    drf = _to_dtype(drf, s.dtype)

    # the simulated drafter: sample y ~ softmax(draft / T); greedy drafter = argmax
    tokens = torch.empty(nd, dtype=torch.int64, device=device)
    t_row = temp[req_of_draft]
    samp = t_row > 0
    if samp.any():
        logits = drf[samp].float() / t_row[samp, None]
        probs = torch.softmax(logits, dim=1)
        tokens[samp] = torch.multinomial(probs, 1, generator=g).squeeze(1)
        del logits, probs
    if (~samp).any():
        tokens[~samp] = drf[~samp].float().argmax(dim=1)

    if s.greedy_copies:
        tgt = torch.cat([tgt, tgt])
        drf = torch.cat([drf, drf])
        tokens = torch.cat([tokens, tokens])
        k = torch.cat([k, k])
        temp = torch.cat([temp, torch.zeros_like(temp)])

    return Batch(name, tgt.contiguous(), drf.contiguous(), tokens.to(torch.int32),
                 k.to(torch.int32), temp.contiguous(), int(s.k), V, s.dtype,
                 info={"spec": s})


def subset(b: Batch, requests) -> Batch:
    """The sub-batch holding the given requests, keyed by their original ids."""
    requests = np.asarray(requests, dtype=np.int64)
    t_off, d_off = b.offsets()
    t_rows, d_rows = [], []
    for r in requests:
        t_rows.extend(range(t_off[r], t_off[r + 1]))
        d_rows.extend(range(d_off[r], d_off[r + 1]))
    dev = b.target.device
    ti = torch.tensor(t_rows, dtype=torch.int64, device=dev)
    di = torch.tensor(d_rows, dtype=torch.int64, device=dev)
    ri = torch.tensor(requests, dtype=torch.int64, device=dev)
    base_ids = (ri if b.request_ids is None else b.request_ids[ri])
    return Batch(b.name + "[subset]", b.target[ti].contiguous(), b.draft[di].contiguous(),
                 b.tokens[di].contiguous(), b.num_draft[ri].contiguous(),
                 b.temperature[ri].contiguous(), b.max_k, b.vocab, b.dtype,
                 base_ids.to(torch.int64), dict(b.info))


# ---------------------------------------------------------------------------
# Drafted token trees (greedy tree verification).
#
#   t0_v151936_bf16 : 64 requests, trees of 32 nodes (a DDTree-sized node
#                     budget), V=151936, bf16; node parents drawn so that depth
#                     grows along the node order (each node hangs off one of the
#                     8 nodes before it, or the root); target rows N(0, 3^2);
#                     a node's token is its parent row's argmax with
#                     probability 0.6 (a drafter that often agrees), else a
#                     uniform token.
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class TreeSpec:
    name: str
    batch: int
    nodes: int
    vocab: int
    dtype: str
    sigma_t: float
    p_agree: float
    gen_seed: int


TREE_SPECS = {
    "t0_v151936_bf16": TreeSpec("t0_v151936_bf16", 64, 32, 151936, "bf16", 3.0, 0.6, 1100),
}


@dataclass
class TreeBatch:
    name: str
    target: torch.Tensor      # [B + sum n, V]
    num_nodes: torch.Tensor   # [B] int32
    parent: torch.Tensor      # [sum n] int32
    tokens: torch.Tensor      # [sum n] int32
    max_nodes: int
    vocab: int
    dtype: str

    @property
    def batch(self) -> int:
        return int(self.num_nodes.shape[0])

    def rows(self) -> int:
        return int(self.target.shape[0])

    def row_bytes(self) -> int:
        return self.vocab * (2 if self.dtype == "bf16" else 4)


def make_tree_batch(name: str, device="cpu", batch: int | None = None) -> TreeBatch:
    spec = TREE_SPECS[name]
    B = spec.batch if batch is None else batch
    g = torch.Generator("cpu").manual_seed(spec.gen_seed)
    rng = np.random.default_rng(spec.gen_seed)
    n = spec.nodes
    num = np.full(B, n, np.int32)
    parents = []
    for _ in range(B):
        parents.append([-1] + [int(rng.integers(max(-1, i - 8), i)) for i in range(1, n)])
    target = torch.randn((B * (n + 1), spec.vocab), generator=g) * spec.sigma_t
    target = _to_dtype(target, spec.dtype)
    # the drafter's token at node i: the parent row's argmax (torch) or uniform noise
    arg = target.float().argmax(dim=1).numpy()
    toks = []
    for r in range(B):
        for i in range(n):
            row = r * (n + 1) + parents[r][i] + 1
            toks.append(int(arg[row]) if rng.random() < spec.p_agree
                        else int(rng.integers(0, spec.vocab)))
    return TreeBatch(name, target.to(device), torch.from_numpy(num).to(device),
                     torch.tensor(sum(parents, []), dtype=torch.int32, device=device),
                     torch.tensor(toks, dtype=torch.int32, device=device), n, spec.vocab,
                     spec.dtype)
