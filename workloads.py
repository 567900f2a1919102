"""Seeded synthetic workloads for the DSA prefill on context-parallel views.

This module holds shapes, request lengths, seeds and random draws only: none
of the method's arithmetic (no split, no metadata, no scores, no softmax).
Both the CUDA path's tests/bench and the CPU oracle take their inputs from
here, so neither ever computes an input for the other.

Workloads (all inputs i.i.d., fp32 draws rounded once to bf16 with
round-to-nearest-even, except w and the sink which stay fp32):

* ``TINY``      1 x 256 tokens, 8 heads, latent 64 (48 nope + 16 rope), value 48,
                indexer 4 x 32, topk 64, cp 2, both split modes; w ~ N(0,1)/2,
                softmax scale 1/sqrt(64).  ``integer=True`` draws q_I, k_I, w
                from {-3..3} so every indexer score is an exact integer.
* ``LONG_8K``   1 x 8192 tokens, DeepSeek-V3.2-like shapes (128 heads, latent
                576 = 512 nope + 64 rope, value 512, indexer 64 x 128, topk
                2048), cp 8 in-seq-split, scale 1/sqrt(192), w ~ N(0,1)*64^-0.5.
* ``VARLEN_4``  lengths {8000, 800, 5, 3000}, cp 4 round-robin, per-head sink.
* ``LONG_64K``  1 x 65536 tokens, cp 8 round-robin.
* ``MIXED_16``  16 requests, lengths round(exp(U(ln 512, ln 32768))) drawn by
                numpy default_rng(4), cp 16, both modes, per-head sink.

The pages measure on no public dataset; these seeded draws stand in for the
prefill batches they describe.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

IN_SEQ_SPLIT = 0
ROUND_ROBIN = 1
HEAD_TAIL = 2
MODE_NAMES = {IN_SEQ_SPLIT: "in-seq-split", ROUND_ROBIN: "round-robin-split", HEAD_TAIL: "head-tail-split"}


def mixed_lengths(seed: int = 4, n: int = 16, lo: int = 512, hi: int = 32768) -> tuple:
    """Request lengths log-uniform in [lo, hi] from numpy's default_rng(seed)."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(math.log(lo), math.log(hi), n)
    return tuple(int(round(math.exp(x))) for x in u)


@dataclass(frozen=True)
class Workload:
    name: str
    lengths: tuple
    H: int
    D: int
    Dv: int
    HI: int
    DI: int
    topk: int
    cp_size: int
    modes: tuple
    sink: bool
    seed: int
    w_std: float
    integer: bool = False
    scale: float = field(default=0.0)

    def __post_init__(self):
        if self.scale == 0.0:
            # 1/sqrt(d_qk) with d_qk = 192 for the V3.2 shapes (128 nope + 64 rope
            # per head before absorption), 1/sqrt(64) for the tiny case.
            object.__setattr__(self, "scale", 1.0 / math.sqrt(64 if self.D == 64 else 192))

    @property
    def num_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def batch(self) -> int:
        return len(self.lengths)

    @property
    def max_len(self) -> int:
        return int(max(self.lengths))

    def query_start_loc(self) -> np.ndarray:
        out = np.zeros(len(self.lengths) + 1, dtype=np.int32)
        out[1:] = np.cumsum(np.asarray(self.lengths, dtype=np.int64))
        return out

    def seq_lens(self) -> np.ndarray:
        return np.asarray(self.lengths, dtype=np.int32)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


BOTH = (IN_SEQ_SPLIT, ROUND_ROBIN)

TINY = Workload("tiny-1x256-cp2", (256,), H=8, D=64, Dv=48, HI=4, DI=32, topk=64,
                cp_size=2, modes=BOTH, sink=False, seed=0, w_std=0.5)
TINY_INT = TINY.with_(name="tiny-1x256-cp2-int", integer=True)
LONG_8K = Workload("long-1x8192-cp8-inseq", (8192,), H=128, D=576, Dv=512, HI=64, DI=128,
                   topk=2048, cp_size=8, modes=(IN_SEQ_SPLIT,), sink=False, seed=1,
                   w_std=64 ** -0.5)
VARLEN_4 = LONG_8K.with_(name="varlen-4req-11805-cp4-rr", lengths=(8000, 800, 5, 3000),
                         cp_size=4, modes=(ROUND_ROBIN,), sink=True, seed=2)
LONG_64K = LONG_8K.with_(name="long-1x65536-cp8-rr", lengths=(65536,), cp_size=8,
                         modes=(ROUND_ROBIN,), sink=False, seed=3)
MIXED_16 = LONG_8K.with_(name="mixed-16req-cp16", lengths=mixed_lengths(4), cp_size=16,
                         modes=BOTH, sink=True, seed=4)

ALL = {w.name: w for w in (TINY, TINY_INT, LONG_8K, VARLEN_4, LONG_64K, MIXED_16)}


def _normal(shape, gen, device, std=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return x * std if std != 1.0 else x


def _small_ints(shape, gen, device):
    return torch.randint(-3, 4, shape, generator=gen, device=device).to(torch.float32)


def draw_inputs(wl: Workload, device: str | torch.device = "cpu", seed_offset: int = 0) -> dict:
    """Draw one batch of inputs for ``wl`` on ``device``.

    Draw order (one generator seeded with ``wl.seed + seed_offset``): q, kv,
    q_idx, k_idx, w, sink.  The same seed on another device type gives other
    values (torch's CPU and CUDA generators differ); tests that need the
    values on both sides copy them.

    Returns bf16 tensors q [T,H,D], kv [T,D], q_idx [T,HI,DI], k_idx [T,DI],
    fp32 w [T,HI], fp32 sink [H] or None.
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed + seed_offset)
    T = wl.num_tokens
    q = _normal((T, wl.H, wl.D), gen, dev).to(torch.bfloat16)
    kv = _normal((T, wl.D), gen, dev).to(torch.bfloat16)
    if wl.integer:
        q_idx = _small_ints((T, wl.HI, wl.DI), gen, dev).to(torch.bfloat16)
        k_idx = _small_ints((T, wl.DI), gen, dev).to(torch.bfloat16)
        w = _small_ints((T, wl.HI), gen, dev)
    else:
        q_idx = _normal((T, wl.HI, wl.DI), gen, dev).to(torch.bfloat16)
        k_idx = _normal((T, wl.DI), gen, dev).to(torch.bfloat16)
        w = _normal((T, wl.HI), gen, dev, std=wl.w_std)
    sink = _normal((wl.H,), gen, dev) if wl.sink else None
    return {"q": q, "kv": kv, "q_idx": q_idx, "k_idx": k_idx, "w": w.contiguous(), "sink": sink}


def draw_index_inputs(wl: Workload, device: str | torch.device = "cpu", seed_offset: int = 0) -> dict:
    """Only the indexer's inputs of ``wl``: q_idx [T,HI,DI], k_idx [T,DI] bf16
    and w [T,HI] fp32, drawn with their own generator (seed ``wl.seed +
    seed_offset + 7919``) in that order; from {-3..3} when ``wl.integer``
    (every score an exact integer), N(0,1) (w: N(0,1) * w_std) otherwise.
    For indexer / top-k tests at sizes where the attention's q would be
    gigabytes."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed + seed_offset + 7919)
    T = wl.num_tokens
    if wl.integer:
        q_idx = _small_ints((T, wl.HI, wl.DI), gen, dev).to(torch.bfloat16)
        k_idx = _small_ints((T, wl.DI), gen, dev).to(torch.bfloat16)
        w = _small_ints((T, wl.HI), gen, dev)
    else:
        q_idx = _normal((T, wl.HI, wl.DI), gen, dev).to(torch.bfloat16)
        k_idx = _normal((T, wl.DI), gen, dev).to(torch.bfloat16)
        w = _normal((T, wl.HI), gen, dev, std=wl.w_std)
    return {"q_idx": q_idx, "k_idx": k_idx, "w": w.contiguous()}


def sample_rows(n_rows_total: int, count: int, seed: int, must=()) -> np.ndarray:
    """A fixed, seeded sample of row indices in [0, n_rows_total): the indices in
    ``must`` that are in range, topped up to ``count`` from a seeded permutation.
    Sorted and unique."""
    rng = np.random.default_rng(seed)
    seen = {int(m) for m in must if 0 <= int(m) < n_rows_total}
    for x in rng.permutation(n_rows_total):
        if len(seen) >= count:
            break
        seen.add(int(x))
    return np.array(sorted(seen), dtype=np.int64)


def chunk_inputs(x: dict, lengths, prefixes) -> tuple:
    """Inputs of a chunked prefill cut from a whole-sequence batch ``x`` (drawn
    for ``lengths``): request b keeps its first ``prefixes[b]`` positions as
    KV only, and its remaining positions are the queries.  q, q_idx and w keep
    the query rows; kv, k_idx and sink stay whole (every request's sequence, in
    order).  Returns (inputs, query lengths, seq_lens)."""
    lengths = [int(n) for n in lengths]
    prefixes = [int(p) for p in prefixes]
    if len(prefixes) != len(lengths) or any(p < 0 or p > n for p, n in zip(prefixes, lengths)):
        raise ValueError("0 <= prefix <= length for every request")
    rows, start = [], 0
    for n, p in zip(lengths, prefixes):
        rows.extend(range(start + p, start + n))
        start += n
    idx = torch.tensor(rows, dtype=torch.long, device=x["q"].device)
    out = dict(x)
    for k in ("q", "q_idx", "w"):
        out[k] = x[k].index_select(0, idx).contiguous()
    return out, [n - p for n, p in zip(lengths, prefixes)], lengths
