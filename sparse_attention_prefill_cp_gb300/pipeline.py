"""All CP views of one prefill batch on one GPU, through the C ABI.

Per batch ("feat: DeepSeek-V4 DSA context-parallel on NPU", 单层前向数据流:
q local, KV full; "[DeepSeek v3.2] 上下文并行详解", 第三部分):
  a1  dsa_cp_build_local_metadata for every view r
  a2  dsa_cp_split of q, q_idx and w into the rank-major layout
  a3  lightning indexer  }  dsa_indexer_topk, per view
  a4  causal top-k       }
  a5  dsa_sparse_attn_prefill, per view
  a6  dsa_cp_rerange of the per-view outputs back to flat token order
``run_headsharded`` instead writes the attention outputs straight into the
head-sharded layout [cp][T][H / cp][Dv] that the head/token all-to-all after
the attention produces (单层前向数据流 (6)), with no a6;
``all_to_all_heads`` is the same permutation as a separate pass over the
per-view outputs.  Buffers are allocated once (the head-sharded one on first
use); the methods only launch kernels on the current stream.  The views
emulate CP ranks: no collective is involved.
"""
from __future__ import annotations

import torch

from . import (CPLocalMetadata, dsa_cp_all_to_all_heads, dsa_cp_build_local_metadata, dsa_cp_geometry,
               dsa_cp_rerange, dsa_cp_split, dsa_indexer_topk, dsa_indexer_topk_workspace_size,
               dsa_sparse_attn_prefill, dsa_sparse_attn_prefill_headsharded)


class DSAPrefill:
    def __init__(self, lengths, cp_size: int, mode: int, H: int, D: int, Dv: int, HI: int, DI: int, topk: int,
                 softmax_scale: float, device=None, workspace_bytes: int | None = None):
        self.device = torch.device(device or "cuda")
        self.lengths = [int(x) for x in lengths]
        self.cp_size, self.mode = int(cp_size), int(mode)
        self.H, self.D, self.Dv, self.HI, self.DI, self.topk = H, D, Dv, HI, DI, topk
        self.scale = float(softmax_scale)
        self.T = sum(self.lengths)
        self.B = len(self.lengths)
        self.max_kv_len = max(self.lengths)
        self.pad, self.tpr = dsa_cp_geometry(self.T, cp_size)
        qsl = [0]
        for n in self.lengths:
            qsl.append(qsl[-1] + n)
        dev = self.device
        self.query_start_loc = torch.tensor(qsl, dtype=torch.int32, device=dev)
        self.seq_lens = torch.tensor(self.lengths, dtype=torch.int32, device=dev)
        self.md = [CPLocalMetadata(self.B, self.T, cp_size, dev) for _ in range(cp_size)]
        cp, tpr = cp_size, self.tpr
        self.q_split = torch.empty((cp, tpr, H, D), dtype=torch.bfloat16, device=dev)
        self.qi_split = torch.empty((cp, tpr, HI, DI), dtype=torch.bfloat16, device=dev)
        self.w_split = torch.empty((cp, tpr, HI), dtype=torch.float32, device=dev)
        self.topk_idx = torch.empty((cp, tpr, topk), dtype=torch.int32, device=dev)
        self.out_split = torch.empty((cp, tpr, H, Dv), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((self.T, H, Dv), dtype=torch.bfloat16, device=dev)
        ws = workspace_bytes or dsa_indexer_topk_workspace_size(tpr, self.max_kv_len, topk)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.out_hs = None  # [cp][T][H / cp][Dv], allocated on first use

    def launches_per_step(self) -> int:
        """Kernel launches of one ``run``: metadata per view, 3 splits, per view
        (indexer + top-k) per workspace chunk and one attention, 1 rerange."""
        ld = (self.max_kv_len + 3) // 4 * 4
        tile = 8 if self.HI == 64 else 128
        rows_fit = (self.workspace.numel() // (ld * 4)) // tile * tile
        chunks = -(-self.tpr // rows_fit)
        return self.cp_size + 3 + self.cp_size * (2 * chunks + 1) + 1

    def metadata(self, stream=None):                                     # a1
        for r in range(self.cp_size):
            dsa_cp_build_local_metadata(self.query_start_loc, self.seq_lens, self.T, self.cp_size, r, self.mode,
                                        self.md[r], stream)

    def split(self, q, q_idx, w, stream=None):                          # a2
        dsa_cp_split(q, self.cp_size, self.mode, -1, self.q_split, stream)
        dsa_cp_split(q_idx, self.cp_size, self.mode, -1, self.qi_split, stream)
        dsa_cp_split(w, self.cp_size, self.mode, -1, self.w_split, stream)

    def view(self, r: int, kv, k_idx, sink=None, stream=None):          # a3 + a4 + a5
        dsa_indexer_topk(self.md[r], self.qi_split[r], k_idx, self.w_split[r], self.topk, self.max_kv_len,
                         self.topk_idx[r], self.workspace, stream)
        dsa_sparse_attn_prefill(self.md[r], self.q_split[r], kv, self.topk_idx[r], self.scale, self.Dv, sink,
                                self.out_split[r], stream)

    def rerange(self, stream=None):                                     # a6
        return dsa_cp_rerange(self.out_split, self.T, self.cp_size, self.mode, self.out, stream)

    def run(self, q, kv, q_idx, k_idx, w, sink=None, stream=None, events=None):
        """One pass of the whole path; returns out [T, H, Dv] (a view of self.out).
        ``events``: optional dict of 4 CUDA events ("start", "core_start",
        "core_end", "end") recorded around the indexer/top-k/attention core."""
        ev = events or {}
        s = stream or torch.cuda.current_stream()
        if "start" in ev:
            ev["start"].record(s)
        self.metadata(stream)
        self.split(q, q_idx, w, stream)
        if "core_start" in ev:
            ev["core_start"].record(s)
        for r in range(self.cp_size):
            self.view(r, kv, k_idx, sink, stream)
        if "core_end" in ev:
            ev["core_end"].record(s)
        out = self.rerange(stream)
        if "end" in ev:
            ev["end"].record(s)
        return out

    def _head_sharded_buffer(self):
        if self.out_hs is None:
            if self.H % self.cp_size:
                raise ValueError("the head count must divide by cp_size")
            self.out_hs = torch.empty((self.cp_size, self.T, self.H // self.cp_size, self.Dv), dtype=torch.bfloat16,
                                      device=self.device)
        return self.out_hs

    def all_to_all_heads(self, stream=None):
        """The per-view outputs of the last ``run`` -> head-sharded [cp, T, H / cp, Dv]."""
        return dsa_cp_all_to_all_heads(self.out_split, self.T, self.cp_size, self.mode, self._head_sharded_buffer(),
                                       stream)

    def run_headsharded(self, q, kv, q_idx, k_idx, w, sink=None, stream=None):
        """a1, a2, then per view a3 + a4 + a5 with the attention writing the
        head-sharded layout directly; returns out_hs [cp, T, H / cp, Dv]."""
        out = self._head_sharded_buffer()
        self.metadata(stream)
        self.split(q, q_idx, w, stream)
        for r in range(self.cp_size):
            dsa_indexer_topk(self.md[r], self.qi_split[r], k_idx, self.w_split[r], self.topk, self.max_kv_len,
                             self.topk_idx[r], self.workspace, stream)
            dsa_sparse_attn_prefill_headsharded(self.md[r], self.q_split[r], kv, self.topk_idx[r], self.scale,
                                                self.Dv, self.cp_size, out, sink, stream)
        return out
