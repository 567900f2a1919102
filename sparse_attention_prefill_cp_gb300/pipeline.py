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

from . import (HEAD_TAIL, IN_SEQ_SPLIT, ROUND_ROBIN, CPLocalMetadata, dsa_cp_all_to_all_heads, dsa_cp_build_local_metadata, dsa_cp_geometry,
               dsa_cp_rerange, dsa_cp_rerange_to_host, dsa_cp_split, dsa_cp_split_from_host, dsa_indexer_topk,
               dsa_indexer_topk_fp8, dsa_indexer_topk_rows, dsa_sparse_attn_prefill_rows,
               dsa_indexer_topk_workspace_size, dsa_kv_fp8_dequantize, dsa_kv_fp8_row_bytes, dsa_sparse_attn_prefill,
               dsa_sparse_attn_prefill_flat, dsa_sparse_attn_prefill_fp8kv, dsa_sparse_attn_prefill_headsharded,
               dsa_sparse_attn_prefill_swa,
               dsa_swa_index)


class DSAPrefill:
    def __init__(self, lengths, cp_size: int, mode: int, H: int, D: int, Dv: int, HI: int, DI: int, topk: int,
                 softmax_scale: float, device=None, workspace_bytes: int | None = None, view_streams: int = 1,
                 prefix_lens=None, kv_fp8: bool = False, fused: bool = False, compress_ratio: int = 1,
                 index_fp8: bool = False, window: int = 0, kv_fp8_direct: bool = False):
        """``lengths``: query tokens per request.  ``prefix_lens`` (chunked
        prefill): KV positions per request that precede its queries; the KV
        and index-key tensors passed to ``run`` then hold every request's
        whole sequence (prefix + queries), requests in order.  ``kv_fp8``:
        the latent KV passed to ``run`` is the FP8 cache (uint8 rows of
        dsa_kv_fp8_row_bytes), dequantised once per batch before the views;
        with ``kv_fp8_direct`` the attention reads the cache itself and
        dequantises in its gather (dsa_sparse_attn_prefill_fp8kv, the same
        results; DeepSeek-V3.2 shapes, no window).
        ``fused``: ``run`` skips the split of q and the rerange of the
        outputs; each view's attention reads its queries from the full q and
        writes its rows of ``out`` in place (dsa_sparse_attn_prefill_flat),
        with the same results.  ``compress_ratio`` c: the latent KV and index
        keys passed to ``run`` are compressed entries, floor(seq_len / c) per
        request in request order (dsa_cp_build_local_metadata_compressed).
        ``index_fp8``: q_idx and k_idx passed to ``run`` are FP8 index rows
        (uint8 [T, HI, row_bytes] and [R, row_bytes], dsa_indexer_fp8_rows)
        and the indexer runs on them (dsa_indexer_topk_fp8).  ``window`` W > 0:
        the sliding window -- each query also attends to the original KV rows
        of its last W positions under the same softmax (dsa_swa_index,
        dsa_sparse_attn_prefill_swa; view layout only); at compress_ratio > 1
        ``run`` then takes the original rows as ``kv_ori``."""
        self.device = torch.device(device or "cuda")
        self.lengths = [int(x) for x in lengths]
        self.prefix_lens = [0] * len(self.lengths) if prefix_lens is None else [int(x) for x in prefix_lens]
        if len(self.prefix_lens) != len(self.lengths) or min(self.prefix_lens, default=0) < 0:
            raise ValueError("one non-negative prefix length per request")
        self.cp_size, self.mode = int(cp_size), int(mode)
        self.H, self.D, self.Dv, self.HI, self.DI, self.topk = H, D, Dv, HI, DI, topk
        self.scale = float(softmax_scale)
        self.T = sum(self.lengths)
        self.B = len(self.lengths)
        self.kv_lens = [n + p for n, p in zip(self.lengths, self.prefix_lens)]
        self.compress_ratio = int(compress_ratio)
        if self.compress_ratio < 1:
            raise ValueError("compress_ratio must be at least 1")
        self.num_kv_rows = sum(n // self.compress_ratio for n in self.kv_lens)
        self.max_kv_len = max(1, max(n // self.compress_ratio for n in self.kv_lens))
        self.pad, self.tpr = dsa_cp_geometry(self.T, cp_size)
        qsl = [0]
        for n in self.lengths:
            qsl.append(qsl[-1] + n)
        dev = self.device
        self.query_start_loc = torch.tensor(qsl, dtype=torch.int32, device=dev)
        self.seq_lens = torch.tensor(self.kv_lens, dtype=torch.int32, device=dev)
        self.md = [CPLocalMetadata(self.B, self.T, cp_size, dev) for _ in range(cp_size)]
        cp, tpr = cp_size, self.tpr
        self.fused = bool(fused)
        self._q_split = None    # [cp][tpr][H][D] and [cp][tpr][H][Dv], allocated on
        self._out_split = None  # first use (never by the fused path)
        self.index_fp8 = bool(index_fp8)
        if self.index_fp8:
            self.qi_split = torch.empty((cp, tpr, HI, dsa_kv_fp8_row_bytes(DI, DI)), dtype=torch.uint8, device=dev)
        else:
            self.qi_split = torch.empty((cp, tpr, HI, DI), dtype=torch.bfloat16, device=dev)
        self.w_split = torch.empty((cp, tpr, HI), dtype=torch.float32, device=dev)
        self.topk_idx = torch.empty((cp, tpr, topk), dtype=torch.int32, device=dev)
        self.out = torch.empty((self.T, H, Dv), dtype=torch.bfloat16, device=dev)
        ws = workspace_bytes or dsa_indexer_topk_workspace_size(tpr, self.max_kv_len, topk)
        # views on several streams: one score workspace per stream, so that the
        # tail of one view's kernels overlaps the start of the next view's
        self.view_streams = max(1, int(view_streams))
        self.workspaces = [torch.empty(ws, dtype=torch.uint8, device=dev) for _ in range(self.view_streams)]
        self.workspace = self.workspaces[0]
        self._side = None
        self.out_hs = None  # [cp][T][H / cp][Dv], allocated on first use
        self.kv_fp8 = bool(kv_fp8)
        self.kv_fp8_direct = bool(kv_fp8_direct)
        if self.kv_fp8_direct and (not self.kv_fp8 or window):
            raise ValueError("kv_fp8_direct needs kv_fp8 and no window")
        self.kv_rows = (torch.empty((self.num_kv_rows, D), dtype=torch.bfloat16, device=dev)
                        if self.kv_fp8 and not self.kv_fp8_direct else None)
        self.attention_events = None  # a list: (view, start, end) CUDA events of every attention launch
        self._q = None
        self.window = int(window)
        if self.window < 0:
            raise ValueError("window must be >= 0")
        if self.window and self.fused:
            raise ValueError("the sliding window runs on the view layout (fused=False)")
        if self.window:
            # extended index rows and their counts; the ratio-1 metadata gives the
            # original KV row of each local request's position 0
            # rows of topk + W entries, padded to a multiple of 4 (16-byte aligned rows and views)
            stride = (topk + self.window + 3) // 4 * 4
            self.ext_idx = torch.empty((cp, tpr, stride), dtype=torch.int32, device=dev)
            self.ext_counts = torch.empty((cp, tpr), dtype=torch.int32, device=dev)
            self.md_ori = (self.md if self.compress_ratio == 1 else
                           [CPLocalMetadata(self.B, self.T, cp_size, dev) for _ in range(cp_size)])
        self._kv_ori = None

    @property
    def q_split(self):
        if self._q_split is None:
            self._q_split = torch.empty((self.cp_size, self.tpr, self.H, self.D), dtype=torch.bfloat16,
                                        device=self.device)
        return self._q_split

    @property
    def out_split(self):
        if self._out_split is None:
            self._out_split = torch.empty((self.cp_size, self.tpr, self.H, self.Dv), dtype=torch.bfloat16,
                                          device=self.device)
        return self._out_split

    def launches_per_step(self) -> int:
        """Kernel launches of one ``run``: metadata per view, 3 splits (2
        fused), the FP8 dequantisation (if any), per view (indexer + top-k) per
        workspace chunk and one attention, 1 rerange (0 fused)."""
        ld = (self.max_kv_len + 3) // 4 * 4
        tile = 8 if self.HI == 64 else 128
        rows_fit = (self.workspace.numel() // (ld * 4)) // tile * tile
        chunks = -(-self.tpr // rows_fit)
        splits, reranges = (2, 0) if self.fused else (3, 1)
        md = self.cp_size * (2 if self.window and self.compress_ratio > 1 else 1)
        swa = self.cp_size if self.window else 0
        dequant = int(self.kv_fp8 and not self.kv_fp8_direct)
        return md + splits + dequant + self.cp_size * (2 * chunks + 1) + swa + reranges

    def metadata(self, stream=None):                                     # a1
        for r in range(self.cp_size):
            dsa_cp_build_local_metadata(self.query_start_loc, self.seq_lens, self.T, self.cp_size, r, self.mode,
                                        self.md[r], stream, self.compress_ratio)
            if self.window and self.compress_ratio > 1:
                dsa_cp_build_local_metadata(self.query_start_loc, self.seq_lens, self.T, self.cp_size, r, self.mode,
                                            self.md_ori[r], stream, 1)

    def split(self, q, q_idx, w, stream=None):                          # a2
        if not self.fused:  # the fused attention reads q in place
            dsa_cp_split(q, self.cp_size, self.mode, -1, self.q_split, stream)
        dsa_cp_split(q_idx, self.cp_size, self.mode, -1, self.qi_split, stream)
        dsa_cp_split(w, self.cp_size, self.mode, -1, self.w_split, stream)

    def indexer(self, r: int, k_idx, stream=None, workspace=None):     # a3 + a4
        ws = self.workspace if workspace is None else workspace
        if self.index_fp8:
            dsa_indexer_topk_fp8(self.md[r], self.qi_split[r], k_idx, self.w_split[r], self.topk, self.max_kv_len,
                                 self.DI, self.topk_idx[r], ws, stream)
        else:
            dsa_indexer_topk(self.md[r], self.qi_split[r], k_idx, self.w_split[r], self.topk, self.max_kv_len,
                             self.topk_idx[r], ws, stream)

    def view(self, r: int, kv, k_idx, sink=None, stream=None, workspace=None):  # a3 + a4 + a5
        self.indexer(r, k_idx, stream, workspace)
        st = stream or torch.cuda.current_stream(self.device)
        ev = self.attention_events
        if ev is not None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)  # on the stream the attention is launched on
        if self.window:
            dsa_swa_index(self.md[r], self.md_ori[r], self.topk_idx[r], self.window, self.num_kv_rows,
                          self.ext_idx[r], self.ext_counts[r], st)
            dsa_sparse_attn_prefill_swa(self.md[r], self.q_split[r], kv, self._kv_ori, self.ext_idx[r],
                                        self.ext_counts[r], self.topk, self.scale, self.Dv, sink, self.out_split[r],
                                        st)
        elif self.kv_fp8_direct:
            q, out = (self._q, self.out) if self.fused else (self.q_split[r], self.out_split[r])
            dsa_sparse_attn_prefill_fp8kv(self.md[r], q, kv, self.topk_idx[r], self.scale, self.D, self.Dv, out, sink,
                                          flat=self.fused, stream=st)
        elif self.fused:
            dsa_sparse_attn_prefill_flat(self.md[r], self._q, kv, self.topk_idx[r], self.scale, self.Dv, self.out,
                                         sink, st)
        else:
            dsa_sparse_attn_prefill(self.md[r], self.q_split[r], kv, self.topk_idx[r], self.scale, self.Dv, sink,
                                    self.out_split[r], st)
        if ev is not None:
            e1.record(st)
            ev.append((r, e0, e1))

    def latent_kv(self, kv, stream=None):
        """The bf16 latent rows the attention reads: ``kv`` itself, or the
        rows an FP8 cache stands for (dequantised into a buffer of this
        object)."""
        if not self.kv_fp8 or self.kv_fp8_direct:
            return kv
        return dsa_kv_fp8_dequantize(kv, self.D, self.Dv, self.kv_rows, stream)

    def side_streams(self):
        if self._side is None:
            self._side = [torch.cuda.Stream(self.device) for _ in range(self.view_streams)]
        return self._side

    def views(self, kv, k_idx, sink, stream):
        """Every view's a3-a5.  With one view stream they run in order on
        ``stream``; with n > 1, view r runs on side stream r % n (forked from
        and joined back into ``stream``), each with its own workspace."""
        if self.view_streams == 1:
            for r in range(self.cp_size):
                self.view(r, kv, k_idx, sink, stream)
            return
        side = self.side_streams()
        fork = torch.cuda.Event()
        fork.record(stream)
        for st in side:
            st.wait_event(fork)
        for r in range(self.cp_size):
            k = r % self.view_streams
            self.view(r, kv, k_idx, sink, side[k], self.workspaces[k])
        for st in side:
            join = torch.cuda.Event()
            join.record(st)
            stream.wait_event(join)

    def rerange(self, stream=None):                                     # a6
        if self.fused:  # the fused attention wrote out in place
            return self.out
        return dsa_cp_rerange(self.out_split, self.T, self.cp_size, self.mode, self.out, stream)

    def run(self, q, kv, q_idx, k_idx, w, sink=None, stream=None, events=None, kv_ori=None):
        """One pass of the whole path; returns out [T, H, Dv] (a view of self.out).
        ``events``: optional dict of 4 CUDA events ("start", "core_start",
        "core_end", "end") recorded around the indexer/top-k/attention core.
        ``kv_ori``: the original latent rows for the sliding window at
        compress_ratio > 1 (at ratio 1 the window reads ``kv``)."""
        if self.window and self.compress_ratio > 1 and kv_ori is None:
            raise ValueError("the sliding window over compressed KV needs the original rows (kv_ori)")
        self._kv_ori = kv_ori if self.window and self.compress_ratio > 1 else None
        ev = events or {}
        s = stream or torch.cuda.current_stream()
        if "start" in ev:
            ev["start"].record(s)
        self.metadata(stream)
        self.split(q, q_idx, w, stream)
        if "core_start" in ev:
            ev["core_start"].record(s)
        self._q = q
        kv = self.latent_kv(kv, s)
        self.views(kv, k_idx, sink, s)
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
        """The per-view outputs of the last ``run`` (not fused) -> head-sharded [cp, T, H / cp, Dv]."""
        return dsa_cp_all_to_all_heads(self.out_split, self.T, self.cp_size, self.mode, self._head_sharded_buffer(),
                                       stream)

    def run_headsharded(self, q, kv, q_idx, k_idx, w, sink=None, stream=None):
        """a1, a2, then per view a3 + a4 + a5 with the attention writing the
        head-sharded layout directly; returns out_hs [cp, T, H / cp, Dv]."""
        if self.kv_fp8_direct:
            raise ValueError("the head-sharded attention reads bf16 rows (build without kv_fp8_direct)")
        out = self._head_sharded_buffer()
        self.metadata(stream)
        self.split(q, q_idx, w, stream)
        if self.fused:  # the head-sharded attention reads the split q
            dsa_cp_split(q, self.cp_size, self.mode, -1, self.q_split, stream)
        kv = self.latent_kv(kv, stream)
        for r in range(self.cp_size):
            self.indexer(r, k_idx, stream)
            dsa_sparse_attn_prefill_headsharded(self.md[r], self.q_split[r], kv, self.topk_idx[r], self.scale,
                                                self.Dv, self.cp_size, out, sink, stream)
        return out


class HostStreamedPrefill:
    """Prefill batches whose inputs and output live in page-locked host memory,
    streamed a chunk of the token stream at a time so that copies and compute
    overlap.

    Per batch: the full-token inputs every view reads (kv, k_idx and the sink)
    go up first; then the token stream is cut into chunks of ``chunk_tokens``
    consecutive tokens (a multiple of cp_size).  A chunk's q, q_idx and w rows
    go up as contiguous copies (the copy engines run contiguous copies at
    about twice the rate of pitched ones), every view then runs its slots
    whose tokens lie in the chunk -- dsa_indexer_topk_rows and
    dsa_sparse_attn_prefill_rows, which read the chunk's q rows and write its
    output rows by token (round-robin: q_idx and w of the chunk are first split
    on the device into per-view slot blocks) -- and the chunk's output rows
    come back as one contiguous copy.  ``depth`` chunk buffer sets rotate, so
    while one chunk computes the next goes up and the previous comes down;
    consecutive batches chain the same way (the full-token buffers alternate
    between two sets).  Streams: one for uploads, ``compute_streams`` for the
    views (view r on stream r mod n, so kernel tails overlap), one for
    read-back.

    ``submit`` only enqueues work; wait on ``done_event(s)`` (or synchronise)
    before reading batch s's host output.  The kernels' arithmetic is that of
    ``DSAPrefill.run``, so the output is the same bit for bit.
    """

    INPUTS = ("q", "kv", "q_idx", "k_idx", "w", "sink")

    def __init__(self, lengths, cp_size: int, mode: int, H: int, D: int, Dv: int, HI: int, DI: int, topk: int,
                 softmax_scale: float, device=None, depth: int = 3, prefix_lens=None, chunk_tokens: int | None = None,
                 compute_streams: int = 2):
        if depth < 1:
            raise ValueError("depth must be at least 1")
        self.device = torch.device(device or "cuda")
        dev = self.device
        self.lengths = [int(x) for x in lengths]
        self.prefix_lens = [0] * len(self.lengths) if prefix_lens is None else [int(x) for x in prefix_lens]
        self.cp_size, self.mode = int(cp_size), int(mode)
        self.H, self.D, self.Dv, self.HI, self.DI, self.topk = H, D, Dv, HI, DI, topk
        self.scale = float(softmax_scale)
        self.T, self.B = sum(self.lengths), len(self.lengths)
        kv_lens = [n + p for n, p in zip(self.lengths, self.prefix_lens)]
        self.num_kv_rows, self.max_kv_len = sum(kv_lens), max(1, max(kv_lens))
        self.pad, self.tpr = dsa_cp_geometry(self.T, cp_size)
        cp = self.cp_size
        qsl = [0]
        for n in self.lengths:
            qsl.append(qsl[-1] + n)
        self.query_start_loc = torch.tensor(qsl, dtype=torch.int32, device=dev)
        self.seq_lens = torch.tensor(kv_lens, dtype=torch.int32, device=dev)
        self.md = [CPLocalMetadata(self.B, self.T, cp_size, dev) for _ in range(cp_size)]
        if chunk_tokens is None:  # about sixteen chunks per batch
            chunk_tokens = -(-self.T // 16)
        C = max(cp, -(-int(chunk_tokens) // cp) * cp)
        self.chunk_tokens = C
        self.chunks = [(t0, min(t0 + C, self.T)) for t0 in range(0, self.T, C)]
        self.depth = depth
        self.q_c = [torch.empty((C, H, D), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        self.qi_c = [torch.empty((C, HI, DI), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        self.w_c = [torch.empty((C, HI), dtype=torch.float32, device=dev) for _ in range(depth)]
        self.out_c = [torch.empty((C, H, Dv), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        rr = self.mode == ROUND_ROBIN
        # round-robin: a chunk's q_idx / w split into per-view slot blocks
        self.qi_s = [torch.empty(C * HI * DI, dtype=torch.bfloat16, device=dev) for _ in range(depth)] if rr else None
        self.w_s = [torch.empty(C * HI, dtype=torch.float32, device=dev) for _ in range(depth)] if rr else None
        self.n_comp = max(1, int(compute_streams))
        max_run = C // cp if rr else min(C, self.tpr)
        self.topk_rows = [torch.empty((max_run, topk), dtype=torch.int32, device=dev) for _ in range(self.n_comp)]
        ws = dsa_indexer_topk_workspace_size(max_run, self.max_kv_len, topk)
        self.workspaces = [torch.empty(ws, dtype=torch.uint8, device=dev) for _ in range(self.n_comp)]
        self.full = [None, None]      # full-token device inputs, by batch parity
        self.h2d = torch.cuda.Stream(dev)
        self.compute = [torch.cuda.Stream(dev) for _ in range(self.n_comp)]
        self.d2h = torch.cuda.Stream(dev)
        self.full_ready = [torch.cuda.Event() for _ in range(2)]
        self.full_free = [torch.cuda.Event() for _ in range(2)]
        self.in_ready = [torch.cuda.Event() for _ in range(depth)]
        self.computed = [torch.cuda.Event() for _ in range(depth)]
        self.read_back = [torch.cuda.Event() for _ in range(depth)]
        self._done = {}
        self._submitted = 0
        self._chunks_done = 0  # chunks enqueued so far (the buffer set of chunk n is n % depth)

    def _runs(self, r, t0, t1):
        """(slot_begin, count, first token) of view r's slots whose tokens lie
        in [t0, t1): whole runs of consecutive slots."""
        T, tpr, cp = self.T, self.tpr, self.cp_size
        if self.mode == ROUND_ROBIN:  # t0 is a multiple of cp: slots t0/cp .., tokens t0 + r, t0 + r + cp, ...
            n = max(0, -(-(min(t1, T) - t0 - r) // cp)) if t0 + r < t1 else 0
            return [(t0 // cp, n, t0 + r)] if n > 0 else []
        if self.mode == IN_SEQ_SPLIT:
            spans = [(r * tpr, 0, tpr)]
        else:  # head-tail: the head run then the tail run
            h, t = (tpr + 1) // 2, tpr // 2
            spans = [(r * h, 0, h), (cp * h + (cp - 1 - r) * t, h, t)]
        out = []
        for g0, s0, n in spans:
            a, b = max(g0, t0), min(g0 + n, t1, T)
            if a < b:
                out.append((s0 + a - g0, b - a, a))
        return out

    def _full_inputs(self, b, host):
        if self.full[b] is None:
            self.full[b] = {n: (torch.empty(host[n].shape, dtype=host[n].dtype, device=self.device)
                                if host.get(n) is not None else None) for n in ("kv", "k_idx", "sink")}
        return self.full[b]

    def submit(self, host: dict, out_host: torch.Tensor, stream=None) -> int:
        """Enqueue one batch: ``host`` maps q, kv, q_idx, k_idx, w (and sink or
        None) to page-locked CPU tensors; ``out_host`` is a page-locked CPU
        tensor [T, H, Dv] bf16 that receives the output.  ``stream``: the
        stream whose prior work the batch waits for (default: the current
        stream).  Returns the batch number."""
        for n in self.INPUTS:
            t = host.get(n)
            if t is not None and (t.device.type != "cpu" or not t.is_pinned()):
                raise ValueError(f"{n}: page-locked host memory expected")
        if out_host.device.type != "cpu" or not out_host.is_pinned():
            raise ValueError("out_host: page-locked host memory expected")
        s = self._submitted
        b = s % 2
        cp, mode, T = self.cp_size, self.mode, self.T
        caller = stream or torch.cuda.current_stream(self.device)
        full = self._full_inputs(b, host)
        # the full-token inputs of batch parity b are free once batch s - 2's views have run
        self.h2d.wait_stream(caller)
        if s >= 2:
            self.h2d.wait_event(self.full_free[b])
        with torch.cuda.stream(self.h2d):
            for n, t in full.items():
                if t is not None:
                    t.copy_(host[n], non_blocking=True)
        self.full_ready[b].record(self.h2d)
        comp0 = self.compute[0]
        comp0.wait_event(self.full_ready[b])
        for r in range(cp):                                                            # a1
            dsa_cp_build_local_metadata(self.query_start_loc, self.seq_lens, T, cp, r, mode, self.md[r], comp0)
        meta = torch.cuda.Event()
        meta.record(comp0)
        for st in self.compute[1:]:
            st.wait_event(meta)
        for (t0, t1) in self.chunks:
            k = self._chunks_done % self.depth
            n = t1 - t0
            if self._chunks_done >= self.depth:  # chunk n - depth has read set k's inputs
                self.h2d.wait_event(self.computed[k])
            with torch.cuda.stream(self.h2d):                                          # a2: contiguous rows
                self.q_c[k][:n].copy_(host["q"][t0:t1], non_blocking=True)
                self.qi_c[k][:n].copy_(host["q_idx"][t0:t1], non_blocking=True)
                self.w_c[k][:n].copy_(host["w"][t0:t1], non_blocking=True)
            self.in_ready[k].record(self.h2d)
            comp0.wait_event(self.in_ready[k])
            if self._chunks_done >= self.depth:  # chunk n - depth's output has been read back
                comp0.wait_event(self.read_back[k])
            if mode == ROUND_ROBIN:  # the chunk's per-view slot blocks of q_idx and w
                ct = -(-n // cp)
                qi_s = self.qi_s[k][:cp * ct * self.HI * self.DI].view(cp, ct, self.HI, self.DI)
                w_s = self.w_s[k][:cp * ct * self.HI].view(cp, ct, self.HI)
                dsa_cp_split(self.qi_c[k][:n], cp, mode, -1, qi_s, comp0)
                dsa_cp_split(self.w_c[k][:n], cp, mode, -1, w_s, comp0)
            fork = torch.cuda.Event()
            fork.record(comp0)
            for st in self.compute[1:]:
                st.wait_event(fork)
            for r in range(cp):
                u = r % self.n_comp
                st = self.compute[u]
                for (s0, cnt, g0) in self._runs(r, t0, t1):
                    if mode == ROUND_ROBIN:
                        qi_rows, w_rows = qi_s[r, :cnt], w_s[r, :cnt]
                    else:
                        qi_rows, w_rows = self.qi_c[k][g0 - t0:g0 - t0 + cnt], self.w_c[k][g0 - t0:g0 - t0 + cnt]
                    rows = self.topk_rows[u][:cnt]
                    dsa_indexer_topk_rows(self.md[r], s0, qi_rows, full["k_idx"], w_rows, self.topk,  # a3 + a4
                                          self.max_kv_len, rows, self.workspaces[u], st)
                    dsa_sparse_attn_prefill_rows(self.md[r], s0, cnt, self.q_c[k][:n], t0, full["kv"], rows,  # a5
                                                 self.scale, self.Dv, self.out_c[k][:n], full["sink"], st)
            for st in self.compute[1:]:
                join = torch.cuda.Event()
                join.record(st)
                comp0.wait_event(join)
            self.computed[k].record(comp0)
            self.d2h.wait_event(self.computed[k])
            with torch.cuda.stream(self.d2h):                                          # a6: contiguous rows
                out_host[t0:t1].copy_(self.out_c[k][:n], non_blocking=True)
            self.read_back[k].record(self.d2h)
            self._chunks_done += 1
        self.full_free[b].record(comp0)
        done = torch.cuda.Event(enable_timing=True)
        done.record(self.d2h)
        self._done[s] = done
        self._submitted += 1
        return s

    def done_event(self, s: int) -> torch.cuda.Event:
        """Recorded on the read-back stream once batch s's output is on the host."""
        return self._done[s]
