"""Plain fp64 CPU oracle for the DSA prefill on context-parallel (CP) views.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference`` arm) may
import this module.  The CUDA product path never imports it, and it imports
nothing from the product path: the two share no code, tables or helpers.

It is deliberately slow and obvious: Python loops over requests and rows,
numpy fp64 matmul / exp / sort as the only library steps, no blocking, no
fusion, no reordering beyond what each definition states.

Pages it follows (cited per function by title and section):

* [xLLM]   "feat: DeepSeek-V4 DSA context-parallel on NPU" (xLLM pull request
           1997): sections "单层前向数据流" (per-layer data flow), "代码实现 /
           2. CP 本地元数据" (build_cp_local_metadata), "8. 单测" (unit tests).
* [blog]   "[DeepSeek v3.2] 上下文并行详解": sections "2.B 核心切分逻辑"
           (round-robin split), "4. 一些细节 / 第一部分" (in-seq-split
           example), "第三部分 KV Cache 的流动" (T0..T7 round-robin data flow,
           gather + rerange).
* [sglang] "NSA Prefill CP 中两次 All-Gather 的作用说明": section
           "第一次 All-Gather" (KV / index key rebuilt in logical order).

Method definitions the pages name but do not write out (DeepSeek Sparse
Attention, named in [xLLM] "背景"): the lightning-indexer score
I[t,s] = sum_j w[t,j] * ReLU(q_I[t,j] . k_I[s]), a causal top-k over s <= t
with ties to the lower index, and MLA sparse attention of every query head
over the selected rows of the shared latent KV (first Dv columns are the
value), with an optional per-head sink logit.

Readings taken where the pages are silent or ambiguous (each listed in the
design notes):
  R1  split granularity is the flat token stream, not per request ([xLLM] 2).
  R2  in-seq-split is contiguous ([blog] 4 第一部分); padding sits at the end.
  R2  head-tail in-seq-split (only named by [xLLM] 7, as a worker-side split):
      the zigzag split.  tokens_per_rank is as for the other modes; the first
      cp*ceil(tpr/2) padded rows are cut into head chunks of ceil(tpr/2) rows
      (rank r: chunk r), the rest into tail chunks of floor(tpr/2) rows given
      out in reverse rank order (rank r: chunk cp-1-r), so a rank pairs an early
      (short-context) chunk with a late one; a rank's slots are its head rows
      then its tail rows, i.e. ascending flat order.
  R3  round-robin indexes the global flat token ([blog] 2.B).
  R4  local_seq_lens is the KV extent visible to the rank's queries of that
      request, i.e. last local in-request position + 1 ([xLLM] 单层前向数据流
      "右对齐"); local_kv_start_loc is its exclusive cumsum.
  R5  requests with no local row are dropped from the local batch.
  R7  KV rows stay in full flat order; request b's key s is flat row qs_b + s.
  R9  top-k ties go to the lower index; -0.0 equals +0.0; rows with p+1 <= k
      select every s <= p and pad with -1; the result is a set (returned in
      ascending order).
  R10 the sink is a logit already in scaled units that adds exp(sink - m) to
      the softmax denominator only; absent means no term.
  R12 chunked prefill ([xLLM] 测试与验证 lists it; 单层前向数据流 (4) gives the
      attention separate KV geometry: cu_seqlens_ori_kv, seqused_kv): request
      b's queries are the last q_len_b positions of its sequence of
      seq_lens[b] >= q_len_b tokens, after a prefix of seq_lens[b] - q_len_b
      positions whose KV is already there.  KV and index keys hold every
      request's whole sequence, requests in order: position s of request b is
      KV row kv_start_b + s, kv_start_b = sum of seq_lens before b.  With no
      prefix kv_start_b = qs_b and this is R7.
  R16 the head/token all-to-all after the attention ([xLLM] 单层前向数据流 (6))
      leaves rank r' with heads r'*H/cp .. (r'+1)*H/cp - 1 of every real token,
      tokens in flat order for both split modes (for in-seq-split the
      rank-major order already is the flat order; for round-robin the rows are
      put back in flat order as by rerange); H must divide by cp.
  R17 the FP8 latent-KV cache ([blog] 1, named only): the OCP E4M3 row layout
      of the FP8 section at the end of this file.
  R18 compressed KV ([xLLM] 背景: compress_ratio in {1, 4, 128}; 5: the sparse
      metadata is built per ratio with the local geometry).  At ratio c a
      request of seq_len tokens has floor(seq_len / c) compressed entries
      (latent rows and index keys, given as inputs: the compressor is out of
      scope); entry e stands for positions [e*c, (e+1)*c).  A query at position
      p sees the entries whose whole group lies at or before p, e <
      floor((p + 1) / c); the indexer, top-k and attention run over those
      entries.  Entries of all requests are stored in request order.  A query
      that sees no entry selects nothing and its output is zero.  c = 1 is
      the uncompressed path.
  R19 FP8 indexer operands (the FP8 path of [blog] 1 applied to the index
      query and keys; the pages fix no format): each DI-wide index row (a key
      k_I[s], or one head q_I[t, j]) is stored like an R17 cache row with
      D = Dv = DI (codes, one fp32 scale per 128 columns, zero padding), and
      stands for the real values decode(code) * scale, taken exactly (no
      rounding to bf16).  The FP8 indexer score is the indexer score of those
      values.
  R20 sliding window (SWA; [xLLM] 背景 names it beside the compressed KV, and
      单层前向数据流 (4) gives the attention the original KV's geometry,
      cu_seqlens_ori_kv / seqused_kv, besides the sparse selection; nothing
      says how the two combine).  Reading taken: a query at position p also
      attends to the original (uncompressed) latent rows of its own request
      at positions max(0, p - W + 1) .. p, and one softmax covers the selected
      entries and those window rows together; at c = 1 the entries are the
      original rows and a row both selected and in the window counts once.
      The original rows are every request's whole sequence in request order
      (R12).  W = 0 is the plain sparse path.

parity pins: every function here is pinned by tests/test_oracle_pins.py
against worked examples from the pages (tests/golden/), closed forms,
invariants, brute force on tiny inputs and independent library routines.
"""
from __future__ import annotations

import numpy as np

IN_SEQ_SPLIT = 0
ROUND_ROBIN = 1
HEAD_TAIL = 2


# --------------------------------------------------------------------------
# CP geometry: which flat rows a rank owns
# --------------------------------------------------------------------------

def padded_geometry(num_tokens: int, cp_size: int) -> tuple[int, int]:
    """(num_tokens_pad, tokens_per_rank).

    [xLLM] 2 (build_cp_local_metadata): the token count is padded up to a
    multiple of cp_size and every rank holds tokens_per_rank = pad / cp_size
    rows.
    """
    if cp_size < 1:
        raise ValueError("cp_size must be >= 1")
    tokens_per_rank = -(-num_tokens // cp_size)  # ceil
    return tokens_per_rank * cp_size, tokens_per_rank


def local_rows(num_tokens: int, cp_size: int, cp_rank: int, mode: int) -> np.ndarray:
    """Flat token index held by each local slot of rank ``cp_rank``; -1 = pad.

    in-seq-split: [blog] 4 第一部分 -- rank k holds a contiguous chunk
      (8000 tokens on 8 ranks: rank k gets 1000k .. 1000k+999); [xLLM] 2 --
      the flattened stream is cut evenly, padding at the end (R1, R2).
    round-robin: [blog] 2.B -- rank r holds arange(r, tokens, cp_size), i.e.
      token g goes to rank g % cp_size, slot g // cp_size (R3).
    head-tail: the zigzag split of R2 ([xLLM] 7 names it only).
    """
    if not 0 <= cp_rank < cp_size:
        raise ValueError("cp_rank out of range")
    _, tpr = padded_geometry(num_tokens, cp_size)
    head, tail = (tpr + 1) // 2, tpr // 2  # R2: head and tail chunk lengths
    rows = np.full(tpr, -1, dtype=np.int64)
    for i in range(tpr):
        if mode == IN_SEQ_SPLIT:
            g = cp_rank * tpr + i
        elif mode == ROUND_ROBIN:
            g = cp_rank + i * cp_size
        elif mode == HEAD_TAIL:
            if i < head:
                g = cp_rank * head + i
            else:
                g = cp_size * head + (cp_size - 1 - cp_rank) * tail + (i - head)
        else:
            raise ValueError("unknown mode")
        if g < num_tokens:
            rows[i] = g
    return rows


# --------------------------------------------------------------------------
# build_cp_local_metadata
# --------------------------------------------------------------------------

def build_local_metadata(query_start_loc, seq_lens, cp_size: int, cp_rank: int, mode: int,
                         compress_ratio: int = 1) -> dict:
    """Local view metadata of one CP rank.

    [xLLM] 2: pad to a multiple of cp_size, tokens_per_rank, local_start /
    local_end; intersect the global cu-seqlens with the rank's rows to get
    local_query_start_loc and local_seq_lens; local_kv_start_loc is the
    right-aligned cumsum of local_seq_lens; cp_size == 1 is the identity.
    [xLLM] 单层前向数据流 (4): the attention call takes cu_seqlens_q =
    local_query_start_loc, cu_seqlens_ori_kv = local_kv_start_loc and
    seqused_kv = local_seq_lens; the local queries see the KV extent that
    ends at their last position (right-aligned) (R4).
    [xLLM] 5: batch_size / max_seqlen_q are replaced by the local geometry.

    Extras (R7, R12): local_req_id (global request index), local_req_kv_base
    (KV row of the request's position 0), local_req_pos_base (a local slot of
    flat query row g is at in-request position g - local_req_pos_base, i.e.
    qs_b minus the request's prefix) and local_token_pos (flat query row of
    every local slot, -1 for pad); num_tokens = T and num_kv_rows = the KV rows
    of the batch (the sum of seq_lens).

    Compressed KV (R18) at ratio c: KV extents, KV bases and the KV row count
    count compressed entries: local_seq_lens = floor(extent / c) of the token
    extent above, request b's entries start at the sum of floor(seq_lens / c)
    before it; query positions stay in tokens.
    """
    c = int(compress_ratio)
    if c < 1:
        raise ValueError("compress_ratio must be at least 1")
    qsl = [int(x) for x in query_start_loc]
    sl = [int(x) for x in seq_lens]
    B = len(sl)
    if len(qsl) != B + 1 or qsl[0] != 0:
        raise ValueError("query_start_loc must have B+1 entries starting at 0")
    prefix, kv_start = [], [0]
    for b in range(B):
        q_len = qsl[b + 1] - qsl[b]
        if q_len < 0 or sl[b] < q_len:
            raise ValueError("seq_lens[b] must be at least the query length of request b (R12)")
        prefix.append(sl[b] - q_len)
        kv_start.append(kv_start[-1] + sl[b] // c)
    T = qsl[B]
    pad, tpr = padded_geometry(T, cp_size)
    rows = local_rows(T, cp_size, cp_rank, mode)

    if mode == IN_SEQ_SPLIT:
        local_start = min(cp_rank * tpr, T)
        local_end = min((cp_rank + 1) * tpr, T)
    elif mode == HEAD_TAIL:
        # the span from the head chunk's start to the tail chunk's end (R2)
        head, tail = (tpr + 1) // 2, tpr // 2
        local_start = min(cp_rank * head, T)
        local_end = max(local_start, min(cp_size * head + (cp_size - cp_rank) * tail, T))
    else:
        # the strided range {local_start + i*cp_size < local_end}
        local_start = min(cp_rank, T)
        local_end = T

    q_lens, kv_lens, req_id, kv_base, pos_base = [], [], [], [], []
    for b in range(B):
        mine = [int(g) for g in rows if g >= 0 and qsl[b] <= g < qsl[b + 1]]
        if not mine:
            continue  # R5
        q_lens.append(len(mine))
        kv_lens.append((prefix[b] + max(mine) - qsl[b] + 1) // c)  # R4: last local position + 1 (R18: entries)
        req_id.append(b)
        kv_base.append(kv_start[b])         # R12: KV row of position 0
        pos_base.append(qsl[b] - prefix[b])  # position of flat row g = g - pos_base

    lqs = [0]
    for n in q_lens:
        lqs.append(lqs[-1] + n)
    lkv = [0]
    for n in kv_lens:
        lkv.append(lkv[-1] + n)

    return {
        "num_tokens_pad": pad,
        "tokens_per_rank": tpr,
        "local_start": local_start,
        "local_end": local_end,
        "local_batch": len(q_lens),
        "local_num_tokens": lqs[-1],
        "local_max_seqlen_q": max(q_lens) if q_lens else 0,
        "local_max_seqlen_kv": max(kv_lens) if kv_lens else 0,
        "local_query_start_loc": lqs,
        "local_seq_lens": kv_lens,
        "local_kv_start_loc": lkv,
        "local_req_id": req_id,
        "local_req_kv_base": kv_base,
        "local_token_pos": [int(g) for g in rows],
        "local_req_pos_base": pos_base,
        "num_tokens": T,
        "num_kv_rows": kv_start[-1],
        "compress_ratio": c,
    }


# --------------------------------------------------------------------------
# split and rerange
# --------------------------------------------------------------------------

def split(x: np.ndarray, cp_size: int, mode: int) -> np.ndarray:
    """Rank-major local layout [cp_size][tokens_per_rank][row...], pad rows zero.

    [blog] 2.B / 第三部分 step 1: each rank gathers its own rows (T0,T4 on
    rank 0 of 4); [blog] 第三部分 step B: concatenated by rank this is the
    all-gathered order T0,T4,T1,T5,...; [xLLM] 单层前向数据流 (6): pad to
    tokens_per_rank.
    """
    T = x.shape[0]
    _, tpr = padded_geometry(T, cp_size)
    out = np.zeros((cp_size, tpr) + x.shape[1:], dtype=x.dtype)
    for r in range(cp_size):
        for i, g in enumerate(local_rows(T, cp_size, r, mode)):
            if g >= 0:
                out[r, i] = x[g]
    return out


def rerange(y: np.ndarray, num_tokens: int, cp_size: int, mode: int) -> np.ndarray:
    """Inverse of :func:`split`: rank-major rows back to logical token order.

    [blog] 第三部分 step B and [sglang] 第一次 All-Gather: after the
    all-gather the rows are in rank order and are re-arranged into the
    original flat order T0, T1, T2, ...; pad rows are dropped.
    """
    out = np.zeros((num_tokens,) + y.shape[2:], dtype=y.dtype)
    for r in range(cp_size):
        for i, g in enumerate(local_rows(num_tokens, cp_size, r, mode)):
            if g >= 0:
                out[g] = y[r, i]
    return out


def all_to_all_heads(y: np.ndarray, num_tokens: int, cp_size: int, mode: int) -> np.ndarray:
    """Head/token transpose of the views' attention outputs (R16).

    [xLLM] 单层前向数据流 (6) and "3. DSAttention 前向": each rank holds its
    attention output [T_local padded to tokens_per_rank, num_heads_full,
    head_dim]; an all_to_all that scatters the head dimension and gathers the
    token dimension leaves rank r' with [tokens, num_heads_full / cp_size,
    head_dim], the pad rows sliced off, ready for the tensor-parallel o_proj.
    y [cp][tpr][H][Dv] -> [cp][num_tokens][H / cp][Dv].
    """
    H = y.shape[2]
    if H % cp_size:
        raise ValueError("the head count must divide by cp_size")
    hc = H // cp_size
    out = np.zeros((cp_size, num_tokens, hc) + y.shape[3:], dtype=y.dtype)
    for r in range(cp_size):  # the view that computed the token
        for i, g in enumerate(local_rows(num_tokens, cp_size, r, mode)):
            if g < 0:
                continue
            for rd in range(cp_size):  # the rank that receives heads rd*hc ..
                out[rd, g] = y[r, i, rd * hc:(rd + 1) * hc]
    return out


# --------------------------------------------------------------------------
# lightning indexer, top-k, sparse attention (one query row at a time)
# --------------------------------------------------------------------------

def indexer_scores(q_idx_row: np.ndarray, w_row: np.ndarray, k_idx_keys: np.ndarray) -> np.ndarray:
    """I[s] = sum_j w[j] * max(0, q_I[j] . k_I[s]) for every key row s given.

    q_idx_row [HI, DI], w_row [HI], k_idx_keys [n, DI] -> fp64 [n].  The
    indexer query and weights are the rank's local rows, the index keys are
    the full-token keys ([xLLM] 单层前向数据流 (2)(3), 4. Indexer full/local).
    """
    q = np.asarray(q_idx_row, dtype=np.float64)
    w = np.asarray(w_row, dtype=np.float64)
    k = np.asarray(k_idx_keys, dtype=np.float64)
    dots = q @ k.T                    # [HI, n]: q_I[j] . k_I[s]
    return w @ np.maximum(dots, 0.0)  # sum over heads j of w[j] * ReLU(.)


def topk_positions(scores: np.ndarray, k: int) -> np.ndarray:
    """The k positions with the largest scores, ties to the lower position.

    R9: a row with n <= k keys selects all of them (never collapses to
    position 0, cf. [xLLM] 5 "top-k 塌缩到 position 0").  Otherwise the k-th
    largest value is the threshold; every position above it is selected and
    the remaining places go to the lowest positions equal to it.  numpy's
    comparison treats -0.0 == +0.0.  Returned ascending.
    """
    s = np.asarray(scores, dtype=np.float64)
    if np.isnan(s).any():
        raise ValueError("NaN score")
    n = s.shape[0]
    if n <= k:
        return np.arange(n, dtype=np.int64)
    threshold = np.sort(s)[n - k]       # k-th largest
    above = np.nonzero(s > threshold)[0]
    equal = np.nonzero(s == threshold)[0]
    chosen = np.concatenate([above, equal[: k - above.shape[0]]])
    return np.sort(chosen)


def sparse_attention(q_row: np.ndarray, kv_sel: np.ndarray, scale: float, Dv: int, sink=None) -> np.ndarray:
    """MLA attention of every head of one query over the selected latent rows.

    q_row [H, D], kv_sel [n, D] (key = the full D-wide latent row, value =
    its first Dv columns), sink [H] or None -> fp64 [H, Dv]:
      l[h, j] = scale * q[h] . kv[j]
      m[h]    = max(max_j l[h, j], sink[h])
      o[h]    = sum_j exp(l[h, j] - m[h]) kv[j, :Dv] / (sum_j exp(l[h, j] - m[h]) + exp(sink[h] - m[h]))
    with the sink terms present only when a sink is given (R10).
    """
    q = np.asarray(q_row, dtype=np.float64)
    kv = np.asarray(kv_sel, dtype=np.float64)
    logits = scale * (q @ kv.T)                       # [H, n]
    m = logits.max(axis=1)
    if sink is not None:
        sk = np.asarray(sink, dtype=np.float64)
        m = np.maximum(m, sk)
    e = np.exp(logits - m[:, None])
    z = e.sum(axis=1)
    if sink is not None:
        z = z + np.exp(sk - m)
    return (e @ kv[:, :Dv]) / z[:, None]


def request_of_slot(md: dict, slot: int) -> int:
    """Local request index j with local_query_start_loc[j] <= slot < [j+1]."""
    lqs = md["local_query_start_loc"]
    for j in range(md["local_batch"]):
        if lqs[j] <= slot < lqs[j + 1]:
            return j
    return -1


def view_row(md: dict, slot: int, q_loc, q_idx_loc, w_loc, kv, k_idx, topk: int, scale: float,
             Dv: int, sink=None):
    """Indexer -> top-k -> sparse attention for one local slot of one view.

    Returns (selected global KV rows ascending [<=topk] int64, scores fp64
    [p+1], output fp64 [H, Dv]); (None, None, zeros) for a pad slot.
    The local query of flat row g in request b, at in-request position
    p = g - local_req_pos_base (= g - qs_b without a prefix), sees the keys at
    positions 0 .. p of its own request, KV rows kv_base .. kv_base + p
    (causal, same request; R7, R12).  At compress ratio c (R18) it sees the
    entries 0 .. floor((p + 1) / c) - 1 instead; with none, nothing is selected
    and the output is zero.
    """
    g = md["local_token_pos"][slot]
    H = np.asarray(q_loc[slot]).shape[0]
    if g < 0:
        return None, None, np.zeros((H, Dv))
    j = request_of_slot(md, slot)
    base = md["local_req_kv_base"][j]
    p = g - md["local_req_pos_base"][j]
    n = (p + 1) // md.get("compress_ratio", 1)
    if n == 0:
        return np.zeros(0, dtype=np.int64), np.zeros(0), np.zeros((H, Dv))
    keys = np.arange(base, base + n)
    scores = indexer_scores(q_idx_loc[slot], w_loc[slot], np.asarray(k_idx)[keys])
    sel = base + topk_positions(scores, topk)
    out = sparse_attention(q_loc[slot], np.asarray(kv)[sel], scale, Dv, sink)
    return sel, scores, out


def prefill_view(md: dict, q_loc, q_idx_loc, w_loc, kv, k_idx, topk: int, scale: float, Dv: int,
                 sink=None, slots=None):
    """One CP view: (topk_idx [tpr, topk] int64 global rows, -1 pad;
    out [tpr, H, Dv] fp64, pad rows 0).  ``slots`` restricts the work to a
    subset of local slots (others stay -1 / 0)."""
    tpr = md["tokens_per_rank"]
    H = np.asarray(q_loc).shape[1]
    idx = np.full((tpr, topk), -1, dtype=np.int64)
    out = np.zeros((tpr, H, Dv))
    for i in (range(tpr) if slots is None else slots):
        sel, _, o = view_row(md, int(i), q_loc, q_idx_loc, w_loc, kv, k_idx, topk, scale, Dv, sink)
        if sel is not None:
            idx[i, : sel.shape[0]] = sel
            out[i] = o
    return idx, out


def prefill(q, kv, q_idx, k_idx, w, query_start_loc, seq_lens, cp_size: int, mode: int, topk: int,
            scale: float, Dv: int, sink=None, compress_ratio: int = 1):
    """The whole prefill through cp_size views: split the local tensors, run
    every view with full KV and index keys, rerange the outputs to flat order
    ([xLLM] 单层前向数据流: q local, KV full).  q, q_idx, w hold the T query
    tokens; kv and k_idx the KV rows of every request's whole sequence (R12;
    the same T rows when seq_lens equal the query lengths).  Returns
    out [T, H, Dv] fp64."""
    q = np.asarray(q, dtype=np.float64)
    q_idx = np.asarray(q_idx, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T = q.shape[0]
    qs, qis, ws = split(q, cp_size, mode), split(q_idx, cp_size, mode), split(w, cp_size, mode)
    _, tpr = padded_geometry(T, cp_size)
    outs = np.zeros((cp_size, tpr, q.shape[1], Dv))
    for r in range(cp_size):
        md = build_local_metadata(query_start_loc, seq_lens, cp_size, r, mode, compress_ratio)
        _, outs[r] = prefill_view(md, qs[r], qis[r], ws[r], kv, k_idx, topk, scale, Dv, sink)
    return rerange(outs, T, cp_size, mode)


# --------------------------------------------------------------------------
# FP8 latent-KV cache (R17)
# --------------------------------------------------------------------------
#
# R17 "FP8 KV Cache" ([blog] 1 核心改动总结: round-robin-split lifts the old
#     restriction that NSA prefill CP could not use an FP8 KV cache) is named
#     without a format.  Reading taken: the published DeepSeek-V3.2 layout of
#     one latent row -- the Dv value ("nope") columns as OCP FP8 E4M3 codes with
#     one fp32 scale per tile of 128 columns (scale = tile max|x| / 448, 1 for
#     an all-zero tile), then the D - Dv rope columns kept as bf16, the row
#     padded with zero bytes to a multiple of 16.  Codes round to nearest even
#     and saturate at +-448; decisions are taken in fp32 (x / scale).  The
#     attention over the cache is the attention over its dequantized rows,
#     bf16(fp32(decode(code)) * scale).

E4M3_MAX = 448.0
FP8_TILE = 128


def e4m3_decode(codes) -> np.ndarray:
    """Values of OCP E4M3 codes (1 sign, 4 exponent bits with bias 7, 3
    mantissa bits; exponent field 0 is subnormal, S.1111.111 is NaN, no
    infinities) as float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = (c >> 7) & 1
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def e4m3_encode(v) -> np.ndarray:
    """Nearest E4M3 code of each finite value, ties to the even mantissa,
    magnitudes above 448 clamped to 448; the sign is kept (also of zero)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1)
    binade = np.maximum(ex - 1, -6)           # subnormals share the 2^-6 binade's step
    step = np.exp2(binade - 3.0)              # 3 mantissa bits
    r = np.rint(a / step) * step              # round half to even (exact scaling)
    r = np.minimum(r, E4M3_MAX)
    _, ex2 = np.frexp(r)
    e_unb = ex2 - 1
    normal = r >= 2.0 ** -6
    e_field = np.where(normal, e_unb + 7, 0)
    m_field = np.where(normal, r / np.exp2(e_unb.astype(np.float64)) * 8.0 - 8.0, r / 2.0 ** -9)
    code = (e_field.astype(np.int64) << 3) | np.rint(m_field).astype(np.int64)
    code = code | (np.signbit(v).astype(np.int64) << 7)
    return code.astype(np.uint8)


def bf16_round(x) -> np.ndarray:
    """fp32 values rounded to the nearest bf16 (ties to even), as float32."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def kv_fp8_row_bytes(D: int, Dv: int) -> int:
    """Bytes of one cache row: Dv codes, 4 bytes per 128-column tile, 2 bytes
    per rope column, padded to a multiple of 16."""
    tiles = -(-Dv // FP8_TILE)
    raw = Dv + 4 * tiles + 2 * (D - Dv)
    return -(-raw // 16) * 16


def kv_fp8_quantize(kv, Dv: int) -> np.ndarray:
    """bf16-valued latent rows kv [R, D] -> cache bytes [R, kv_fp8_row_bytes]."""
    x = np.asarray(kv, dtype=np.float32)
    R, D = x.shape
    tiles = -(-Dv // FP8_TILE)
    out = np.zeros((R, kv_fp8_row_bytes(D, Dv)), dtype=np.uint8)
    for t in range(tiles):
        cols = slice(t * FP8_TILE, min((t + 1) * FP8_TILE, Dv))
        amax = np.abs(x[:, cols]).max(axis=1)
        scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        v = (x[:, cols] / scale[:, None]).astype(np.float32)   # fp32 division, rounded to nearest
        out[:, cols] = e4m3_encode(v)
        out[:, Dv + 4 * t: Dv + 4 * t + 4] = scale.view(np.uint8).reshape(R, 4)
    rope = x[:, Dv:].astype(np.float32).view(np.uint32) >> 16     # bf16-valued: the upper half
    off = Dv + 4 * tiles
    out[:, off: off + 2 * (D - Dv)] = rope.astype(np.uint16).view(np.uint8).reshape(R, 2 * (D - Dv))
    return out


def kv_fp8_dequantize(cache, D: int, Dv: int) -> np.ndarray:
    """Cache bytes [R, row_bytes] -> the latent rows [R, D] it stands for
    (bf16 values as float64): value column c of tile t is
    bf16(fp32(decode(code)) * scale_t), rope columns are the stored bf16."""
    b = np.asarray(cache, dtype=np.uint8)
    R = b.shape[0]
    tiles = -(-Dv // FP8_TILE)
    out = np.zeros((R, D), dtype=np.float64)
    for t in range(tiles):
        cols = slice(t * FP8_TILE, min((t + 1) * FP8_TILE, Dv))
        scale = np.ascontiguousarray(b[:, Dv + 4 * t: Dv + 4 * t + 4]).view(np.float32).reshape(R)
        val = e4m3_decode(b[:, cols]).astype(np.float32) * scale[:, None]    # fp32 product, rounded
        out[:, cols] = bf16_round(val)
    off = Dv + 4 * tiles
    rope16 = np.ascontiguousarray(b[:, off: off + 2 * (D - Dv)]).view(np.uint16).astype(np.uint32) << 16
    out[:, Dv:] = rope16.view(np.float32)
    return out


# --------------------------------------------------------------------------
# FP8 indexer operands (R19)
# --------------------------------------------------------------------------

def index_fp8_values(rows, DI: int) -> np.ndarray:
    """FP8 index rows [R, kv_fp8_row_bytes(DI, DI)] -> the values they stand
    for, [R, DI] float64: decode(code) * scale of the code's 128-column tile,
    exact (an E4M3 value has 4 significant bits, an fp32 scale 24)."""
    b = np.asarray(rows, dtype=np.uint8)
    R = b.shape[0]
    tiles = -(-DI // FP8_TILE)
    out = np.zeros((R, DI), dtype=np.float64)
    for t in range(tiles):
        cols = slice(t * FP8_TILE, min((t + 1) * FP8_TILE, DI))
        scale = np.ascontiguousarray(b[:, DI + 4 * t: DI + 4 * t + 4]).view(np.float32).reshape(R)
        out[:, cols] = e4m3_decode(b[:, cols]) * scale.astype(np.float64)[:, None]
    return out


def indexer_scores_fp8(q_idx_row8, w_row, k_idx_keys8, DI: int) -> np.ndarray:
    """The indexer score (indexer_scores) of the values FP8 index rows stand
    for: q_idx_row8 [HI, row_bytes] (one query's heads), k_idx_keys8
    [n, row_bytes] -> fp64 [n]."""
    return indexer_scores(index_fp8_values(q_idx_row8, DI), w_row, index_fp8_values(k_idx_keys8, DI))


# --------------------------------------------------------------------------
# Sliding window over the original KV (R20)
# --------------------------------------------------------------------------

def window_rows(p: int, ori_start: int, window: int) -> np.ndarray:
    """Original KV rows of the positions max(0, p - W + 1) .. p of a request
    whose position 0 is original row ori_start (none for W = 0)."""
    if window <= 0:
        return np.zeros(0, dtype=np.int64)
    return np.arange(ori_start + max(0, p - window + 1), ori_start + p + 1, dtype=np.int64)


def view_row_swa(md: dict, slot: int, q_loc, q_idx_loc, w_loc, kv, k_idx, topk: int, scale: float, Dv: int,
                 window: int, kv_ori, ori_starts, sink=None):
    """One local slot with the sliding window (R20): the selection of view_row
    over the (compressed) rows ``kv``, plus the window rows of ``kv_ori``
    (the original rows; request b starts at ori_starts[b]), one softmax over
    both.  Returns (selected rows, window rows, output fp64 [H, Dv]); (None,
    None, zeros) for a pad slot."""
    sel, _, _ = view_row(md, slot, q_loc, q_idx_loc, w_loc, kv, k_idx, topk, scale, Dv, sink)
    H = np.asarray(q_loc[slot]).shape[0]
    if sel is None:
        return None, None, np.zeros((H, Dv))
    j = request_of_slot(md, slot)
    p = md["local_token_pos"][slot] - md["local_req_pos_base"][j]
    win = window_rows(p, ori_starts[md["local_req_id"][j]], window)
    if md.get("compress_ratio", 1) == 1:  # the same rows: their union
        rows = np.asarray(kv)[np.union1d(sel, win)]
    else:
        rows = np.concatenate([np.asarray(kv)[sel], np.asarray(kv_ori)[win]])
    if rows.shape[0] == 0:
        return sel, win, np.zeros((H, Dv))
    return sel, win, sparse_attention(q_loc[slot], rows, scale, Dv, sink)


def prefill_swa(q, kv, q_idx, k_idx, w, query_start_loc, seq_lens, cp_size: int, mode: int, topk: int,
                scale: float, Dv: int, window: int, kv_ori=None, sink=None, compress_ratio: int = 1):
    """prefill with the sliding window (R20): ``kv`` / ``k_idx`` are the rows
    the indexer selects from (compressed entries at compress_ratio > 1),
    ``kv_ori`` the original rows of every request's whole sequence (``kv``
    itself when omitted, as at c = 1).  Returns out [T, H, Dv] fp64."""
    q = np.asarray(q, dtype=np.float64)
    q_idx = np.asarray(q_idx, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    kv_ori = kv if kv_ori is None else kv_ori
    ori_starts = np.concatenate([[0], np.cumsum(seq_lens)]).astype(np.int64)
    T = q.shape[0]
    qs, qis, ws = split(q, cp_size, mode), split(q_idx, cp_size, mode), split(w, cp_size, mode)
    _, tpr = padded_geometry(T, cp_size)
    outs = np.zeros((cp_size, tpr, q.shape[1], Dv))
    for r in range(cp_size):
        md = build_local_metadata(query_start_loc, seq_lens, cp_size, r, mode, compress_ratio)
        for i in range(tpr):
            _, _, outs[r, i] = view_row_swa(md, i, qs[r], qis[r], ws[r], kv, k_idx, topk, scale, Dv, window,
                                            kv_ori, ori_starts, sink)
    return rerange(outs, T, cp_size, mode)
