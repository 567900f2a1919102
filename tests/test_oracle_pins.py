"""Pins for the fp64 oracle, against things other than the oracle itself:
worked examples printed on the pages (tests/golden/), hand-derived cases,
closed forms, invariants the pages state, and independent library routines
(torch's scaled_dot_product_attention, Python's stable ``sorted``).

Each pin is chosen so that a plausible slip in the oracle (an off-by-one in
the causal extent, a dropped ReLU, a transposed operand, a wrong tie rule, a
sink added to the numerator, a wrong rank-row mapping) fails at least one test.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden, read_golden_lines
from oracle import dsa_oracle as O
from workloads import HEAD_TAIL, IN_SEQ_SPLIT, ROUND_ROBIN, TINY, TINY_INT, chunk_inputs, draw_inputs

MODES = (IN_SEQ_SPLIT, ROUND_ROBIN, HEAD_TAIL)


def _f64(t):
    return t.to(torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, dtype=np.float64)


# ---------------------------------------------------------------- split geometry

def test_round_robin_worked_example():
    g = read_golden("round_robin_cp4_t8.txt")
    T, cp = g["num_tokens"][0], g["cp_size"][0]
    for r in range(cp):
        assert list(O.local_rows(T, cp, r, ROUND_ROBIN)) == g[f"rank{r}"]
    x = np.arange(T)
    gathered = O.split(x, cp, ROUND_ROBIN).reshape(-1)
    assert list(gathered) == g["gathered_order"]
    assert list(O.rerange(gathered.reshape(cp, -1), T, cp, ROUND_ROBIN)) == g["reranged_order"]


def test_in_seq_worked_example():
    g = read_golden("in_seq_cp8_t8000.txt")
    T, cp = g["num_tokens"][0], g["cp_size"][0]
    for r in range(cp):
        rows = O.local_rows(T, cp, r, IN_SEQ_SPLIT)
        assert rows[0] == g["first"][r] and rows[-1] == g["last"][r]
        assert np.all(np.diff(rows) == 1)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,cp", [(1, 1), (7, 2), (12, 3), (13, 4), (5, 16), (100, 8), (257, 2)])
def test_split_rerange_identity_and_padding(T, cp, mode):
    x = np.arange(T * 3, dtype=np.int64).reshape(T, 3) + 1  # no zero rows
    y = O.split(x, cp, mode)
    pad, tpr = O.padded_geometry(T, cp)
    assert y.shape == (cp, tpr, 3) and pad == tpr * cp and pad - T < cp
    assert np.array_equal(O.rerange(y, T, cp, mode), x)
    # every real row appears exactly once, pad rows are zero
    flat = y.reshape(-1, 3)
    nonzero = flat[np.any(flat != 0, axis=1)]
    assert nonzero.shape[0] == T and np.all(flat[np.all(flat == 0, axis=1)] == 0)


@pytest.mark.parametrize("T,cp", [(8, 4), (11805, 4), (65536, 8), (5, 16), (184265, 16)])
def test_round_robin_counts_differ_by_at_most_one(T, cp):
    counts = [int(np.sum(O.local_rows(T, cp, r, ROUND_ROBIN) >= 0)) for r in range(cp)]
    assert sum(counts) == T and max(counts) - min(counts) <= 1


def test_head_tail_hand_examples():
    # zigzag: tokens_per_rank as for the other modes; head chunks of ceil(tpr/2)
    # rows, tail chunks of floor(tpr/2) rows in reverse rank order
    assert O.local_rows(10, 2, 0, HEAD_TAIL).tolist() == [0, 1, 2, 8, 9]
    assert O.local_rows(10, 2, 1, HEAD_TAIL).tolist() == [3, 4, 5, 6, 7]
    assert O.local_rows(9, 2, 0, HEAD_TAIL).tolist() == [0, 1, 2, 8, -1]
    assert O.local_rows(8, 2, 0, HEAD_TAIL).tolist() == [0, 1, 6, 7]
    assert O.local_rows(8, 2, 1, HEAD_TAIL).tolist() == [2, 3, 4, 5]


@pytest.mark.parametrize("T,cp", [(16, 2), (64, 4), (96, 8), (48, 3)])
def test_head_tail_is_the_textbook_zigzag_for_even_chunks(T, cp):
    # with T a multiple of 2*cp, rank r holds equal chunks r and 2cp-1-r of the
    # stream cut into 2cp pieces (numpy's array_split)
    chunks = np.array_split(np.arange(T), 2 * cp)
    for r in range(cp):
        want = np.concatenate([chunks[r], chunks[2 * cp - 1 - r]])
        assert np.array_equal(O.local_rows(T, cp, r, HEAD_TAIL), want)


@pytest.mark.parametrize("T,cp", [(11805, 4), (65536, 8), (184265, 16)])
def test_head_tail_balances_causal_work(T, cp):
    # the sum of in-stream positions (a proxy for causal attention work) per rank
    # is far more even than with the contiguous in-seq-split
    def spread(mode):
        work = [int(np.sum(r[r >= 0])) for r in (O.local_rows(T, cp, k, mode) for k in range(cp))]
        return max(work) / max(1, min(work))
    assert spread(HEAD_TAIL) < 1.2 < spread(IN_SEQ_SPLIT)


# ---------------------------------------------------------------- head/token all-to-all

def test_all_to_all_hand_example():
    # 3 tokens, cp 2, 2 heads, head_dim 2; y[r][i][h][d] = 1000r + 100i + 10h + d
    y = np.zeros((2, 2, 2, 2), dtype=np.int64)
    for r in range(2):
        for i in range(2):
            for h in range(2):
                for d in range(2):
                    y[r, i, h, d] = 1000 * r + 100 * i + 10 * h + d
    names = {"in_seq": IN_SEQ_SPLIT, "round_robin": ROUND_ROBIN}
    outs = {m: O.all_to_all_heads(y, 3, 2, mode) for m, mode in names.items()}
    lines = read_golden_lines("all_to_all_hand_example.txt")
    assert len(lines) == 12
    for line in lines:
        m, rank, tok, d0, d1 = line.split()
        assert list(outs[m][int(rank), int(tok), 0]) == [int(d0), int(d1)], line


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,cp,H", [(1, 1, 4), (7, 2, 4), (13, 4, 8), (5, 8, 8), (33, 4, 128)])
def test_all_to_all_of_split_is_a_head_transpose(T, cp, H, mode):
    # split then all-to-all == reshaping the full [T][H][Dv] tensor into
    # [T][cp][H/cp][Dv] and moving the rank axis first (plain numpy)
    rng = np.random.default_rng(T * 100 + cp)
    x = rng.integers(-1000, 1000, size=(T, H, 3))
    out = O.all_to_all_heads(O.split(x, cp, mode), T, cp, mode)
    assert np.array_equal(out, np.moveaxis(x.reshape(T, cp, H // cp, 3), 1, 0))


@pytest.mark.parametrize("mode", MODES)
def test_all_to_all_is_a_permutation_of_the_real_rows(mode):
    T, cp, H = 10, 4, 8
    _, tpr = O.padded_geometry(T, cp)
    y = np.arange(1, cp * tpr * H * 2 + 1, dtype=np.int64).reshape(cp, tpr, H, 2)
    out = O.all_to_all_heads(y, T, cp, mode)
    real = np.concatenate([y[r, O.local_rows(T, cp, r, mode) >= 0].ravel() for r in range(cp)])
    assert out.shape == (cp, T, H // cp, 2)
    assert np.array_equal(np.sort(out.ravel()), np.sort(real))


def test_all_to_all_cp1_is_identity_and_rejects_indivisible_heads():
    x = np.arange(5 * 6 * 2).reshape(5, 6, 2)
    assert np.array_equal(O.all_to_all_heads(x[None], 5, 1, IN_SEQ_SPLIT)[0], x)
    with pytest.raises(ValueError):
        O.all_to_all_heads(O.split(x, 4, ROUND_ROBIN), 5, 4, ROUND_ROBIN)


# ---------------------------------------------------------------- metadata

_CASES = {"A": [5, 3, 4], "B": [3, 4], "C": [5, 1]}
_CP = {"A": 3, "B": 2, "C": 4}


def _qsl(lengths):
    return [0] + list(np.cumsum(lengths))


def _ints(s):
    s = s.strip()
    return [] if s == "-" else [int(x) for x in s.split()]


def test_metadata_hand_cases():
    for line in read_golden_lines("metadata_hand_cases.txt"):
        head, lqs, kvl, lkv, rid, base, pos = line.split("|")
        case, mode_s, rank = head.split()
        lengths = _CASES[case]
        mode = {"inseq": IN_SEQ_SPLIT, "rr": ROUND_ROBIN, "ht": HEAD_TAIL}[mode_s]
        md = O.build_local_metadata(_qsl(lengths), lengths, _CP[case], int(rank), mode)
        assert md["local_query_start_loc"] == _ints(lqs), line
        assert md["local_seq_lens"] == _ints(kvl), line
        assert md["local_kv_start_loc"] == _ints(lkv), line
        assert md["local_req_id"] == _ints(rid), line
        assert md["local_req_kv_base"] == _ints(base), line
        assert md["local_token_pos"] == _ints(pos), line
        assert md["local_batch"] == len(_ints(kvl))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("lengths,cp", [([8000, 800, 5, 3000], 4), ([5, 3, 4], 3), ([1, 1, 1], 8),
                                        ([256], 2), ([17, 1, 30, 2], 5)])
def test_metadata_partitions_all_query_tokens(lengths, cp, mode):
    qsl = _qsl(lengths)
    T = qsl[-1]
    owner = np.zeros(T, dtype=np.int64)
    total = 0
    for r in range(cp):
        md = O.build_local_metadata(qsl, lengths, cp, r, mode)
        total += md["local_num_tokens"]
        for g in md["local_token_pos"]:
            if g >= 0:
                owner[g] += 1
        # local_kv_start_loc is the exclusive cumsum of local_seq_lens
        assert md["local_kv_start_loc"] == [0] + list(np.cumsum(md["local_seq_lens"]))
        # every local query's position is inside its request's visible extent
        for j in range(md["local_batch"]):
            for slot in range(md["local_query_start_loc"][j], md["local_query_start_loc"][j + 1]):
                p = md["local_token_pos"][slot] - md["local_req_pos_base"][j]
                assert 0 <= p < md["local_seq_lens"][j]
    assert total == T and np.all(owner == 1)


@pytest.mark.parametrize("mode", MODES)
def test_metadata_cp1_is_identity(mode):
    lengths = [8000, 800, 5, 3000]
    qsl = _qsl(lengths)
    md = O.build_local_metadata(qsl, lengths, 1, 0, mode)
    assert md["local_query_start_loc"] == qsl
    assert md["local_kv_start_loc"] == qsl
    assert md["local_seq_lens"] == lengths
    assert md["local_token_pos"] == list(range(qsl[-1]))
    assert md["tokens_per_rank"] == qsl[-1] == md["num_tokens_pad"]


def test_metadata_in_seq_right_aligned_extent():
    # the last in-seq rank sees the full KV stream of the last request; every
    # other rank's extent ends at its own last local token
    lengths = [8192]
    for cp in (2, 4, 8):
        for r in range(cp):
            md = O.build_local_metadata([0, 8192], lengths, cp, r, IN_SEQ_SPLIT)
            assert md["local_seq_lens"] == [8192 // cp * (r + 1)]
            assert md["local_start"] == 8192 // cp * r and md["local_end"] == 8192 // cp * (r + 1)


def test_metadata_rejects_seq_lens_shorter_than_queries():
    with pytest.raises(ValueError):
        O.build_local_metadata([0, 4], [3], 2, 0, IN_SEQ_SPLIT)


_PREFIX_CASES = {"P": ([3, 2], [5, 2], 2), "Q": ([4], [10], 3)}  # q_lens, seq_lens, cp


def test_metadata_prefix_hand_cases():
    seen = set()
    for line in read_golden_lines("metadata_prefix_hand_cases.txt"):
        head, lqs, kvl, lkv, rid, base, pbase, pos = line.split("|")
        case, mode_s, rank = head.split()
        q_lens, seq_lens, cp = _PREFIX_CASES[case]
        mode = {"inseq": IN_SEQ_SPLIT, "rr": ROUND_ROBIN, "ht": HEAD_TAIL}[mode_s]
        md = O.build_local_metadata(_qsl(q_lens), seq_lens, cp, int(rank), mode)
        assert md["local_query_start_loc"] == _ints(lqs), line
        assert md["local_seq_lens"] == _ints(kvl), line
        assert md["local_kv_start_loc"] == _ints(lkv), line
        assert md["local_req_id"] == _ints(rid), line
        assert md["local_req_kv_base"] == _ints(base), line
        assert md["local_req_pos_base"] == _ints(pbase), line
        assert md["local_token_pos"] == _ints(pos), line
        assert md["num_tokens"] == sum(q_lens) and md["num_kv_rows"] == sum(seq_lens)
        seen.add((case, mode_s, int(rank)))
    assert len(seen) == 12


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("q_lens,prefixes,cp", [([37, 20, 9], [25, 0, 4], 3), ([5, 1, 12], [0, 30, 3], 4),
                                                ([64], [192], 8)])
def test_metadata_prefix_extents(q_lens, prefixes, cp, mode):
    # with a prefix the extents stay right-aligned: every local query sits inside
    # its request's visible extent, the extents of a request over all ranks end at
    # its seq_len, and the KV base of request b is the sum of the seq_lens before it
    seq_lens = [n + p for n, p in zip(q_lens, prefixes)]
    qsl = _qsl(q_lens)
    widest = [0] * len(q_lens)
    for r in range(cp):
        md = O.build_local_metadata(qsl, seq_lens, cp, r, mode)
        for j in range(md["local_batch"]):
            b = md["local_req_id"][j]
            assert md["local_req_kv_base"][j] == sum(seq_lens[:b])
            assert md["local_req_pos_base"][j] == qsl[b] - prefixes[b]
            widest[b] = max(widest[b], md["local_seq_lens"][j])
            for slot in range(md["local_query_start_loc"][j], md["local_query_start_loc"][j + 1]):
                p = md["local_token_pos"][slot] - md["local_req_pos_base"][j]
                assert prefixes[b] <= p < md["local_seq_lens"][j] <= seq_lens[b]
    assert widest == seq_lens


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("cp", [1, 2, 3])
def test_chunked_prefill_rows_equal_whole_prefill(cp, mode):
    # a request processed as prefix (KV only) + chunk (queries) gives exactly the
    # chunk's rows of the whole-sequence prefill: the same keys, scores, top-k and
    # attention per row, only the geometry differs
    lengths, prefixes = [37, 20, 9], [25, 0, 4]
    wl = TINY.with_(name="tiny-chunk", lengths=tuple(lengths), topk=8, sink=True)
    x = draw_inputs(wl)
    xf = {k: (_f64(v) if v is not None else None) for k, v in x.items()}
    whole = O.prefill(xf["q"], xf["kv"], xf["q_idx"], xf["k_idx"], xf["w"], _qsl(lengths), lengths, cp, mode,
                      wl.topk, wl.scale, wl.Dv, xf["sink"])
    xc, q_lens, seq_lens = chunk_inputs(x, lengths, prefixes)
    xcf = {k: (_f64(v) if v is not None else None) for k, v in xc.items()}
    chunk = O.prefill(xcf["q"], xcf["kv"], xcf["q_idx"], xcf["k_idx"], xcf["w"], _qsl(q_lens), seq_lens, cp, mode,
                      wl.topk, wl.scale, wl.Dv, xcf["sink"])
    rows = [g for b, (n, p) in enumerate(zip(lengths, prefixes)) for g in range(sum(lengths[:b]) + p,
                                                                                 sum(lengths[:b]) + n)]
    assert chunk.shape[0] == sum(q_lens)
    np.testing.assert_allclose(chunk, whole[rows], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- indexer

def test_indexer_hand_example():
    g = read_golden("indexer_hand_example.txt")
    q = np.array(g["q_idx"], dtype=float).reshape(2, 2)
    k = np.array(g["k_idx"], dtype=float).reshape(-1, 2)
    s = O.indexer_scores(q, g["w"], k)
    assert np.array_equal(s, np.array(g["scores"], dtype=float))
    for kk in (2, 3, 4):
        assert list(O.topk_positions(s, kk)) == g[f"top{kk}"]


def test_indexer_closed_form_unit_queries():
    # head j reads dim j only (q_I[j] = e_j); k_I[s, j] = (j + 1) * (s - 2j - 1)
    # => I[s] = sum_j w[j] (j+1) max(0, s - 2j - 1): a ramp per head that turns on
    # at s = 2j + 2.  A transposed q/k, a dropped ReLU or a wrong w index breaks it.
    HI = DI = 4
    n = 12
    q = np.eye(HI, DI)
    w = np.array([0.5, -1.0, 2.0, 0.25])
    k = np.array([[(j + 1) * (s - 2 * j - 1) for j in range(DI)] for s in range(n)], dtype=float)
    expect = np.array([sum(w[j] * (j + 1) * max(0, s - 2 * j - 1) for j in range(HI)) for s in range(n)])
    assert np.array_equal(O.indexer_scores(q, w, k), expect)


def test_indexer_relu_kills_negative_dots_and_w_scales():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, 8))
    k = -np.abs(rng.standard_normal((10, 8)))
    q = np.abs(q)                     # every dot q . k < 0 -> ReLU 0
    assert np.all(O.indexer_scores(q, [1.0, 2.0, 3.0], k) == 0.0)
    k2 = rng.standard_normal((10, 8))
    w = rng.standard_normal(3)
    s1 = O.indexer_scores(q, w, k2)
    assert np.array_equal(O.indexer_scores(q, 2.0 * w, k2), 2.0 * s1)
    assert np.array_equal(O.indexer_scores(q, -w, k2), -s1)


# ---------------------------------------------------------------- top-k

def test_topk_ties_and_short_rows():
    assert list(O.topk_positions([5, 3, 3, 1, 3, 7], 3)) == [0, 1, 5]
    assert list(O.topk_positions([2.0] * 10, 4)) == [0, 1, 2, 3]
    assert list(O.topk_positions([-0.0, 0.0], 1)) == [0]
    assert list(O.topk_positions([0.0, -0.0, -1.0], 1)) == [0]
    assert list(O.topk_positions([1.0, 2.0, 3.0], 64)) == [0, 1, 2]   # p+1 <= k: all
    assert list(O.topk_positions([9.0, 1.0], 2)) == [0, 1]


@pytest.mark.parametrize("seed", range(6))
def test_topk_equals_stable_sort(seed):
    # library route: Python's stable sort by (score desc, position asc), take k
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 400))
    k = int(rng.integers(1, 80))
    s = rng.integers(-4, 5, n).astype(float)            # many ties
    ref = sorted(sorted(range(n), key=lambda i: -s[i])[:k])
    assert list(O.topk_positions(s, k)) == ref


# ---------------------------------------------------------------- attention

def _sdpa_causal(q, kv, Dv, scale, sink=None):
    """torch fp64 scaled_dot_product_attention, causal, KV shared by all heads;
    the sink is an extra key with logit sink[h] and a zero value."""
    T, H, D = q.shape
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                 # [1,H,T,D]
    k = torch.from_numpy(kv)[None, None].expand(1, H, T, D)
    v = torch.from_numpy(kv[:, :Dv])[None, None].expand(1, H, T, Dv)
    mask = torch.full((T, T), -math.inf, dtype=torch.float64).triu(1)  # s > t masked
    mask = mask[None, None].expand(1, H, T, T)
    if sink is not None:
        k = torch.cat([k, torch.zeros(1, H, 1, D, dtype=torch.float64)], dim=2)
        v = torch.cat([v, torch.zeros(1, H, 1, Dv, dtype=torch.float64)], dim=2)
        extra = torch.from_numpy(sink)[None, :, None, None].expand(1, H, T, 1)
        mask = torch.cat([mask, extra], dim=3)
    o = torch.nn.functional.scaled_dot_product_attention(qt, k, v, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("with_sink", [False, True])
@pytest.mark.parametrize("mode", MODES)
def test_attention_with_full_topk_is_dense_causal(mode, with_sink):
    rng = np.random.default_rng(11)
    T, H, D, Dv, HI, DI = 40, 3, 10, 6, 2, 4
    q = rng.standard_normal((T, H, D))
    kv = rng.standard_normal((T, D))
    qi = rng.standard_normal((T, HI, DI))
    ki = rng.standard_normal((T, DI))
    w = rng.standard_normal((T, HI))
    sink = rng.standard_normal(H) if with_sink else None
    lengths = [17, 23]
    qsl = _qsl(lengths)
    out = O.prefill(q, kv, qi, ki, w, qsl, lengths, 3, mode, topk=64, scale=0.3, Dv=Dv, sink=sink)
    for b, L in enumerate(lengths):
        lo, hi = qsl[b], qsl[b + 1]
        ref = _sdpa_causal(q[lo:hi], kv[lo:hi], Dv, 0.3, sink)
        assert np.allclose(out[lo:hi], ref, rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(3)
    H, D, Dv = 4, 8, 5
    kv = rng.standard_normal((6, D))
    q = rng.standard_normal((H, D))
    # one selected row: the output is that row's value, whatever q is
    assert np.allclose(O.sparse_attention(q, kv[2:3], 0.7, Dv), np.tile(kv[2, :Dv], (H, 1)), atol=1e-15)
    # q = 0: equal logits -> the mean of the selected values
    assert np.allclose(O.sparse_attention(np.zeros((H, D)), kv, 0.7, Dv), np.tile(kv[:, :Dv].mean(0), (H, 1)))
    # q = 0, sink = 0: the sink takes one share of n+1 in the denominator only
    assert np.allclose(O.sparse_attention(np.zeros((H, D)), kv, 0.7, Dv, np.zeros(H)),
                       np.tile(kv[:, :Dv].sum(0) / 7.0, (H, 1)))
    # sink -> -inf is no sink; permuting the selected rows changes nothing
    base = O.sparse_attention(q, kv, 0.7, Dv)
    assert np.allclose(O.sparse_attention(q, kv, 0.7, Dv, np.full(H, -np.inf)), base, atol=1e-15)
    assert np.allclose(O.sparse_attention(q, kv[::-1], 0.7, Dv), base, atol=1e-14)
    # scale equivariance: (2q, scale/2) == (q, scale)
    assert np.allclose(O.sparse_attention(2 * q, kv, 0.35, Dv), base, atol=1e-14)
    # without a sink the output is a convex combination of the values
    assert np.all(base <= kv[:, :Dv].max(0) + 1e-12) and np.all(base >= kv[:, :Dv].min(0) - 1e-12)


# ---------------------------------------------------------------- CP views

@pytest.mark.parametrize("wl", [TINY, TINY_INT], ids=lambda w: w.name)
@pytest.mark.parametrize("mode", MODES)
def test_cp_views_rerange_to_single_view(wl, mode):
    x = draw_inputs(wl)
    args = [_f64(x[k]) for k in ("q", "kv", "q_idx", "k_idx", "w")]
    qsl, sl = wl.query_start_loc(), wl.seq_lens()
    kw = dict(topk=wl.topk, scale=wl.scale, Dv=wl.Dv, sink=None if x["sink"] is None else _f64(x["sink"]))
    single = O.prefill(*args, qsl, sl, 1, mode, **kw)
    views = O.prefill(*args, qsl, sl, wl.cp_size, mode, **kw)
    assert np.array_equal(single, views)


def test_short_rows_select_everything():
    # rows with p + 1 <= topk select every causal key, in order, padded with -1
    wl = TINY
    x = draw_inputs(wl)
    md = O.build_local_metadata(wl.query_start_loc(), wl.seq_lens(), 1, 0, IN_SEQ_SPLIT)
    idx, _ = O.prefill_view(md, _f64(x["q"]), _f64(x["q_idx"]), _f64(x["w"]), _f64(x["kv"]),
                            _f64(x["k_idx"]), wl.topk, wl.scale, wl.Dv, slots=[0, 5, 63, 64, 200])
    assert list(idx[0]) == [0] + [-1] * 63
    assert list(idx[5][:6]) == list(range(6)) and np.all(idx[5][6:] == -1)
    assert list(idx[63]) == list(range(64))
    assert np.all(idx[64] >= 0) and len(set(idx[64])) == 64 and idx[64].max() <= 64
    assert np.all(idx[200] >= 0) and np.all(np.diff(idx[200]) > 0) and idx[200].max() <= 200


# ---------------------------------------------------------------- FP8 latent-KV cache (R17)
# The pages name an FP8 KV cache without a format; the reading is the OCP E4M3
# code with per-128-column fp32 scales and bf16 rope columns.  Pins: values the
# E4M3 format fixes, torch's own float8_e4m3fn conversion (a library routine),
# round trips and the quantisation error bound.

def test_e4m3_format_values():
    # sign | exponent (bias 7) | 3 mantissa bits; exponent 0 is subnormal
    pairs = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0,
             0x3C: 1.5, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in pairs.items():
        assert O.e4m3_decode([c])[0] == v, hex(c)
    assert np.isnan(O.e4m3_decode([0x7F, 0xFF])).all()
    assert np.signbit(O.e4m3_decode([0x80])[0]) and O.e4m3_decode([0x80])[0] == 0.0
    vals = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(vals) > 0)  # positive codes are ordered by value


def test_e4m3_encode_matches_torch_and_rounds_ties_to_even():
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert np.array_equal(O.e4m3_encode(vals[finite]), codes[finite])
    pos = np.sort(vals[(vals > 0) & finite])
    mids = (pos[:-1] + pos[1:]) / 2          # exact ties between neighbours
    got = O.e4m3_decode(O.e4m3_encode(mids))
    lo_even = (O.e4m3_encode(pos[:-1]) & 1) == 0
    assert np.array_equal(got, np.where(lo_even, pos[:-1], pos[1:]))
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(100000) * np.exp2(rng.uniform(-14, 8, 100000))).astype(np.float32)
    v = np.clip(v, -447.0, 447.0).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(v), ref)
    assert O.e4m3_encode([500.0, -1e6, 449.0])[0] == 0x7E and O.e4m3_encode([-1e6])[0] == 0xFE


def test_bf16_round_matches_torch():
    x = np.concatenate([np.random.default_rng(8).standard_normal(20000).astype(np.float32),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], dtype=np.float32)])
    assert np.array_equal(O.bf16_round(x), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("D,Dv", [(576, 512), (64, 48)])
def test_kv_fp8_cache_layout_and_error_bound(D, Dv):
    gen = torch.Generator().manual_seed(11)
    kv = (torch.randn(300, D, generator=gen) * torch.exp2(torch.randn(300, 1, generator=gen) * 3)).to(torch.bfloat16)
    kv[7, :] = 0.0  # an all-zero row: scale 1, codes 0
    x = kv.float().numpy()
    c = O.kv_fp8_quantize(x, Dv)
    tiles = -(-Dv // 128)
    assert c.shape == (300, O.kv_fp8_row_bytes(D, Dv)) and c.shape[1] % 16 == 0
    assert O.kv_fp8_row_bytes(576, 512) == 656
    rope = np.ascontiguousarray(c[:, Dv + 4 * tiles: Dv + 4 * tiles + 2 * (D - Dv)]).view(np.uint16)
    assert np.array_equal(rope, kv[:, Dv:].view(torch.int16).numpy().view(np.uint16))
    assert np.all(c[:, Dv + 4 * tiles + 2 * (D - Dv):] == 0)
    d = O.kv_fp8_dequantize(c, D, Dv)
    assert np.array_equal(d[:, Dv:], x[:, Dv:])
    for t in range(tiles):
        cols = slice(t * 128, min((t + 1) * 128, Dv))
        scale = np.ascontiguousarray(c[:, Dv + 4 * t: Dv + 4 * t + 4]).view(np.float32).reshape(-1)
        amax = np.abs(x[:, cols]).max(axis=1)
        assert np.array_equal(scale, np.where(amax > 0, (amax / np.float32(448)).astype(np.float32), 1.0))
        # the largest magnitude of a tile encodes to +-448
        j = np.abs(x[:, cols]).argmax(axis=1)
        top = c[np.arange(300), t * 128 + j]
        nz = amax > 0
        assert np.all((top[nz] & 0x7F) == 0x7E)
        # error: half an E4M3 step at the value's binade (scaled) plus half a bf16 ulp
        v = np.abs(x[:, cols]) / scale[:, None]
        half_step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(v, 2.0 ** -20))), -6) - 4) * scale[:, None]
        bound = half_step + np.abs(d[:, cols]) * 2.0 ** -8 + 1e-30
        assert np.all(np.abs(d[:, cols] - x[:, cols]) <= bound)
    assert np.all(c[7, :Dv] == 0) and np.all(d[7] == 0)


# ---------------------------------------------------------------- FP8 indexer operands (R19)
# Index rows in the FP8 cache row format with D = Dv = DI; the score is the
# indexer score of decode(code) * scale.  Pins: the hand example with its
# operands as hand-encoded bytes, a closed form with distinct per-row scales,
# and exact agreement with the plain indexer where quantisation is exact.

def _golden_fp8_rows(name):
    out = {}
    for line in read_golden_lines(name):
        k, v = (x.strip() for x in line.split("=", 1))
        out[k] = v.split()
    return out


def test_indexer_fp8_hand_example():
    g = _golden_fp8_rows("indexer_fp8_hand_example.txt")
    q8 = np.array([int(x, 16) for x in g["q_rows"]], dtype=np.uint8).reshape(2, 16)
    k8 = np.array([int(x, 16) for x in g["k_rows"]], dtype=np.uint8).reshape(5, 16)
    assert O.kv_fp8_row_bytes(2, 2) == 16
    assert np.array_equal(O.index_fp8_values(q8, 2).reshape(-1), np.array(g["values_q"], dtype=float))
    assert np.array_equal(O.index_fp8_values(k8, 2).reshape(-1), np.array(g["values_k"], dtype=float))
    w = np.array(g["w"], dtype=float)
    assert np.array_equal(O.indexer_scores_fp8(q8, w, k8, 2), np.array(g["scores"], dtype=float))
    # the same scores as the plain hand example
    assert np.array_equal(O.indexer_scores_fp8(q8, w, k8, 2),
                          np.array(read_golden("indexer_hand_example.txt")["scores"], dtype=float))


def test_indexer_fp8_closed_form_row_scales():
    # every code 1.0 (0x38); head j has scale a_j, key s scale b_s: q . k = DI a_j b_s,
    # so I[s] = DI b_s sum_j w_j a_j (all dots positive).  A scale read from the
    # wrong row or operand, or a dropped scale, breaks it.
    HI, DI, n = 3, 128, 5
    # 1 + 2^-10 has more significant bits than bf16: values decode(code) * scale
    # are taken exactly, so rounding them to bf16 would also break the form
    a = np.array([0.5, 2.0, 1 + 2.0 ** -10], dtype=np.float32)
    b = np.array([1.0, 0.25, 4.0, 3.0, 0.75], dtype=np.float32)
    def rows(scales):
        r = np.zeros((len(scales), O.kv_fp8_row_bytes(DI, DI)), dtype=np.uint8)
        r[:, :DI] = 0x38
        r[:, DI:DI + 4] = scales.view(np.uint8).reshape(-1, 4)
        return r
    w = np.array([1.0, -0.5, 3.0])
    expect = DI * b.astype(float) * float((w * a).sum())
    assert np.array_equal(O.indexer_scores_fp8(rows(a), w, rows(b), DI), expect)
    assert O.indexer_scores_fp8(rows(a), w, rows(b), DI).shape == (n,)


def test_indexer_fp8_exact_where_quantisation_is_exact():
    # rows made of E4M3 values times a power of two, each row holding +-448 times
    # it: the quantiser's scale is that power of two and every code is exact, so
    # the FP8 score equals the plain indexer score of the original rows.
    rng = np.random.default_rng(21)
    HI, DI, n = 4, 128, 40
    def exact_rows(R):
        vals = O.e4m3_decode(rng.integers(0, 0x7F, size=(R, DI)).astype(np.uint8) | (rng.integers(0, 2, (R, DI)) << 7).astype(np.uint8))
        vals[:, 5] = 448.0 * np.where(rng.integers(0, 2, R) == 1, 1.0, -1.0)
        return vals * np.exp2(rng.integers(-12, -4, size=(R, 1)))
    q, k = exact_rows(HI), exact_rows(n)
    q8, k8 = O.kv_fp8_quantize(q.astype(np.float32), DI), O.kv_fp8_quantize(k.astype(np.float32), DI)
    assert np.array_equal(O.index_fp8_values(q8, DI), q) and np.array_equal(O.index_fp8_values(k8, DI), k)
    w = rng.standard_normal(HI)
    assert np.array_equal(O.indexer_scores_fp8(q8, w, k8, DI), O.indexer_scores(q, w, k))
    # general rows: within the quantisation error of the plain score
    qf = O.bf16_round(rng.standard_normal((HI, DI)).astype(np.float32)).astype(float)
    kf = O.bf16_round(rng.standard_normal((n, DI)).astype(np.float32)).astype(float)
    s8 = O.indexer_scores_fp8(O.kv_fp8_quantize(qf.astype(np.float32), DI), w, O.kv_fp8_quantize(kf.astype(np.float32), DI), DI)
    s = O.indexer_scores(qf, w, kf)
    bound = np.abs(w) @ (np.abs(qf) @ np.abs(kf).T) * (2 * 2.0 ** -4 + 2.0 ** -8)
    assert np.all(np.abs(s8 - s) <= bound) and not np.array_equal(s8, s)


# ---------------------------------------------------------------- compressed KV (R18)

_COMPRESSED_CASES = {"C": ([9, 6], [9, 6], 2, 4), "D": ([5, 3], [135, 3], 2, 128)}  # q_lens, seq_lens, cp, c


def test_metadata_compressed_hand_cases():
    seen = 0
    for line in read_golden_lines("metadata_compressed_hand_cases.txt"):
        head, lqs, kvl, lkv, rid, base, pbase, pos = line.split("|")
        case, mode_s, rank = head.split()
        q_lens, seq_lens, cp, c = _COMPRESSED_CASES[case]
        mode = {"inseq": IN_SEQ_SPLIT, "rr": ROUND_ROBIN}[mode_s]
        md = O.build_local_metadata(_qsl(q_lens), seq_lens, cp, int(rank), mode, compress_ratio=c)
        assert md["local_query_start_loc"] == _ints(lqs), line
        assert md["local_seq_lens"] == _ints(kvl), line
        assert md["local_kv_start_loc"] == _ints(lkv), line
        assert md["local_req_id"] == _ints(rid), line
        assert md["local_req_kv_base"] == _ints(base), line
        assert md["local_req_pos_base"] == _ints(pbase), line
        assert md["local_token_pos"] == _ints(pos), line
        assert md["num_kv_rows"] == sum(n // c for n in seq_lens) and md["compress_ratio"] == c
        seen += 1
    assert seen == 6


@pytest.mark.parametrize("with_sink", [False, True])
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("c", [1, 4, 7])
def test_compressed_attention_with_full_topk_is_masked_dense(c, mode, with_sink):
    # with topk above every entry count, each query attends to all entries it
    # sees: torch's fp64 scaled_dot_product_attention over the compressed rows
    # with the mask "entry e visible from position p iff (e + 1) c <= p + 1";
    # a query that sees no entry outputs zero
    rng = np.random.default_rng(13)
    H, D, Dv, HI, DI = 3, 10, 6, 2, 4
    q_lens, prefixes = [17, 23], [5, 0]
    seq_lens = [n + p for n, p in zip(q_lens, prefixes)]
    ents = [n // c for n in seq_lens]
    T, R = sum(q_lens), sum(ents)
    q = rng.standard_normal((T, H, D))
    kv = rng.standard_normal((R, D))
    qi = rng.standard_normal((T, HI, DI))
    ki = rng.standard_normal((R, DI))
    w = rng.standard_normal((T, HI))
    sink = rng.standard_normal(H) if with_sink else None
    qsl = _qsl(q_lens)
    out = O.prefill(q, kv, qi, ki, w, qsl, seq_lens, 3, mode, topk=64, scale=0.3, Dv=Dv, sink=sink,
                    compress_ratio=c)
    for b in range(2):
        rows = kv[sum(ents[:b]): sum(ents[:b]) + ents[b]]
        for t in range(q_lens[b]):
            g, p = qsl[b] + t, prefixes[b] + t
            n = (p + 1) // c
            if n == 0:
                assert np.all(out[g] == 0)
                continue
            qt = torch.from_numpy(q[g])[None, :, None, :]                    # [1,H,1,D]
            k = torch.from_numpy(rows)[None, None].expand(1, H, len(rows), D)
            v = torch.from_numpy(rows[:, :Dv])[None, None].expand(1, H, len(rows), Dv)
            mask = torch.full((1, H, 1, len(rows)), -math.inf, dtype=torch.float64)
            mask[..., :n] = 0.0
            if sink is not None:
                k = torch.cat([k, torch.zeros(1, H, 1, D, dtype=torch.float64)], dim=2)
                v = torch.cat([v, torch.zeros(1, H, 1, Dv, dtype=torch.float64)], dim=2)
                mask = torch.cat([mask, torch.from_numpy(sink)[None, :, None, None]], dim=3)
            ref = torch.nn.functional.scaled_dot_product_attention(qt, k, v, attn_mask=mask, scale=0.3)
            assert np.allclose(out[g], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12), (b, t)


@pytest.mark.parametrize("mode", MODES)
def test_compressed_metadata_extents(mode):
    # entry extents stay right-aligned: the widest local extent of a request over
    # all ranks is its entry count, and every local query sees at most that many
    q_lens, prefixes, cp, c = [37, 20, 9, 300], [25, 0, 4, 900], 4, 128
    seq_lens = [n + p for n, p in zip(q_lens, prefixes)]
    widest = [0] * 4
    for r in range(cp):
        md = O.build_local_metadata(_qsl(q_lens), seq_lens, cp, r, mode, compress_ratio=c)
        for j in range(md["local_batch"]):
            b = md["local_req_id"][j]
            widest[b] = max(widest[b], md["local_seq_lens"][j])
            assert md["local_req_kv_base"][j] == sum(n // c for n in seq_lens[:b])
    assert widest == [n // c for n in seq_lens]


# ---------------------------------------------------------------- sliding window (R20)
# A query at position p also attends to the original rows of positions
# max(0, p - W + 1) .. p; one softmax over the selected entries and the window
# rows (a row both selected and in the window counts once at c = 1).

def test_swa_hand_example():
    # 1 request of 3 tokens, H = 1, D = Dv = 1, q = 1, latent rows [1], [2], [3],
    # scale 1 (logit = row value); index keys 3, 2, 1 with q_I = w = 1 -> scores
    # 3, 2, 1: the top-1 is always key 0.  Window W = 2:
    #   p = 0: {0}             -> out = 1
    #   p = 1: {0} u {0, 1}    -> (1 e + 2 e^2) / (e + e^2) = (1 + 2e) / (1 + e)
    #          (counting key 0 twice would give (2 + 2e) / (2 + e) instead)
    #   p = 2: {0} u {1, 2}    -> (e + 2 e^2 + 3 e^3) / (e + e^2 + e^3)
    e = math.e
    q, kv = np.ones((3, 1, 1)), np.array([[1.0], [2.0], [3.0]])
    qi, ki, w = np.ones((3, 1, 1)), np.array([[3.0], [2.0], [1.0]]), np.ones((3, 1))
    out = O.prefill_swa(q, kv, qi, ki, w, [0, 3], [3], 1, O.IN_SEQ_SPLIT, topk=1, scale=1.0, Dv=1, window=2)
    expect = [1.0, (1 + 2 * e) / (1 + e), (e + 2 * e ** 2 + 3 * e ** 3) / (e + e ** 2 + e ** 3)]
    assert np.allclose(out[:, 0, 0], expect, rtol=1e-15, atol=0)
    assert not np.isclose(out[1, 0, 0], (2 + 2 * e) / (2 + e))


def _swa_case(c, seed=17, prefixes=(0, 0)):
    """Queries of two requests (lengths 19, 26) after the given prefixes; the
    original rows hold the whole sequences, the entries floor(seq_len / c)
    rows per request (the original rows themselves at c = 1)."""
    rng = np.random.default_rng(seed)
    H, D, Dv, HI, DI = 3, 10, 6, 2, 4
    lens = [19, 26]
    seq = [n + p for n, p in zip(lens, prefixes)]
    ents = [n // c for n in seq]
    T, S, R = sum(lens), sum(seq), sum(ents)
    x = dict(q=rng.standard_normal((T, H, D)), kv_ori=rng.standard_normal((S, D)),
             qi=rng.standard_normal((T, HI, DI)), w=rng.standard_normal((T, HI)), sink=rng.standard_normal(H))
    x["kv"] = x["kv_ori"] if c == 1 else rng.standard_normal((R, D))
    x["ki"] = rng.standard_normal((S if c == 1 else R, DI))
    return x, lens, seq, ents, (H, D, Dv)


@pytest.mark.parametrize("c", [1, 4])
@pytest.mark.parametrize("mode", [O.IN_SEQ_SPLIT, O.ROUND_ROBIN, O.HEAD_TAIL])
def test_swa_window_zero_is_the_sparse_path(c, mode):
    x, lens, _, _, (H, D, Dv) = _swa_case(c)
    qsl = _qsl(lens)
    a = O.prefill_swa(x["q"], x["kv"], x["qi"], x["ki"], x["w"], qsl, lens, 3, mode, topk=5, scale=0.3, Dv=Dv,
                      window=0, kv_ori=x["kv_ori"], sink=x["sink"], compress_ratio=c)
    b = O.prefill(x["q"], x["kv"], x["qi"], x["ki"], x["w"], qsl, lens, 3, mode, topk=5, scale=0.3, Dv=Dv,
                  sink=x["sink"], compress_ratio=c)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("prefixes", [(0, 0), (6, 3)])
@pytest.mark.parametrize("c,window", [(1, 4), (4, 3), (4, 7)])
@pytest.mark.parametrize("mode", [O.IN_SEQ_SPLIT, O.ROUND_ROBIN])
def test_swa_is_masked_dense_attention(c, window, mode, prefixes):
    # against torch's fp64 scaled_dot_product_attention over all candidate rows
    # (the compressed entries, then the original rows) with the mask "selected
    # entry, or original position in the window"; the selection is the plain
    # path's (view_row), the sink an extra key of zero value; with a prefix the
    # original rows of request b start at the sum of the earlier seq_lens
    x, lens, seq, ents, (H, D, Dv) = _swa_case(c, seed=23, prefixes=prefixes)
    qsl, topk, scale = _qsl(lens), 5, 0.3
    out = O.prefill_swa(x["q"], x["kv"], x["qi"], x["ki"], x["w"], qsl, seq, 2, mode, topk=topk, scale=scale,
                        Dv=Dv, window=window, kv_ori=x["kv_ori"], sink=x["sink"], compress_ratio=c)
    for r in range(2):
        md = O.build_local_metadata(qsl, seq, 2, r, mode, compress_ratio=c)
        qs, qis, ws = (O.split(x[k], 2, mode)[r] for k in ("q", "qi", "w"))
        for i, g in enumerate(md["local_token_pos"]):
            if g < 0:
                continue
            sel, _, _ = O.view_row(md, i, qs, qis, ws, x["kv"], x["ki"], topk, scale, Dv, x["sink"])
            b = 0 if g < lens[0] else 1
            p = prefixes[b] + g - qsl[b]
            ent0, ori0 = sum(ents[:b]), sum(seq[:b])
            if c == 1:
                keys = x["kv_ori"][ori0: ori0 + p + 1]
                allowed = np.zeros(p + 1, dtype=bool)
                allowed[sel - ori0] = True
                allowed[max(0, p - window + 1):] = True
            else:
                keys = np.concatenate([x["kv"][ent0: ent0 + ents[b]], x["kv_ori"][ori0: ori0 + p + 1]])
                allowed = np.zeros(keys.shape[0], dtype=bool)
                allowed[sel - ent0] = True
                allowed[ents[b] + max(0, p - window + 1):] = True
            qt = torch.from_numpy(x["q"][g])[None, :, None, :]
            k = torch.from_numpy(keys)[None, None].expand(1, H, len(keys), D)
            v = torch.from_numpy(keys[:, :Dv])[None, None].expand(1, H, len(keys), Dv)
            mask = torch.where(torch.from_numpy(allowed), 0.0, -math.inf).to(torch.float64)
            mask = mask[None, None, None].expand(1, H, 1, len(keys))
            k = torch.cat([k, torch.zeros(1, H, 1, D, dtype=torch.float64)], dim=2)
            v = torch.cat([v, torch.zeros(1, H, 1, Dv, dtype=torch.float64)], dim=2)
            mask = torch.cat([mask, torch.from_numpy(x["sink"])[None, :, None, None]], dim=3)
            ref = torch.nn.functional.scaled_dot_product_attention(qt, k, v, attn_mask=mask, scale=scale)
            assert np.allclose(out[g], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12), (r, i)


def test_swa_full_window_is_dense_causal():
    # c = 1 and a window as long as the request: every causal key, whatever the
    # selection -- torch's causal attention
    x, lens, _, _, (H, D, Dv) = _swa_case(1, seed=29)
    qsl = _qsl(lens)
    out = O.prefill_swa(x["q"], x["kv"], x["qi"], x["ki"], x["w"], qsl, lens, 4, O.ROUND_ROBIN, topk=2,
                        scale=0.3, Dv=Dv, window=max(lens))
    for b in range(2):
        qb = torch.from_numpy(x["q"][qsl[b]: qsl[b + 1]]).permute(1, 0, 2)[None]          # [1,H,n,D]
        kb = torch.from_numpy(x["kv"][qsl[b]: qsl[b + 1]])[None, None].expand(1, H, lens[b], D)
        vb = torch.from_numpy(x["kv"][qsl[b]: qsl[b + 1], :Dv])[None, None].expand(1, H, lens[b], Dv)
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, is_causal=True, scale=0.3)
        assert np.allclose(out[qsl[b]: qsl[b + 1]], ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
