"""Host-side schedule of the host-streamed prefill, without a GPU.

HostStreamedPrefill cuts the token stream into chunks of consecutive tokens (a
multiple of cp_size) and, per chunk, runs each view over the runs of its slots
whose tokens lie in the chunk.  Over all chunks, every real slot of every view
must be computed exactly once and with its own token; pad slots never.  The
slot -> token map is the oracle's (local_rows: the split modes of "[DeepSeek
v3.2] 上下文并行详解" 2.B and 4 第一部分, and the head-tail zigzag), and the
geometry is the library's own dsa_cp_geometry.
"""
import types

import numpy as np
import pytest

from oracle import dsa_oracle as O
from sparse_attention_prefill_cp_gb300 import dsa_cp_geometry
from sparse_attention_prefill_cp_gb300.pipeline import HostStreamedPrefill
from workloads import HEAD_TAIL, IN_SEQ_SPLIT, ROUND_ROBIN

# (tokens, cp_size, requested chunk tokens): exact and ragged tails, chunks
# smaller than cp_size, a single chunk, tokens fewer than ranks, and the
# 16-request batch's geometry with the chunk size the bench uses
CASES = [
    (8192, 8, 512),
    (11805, 4, 740),
    (11805, 4, 11805),
    (5, 4, 1),
    (7, 2, 3),
    (33, 8, 8),
    (1000, 16, 64),
    (3, 8, 8),
    (184265, 16, 11520),
]


@pytest.mark.parametrize("mode", [IN_SEQ_SPLIT, ROUND_ROBIN, HEAD_TAIL])
@pytest.mark.parametrize("T,cp,chunk", CASES)
def test_chunk_runs_cover_every_slot_once(T, cp, chunk, mode):
    pad, tpr = dsa_cp_geometry(T, cp)
    assert (pad, tpr) == O.padded_geometry(T, cp)
    fake = types.SimpleNamespace(T=T, tpr=tpr, cp_size=cp, mode=mode)
    C = max(cp, -(-chunk // cp) * cp)  # the class rounds the chunk up to a multiple of cp_size
    chunks = [(t0, min(t0 + C, T)) for t0 in range(0, T, C)]
    step = cp if mode == ROUND_ROBIN else 1
    for r in range(cp):
        rows = O.local_rows(T, cp, r, mode)
        seen = np.zeros(tpr, dtype=np.int64)
        for t0, t1 in chunks:
            for s0, n, g0 in HostStreamedPrefill._runs(fake, r, t0, t1):
                assert n > 0 and 0 <= s0 and s0 + n <= tpr
                slots = np.arange(s0, s0 + n)
                toks = g0 + step * np.arange(n)
                assert np.array_equal(rows[slots], toks), (r, t0, t1, s0, n, g0)
                assert toks.min() >= t0 and toks.max() < t1
                seen[slots] += 1
        assert np.array_equal(seen, (rows >= 0).astype(np.int64)), (r, np.flatnonzero(seen != (rows >= 0)))
