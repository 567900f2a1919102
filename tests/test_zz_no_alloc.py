"""The allocation-free indexer entry point (dsa_indexer_topk_noalloc).

Callers that cannot allocate device memory where they run the indexer use
this variant: its score workspace is a fixed array inside the library.  The
test calls it through the C ABI twice in a row (the second call finds the
first call's scores still in the shared array) and checks each result
against dsa_indexer_topk with its own workspace; the top-k index sets must
be identical.  This file is collected last on purpose."""
import pytest
import torch

import sparse_attention_prefill_cp_gb300 as dsa
from sparse_attention_prefill_cp_gb300.pipeline import DSAPrefill
from workloads import IN_SEQ_SPLIT, ROUND_ROBIN, LONG_8K, TINY, draw_index_inputs, draw_inputs

pytestmark = pytest.mark.gpu

CASES = [
    (TINY, IN_SEQ_SPLIT),
    (LONG_8K.with_(name="noalloc-full-2x", lengths=(2500, 700), cp_size=2, seed=21), ROUND_ROBIN),
    # 4096 query rows of 8192-key scores (128 MiB) per view: four passes over
    # the 32 MiB array within one call
    (LONG_8K.with_(name="noalloc-multipass", cp_size=2, seed=22), IN_SEQ_SPLIT),
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    dsa.load()


@pytest.mark.parametrize("wl,mode", CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_noalloc_matches_workspace_entry_point_twice(wl, mode):
    for call in range(2):
        x = draw_index_inputs(wl, device="cuda", seed_offset=call)
        pipe = DSAPrefill(wl.lengths, wl.cp_size, mode, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale,
                          fused=True)
        pipe.metadata()
        pipe.split(None, x["q_idx"], x["w"])
        for r in range(wl.cp_size):
            ref = dsa.dsa_indexer_topk(pipe.md[r], pipe.qi_split[r], x["k_idx"], pipe.w_split[r], wl.topk,
                                       pipe.max_kv_len)
            got = dsa.dsa_indexer_topk_noalloc(pipe.md[r], pipe.qi_split[r], x["k_idx"], pipe.w_split[r],
                                               wl.topk, pipe.max_kv_len)
            dsa.dsa_poll_device_error()
            assert torch.equal(got, ref), (call, r)


def test_noalloc_rejects_rows_beyond_its_array():
    wl = TINY
    x = {k: (v.cuda() if v is not None else None) for k, v in draw_inputs(wl).items()}
    pipe = DSAPrefill(wl.lengths, wl.cp_size, IN_SEQ_SPLIT, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale)
    pipe.metadata()
    pipe.split(x["q"], x["q_idx"], x["w"])
    with pytest.raises(dsa.DSAError) as e:
        dsa.dsa_indexer_topk_noalloc(pipe.md[0], pipe.qi_split[0], x["k_idx"], pipe.w_split[0], wl.topk,
                                     70000)
    assert e.value.status == 4
