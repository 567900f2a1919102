"""CPU-only checks of the C ABI: the library builds and loads, exports every
function include/dsa_cp.h declares, and its host-side logic (geometry,
metadata sizing, argument validation) answers without touching a GPU."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT
import sparse_attention_prefill_cp_gb300 as dsa
from sparse_attention_prefill_cp_gb300 import _lib
from oracle import dsa_oracle as O

HEADER = os.path.join(ROOT, "include", "dsa_cp.h")


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(dsa_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_abi_version_and_status_strings(lib):
    assert lib.dsa_abi_version() == 9
    for code, name in _lib.STATUS.items():
        assert lib.dsa_status_string(code).decode().startswith(name)


@pytest.mark.parametrize("T,cp", [(0, 1), (1, 1), (12, 3), (13, 4), (11805, 4), (184265, 16), (65536, 8)])
def test_geometry_matches_oracle(T, cp):
    assert dsa.dsa_cp_geometry(T, cp) == O.padded_geometry(T, cp)


def test_metadata_sizes_and_bind(lib):
    B, T, cp = 4, 11805, 4
    n = dsa.dsa_cp_metadata_sizes(B, T, cp)
    tpr = O.padded_geometry(T, cp)[1]
    assert n == 11 + 2 * (B + 1) + 4 * B + tpr
    md = _lib.LocalMetadata()
    base = 0x10000
    assert lib.dsa_cp_metadata_bind(C.c_void_p(base), B, T, cp, C.byref(md)) == 0
    offs = [md.scalars, md.local_query_start_loc, md.local_seq_lens, md.local_kv_start_loc, md.local_req_id,
            md.local_req_kv_base, md.local_req_pos_base, md.local_token_pos]
    assert [(o - base) // 4 for o in offs] == [0, 11, 11 + B + 1, 11 + 2 * B + 1, 11 + 3 * B + 2, 11 + 4 * B + 2,
                                                11 + 5 * B + 2, 11 + 6 * B + 2]
    assert (md.local_token_pos - base) // 4 + tpr == n


def test_workspace_size_holds_a_tile():
    big = dsa.dsa_indexer_topk_workspace_size(1024, 8192, 2048)
    assert big == 1024 * 8192 * 4
    assert dsa.dsa_indexer_topk_workspace_size(8192, 65536, 2048) <= (1 << 30)
    assert dsa.dsa_indexer_topk_workspace_size(1, 3, 2048) == 8 * 4 * 4  # one 8-row tile, ld rounded to 4


def test_host_validation_rejects_before_any_launch(lib):
    md = _lib.LocalMetadata()
    assert lib.dsa_cp_metadata_bind(C.c_void_p(0x10000), 1, 16, 2, C.byref(md)) == 0
    p = C.c_void_p(0x10000)
    # null pointers, bad rank / mode / sizes
    assert lib.dsa_cp_split(None, 16, 10, 2, 0, -1, p, None) == 1
    assert lib.dsa_cp_split(p, 16, 10, 2, 7, -1, p, None) == 1
    assert lib.dsa_cp_split(p, 16, 10, 2, 0, 2, p, None) == 1
    assert lib.dsa_cp_split(p, 0, 10, 2, 0, -1, p, None) == 2
    assert lib.dsa_cp_rerange(p, 16, -1, 2, 1, p, None) == 2
    assert lib.dsa_cp_build_local_metadata(p, p, 1, 16, 2, 2, 0, C.byref(md), None) == 1
    assert lib.dsa_cp_build_local_metadata(p, p, 1, 16, 0, 0, 0, C.byref(md), None) == 1
    assert lib.dsa_cp_build_local_metadata_compressed(p, p, 1, 16, 2, 0, 0, 0, C.byref(md), None) == 1
    assert lib.dsa_cp_geometry(5, 0, C.byref(C.c_int32()), C.byref(C.c_int32())) == 1
    # dimension sets that are not compiled
    assert lib.dsa_indexer_topk(C.byref(md), 1, 8, 16, p, p, p, 16, 32, 128, 2048, p, p, 1 << 20, None) == 3
    assert lib.dsa_indexer_topk(C.byref(md), 1, 8, 16, p, p, p, 16, 64, 128, 1024, p, p, 1 << 20, None) == 3
    assert lib.dsa_sparse_attn_prefill(C.byref(md), 1, 8, p, p, 16, p, 2048, None, C.c_float(0.07), 64, 576,
                                       512, p, None) == 3
    # misaligned tensors and a non-positive scale
    q = C.c_void_p(0x10008)
    assert lib.dsa_sparse_attn_prefill(C.byref(md), 1, 8, q, p, 16, p, 2048, None, C.c_float(0.07), 128, 576,
                                       512, p, None) == 1
    assert lib.dsa_sparse_attn_prefill(C.byref(md), 1, 8, p, p, 16, p, 2048, None, C.c_float(-1.0), 128, 576,
                                       512, p, None) == 1
    assert lib.dsa_indexer_topk(None, 1, 8, 16, p, p, p, 16, 64, 128, 2048, p, p, 1 << 20, None) == 1
    # head/token all-to-all: null, bad mode / cp, heads not divisible by cp
    assert lib.dsa_cp_all_to_all_heads(None, 128, 1024, 10, 8, 0, p, None) == 1
    assert lib.dsa_cp_all_to_all_heads(p, 128, 1024, 10, 8, 5, p, None) == 1
    assert lib.dsa_cp_all_to_all_heads(p, 128, 1024, 10, 0, 0, p, None) == 1
    assert lib.dsa_cp_all_to_all_heads(p, 128, 1024, 10, 3, 0, p, None) == 2
    assert lib.dsa_cp_all_to_all_heads(p, 128, 0, 10, 8, 0, p, None) == 2
    # fused head-sharded attention: cp_size < 1, heads not divisible by cp, uncompiled dims
    assert lib.dsa_sparse_attn_prefill_headsharded(C.byref(md), 1, 8, p, p, 16, p, 2048, None, C.c_float(0.07), 128,
                                                   576, 512, 0, p, None) == 1
    assert lib.dsa_sparse_attn_prefill_headsharded(C.byref(md), 1, 8, p, p, 16, p, 2048, None, C.c_float(0.07), 128,
                                                   576, 512, 3, p, None) == 2
    assert lib.dsa_sparse_attn_prefill_headsharded(C.byref(md), 1, 8, p, p, 16, p, 2048, None, C.c_float(0.07), 64,
                                                   576, 512, 2, p, None) == 3


def test_flat_attention_and_fp8_cache_validation(lib):
    md = _lib.LocalMetadata()
    assert lib.dsa_cp_metadata_bind(C.c_void_p(0x10000), 1, 16, 2, C.byref(md)) == 0
    p, odd = C.c_void_p(0x10000), C.c_void_p(0x10008)
    f = C.c_float(0.07)
    # flat-layout attention: misaligned q, negative token count, nothing to do, uncompiled dims
    assert lib.dsa_sparse_attn_prefill_flat(C.byref(md), 1, 8, odd, 16, p, 16, p, 2048, None, f, 128, 576, 512, p,
                                            None) == 1
    assert lib.dsa_sparse_attn_prefill_flat(C.byref(md), 1, 8, p, -1, p, 16, p, 2048, None, f, 128, 576, 512, p,
                                            None) == 2
    assert lib.dsa_sparse_attn_prefill_flat(C.byref(md), 1, 8, p, 0, p, 16, p, 2048, None, f, 128, 576, 512, p,
                                            None) == 0
    assert lib.dsa_sparse_attn_prefill_flat(C.byref(md), 1, 8, p, 16, p, 16, p, 2048, None, f, 96, 576, 512, p,
                                            None) == 3
    # FP8 cache: row sizes, null / misaligned buffers, shapes, nothing to do
    n = C.c_size_t()
    assert lib.dsa_kv_fp8_row_bytes(576, 512, C.byref(n)) == 0 and n.value == 656
    assert lib.dsa_kv_fp8_row_bytes(64, 48, C.byref(n)) == 0 and n.value == 96 == O.kv_fp8_row_bytes(64, 48)
    assert lib.dsa_kv_fp8_row_bytes(576, 500, C.byref(n)) == 2
    assert lib.dsa_kv_fp8_row_bytes(512, 576, C.byref(n)) == 2
    assert lib.dsa_kv_fp8_row_bytes(576, 512, None) == 1
    assert lib.dsa_kv_fp8_quantize(None, 4, 576, 512, p, None) == 1
    assert lib.dsa_kv_fp8_quantize(odd, 4, 576, 512, p, None) == 1
    assert lib.dsa_kv_fp8_quantize(p, -1, 576, 512, p, None) == 2
    assert lib.dsa_kv_fp8_quantize(p, 4, 576, 12, p, None) == 2
    assert lib.dsa_kv_fp8_quantize(p, 0, 576, 512, p, None) == 0
    assert lib.dsa_kv_fp8_dequantize(p, 4, 576, 512, None, None) == 1
    assert lib.dsa_kv_fp8_dequantize(p, 0, 64, 48, p, None) == 0


def test_fp8_indexer_validation(lib):
    md = _lib.LocalMetadata()
    assert lib.dsa_cp_metadata_bind(C.c_void_p(0x10000), 1, 16, 2, C.byref(md)) == 0
    p, odd = C.c_void_p(0x10000), C.c_void_p(0x10008)
    # null / misaligned operands, then dimension sets without an FP8 build (tiny shapes, other topk)
    assert lib.dsa_indexer_topk_fp8(C.byref(md), 1, 8, 16, None, p, p, 16, 64, 128, 2048, p, p, 1 << 20, None) == 1
    assert lib.dsa_indexer_topk_fp8(C.byref(md), 1, 8, 16, odd, p, p, 16, 64, 128, 2048, p, p, 1 << 20, None) == 1
    assert lib.dsa_indexer_topk_fp8(C.byref(md), 1, 8, 16, p, p, p, 16, 4, 32, 64, p, p, 1 << 20, None) == 3
    assert lib.dsa_indexer_topk_fp8(C.byref(md), 1, 8, 16, p, p, p, 16, 64, 128, 1024, p, p, 1 << 20, None) == 3
    assert lib.dsa_indexer_topk_fp8(C.byref(md), 1, 0, 16, p, p, p, 16, 64, 128, 2048, p, p, 1 << 20, None) == 0
    assert lib.dsa_indexer_scores_fp8(C.byref(md), 1, 8, 16, p, p, p, 16, 4, 32, 0, 8, p, None) == 3
    assert lib.dsa_indexer_scores_fp8(C.byref(md), 1, 8, 16, p, p, p, 16, 64, 128, 4, 8, p, None) == 2
    assert lib.dsa_indexer_scores_fp8(C.byref(md), 1, 8, 16, p, p, None, 16, 64, 128, 0, 8, p, None) == 1
    # the FP8 index row is the FP8 cache row with D = Dv = DI
    n = C.c_size_t()
    assert lib.dsa_kv_fp8_row_bytes(128, 128, C.byref(n)) == 0 and n.value == 144 == O.kv_fp8_row_bytes(128, 128)



def test_host_row_copies_validation(lib):
    # one rank's rows between host memory and the device: null pointers, bad
    # mode or rank (-1 = all ranks is not a host-copy rank), bad sizes; all
    # answered on the host before any copy is issued
    p = C.c_void_p(0x10000)
    for fn in (lib.dsa_cp_split_from_host, lib.dsa_cp_rerange_to_host):
        assert fn(None, 16, 10, 2, 0, 0, p, None) == 1
        assert fn(p, 16, 10, 2, 0, 0, None, None) == 1
        assert fn(p, 16, 10, 2, 9, 0, p, None) == 1
        assert fn(p, 16, 10, 2, 0, -1, p, None) == 1
        assert fn(p, 16, 10, 2, 0, 2, p, None) == 1
        assert fn(p, 16, 10, 0, 0, 0, p, None) == 1
        assert fn(p, 0, 10, 2, 0, 0, p, None) == 2
        assert fn(p, 16, -3, 2, 0, 0, p, None) == 2
        assert fn(p, 1 << 40, 10, 2, 1, 0, p, None) == 2


def test_slot_range_and_window_validation(lib):
    # slot ranges, the window's extended rows and its attention: null pointers,
    # ranges past the view, bad windows and strides, answered on the host
    md = _lib.LocalMetadata()
    assert lib.dsa_cp_metadata_bind(C.c_void_p(0x10000), 1, 16, 2, C.byref(md)) == 0
    p = C.c_void_p(0x10000)
    f = C.c_float(0.07)
    # indexer over a slot range: the range must lie inside the view (tpr 8)
    assert lib.dsa_indexer_topk_rows(C.byref(md), 1, 8, 16, 4, 5, p, p, p, 16, 64, 128, 2048, p, p, 1 << 20,
                                     None) == 2
    assert lib.dsa_indexer_topk_rows(C.byref(md), 1, 8, 16, -1, 2, p, p, p, 16, 64, 128, 2048, p, p, 1 << 20,
                                     None) == 2
    assert lib.dsa_indexer_topk_rows(C.byref(md), 1, 8, 16, 0, -1, p, p, p, 16, 64, 128, 2048, p, p, 1 << 20,
                                     None) == 2
    assert lib.dsa_indexer_topk_rows(C.byref(md), 1, 8, 16, 2, 0, p, p, p, 16, 64, 128, 2048, p, p, 1 << 20,
                                     None) == 0
    assert lib.dsa_indexer_topk_rows(C.byref(md), 1, 8, 16, 2, 3, p, p, p, 16, 32, 128, 2048, p, p, 1 << 20,
                                     None) == 3
    # attention over a slot range and a token window
    assert lib.dsa_sparse_attn_prefill_rows(C.byref(md), 1, 8, 6, 3, p, 0, 16, p, 16, p, 2048, None, f, 128, 576,
                                            512, p, None) == 2
    assert lib.dsa_sparse_attn_prefill_rows(C.byref(md), 1, 8, 0, 3, p, -1, 16, p, 16, p, 2048, None, f, 128, 576,
                                            512, p, None) == 2
    assert lib.dsa_sparse_attn_prefill_rows(C.byref(md), 1, 8, 0, 3, p, 0, 0, p, 16, p, 2048, None, f, 128, 576,
                                            512, p, None) == 2
    assert lib.dsa_sparse_attn_prefill_rows(C.byref(md), 1, 8, 0, 0, p, 0, 0, p, 16, p, 2048, None, f, 128, 576,
                                            512, p, None) == 0
    assert lib.dsa_sparse_attn_prefill_rows(C.byref(md), 1, 8, 0, 3, p, 0, 16, p, 16, p, 2048, None, f, 96, 576,
                                            512, p, None) == 3
    # the window's extended rows: null pointers, W < 1, a stride below topk + W
    assert lib.dsa_swa_index(C.byref(md), 1, 8, None, 16, p, 2048, 128, 2176, p, p, None) == 1
    assert lib.dsa_swa_index(C.byref(md), 1, 8, p, 16, p, 2048, 0, 2176, p, p, None) == 2
    assert lib.dsa_swa_index(C.byref(md), 1, 8, p, 16, p, 2048, 128, 2175, p, p, None) == 2
    assert lib.dsa_swa_index(C.byref(md), 1, 0, p, 16, p, 2048, 128, 2176, p, p, None) == 0
    # its attention: counts missing, a second source without rows' pointer, stride below topk
    assert lib.dsa_sparse_attn_prefill_swa(C.byref(md), 1, 8, p, p, 16, None, 0, p, 2176, None, 2048, None, f, 128,
                                           576, 512, p, None) == 1
    assert lib.dsa_sparse_attn_prefill_swa(C.byref(md), 1, 8, p, p, 16, C.c_void_p(0x10008), 4, p, 2176, p, 2048,
                                           None, f, 128, 576, 512, p, None) == 1
    assert lib.dsa_sparse_attn_prefill_swa(C.byref(md), 1, 8, p, p, 16, None, 0, p, 2000, p, 2048, None, f, 128,
                                           576, 512, p, None) == 2
