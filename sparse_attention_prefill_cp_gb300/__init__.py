"""GB300-native DeepSeek Sparse Attention (DSA) prefill on context-parallel views.

Thin PyTorch binding of libdsa_cp.so (include/dsa_cp.h): each function has
the C entry point's name, checks and marshals its tensors (device, dtype,
contiguity) and passes raw pointers plus the current CUDA stream.  Every
step of the path runs in the library's sm_103a kernels; if the library is
missing it is built, and if it cannot be built or loaded the call raises.
PyTorch only provides device memory and streams.
"""
from __future__ import annotations

import ctypes as C

import torch

from ._lib import DSAError, LocalMetadata, check, load  # noqa: F401

IN_SEQ_SPLIT = 0
ROUND_ROBIN = 1
HEAD_TAIL = 2

__all__ = [
    "IN_SEQ_SPLIT", "ROUND_ROBIN", "HEAD_TAIL", "DSAError", "CPLocalMetadata", "load",
    "dsa_cp_geometry", "dsa_cp_metadata_sizes", "dsa_cp_build_local_metadata", "dsa_cp_split",
    "dsa_cp_rerange", "dsa_cp_split_from_host", "dsa_cp_rerange_to_host", "dsa_cp_all_to_all_heads", "dsa_indexer_topk_workspace_size", "dsa_indexer_topk",
    "dsa_indexer_topk_rows", "dsa_indexer_scores", "dsa_indexer_fp8_rows", "dsa_indexer_topk_fp8", "dsa_indexer_scores_fp8",
    "dsa_sparse_attn_prefill", "dsa_sparse_attn_prefill_headsharded", "dsa_sparse_attn_prefill_rows",
    "dsa_swa_index",
    "dsa_sparse_attn_prefill_swa", "dsa_poll_device_error",
]


def _stream(stream) -> C.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _ptr(t) -> C.c_void_p | None:
    return None if t is None else C.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, dtype: torch.dtype, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def dsa_cp_geometry(num_tokens: int, cp_size: int) -> tuple[int, int]:
    """(num_tokens_pad, tokens_per_rank)."""
    pad, tpr = C.c_int32(), C.c_int32()
    check(load().dsa_cp_geometry(num_tokens, cp_size, C.byref(pad), C.byref(tpr)), "dsa_cp_geometry")
    return pad.value, tpr.value


def dsa_cp_metadata_sizes(batch: int, num_tokens: int, cp_size: int) -> int:
    n = C.c_size_t()
    check(load().dsa_cp_metadata_sizes(batch, num_tokens, cp_size, C.byref(n)), "dsa_cp_metadata_sizes")
    return n.value


class CPLocalMetadata:
    """One CP view's local metadata: a device int32 buffer and the C struct
    of pointers into it (dsa_cp_local_metadata)."""

    FIELDS = ("local_query_start_loc", "local_seq_lens", "local_kv_start_loc", "local_req_id",
              "local_req_kv_base", "local_token_pos", "local_req_pos_base")
    SCALARS = ("num_tokens_pad", "tokens_per_rank", "local_start", "local_end", "local_batch",
               "local_num_tokens", "local_max_seqlen_q", "local_max_seqlen_kv", "num_tokens", "num_kv_rows",
               "compress_ratio")

    def __init__(self, batch: int, num_tokens: int, cp_size: int, device=None):
        self.batch, self.num_tokens, self.cp_size = int(batch), int(num_tokens), int(cp_size)
        self.num_tokens_pad, self.tokens_per_rank = dsa_cp_geometry(num_tokens, cp_size)
        n = dsa_cp_metadata_sizes(batch, num_tokens, cp_size)
        self.buffer = torch.zeros(n, dtype=torch.int32, device=device or torch.device("cuda"))
        self.struct = LocalMetadata()
        check(load().dsa_cp_metadata_bind(_ptr(self.buffer), batch, num_tokens, cp_size, C.byref(self.struct)),
              "dsa_cp_metadata_bind")

    def to_host(self) -> dict:
        """Read the view back (synchronises); lists trimmed to their valid length."""
        b = self.buffer.cpu().tolist()
        B, tpr = self.batch, self.tokens_per_rank
        ns = len(self.SCALARS)
        out = dict(zip(self.SCALARS, b[:ns]))
        o = ns
        nb = out["local_batch"]
        # the order of dsa_cp_metadata_bind's carve-up
        for name, size, valid in (("local_query_start_loc", B + 1, nb + 1), ("local_seq_lens", B, nb),
                                  ("local_kv_start_loc", B + 1, nb + 1), ("local_req_id", B, nb),
                                  ("local_req_kv_base", B, nb), ("local_req_pos_base", B, nb),
                                  ("local_token_pos", tpr, tpr)):
            out[name] = b[o:o + valid]
            o += size
        return out


def dsa_cp_build_local_metadata(query_start_loc: torch.Tensor, seq_lens: torch.Tensor, num_tokens: int,
                                cp_size: int, cp_rank: int, mode: int, md: CPLocalMetadata | None = None,
                                stream=None, compress_ratio: int = 1) -> CPLocalMetadata:
    _need(query_start_loc, torch.int32, "query_start_loc")
    _need(seq_lens, torch.int32, "seq_lens")
    batch = seq_lens.numel()
    if query_start_loc.numel() != batch + 1:
        raise ValueError("query_start_loc must have batch + 1 entries")
    if md is None:
        md = CPLocalMetadata(batch, num_tokens, cp_size, query_start_loc.device)
    elif (md.batch, md.num_tokens, md.cp_size) != (batch, num_tokens, cp_size):
        raise ValueError("metadata buffer was sized for another batch / token count / cp_size")
    check(load().dsa_cp_build_local_metadata_compressed(_ptr(query_start_loc), _ptr(seq_lens), batch, num_tokens,
                                                        cp_size, cp_rank, mode, int(compress_ratio),
                                                        C.byref(md.struct), _stream(stream)),
          "dsa_cp_build_local_metadata")
    return md


def _row_bytes(t: torch.Tensor) -> int:
    return t[0].numel() * t.element_size() if t.dim() > 1 else t.element_size()


def dsa_cp_split(src: torch.Tensor, cp_size: int, mode: int, cp_rank: int = -1, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """src [T, ...] -> [cp_size, tpr, ...] (cp_rank == -1) or [tpr, ...]."""
    if not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA tensor")
    T = src.shape[0]
    _, tpr = dsa_cp_geometry(T, cp_size)
    shape = ((cp_size, tpr) if cp_rank < 0 else (tpr,)) + tuple(src.shape[1:])
    if out is None:
        out = torch.empty(shape, dtype=src.dtype, device=src.device)
    elif tuple(out.shape) != shape or out.dtype != src.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {src.dtype} tensor of shape {shape}")
    check(load().dsa_cp_split(_ptr(src), _row_bytes(src), T, cp_size, mode, cp_rank, _ptr(out), _stream(stream)),
          "dsa_cp_split")
    return out


def dsa_cp_rerange(src: torch.Tensor, num_tokens: int, cp_size: int, mode: int, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """src [cp_size, tpr, ...] -> [num_tokens, ...]."""
    if not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA tensor")
    _, tpr = dsa_cp_geometry(num_tokens, cp_size)
    if tuple(src.shape[:2]) != (cp_size, tpr):
        raise ValueError(f"src must be [cp_size={cp_size}, tpr={tpr}, ...]")
    shape = (num_tokens,) + tuple(src.shape[2:])
    if out is None:
        out = torch.empty(shape, dtype=src.dtype, device=src.device)
    elif tuple(out.shape) != shape or out.dtype != src.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {src.dtype} tensor of shape {shape}")
    row = src[0, 0].numel() * src.element_size() if src.dim() > 2 else src.element_size()
    check(load().dsa_cp_rerange(_ptr(src), row, num_tokens, cp_size, mode, _ptr(out), _stream(stream)),
          "dsa_cp_rerange")
    return out


def _host_rows(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host (CPU) tensor, page-locked for asynchronous copies")
    return t


def dsa_cp_split_from_host(host_src: torch.Tensor, cp_size: int, mode: int, cp_rank: int, out: torch.Tensor,
                           stream=None) -> torch.Tensor:
    """Rows of rank ``cp_rank`` of host_src [T, ...] (host memory) -> out
    [tpr, ...] (device) by the copy engines; pad rows of ``out`` untouched."""
    _host_rows(host_src, "host_src")
    T = host_src.shape[0]
    _, tpr = dsa_cp_geometry(T, cp_size)
    shape = (tpr,) + tuple(host_src.shape[1:])
    if not out.is_cuda or tuple(out.shape) != shape or out.dtype != host_src.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous CUDA {host_src.dtype} tensor of shape {shape}")
    check(load().dsa_cp_split_from_host(_ptr(host_src), _row_bytes(host_src), T, cp_size, mode, cp_rank, _ptr(out),
                                        _stream(stream)), "dsa_cp_split_from_host")
    return out


def dsa_cp_rerange_to_host(src: torch.Tensor, num_tokens: int, cp_size: int, mode: int, cp_rank: int,
                           host_out: torch.Tensor, stream=None) -> torch.Tensor:
    """Rank ``cp_rank``'s rows src [tpr, ...] (device) -> their token rows of
    host_out [num_tokens, ...] (host memory) by the copy engines."""
    _host_rows(host_out, "host_out")
    if not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA tensor")
    _, tpr = dsa_cp_geometry(num_tokens, cp_size)
    if src.shape[0] != tpr or tuple(host_out.shape) != (num_tokens,) + tuple(src.shape[1:]) or \
            host_out.dtype != src.dtype:
        raise ValueError("src must be [tpr, ...] and host_out [num_tokens, ...] of the same row shape and dtype")
    check(load().dsa_cp_rerange_to_host(_ptr(src), _row_bytes(src), num_tokens, cp_size, mode, cp_rank,
                                        _ptr(host_out), _stream(stream)), "dsa_cp_rerange_to_host")
    return host_out


def dsa_cp_all_to_all_heads(src: torch.Tensor, num_tokens: int, cp_size: int, mode: int,
                            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """src [cp_size, tpr, H, ...] (every view's output) -> [cp_size, num_tokens, H / cp_size, ...]."""
    if not src.is_cuda or not src.is_contiguous() or src.dim() < 3:
        raise ValueError("src must be a contiguous CUDA tensor [cp_size, tpr, H, ...]")
    _, tpr = dsa_cp_geometry(num_tokens, cp_size)
    H = src.shape[2]
    if tuple(src.shape[:2]) != (cp_size, tpr) or H % cp_size:
        raise ValueError(f"src must be [cp_size={cp_size}, tpr={tpr}, H divisible by cp_size, ...]")
    shape = (cp_size, num_tokens, H // cp_size) + tuple(src.shape[3:])
    if out is None:
        out = torch.empty(shape, dtype=src.dtype, device=src.device)
    elif tuple(out.shape) != shape or out.dtype != src.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {src.dtype} tensor of shape {shape}")
    head = src[0, 0, 0].numel() * src.element_size()
    check(load().dsa_cp_all_to_all_heads(_ptr(src), H, head, num_tokens, cp_size, mode, _ptr(out),
                                         _stream(stream)), "dsa_cp_all_to_all_heads")
    return out


def dsa_indexer_topk_workspace_size(tokens_per_rank: int, max_kv_len: int, topk: int) -> int:
    n = C.c_size_t()
    check(load().dsa_indexer_topk_workspace_size(tokens_per_rank, max_kv_len, topk, C.byref(n)),
          "dsa_indexer_topk_workspace_size")
    return n.value


def dsa_indexer_topk(md: CPLocalMetadata, q_idx: torch.Tensor, k_idx: torch.Tensor, w: torch.Tensor, topk: int,
                     max_kv_len: int, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """q_idx bf16 [tpr, HI, DI], k_idx bf16 [T, DI], w fp32 [tpr, HI] -> int32 [tpr, topk]."""
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(k_idx, torch.bfloat16, "k_idx")
    _need(w, torch.float32, "w")
    tpr, HI, DI = q_idx.shape
    if tpr != md.tokens_per_rank or tuple(w.shape) != (tpr, HI) or k_idx.shape[1] != DI:
        raise ValueError("q_idx / w / k_idx shapes do not match the view")
    if out is None:
        out = torch.empty((tpr, topk), dtype=torch.int32, device=q_idx.device)
    _need(out, torch.int32, "out")
    if workspace is None:
        workspace = torch.empty(dsa_indexer_topk_workspace_size(tpr, max_kv_len, topk), dtype=torch.uint8,
                                device=q_idx.device)
    check(load().dsa_indexer_topk(C.byref(md.struct), md.batch, tpr, max_kv_len, _ptr(q_idx), _ptr(k_idx), _ptr(w),
                                  k_idx.shape[0], HI, DI, topk, _ptr(out), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
          "dsa_indexer_topk")
    return out


def dsa_indexer_topk_rows(md: CPLocalMetadata, slot_begin: int, q_idx_rows: torch.Tensor, k_idx: torch.Tensor,
                          w_rows: torch.Tensor, topk: int, max_kv_len: int, out: torch.Tensor | None = None,
                          workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dsa_indexer_topk for the slots [slot_begin, slot_begin + n): q_idx_rows
    bf16 [n, HI, DI], w_rows fp32 [n, HI] -> int32 [n, topk]."""
    _need(q_idx_rows, torch.bfloat16, "q_idx_rows")
    _need(k_idx, torch.bfloat16, "k_idx")
    _need(w_rows, torch.float32, "w_rows")
    n, HI, DI = q_idx_rows.shape
    if tuple(w_rows.shape) != (n, HI) or k_idx.shape[1] != DI:
        raise ValueError("q_idx_rows / w_rows / k_idx shapes do not match")
    if out is None:
        out = torch.empty((n, topk), dtype=torch.int32, device=q_idx_rows.device)
    _need(out, torch.int32, "out")
    if workspace is None:
        workspace = torch.empty(dsa_indexer_topk_workspace_size(max(n, 1), max_kv_len, topk), dtype=torch.uint8,
                                device=q_idx_rows.device)
    check(load().dsa_indexer_topk_rows(C.byref(md.struct), md.batch, md.tokens_per_rank, max_kv_len, int(slot_begin),
                                       n, _ptr(q_idx_rows), _ptr(k_idx), _ptr(w_rows), k_idx.shape[0], HI, DI, topk,
                                       _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "dsa_indexer_topk_rows")
    return out


def dsa_indexer_topk_noalloc(md: CPLocalMetadata, q_idx: torch.Tensor, k_idx: torch.Tensor, w: torch.Tensor,
                             topk: int, max_kv_len: int, out: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """dsa_indexer_topk for callers that cannot allocate device memory at the
    call site: the score workspace is the library's fixed 32 MiB device array.
    ``out`` should be passed pre-allocated by such callers (when omitted it is
    allocated here, for convenience in tests).  Calls that overlap on the GPU
    share that array and race; the first call on a device should come before
    any stream capture."""
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(k_idx, torch.bfloat16, "k_idx")
    _need(w, torch.float32, "w")
    tpr, HI, DI = q_idx.shape
    if tpr != md.tokens_per_rank or tuple(w.shape) != (tpr, HI) or k_idx.shape[1] != DI:
        raise ValueError("q_idx / w / k_idx shapes do not match the view")
    if out is None:
        out = torch.empty((tpr, topk), dtype=torch.int32, device=q_idx.device)
    _need(out, torch.int32, "out")
    check(load().dsa_indexer_topk_noalloc(C.byref(md.struct), md.batch, tpr, max_kv_len, _ptr(q_idx),
                                          _ptr(k_idx), _ptr(w), k_idx.shape[0], HI, DI, topk, _ptr(out),
                                          _stream(stream)),
          "dsa_indexer_topk_noalloc")
    return out


def dsa_indexer_scores(md: CPLocalMetadata, q_idx: torch.Tensor, k_idx: torch.Tensor, w: torch.Tensor,
                       max_kv_len: int, row_begin: int = 0, row_count: int | None = None,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Test hook: fp32 scores [row_count, max_kv_len], -inf beyond each row's causal extent."""
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(k_idx, torch.bfloat16, "k_idx")
    _need(w, torch.float32, "w")
    tpr, HI, DI = q_idx.shape
    if row_count is None:
        row_count = tpr - row_begin
    if out is None:
        out = torch.empty((row_count, max_kv_len), dtype=torch.float32, device=q_idx.device)
    _need(out, torch.float32, "out")
    check(load().dsa_indexer_scores(C.byref(md.struct), md.batch, tpr, max_kv_len, _ptr(q_idx), _ptr(k_idx),
                                    _ptr(w), k_idx.shape[0], HI, DI, row_begin, row_count, _ptr(out),
                                    _stream(stream)),
          "dsa_indexer_scores")
    return out


def dsa_indexer_fp8_rows(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Index rows bf16 [..., DI] -> FP8 index rows uint8 [..., row_bytes]: the
    FP8 cache row with D = Dv = DI (E4M3 codes, one fp32 scale, zero padding),
    written by dsa_kv_fp8_quantize."""
    _need(x, torch.bfloat16, "x")
    DI = x.shape[-1]
    rb = dsa_kv_fp8_row_bytes(DI, DI)
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (rb,), dtype=torch.uint8, device=x.device)
    _need(out, torch.uint8, "out")
    if tuple(out.shape) != tuple(x.shape[:-1]) + (rb,):
        raise ValueError("out must have x's leading shape and FP8 rows")
    dsa_kv_fp8_quantize(x.reshape(-1, DI), DI, out.view(-1, rb), stream=stream)
    return out


def _fp8_index_shapes(md, q_idx8, k_idx8, w, DI):
    _need(q_idx8, torch.uint8, "q_idx8")
    _need(k_idx8, torch.uint8, "k_idx8")
    _need(w, torch.float32, "w")
    rb = dsa_kv_fp8_row_bytes(DI, DI)
    tpr, HI, qrb = q_idx8.shape
    if qrb != rb or k_idx8.dim() != 2 or k_idx8.shape[1] != rb or tuple(w.shape) != (tpr, HI):
        raise ValueError("q_idx8 / k_idx8 must be FP8 index rows of DI and w [tpr, HI]")
    if tpr != md.tokens_per_rank:
        raise ValueError("q_idx8 rows do not match the view")
    return tpr, HI


def dsa_indexer_topk_fp8(md: CPLocalMetadata, q_idx8: torch.Tensor, k_idx8: torch.Tensor, w: torch.Tensor,
                         topk: int, max_kv_len: int, DI: int = 128, out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q_idx8 uint8 [tpr, HI, row_bytes], k_idx8 uint8 [T, row_bytes] (FP8 index
    rows, dsa_indexer_fp8_rows), w fp32 [tpr, HI] -> int32 [tpr, topk]."""
    tpr, HI = _fp8_index_shapes(md, q_idx8, k_idx8, w, DI)
    if out is None:
        out = torch.empty((tpr, topk), dtype=torch.int32, device=q_idx8.device)
    _need(out, torch.int32, "out")
    if workspace is None:
        workspace = torch.empty(dsa_indexer_topk_workspace_size(tpr, max_kv_len, topk), dtype=torch.uint8,
                                device=q_idx8.device)
    check(load().dsa_indexer_topk_fp8(C.byref(md.struct), md.batch, tpr, max_kv_len, _ptr(q_idx8), _ptr(k_idx8),
                                      _ptr(w), k_idx8.shape[0], HI, DI, topk, _ptr(out), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
          "dsa_indexer_topk_fp8")
    return out


def dsa_indexer_scores_fp8(md: CPLocalMetadata, q_idx8: torch.Tensor, k_idx8: torch.Tensor, w: torch.Tensor,
                           max_kv_len: int, DI: int = 128, row_begin: int = 0, row_count: int | None = None,
                           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Test hook: dsa_indexer_scores over FP8 index rows."""
    tpr, HI = _fp8_index_shapes(md, q_idx8, k_idx8, w, DI)
    if row_count is None:
        row_count = tpr - row_begin
    if out is None:
        out = torch.empty((row_count, max_kv_len), dtype=torch.float32, device=q_idx8.device)
    _need(out, torch.float32, "out")
    check(load().dsa_indexer_scores_fp8(C.byref(md.struct), md.batch, tpr, max_kv_len, _ptr(q_idx8),
                                        _ptr(k_idx8), _ptr(w), k_idx8.shape[0], HI, DI, row_begin, row_count,
                                        _ptr(out), _stream(stream)),
          "dsa_indexer_scores_fp8")
    return out


def dsa_sparse_attn_prefill(md: CPLocalMetadata, q: torch.Tensor, kv: torch.Tensor, topk_idx: torch.Tensor,
                            softmax_scale: float, Dv: int, attn_sink: torch.Tensor | None = None,
                            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q bf16 [tpr, H, D], kv bf16 [T, D], topk_idx int32 [tpr, topk] -> bf16 [tpr, H, Dv]."""
    _need(q, torch.bfloat16, "q")
    _need(kv, torch.bfloat16, "kv")
    _need(topk_idx, torch.int32, "topk_idx")
    if attn_sink is not None:
        _need(attn_sink, torch.float32, "attn_sink")
    tpr, H, D = q.shape
    if tpr != md.tokens_per_rank or kv.shape[1] != D or topk_idx.shape[0] != tpr:
        raise ValueError("q / kv / topk_idx shapes do not match the view")
    if out is None:
        out = torch.empty((tpr, H, Dv), dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out")
    check(load().dsa_sparse_attn_prefill(C.byref(md.struct), md.batch, tpr, _ptr(q), _ptr(kv), kv.shape[0],
                                         _ptr(topk_idx), topk_idx.shape[1], _ptr(attn_sink), float(softmax_scale),
                                         H, D, Dv, _ptr(out), _stream(stream)),
          "dsa_sparse_attn_prefill")
    return out


def dsa_sparse_attn_prefill_headsharded(md: CPLocalMetadata, q: torch.Tensor, kv: torch.Tensor,
                                        topk_idx: torch.Tensor, softmax_scale: float, Dv: int, cp_size: int,
                                        out: torch.Tensor, attn_sink: torch.Tensor | None = None,
                                        stream=None) -> torch.Tensor:
    """As dsa_sparse_attn_prefill, writing into the head-sharded out bf16 [cp_size, T, H / cp_size, Dv]
    (shared by every view of the batch; each view fills the rows of its own tokens)."""
    _need(q, torch.bfloat16, "q")
    _need(kv, torch.bfloat16, "kv")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(out, torch.bfloat16, "out")
    if attn_sink is not None:
        _need(attn_sink, torch.float32, "attn_sink")
    tpr, H, D = q.shape
    if tpr != md.tokens_per_rank or kv.shape[1] != D or topk_idx.shape[0] != tpr:
        raise ValueError("q / kv / topk_idx shapes do not match the view")
    if cp_size < 1 or H % cp_size or tuple(out.shape) != (cp_size, md.num_tokens, H // cp_size, Dv):
        raise ValueError("out must be [cp_size, T, H / cp_size, Dv] with H divisible by cp_size")
    check(load().dsa_sparse_attn_prefill_headsharded(C.byref(md.struct), md.batch, tpr, _ptr(q), _ptr(kv),
                                                     kv.shape[0], _ptr(topk_idx), topk_idx.shape[1],
                                                     _ptr(attn_sink), float(softmax_scale), H, D, Dv, cp_size,
                                                     _ptr(out), _stream(stream)),
          "dsa_sparse_attn_prefill_headsharded")
    return out


def dsa_sparse_attn_prefill_flat(md: CPLocalMetadata, q: torch.Tensor, kv: torch.Tensor, topk_idx: torch.Tensor,
                                 softmax_scale: float, Dv: int, out: torch.Tensor,
                                 attn_sink: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One view's attention on the flat layout: q bf16 [T, H, D] (every token
    of the batch), out bf16 [T, H, Dv] shared by the views of the batch; the
    view's rows are reached through its local_token_pos."""
    _need(q, torch.bfloat16, "q")
    _need(kv, torch.bfloat16, "kv")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(out, torch.bfloat16, "out")
    if attn_sink is not None:
        _need(attn_sink, torch.float32, "attn_sink")
    T, H, D = q.shape
    tpr = md.tokens_per_rank
    if T != md.num_tokens or kv.shape[1] != D or tuple(topk_idx.shape[:1]) != (tpr,):
        raise ValueError("q / kv / topk_idx shapes do not match the view")
    if tuple(out.shape) != (T, H, Dv):
        raise ValueError("out must be [T, H, Dv]")
    check(load().dsa_sparse_attn_prefill_flat(C.byref(md.struct), md.batch, tpr, _ptr(q), T, _ptr(kv), kv.shape[0],
                                              _ptr(topk_idx), topk_idx.shape[1], _ptr(attn_sink),
                                              float(softmax_scale), H, D, Dv, _ptr(out), _stream(stream)),
          "dsa_sparse_attn_prefill_flat")
    return out


def dsa_sparse_attn_prefill_rows(md: CPLocalMetadata, slot_begin: int, slot_count: int, q_rows: torch.Tensor,
                                 q_row0: int, kv: torch.Tensor, topk_rows: torch.Tensor, softmax_scale: float,
                                 Dv: int, out_rows: torch.Tensor, attn_sink: torch.Tensor | None = None,
                                 stream=None) -> torch.Tensor:
    """The attention of the slots [slot_begin, slot_begin + slot_count) whose
    tokens lie in q_rows bf16 [n, H, D] (tokens q_row0 .. q_row0 + n - 1,
    flat order); their rows of out_rows bf16 [n, H, Dv] are written."""
    _need(q_rows, torch.bfloat16, "q_rows")
    _need(kv, torch.bfloat16, "kv")
    _need(topk_rows, torch.int32, "topk_rows")
    _need(out_rows, torch.bfloat16, "out_rows")
    if attn_sink is not None:
        _need(attn_sink, torch.float32, "attn_sink")
    n, H, D = q_rows.shape
    if kv.shape[1] != D or topk_rows.shape[0] < slot_count or tuple(out_rows.shape) != (n, H, Dv):
        raise ValueError("q_rows / kv / topk_rows / out_rows shapes do not match")
    check(load().dsa_sparse_attn_prefill_rows(C.byref(md.struct), md.batch, md.tokens_per_rank, int(slot_begin),
                                              int(slot_count), _ptr(q_rows), int(q_row0), n, _ptr(kv), kv.shape[0],
                                              _ptr(topk_rows), topk_rows.shape[1], _ptr(attn_sink),
                                              float(softmax_scale), H, D, Dv, _ptr(out_rows), _stream(stream)),
          "dsa_sparse_attn_prefill_rows")
    return out_rows


def dsa_swa_index(md: CPLocalMetadata, ori_md: CPLocalMetadata, topk_idx: torch.Tensor, window: int,
                  num_kv_rows: int, ext_idx: torch.Tensor | None = None, counts: torch.Tensor | None = None,
                  stream=None) -> tuple:
    """Extended index rows for the sliding window: (ext_idx int32 [tpr,
    stride], counts int32 [tpr]), stride = topk + window rounded up to a
    multiple of 4 (16-byte aligned rows) unless ``ext_idx`` is given.  ``ori_md``: the same view's
    metadata built with compress ratio 1 (``md`` itself at ratio 1), whose
    local_req_kv_base gives the original KV row of each local request."""
    _need(topk_idx, torch.int32, "topk_idx")
    tpr, topk = topk_idx.shape
    if tpr != md.tokens_per_rank or ori_md.tokens_per_rank != tpr or ori_md.batch != md.batch:
        raise ValueError("topk_idx / ori_md do not match the view")
    stride = (topk + int(window) + 3) // 4 * 4
    if ext_idx is None:
        ext_idx = torch.empty((tpr, stride), dtype=torch.int32, device=topk_idx.device)
    if counts is None:
        counts = torch.empty(tpr, dtype=torch.int32, device=topk_idx.device)
    _need(ext_idx, torch.int32, "ext_idx")
    _need(counts, torch.int32, "counts")
    if ext_idx.shape[0] != tpr or ext_idx.shape[1] < topk + int(window) or counts.numel() != tpr:
        raise ValueError("ext_idx must be [tpr, >= topk + window] and counts [tpr]")
    check(load().dsa_swa_index(C.byref(md.struct), md.batch, tpr, C.c_void_p(ori_md.struct.local_req_kv_base),
                               int(num_kv_rows), _ptr(topk_idx), topk, int(window), ext_idx.shape[1], _ptr(ext_idx),
                               _ptr(counts), _stream(stream)), "dsa_swa_index")
    return ext_idx, counts


def dsa_sparse_attn_prefill_swa(md: CPLocalMetadata, q: torch.Tensor, kv: torch.Tensor, kv_ori: torch.Tensor | None,
                                ext_idx: torch.Tensor, counts: torch.Tensor, topk: int, softmax_scale: float, Dv: int,
                                attn_sink: torch.Tensor | None = None, out: torch.Tensor | None = None,
                                stream=None) -> torch.Tensor:
    """One view's attention over its extended index rows (selected entries
    of ``kv`` plus window rows, of ``kv_ori`` when given): bf16 [tpr, H, Dv]."""
    _need(q, torch.bfloat16, "q")
    _need(kv, torch.bfloat16, "kv")
    _need(ext_idx, torch.int32, "ext_idx")
    _need(counts, torch.int32, "counts")
    if kv_ori is not None:
        _need(kv_ori, torch.bfloat16, "kv_ori")
    if attn_sink is not None:
        _need(attn_sink, torch.float32, "attn_sink")
    tpr, H, D = q.shape
    if tpr != md.tokens_per_rank or kv.shape[1] != D or ext_idx.shape[0] != tpr or counts.numel() != tpr:
        raise ValueError("q / kv / ext_idx / counts shapes do not match the view")
    if out is None:
        out = torch.empty((tpr, H, Dv), dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out")
    n_ori = 0 if kv_ori is None else kv_ori.shape[0]
    check(load().dsa_sparse_attn_prefill_swa(C.byref(md.struct), md.batch, tpr, _ptr(q), _ptr(kv), kv.shape[0],
                                             _ptr(kv_ori), n_ori, _ptr(ext_idx), ext_idx.shape[1], _ptr(counts),
                                             int(topk), _ptr(attn_sink), float(softmax_scale), H, D, Dv, _ptr(out),
                                             _stream(stream)), "dsa_sparse_attn_prefill_swa")
    return out


def dsa_kv_fp8_row_bytes(D: int, Dv: int) -> int:
    """Bytes of one FP8 latent-KV cache row (include/dsa_cp.h)."""
    n = C.c_size_t()
    check(load().dsa_kv_fp8_row_bytes(D, Dv, C.byref(n)), "dsa_kv_fp8_row_bytes")
    return n.value


def dsa_sparse_attn_prefill_fp8kv(md: CPLocalMetadata, q: torch.Tensor, kv_cache: torch.Tensor,
                                  topk_idx: torch.Tensor, softmax_scale: float, D: int, Dv: int, out: torch.Tensor,
                                  attn_sink: torch.Tensor | None = None, flat: bool = False,
                                  stream=None) -> torch.Tensor:
    """The attention over an FP8 latent cache uint8 [R, row_bytes] (as
    dsa_kv_fp8_quantize writes it), dequantised by the gather.  flat=False:
    the view layout (q [tpr, H, D], out [tpr, H, Dv]); flat=True: q [T, H, D]
    and out [T, H, Dv] in token order, as dsa_sparse_attn_prefill_flat."""
    _need(q, torch.bfloat16, "q")
    _need(kv_cache, torch.uint8, "kv_cache")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(out, torch.bfloat16, "out")
    if attn_sink is not None:
        _need(attn_sink, torch.float32, "attn_sink")
    rows, H, Dq = q.shape
    tpr = md.tokens_per_rank
    if Dq != D or kv_cache.dim() != 2 or kv_cache.shape[1] != dsa_kv_fp8_row_bytes(D, Dv):
        raise ValueError("q / kv_cache do not match (D, Dv)")
    if rows != (md.num_tokens if flat else tpr) or topk_idx.shape[0] != tpr or tuple(out.shape) != (rows, H, Dv):
        raise ValueError("q / topk_idx / out shapes do not match the view")
    check(load().dsa_sparse_attn_prefill_fp8kv(C.byref(md.struct), md.batch, tpr, _ptr(q), rows if flat else 0,
                                               _ptr(kv_cache), kv_cache.shape[0], _ptr(topk_idx), topk_idx.shape[1],
                                               _ptr(attn_sink), float(softmax_scale), H, D, Dv, _ptr(out),
                                               _stream(stream)),
          "dsa_sparse_attn_prefill_fp8kv")
    return out


def dsa_kv_fp8_quantize(kv: torch.Tensor, Dv: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kv bf16 [R, D] -> FP8 cache uint8 [R, row_bytes]."""
    _need(kv, torch.bfloat16, "kv")
    R, D = kv.shape
    rb = dsa_kv_fp8_row_bytes(D, Dv)
    if out is None:
        out = torch.empty((R, rb), dtype=torch.uint8, device=kv.device)
    _need(out, torch.uint8, "out")
    if tuple(out.shape) != (R, rb):
        raise ValueError(f"out must be [{R}, {rb}]")
    check(load().dsa_kv_fp8_quantize(_ptr(kv), R, D, Dv, _ptr(out), _stream(stream)), "dsa_kv_fp8_quantize")
    return out


def dsa_kv_fp8_dequantize(cache: torch.Tensor, D: int, Dv: int, out: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """FP8 cache uint8 [R, row_bytes] -> the bf16 rows [R, D] it stands for."""
    _need(cache, torch.uint8, "cache")
    R = cache.shape[0]
    if cache.dim() != 2 or cache.shape[1] != dsa_kv_fp8_row_bytes(D, Dv):
        raise ValueError("cache rows do not have the FP8 row size of (D, Dv)")
    if out is None:
        out = torch.empty((R, D), dtype=torch.bfloat16, device=cache.device)
    _need(out, torch.bfloat16, "out")
    if tuple(out.shape) != (R, D):
        raise ValueError(f"out must be [{R}, {D}]")
    check(load().dsa_kv_fp8_dequantize(_ptr(cache), R, D, Dv, _ptr(out), _stream(stream)), "dsa_kv_fp8_dequantize")
    return out


def dsa_poll_device_error(stream=None) -> None:
    """Synchronise and raise DSAError if a kernel recorded a device-side error
    (with the site that recorded it)."""
    detail = (C.c_int32 * 3)()
    status = load().dsa_poll_device_error_detail(_stream(stream), detail)
    if status != 0:
        raise DSAError(status, "dsa_poll_device_error", tuple(detail))
