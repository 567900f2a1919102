/*
 * dsa_cp.h -- C ABI of libdsa_cp.so: DeepSeek Sparse Attention (DSA) prefill
 * on context-parallel (CP) local query views, for GB300 (sm_103a).
 *
 * The hot path per CP view: lightning-indexer scores of the view's local
 * queries against the FULL index keys, a causal top-k per query, and MLA
 * sparse attention of every query head over the selected rows of the FULL
 * shared latent KV ("q local, KV full"); around it the CP geometry: the
 * local metadata of a rank, and the split / rerange permutations.
 *
 * Sources (pages, cited by title and section):
 *   [xLLM]   "feat: DeepSeek-V4 DSA context-parallel on NPU" (xLLM PR 1997)
 *   [blog]   "[DeepSeek v3.2] 上下文并行详解"
 *   [sglang] "NSA Prefill CP 中两次 All-Gather 的作用说明"
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers unless marked "host".  The
 *     caller owns and allocates every buffer; the library never allocates,
 *     frees or synchronises (except dsa_poll_device_error, which syncs).
 *   - Every call is asynchronous on the caller's CUDA stream (`stream`,
 *     a cudaStream_t; NULL = the legacy default stream).
 *   - Arguments are validated on the host before any launch; on an error
 *     the call returns a status and nothing is written or launched.
 *   - Device kernels never trap.  A bounds violation found on the device,
 *     a metadata inconsistency, or a wait that ran past its limit (about
 *     one second) sets a device error word and the kernel returns early;
 *     dsa_poll_device_error reports it.
 *   - bf16 tensors are row-major, contiguous, 16-byte aligned.
 *   - The library looks up the device addresses of its own static device
 *     arrays (the error record, the no-allocation scratch) once per device
 *     and keeps them for the life of the process.  They belong to the
 *     device's primary context: after a cudaDeviceReset of that device the
 *     kept addresses are stale, so do not use the library on that device
 *     again in the same process.
 *   - Supported dimension sets (others return DSA_ERR_UNSUPPORTED):
 *       DeepSeek-V3.2 shapes: H=128, D=576, Dv=512, HI=64, DI=128, topk=2048
 *       tiny shapes:          H=8,   D=64,  Dv=48,  HI=4,  DI=32,  topk=64
 */
#ifndef DSA_CP_H
#define DSA_CP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_CP_ABI_VERSION 9

typedef struct CUstream_st *dsa_stream_t; /* same type as cudaStream_t */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,    /* null pointer, rank out of range, bad mode  */
  DSA_ERR_SHAPE = 2,          /* sizes inconsistent or out of range         */
  DSA_ERR_UNSUPPORTED = 3,    /* dimension set not compiled                 */
  DSA_ERR_WORKSPACE = 4,      /* workspace too small                        */
  DSA_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed          */
  DSA_ERR_DEVICE_TIMEOUT = 6, /* a device wait ran past its limit           */
  DSA_ERR_DEVICE_BOUNDS = 7,  /* a device-side index was out of range       */
  DSA_ERR_DEVICE_SEQ_LENS = 8 /* metadata: a seq_lens below its query length */
} dsa_status;

typedef enum { DSA_CP_IN_SEQ_SPLIT = 0, DSA_CP_ROUND_ROBIN = 1, DSA_CP_HEAD_TAIL = 2 } dsa_cp_mode;

/* Indices into dsa_cp_local_metadata.scalars. */
enum {
  DSA_MD_NUM_TOKENS_PAD = 0,
  DSA_MD_TOKENS_PER_RANK = 1,
  DSA_MD_LOCAL_START = 2,
  DSA_MD_LOCAL_END = 3,
  DSA_MD_LOCAL_BATCH = 4,
  DSA_MD_LOCAL_NUM_TOKENS = 5,
  DSA_MD_LOCAL_MAX_SEQLEN_Q = 6,
  DSA_MD_LOCAL_MAX_SEQLEN_KV = 7,
  DSA_MD_NUM_TOKENS = 8,   /* query tokens T of the batch        */
  DSA_MD_NUM_KV_ROWS = 9,  /* KV rows of the batch = sum seq_lens / ratio */
  DSA_MD_COMPRESS_RATIO = 10,  /* compress_ratio c (1 = uncompressed) */
  DSA_MD_NUM_SCALARS = 11
};

/*
 * Local view of one CP rank ([xLLM] "代码实现 / 2. CP 本地元数据",
 * DSACPMetadata, without the RoPE tables).  All members are device int32
 * arrays owned by the caller; dsa_cp_metadata_bind carves them out of one
 * buffer of dsa_cp_metadata_sizes() ints.  B = global batch size,
 * tpr = tokens_per_rank.
 *   scalars[11]                 see DSA_MD_*; in round-robin mode the local
 *                               rows are {local_start + i*cp_size < local_end}
 *   local_query_start_loc[B+1]  cu-seqlens of the local queries (first
 *                               local_batch+1 entries valid)
 *   local_seq_lens[B]           KV extent seen by the local queries of each
 *                               local request = last local position + 1
 *                               (right-aligned, [xLLM] 单层前向数据流 (4))
 *   local_kv_start_loc[B+1]     exclusive cumsum of local_seq_lens
 *   local_req_id[B]             global request index of each local request
 *   local_req_kv_base[B]        KV row of that request's position 0 (KV and
 *                               index keys hold every request's whole
 *                               sequence, requests in order: the sum of the
 *                               seq_lens before it; = its first query row
 *                               when there is no prefix)
 *   local_token_pos[tpr]        flat query row of every local slot, -1 = pad
 *   local_req_pos_base[B]       a local slot of flat query row g in that
 *                               request is at position g - local_req_pos_base
 *                               (= first query row - prefix length)
 * Requests with no local row are not in the local batch.
 */
typedef struct {
  int32_t *scalars;
  int32_t *local_query_start_loc;
  int32_t *local_seq_lens;
  int32_t *local_kv_start_loc;
  int32_t *local_req_id;
  int32_t *local_req_kv_base;
  int32_t *local_token_pos;
  int32_t *local_req_pos_base;
} dsa_cp_local_metadata;

/* Host only.  num_tokens_pad = ceil(num_tokens / cp_size) * cp_size and
 * tokens_per_rank = num_tokens_pad / cp_size ([xLLM] 2).  Outputs are host
 * pointers.  Errors: DSA_ERR_INVALID_ARG (null output, cp_size < 1),
 * DSA_ERR_SHAPE (num_tokens < 0 or the padded count overflows int32). */
dsa_status dsa_cp_geometry(int32_t num_tokens, int32_t cp_size, int32_t *num_tokens_pad,
                           int32_t *tokens_per_rank);

/* Host only.  Number of int32 elements one view's metadata needs:
 * 11 + 2*(batch+1) + 4*batch + tokens_per_rank.  `ints_needed` is a host
 * pointer. */
dsa_status dsa_cp_metadata_sizes(int32_t batch, int32_t num_tokens, int32_t cp_size,
                                 size_t *ints_needed);

/* Host only.  Fill `out` (host struct) with pointers into `buffer` (device,
 * at least dsa_cp_metadata_sizes() ints, 4-byte aligned); no memory access. */
dsa_status dsa_cp_metadata_bind(int32_t *buffer, int32_t batch, int32_t num_tokens, int32_t cp_size,
                                dsa_cp_local_metadata *out);

/*
 * build_cp_local_metadata ([xLLM] "代码实现 / 2", [blog] "2.B"): the local
 * view of rank cp_rank.  query_start_loc [batch+1] and seq_lens [batch] are
 * device arrays with query_start_loc[0] = 0, query_start_loc[batch] =
 * num_tokens and seq_lens[b] = the KV length of request b, at least its
 * query length q_len_b.  Chunked prefill ([xLLM] 测试与验证; the separate KV
 * geometry of 单层前向数据流 (4)): the queries of request b are the last
 * q_len_b positions of its seq_lens[b]-token sequence, after a prefix of
 * seq_lens[b] - q_len_b positions whose KV is already present; KV and index
 * keys hold every request's whole sequence, requests in order.  With
 * seq_lens = query lengths there is no prefix.  A seq_lens below its query
 * length, or sum(seq_lens) beyond int32, is reported as
 * DSA_ERR_DEVICE_SEQ_LENS through dsa_poll_device_error, and inconsistent
 * query_start_loc as DSA_ERR_DEVICE_BOUNDS.  `out` is a host struct of
 * device pointers.  The local KV extent of a request (local_seq_lens) is its
 * prefix plus the positions up to its last local query (right-aligned).
 * Split of the flat token stream (padded at the end to a multiple of
 * cp_size):
 *   DSA_CP_IN_SEQ_SPLIT: rank r holds rows [r*tpr, (r+1)*tpr)
 *   DSA_CP_ROUND_ROBIN:  rank r holds rows g with g % cp_size == r, slot g / cp_size.
 *   DSA_CP_HEAD_TAIL:    the zigzag split ([xLLM] "7. Worker 侧 gate" names
 *                        "head-tail" only): with h = ceil(tpr/2), t = floor(tpr/2),
 *                        rank r holds rows [r*h, (r+1)*h) then
 *                        [cp*h + (cp-1-r)*t, cp*h + (cp-r)*t), both clipped to
 *                        [0, num_tokens) -- an early chunk paired with a late one,
 *                        which evens out the causal work.
 * cp_size == 1 gives the identity view.
 */
dsa_status dsa_cp_build_local_metadata(const int32_t *query_start_loc, const int32_t *seq_lens,
                                       int32_t batch, int32_t num_tokens, int32_t cp_size,
                                       int32_t cp_rank, dsa_cp_mode mode,
                                       const dsa_cp_local_metadata *out, dsa_stream_t stream);

/*
 * dsa_cp_build_local_metadata for compressed KV ([xLLM] "背景": compress_ratio
 * in {1, 4, 128}; "5. 模型前向装配": the sparse metadata of every ratio is
 * built with the local geometry).  At ratio c (>= 1, else
 * DSA_ERR_INVALID_ARG) a request of seq_lens[b] tokens has seq_lens[b] / c
 * (rounded down) compressed entries, entry e standing for positions
 * [e*c, (e+1)*c); the compressed latent rows and index keys of all requests
 * are stored in request order.  A query at position p sees the entries
 * e < (p + 1) / c (rounded down).  local_seq_lens, local_kv_start_loc,
 * local_req_kv_base and scalars[DSA_MD_NUM_KV_ROWS] count entries; query
 * positions (local_req_pos_base) stay in tokens; scalars[DSA_MD_COMPRESS_RATIO]
 * = c.  The indexer, top-k and attention read c from the metadata: their
 * k_idx / kv are then the compressed rows, and a query that sees no entry
 * selects nothing (-1) and gets a zero output row.  c = 1 is
 * dsa_cp_build_local_metadata.
 */
dsa_status dsa_cp_build_local_metadata_compressed(const int32_t *query_start_loc, const int32_t *seq_lens,
                                                  int32_t batch, int32_t num_tokens, int32_t cp_size,
                                                  int32_t cp_rank, dsa_cp_mode mode, int32_t compress_ratio,
                                                  const dsa_cp_local_metadata *out, dsa_stream_t stream);

/*
 * Split ([blog] "2.B" and "第三部分" step 1; [sglang] cp_split_and_rebuild):
 * gather the rows of src [num_tokens][row_bytes] that rank cp_rank holds
 * into dst [tpr][row_bytes] (cp_rank >= 0), or every rank's rows into the
 * rank-major layout dst [cp_size][tpr][row_bytes] (cp_rank == -1; this is
 * also the all-gathered order T0,T4,T1,T5,... of [blog] "第三部分" step B).
 * Pad rows are zero.  A byte copy: results are bit-exact.  row_bytes > 0.
 */
dsa_status dsa_cp_split(const void *src, int64_t row_bytes, int32_t num_tokens, int32_t cp_size,
                        dsa_cp_mode mode, int32_t cp_rank, void *dst, dsa_stream_t stream);

/*
 * Rerange ([blog] "第三部分" step B, [sglang] "第一次 All-Gather",
 * cp_all_gather_rerange_output): the inverse of the all-rank split, from
 * the rank-major src [cp_size][tpr][row_bytes] back to logical token order
 * dst [num_tokens][row_bytes]; pad rows are dropped.  Bit-exact.
 */
dsa_status dsa_cp_rerange(const void *src, int64_t row_bytes, int32_t num_tokens, int32_t cp_size,
                          dsa_cp_mode mode, void *dst, dsa_stream_t stream);

/*
 * The split and the rerange of ONE rank's rows between HOST memory and the
 * device, done by the copy engines (cudaMemcpy2DAsync: no kernel, no
 * allocation), for inputs and outputs that live on the host ([blog]
 * "第三部分": a rank receives its own rows of the token stream and its
 * outputs go back to logical token order).
 *   dsa_cp_split_from_host:  host_src [num_tokens][row_bytes] (host) ->
 *       dst [tpr][row_bytes] (device): the rows of rank cp_rank, slot order
 *       as in dsa_cp_split with that cp_rank.
 *   dsa_cp_rerange_to_host:  src [tpr][row_bytes] (device, rank cp_rank's
 *       slots) -> host_dst [num_tokens][row_bytes] (host): each real slot's
 *       row to its flat token row; other rows of host_dst are not written.
 * Pad slots are neither read nor written (the device buffer's pad rows keep
 * what they held).  A rank's rows are at most two runs of evenly spaced flat
 * rows (in-seq: one contiguous run; round-robin: stride cp_size rows;
 * head-tail: a head run and a tail run), so a call issues at most two 2D
 * copies on `stream`.  The host buffer should be page-locked
 * (cudaHostAlloc / cudaHostRegister) for the copy to be asynchronous;
 * pageable memory works but the copy then blocks the calling thread.
 * 0 <= cp_rank < cp_size.  Byte copies: bit-exact.  A failing copy returns
 * DSA_ERR_CUDA.
 */
dsa_status dsa_cp_split_from_host(const void *host_src, int64_t row_bytes, int32_t num_tokens, int32_t cp_size,
                                  dsa_cp_mode mode, int32_t cp_rank, void *dst, dsa_stream_t stream);
dsa_status dsa_cp_rerange_to_host(const void *src, int64_t row_bytes, int32_t num_tokens, int32_t cp_size,
                                  dsa_cp_mode mode, int32_t cp_rank, void *host_dst, dsa_stream_t stream);

/*
 * Head/token all-to-all of the attention outputs ([xLLM] 单层前向数据流 (6)
 * and "3. DSAttention 前向": all_to_all_4D with the head dimension scattered
 * and the token dimension gathered, pad rows sliced off), emulated for all
 * views on one device: from every view's output src [cp_size][tpr][num_heads]
 * [head_bytes] (the rank-major layout, pad slots ignored) to
 * dst [cp_size][num_tokens][num_heads / cp_size][head_bytes], where rank rd
 * holds heads rd * num_heads / cp_size .. (rd + 1) * num_heads / cp_size - 1
 * of every real token, tokens in flat order for both split modes (for
 * round-robin the rows are put back in flat order as by dsa_cp_rerange).
 * num_heads must divide by cp_size (else DSA_ERR_SHAPE).  A byte copy:
 * results are bit-exact.  The caller owns both buffers; the call is
 * asynchronous on `stream`.
 */
dsa_status dsa_cp_all_to_all_heads(const void *src, int32_t num_heads, int64_t head_bytes, int32_t num_tokens,
                                   int32_t cp_size, dsa_cp_mode mode, void *dst, dsa_stream_t stream);

/* Host only.  Recommended workspace bytes for dsa_indexer_topk: room for the
 * fp32 indexer scores of a block of local rows (rows x round_up(max_kv_len, 4)
 * x 4 bytes, at most 1 GiB, at least one 8-row tile).  Any size holding one
 * tile works; smaller workspaces take more launches. */
dsa_status dsa_indexer_topk_workspace_size(int32_t tokens_per_rank, int32_t max_kv_len, int32_t topk,
                                           size_t *bytes);

/*
 * Lightning indexer + causal top-k for one CP view ([xLLM] 单层前向数据流
 * (3) and "4. Indexer full/local 分离": local queries and weights, full
 * index keys).  For every local slot i with flat query row g in request b,
 * in-request position p = g - local_req_pos_base[b] and KV base
 * kb = local_req_kv_base[b] (p = g - qs_b and kb = qs_b without a prefix):
 *   I[i, s] = sum_j w[i, j] * ReLU(q_idx[i, j, :] . k_idx[kb + s, :]),  s = 0..p
 * and topk_idx[i, :] = the KV rows kb + s of the topk largest
 * I[i, s], ties to the lower s, in ascending order; rows with p + 1 <= topk
 * select every s; unused entries and pad slots are -1.
 *   md           host struct of device pointers (dsa_cp_build_local_metadata)
 *   batch        global batch size B (capacity of the md arrays)
 *   tpr          tokens_per_rank
 *   max_kv_len   host upper bound of every local_seq_lens entry (e.g. the
 *                longest request); a larger extent on the device is a
 *                DSA_ERR_DEVICE_BOUNDS
 *   q_idx        bf16 [tpr][HI][DI]   (local, split)
 *   k_idx        bf16 [num_kv_rows][DI] (full: every request's whole sequence)
 *   w            fp32 [tpr][HI]        (local, split)
 *   topk_idx     int32 [tpr][topk]     output
 *   workspace    device scratch of ws_bytes bytes (16-byte aligned)
 * Scores accumulate in fp32 on the tensor cores (bf16 inputs).
 */
dsa_status dsa_indexer_topk(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                            int32_t max_kv_len, const void *q_idx, const void *k_idx, const float *w,
                            int32_t num_kv_rows, int32_t HI, int32_t DI, int32_t topk, int32_t *topk_idx,
                            void *workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * dsa_indexer_topk over a range of the view's slots, [slot_begin,
 * slot_begin + slot_count): q_idx_rows bf16 [slot_count][HI][DI] and w_rows
 * fp32 [slot_count][HI] hold those slots' rows, topk_rows int32
 * [slot_count][topk] receives theirs; the metadata, keys and results are
 * those of dsa_indexer_topk (the same rows of its output).  For inputs that
 * arrive in pieces (a chunk of the token stream at a time).  0 <= slot_begin,
 * slot_begin + slot_count <= tpr.
 */
dsa_status dsa_indexer_topk_rows(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr, int32_t max_kv_len,
                                 int32_t slot_begin, int32_t slot_count, const void *q_idx_rows, const void *k_idx,
                                 const float *w_rows, int32_t num_kv_rows, int32_t HI, int32_t DI, int32_t topk,
                                 int32_t *topk_rows, void *workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * dsa_indexer_topk without a workspace argument, for callers that cannot
 * allocate device memory where they call it (inside an allocator or memory
 * pool callback, in a runtime whose memory is all owned by a pool, or from
 * a framework hook that must not call cudaMalloc).  The pages have no
 * counterpart; this is a deployment convenience.  Same inputs, outputs and
 * results as dsa_indexer_topk; the score workspace is a fixed 32 MiB array
 * inside the library (static device memory, held by every GPU that loads the
 * library until the process exits).  It allocates nothing: no cudaMalloc,
 * no cudaFree, no allocating library call.
 *   - Limit: the array must hold one query tile of scores, so
 *     max_kv_len <= 1,048,576 for the DeepSeek-V3.2 shapes (8-query tiles)
 *     and <= 65,536 for the tiny shapes (128-query tiles); larger values
 *     return DSA_ERR_WORKSPACE without launching.  Rows beyond what fits in
 *     one pass are processed in several passes over the same array.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps whatever the
 *     last call left in it.  Nothing needs to start at zero: each pass writes
 *     every score it later reads.  Calls whose kernels overlap on the GPU
 *     (other streams, other host threads) race on the array and give wrong
 *     results: serialise them.
 */
dsa_status dsa_indexer_topk_noalloc(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                    int32_t max_kv_len, const void *q_idx, const void *k_idx,
                                    const float *w, int32_t num_kv_rows, int32_t HI, int32_t DI,
                                    int32_t topk, int32_t *topk_idx, dsa_stream_t stream);

/*
 * Test hook: the indexer scores themselves for local slots
 * [row_begin, row_begin + row_count): scores [row_count][max_kv_len] fp32,
 * entry s of a row = I[i, s] for s <= p, -inf for s > p and for pad slots.
 * Same inputs and meaning as dsa_indexer_topk.
 */
dsa_status dsa_indexer_scores(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                              int32_t max_kv_len, const void *q_idx, const void *k_idx, const float *w,
                              int32_t num_kv_rows, int32_t HI, int32_t DI, int32_t row_begin,
                              int32_t row_count, float *scores, dsa_stream_t stream);

/*
 * FP8 indexer operands (the FP8 path that "[DeepSeek v3.2] 上下文并行详解",
 * section 1, opens with round-robin-split, applied to the index query and
 * keys; the page fixes no format).  q_idx8 and k_idx8 hold every DI-wide
 * index row -- one head of one local query, or one key -- in the FP8 cache
 * row format with D = Dv = DI (dsa_kv_fp8_quantize with D = Dv = DI writes
 * it): DI OCP E4M3 codes, the row's fp32 scale, zero bytes to a multiple of
 * 16 (144 bytes at DI = 128).  A row stands for decode(code) * scale, and
 * the score is the indexer score of those values:
 *   I[i, s] = sum_j w[i, j] * sq[i, j] * sk[kb + s]
 *                           * ReLU(codes_q[i, j, :] . codes_k[kb + s, :])
 * (sq, sk the row scales, positive), with the E4M3 products accumulated in
 * fp32 by tcgen05 kind::f8f6f4.  Otherwise the same as dsa_indexer_topk:
 *   q_idx8       FP8 rows [tpr][HI][row_bytes]          (local, split)
 *   k_idx8       FP8 rows [num_kv_rows][row_bytes]      (full)
 * Only HI = 64, DI = 128, topk = 2048 is compiled (DSA_ERR_UNSUPPORTED
 * otherwise).  Same workspace rule, same errors.
 */
dsa_status dsa_indexer_topk_fp8(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                int32_t max_kv_len, const void *q_idx8, const void *k_idx8, const float *w,
                                int32_t num_kv_rows, int32_t HI, int32_t DI, int32_t topk, int32_t *topk_idx,
                                void *workspace, size_t ws_bytes, dsa_stream_t stream);

/* Test hook: dsa_indexer_scores over FP8 operands (inputs as dsa_indexer_topk_fp8). */
dsa_status dsa_indexer_scores_fp8(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                  int32_t max_kv_len, const void *q_idx8, const void *k_idx8, const float *w,
                                  int32_t num_kv_rows, int32_t HI, int32_t DI, int32_t row_begin,
                                  int32_t row_count, float *scores, dsa_stream_t stream);

/*
 * MLA sparse attention prefill for one CP view ([xLLM] 单层前向数据流 (4):
 * local queries, full latent KV, output [T_local, num_heads_FULL, Dv]).
 * For every local slot i and head h over the valid selected rows J of
 * topk_idx[i, :]:
 *   l_j = softmax_scale * q[i, h, :] . kv[j, :]            (D-wide latent)
 *   out[i, h, :] = sum_j e^(l_j - m) kv[j, :Dv] / (sum_j e^(l_j - m) + e^(sink_h - m))
 * with m any common shift and the sink term present only when attn_sink
 * is non-NULL (a logit in scaled units that adds to the denominator only).
 *   q          bf16 [tpr][H][D] (local, split)
 *   kv         bf16 [num_kv_rows][D] (full: every request's whole sequence);
 *              value = the first Dv columns
 *   topk_idx   int32 [tpr][topk] KV rows, -1 = unused (as produced by
 *              dsa_indexer_topk: the valid entries first); a row outside
 *              [0, num_kv_rows) is a DSA_ERR_DEVICE_BOUNDS and is not read
 *   attn_sink  fp32 [H] or NULL
 *   out        bf16 [tpr][H][Dv]; pad slots are written as zeros
 * QK and PV run on the tensor cores (bf16 operands, fp32 accumulate); the
 * softmax is fp32.  Each view's per-token arithmetic is independent of the
 * view, so reranged views reproduce the single-view result.
 */
dsa_status dsa_sparse_attn_prefill(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                   const void *q, const void *kv, int32_t num_kv_rows,
                                   const int32_t *topk_idx, int32_t topk, const float *attn_sink,
                                   float softmax_scale, int32_t H, int32_t D, int32_t Dv, void *out,
                                   dsa_stream_t stream);

/*
 * dsa_sparse_attn_prefill with the head/token all-to-all fused into the
 * output stores ([xLLM] 单层前向数据流 (4) then (6)): same inputs and
 * arithmetic (the results are bit-identical to dsa_sparse_attn_prefill
 * followed by dsa_cp_all_to_all_heads), but each head row is written
 * straight to its place in out bf16 [cp_size][T][H / cp_size][Dv], with
 * T = the batch's query tokens (scalars[DSA_MD_NUM_TOKENS]): rank
 * h / (H / cp_size), token local_token_pos[i], head h % (H / cp_size).
 * Pad slots write nothing.  Every view of a batch writes into the same out;
 * their rows do not overlap.  cp_size >= 1 (else DSA_ERR_INVALID_ARG) and H
 * must divide by cp_size (else DSA_ERR_SHAPE).
 */
dsa_status dsa_sparse_attn_prefill_headsharded(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                               const void *q, const void *kv, int32_t num_kv_rows,
                                               const int32_t *topk_idx, int32_t topk, const float *attn_sink,
                                               float softmax_scale, int32_t H, int32_t D, int32_t Dv,
                                               int32_t cp_size, void *out, dsa_stream_t stream);

/*
 * dsa_sparse_attn_prefill on the flat token layout: q bf16 [num_tokens][H][D]
 * and out bf16 [num_tokens][H][Dv] hold every token of the batch in flat
 * order, and a view reads its local queries and writes its output rows at
 * local_token_pos[i].  Same arithmetic and results as the split of q
 * ([blog] "2.B"), dsa_sparse_attn_prefill and the rerange of the outputs
 * ([blog] "第三部分" step B) in sequence, without the two copies; every view
 * of a batch writes into the same out, their rows do not overlap, and pad
 * slots write nothing.  num_tokens = T of the metadata (a local_token_pos
 * at or beyond it is a DSA_ERR_DEVICE_BOUNDS).
 */
dsa_status dsa_sparse_attn_prefill_flat(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                        const void *q, int32_t num_tokens, const void *kv, int32_t num_kv_rows,
                                        const int32_t *topk_idx, int32_t topk, const float *attn_sink,
                                        float softmax_scale, int32_t H, int32_t D, int32_t Dv, void *out,
                                        dsa_stream_t stream);

/*
 * dsa_sparse_attn_prefill_flat over a range of the view's slots and a window
 * of the token stream: the slots [slot_begin, slot_begin + slot_count) with
 * their index rows topk_rows [slot_count][topk]; q_rows bf16
 * [num_q_rows][H][D] and out_rows bf16 [num_q_rows][H][Dv] hold the tokens
 * q_row0 .. q_row0 + num_q_rows - 1 in flat order, and a slot reads and
 * writes the row of its token (local_token_pos) there.  Every slot's token
 * must lie in that window (otherwise DSA_ERR_DEVICE_BOUNDS and nothing is
 * written for it); pad slots write nothing.  Same arithmetic and results as
 * the whole-view calls.  For inputs and outputs streamed a chunk of tokens
 * at a time.
 */
dsa_status dsa_sparse_attn_prefill_rows(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                        int32_t slot_begin, int32_t slot_count, const void *q_rows, int32_t q_row0,
                                        int32_t num_q_rows, const void *kv, int32_t num_kv_rows,
                                        const int32_t *topk_rows, int32_t topk, const float *attn_sink,
                                        float softmax_scale, int32_t H, int32_t D, int32_t Dv, void *out_rows,
                                        dsa_stream_t stream);

/*
 * Sliding window (SWA; [xLLM] "背景" names it beside the compressed KV, and
 * "单层前向数据流" (4) hands the attention the original KV's geometry besides
 * the sparse selection; the page does not say how the two combine).  Reading
 * taken: a query at in-request position p (tokens) also attends to the
 * ORIGINAL latent rows of its own request at positions max(0, p - W + 1) ..
 * p, under one softmax with its selected entries (and the sink, if any); at
 * compress ratio 1 the entries are those same rows and a row both selected
 * and in the window counts once.  Two calls:
 *
 * dsa_swa_index: for every local slot, the extended index row
 *   ext_idx [tpr][ext_stride] int32 = the slot's top-k row as dsa_indexer_topk
 *   wrote it (its valid entries, ascending), then its window rows, then -1;
 *   counts [tpr] int32 = the number of valid entries.  Window rows are KV row
 *   numbers: at ratio 1 (from md) local_req_kv_base[j] + position, only those
 *   the selection does not hold; at ratio c > 1, num_kv_rows +
 *   ori_req_kv_base[j] + position (rows of the original KV, numbered after
 *   the num_kv_rows compressed rows).
 *     md               the view's metadata (ratio c) that the top-k used
 *     ori_req_kv_base  [local batch] original KV row of each local request's
 *                      position 0: local_req_kv_base of the same view's
 *                      metadata built with ratio 1 (md's own at ratio 1)
 *     topk_idx         [tpr][topk] from dsa_indexer_topk
 *     window           W >= 1;  ext_stride >= topk + W (a multiple of 4 keeps
 *                      every row 16-byte aligned, which the attention needs)
 *   Integer work, exact.  Pad slots get count 0 and a row of -1.
 *
 * dsa_sparse_attn_prefill_swa: dsa_sparse_attn_prefill over the extended
 *   rows: entry e < num_kv_rows reads kv row e, entry e >= num_kv_rows reads
 *   kv_ori row e - num_kv_rows (kv_ori [num_ori_rows][D] bf16, every
 *   request's whole sequence in request order; NULL with num_ori_rows = 0 at
 *   ratio 1, where every entry is a kv row).  A slot's count replaces the
 *   causal key count (a query with no visible entry still attends to its
 *   window).  Output, layout, sink and precision as dsa_sparse_attn_prefill;
 *   an entry outside both sources is a DSA_ERR_DEVICE_BOUNDS (zero row used).
 */
dsa_status dsa_swa_index(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                         const int32_t *ori_req_kv_base, int32_t num_kv_rows, const int32_t *topk_idx,
                         int32_t topk, int32_t window, int32_t ext_stride, int32_t *ext_idx, int32_t *counts,
                         dsa_stream_t stream);
dsa_status dsa_sparse_attn_prefill_swa(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                       const void *q, const void *kv, int32_t num_kv_rows, const void *kv_ori,
                                       int32_t num_ori_rows, const int32_t *ext_idx, int32_t ext_stride,
                                       const int32_t *counts, int32_t topk, const float *attn_sink,
                                       float softmax_scale, int32_t H, int32_t D, int32_t Dv, void *out,
                                       dsa_stream_t stream);

/*
 * FP8 latent-KV cache ([blog] "1 核心改动总结": round-robin-split lifts the
 * restriction that NSA prefill CP could not use an FP8 KV cache; the page
 * gives no format).  Row layout taken (the published DeepSeek-V3.2 one):
 *   bytes [0, Dv)                  the Dv value columns as OCP FP8 E4M3 codes
 *   bytes [Dv, Dv + 4*tiles)       one fp32 scale per tile of 128 value columns
 *                                  (tiles = ceil(Dv / 128)); scale = tile
 *                                  max|x| / 448, 1 for an all-zero tile
 *   next 2*(D - Dv) bytes          the rope columns, bf16 as given
 *   zero bytes up to row_bytes     (a multiple of 16; 656 for D 576, Dv 512)
 * Codes are round-to-nearest-even of x / scale (fp32, IEEE division),
 * saturated at +-448.  Supported: 1 <= Dv <= D <= 65536, Dv and D - Dv
 * multiples of 8 (else DSA_ERR_SHAPE).  Byte-exact results.
 */
/* Host only: bytes of one cache row. */
dsa_status dsa_kv_fp8_row_bytes(int32_t D, int32_t Dv, size_t *bytes);

/* Quantise kv bf16 [num_rows][D] into cache [num_rows][row_bytes] (device
 * buffers, 16-byte aligned, caller-owned; asynchronous on `stream`). */
dsa_status dsa_kv_fp8_quantize(const void *kv, int32_t num_rows, int32_t D, int32_t Dv, void *cache,
                               dsa_stream_t stream);

/* The rows a cache stands for: kv bf16 [num_rows][D] with value column c of
 * tile t = bf16(fp32(decode(code)) * scale_t) (one fp32 rounding, then round
 * to nearest bf16) and the rope columns as stored.  The sparse attention over
 * an FP8 cache reads these rows. */
dsa_status dsa_kv_fp8_dequantize(const void *cache, int32_t num_rows, int32_t D, int32_t Dv, void *kv,
                                 dsa_stream_t stream);

/* dsa_sparse_attn_prefill (num_tokens = 0: the view layout) or
 * dsa_sparse_attn_prefill_flat (num_tokens > 0: q and out in flat token
 * order) over an FP8 latent cache instead of bf16 rows ([blog] 1 核心改动总结:
 * round-robin-split lets CP prefill use an FP8 KV cache):
 *   kv_cache   [num_kv_rows][row_bytes] in the layout above
 *              (dsa_kv_fp8_quantize writes it; row_bytes from
 *              dsa_kv_fp8_row_bytes), 16-byte aligned
 * The gather dequantises each selected row exactly as dsa_kv_fp8_dequantize
 * does, so the result equals dsa_sparse_attn_prefill over the dequantised
 * rows bit for bit; the cache is read instead of bf16 rows (328 instead of
 * 576 bytes per row and CTA).  Only H = 128, D = 576, Dv = 512, topk = 2048
 * is compiled (DSA_ERR_UNSUPPORTED otherwise).  Same errors as
 * dsa_sparse_attn_prefill. */
dsa_status dsa_sparse_attn_prefill_fp8kv(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                         const void *q, int32_t num_tokens, const void *kv_cache,
                                         int32_t num_kv_rows, const int32_t *topk_idx, int32_t topk,
                                         const float *attn_sink, float softmax_scale, int32_t H, int32_t D,
                                         int32_t Dv, void *out, dsa_stream_t stream);

/* Synchronise `stream`, then return (and clear) the first error a kernel
 * recorded on the current device since the last poll: DSA_OK, or
 * DSA_ERR_DEVICE_TIMEOUT / _BOUNDS / _SEQ_LENS; DSA_ERR_CUDA if the sync
 * itself failed (the message is in dsa_last_cuda_error()). */
dsa_status dsa_poll_device_error(dsa_stream_t stream);

/* As dsa_poll_device_error, and when an error is returned, `detail` (host,
 * 3 ints, may be NULL) receives where it was recorded: {site, site detail,
 * linear CTA index}.  Site codes: 11-18 indexer waits, 19-37 attention waits
 * (the detail is the key block), 41-46 bounds checks (indexer slot, top-k
 * slot, top-k overflow, attention slot, attention index, metadata). */
dsa_status dsa_poll_device_error_detail(dsa_stream_t stream, int32_t *detail);

/* Static string for a status code. */
const char *dsa_status_string(dsa_status status);

/* Static string of the last CUDA error a call returned DSA_ERR_CUDA for
 * (per thread; "" if none). */
const char *dsa_last_cuda_error(void);

/* DSA_CP_ABI_VERSION of the built library. */
int32_t dsa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_CP_H */
