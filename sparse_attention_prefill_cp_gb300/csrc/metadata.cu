// build_cp_local_metadata on the device ("feat: DeepSeek-V4 DSA
// context-parallel on NPU", section 代码实现 / 2; round-robin split of
// "[DeepSeek v3.2] 上下文并行详解", section 2.B).
//
// One CTA per call.  Per request b the number of local rows and the last
// local position come from closed forms (an interval intersection for
// in-seq-split, two for the head-tail zigzag, an arithmetic progression for
// round-robin); a block-wide exclusive scan compacts the requests that have
// local rows and accumulates the KV start of every request (the sum of the
// seq_lens before it).  In every mode a rank's slots are in ascending flat
// order, so the local rows of a request are consecutive slots.
//
// Chunked prefill (section 测试与验证 lists it; section 单层前向数据流 (4)
// gives the attention its own KV geometry): seq_lens[b] may exceed the query
// length; the queries are then the last positions of the request's sequence
// and its KV extent includes the prefix.
#include "dsa_common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Per request: a = has local rows, b = local rows, c = local KV extent,
// d = seq_lens (every request, for the KV starts).
struct Quad {
  int a, b, c, d;
  __device__ void add(const Quad &o) {
    a += o.a;
    b += o.b;
    c += o.c;
    d += o.d;
  }
};

// Exclusive scan of Quad over the block; returns the block totals in `tot`.
__device__ Quad block_exclusive_scan(Quad v, Quad &tot) {
  __shared__ Quad warp_tot[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Quad inc = v;
  for (int off = 1; off < 32; off <<= 1) {
    const Quad o = {__shfl_up_sync(0xffffffffu, inc.a, off), __shfl_up_sync(0xffffffffu, inc.b, off),
                    __shfl_up_sync(0xffffffffu, inc.c, off), __shfl_up_sync(0xffffffffu, inc.d, off)};
    if (lane >= off) inc.add(o);
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  Quad before = {0, 0, 0, 0};
  tot = {0, 0, 0, 0};
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before.add(warp_tot[w]);
    tot.add(warp_tot[w]);
  }
  __syncthreads();
  return {before.a + inc.a - v.a, before.b + inc.b - v.b, before.c + inc.c - v.c, before.d + inc.d - v.d};
}

__global__ void __launch_bounds__(kThreads) cp_metadata_kernel(const int32_t *__restrict__ qsl,
                                                               const int32_t *__restrict__ seq_lens, int B,
                                                               int T, int cp, int rank, int mode, int ratio,
                                                               dsa_cp_local_metadata md, int *err) {
  __shared__ int s_bad;
  __shared__ int s_run[4];  // running local_batch, query total, kv extent total, kv rows
  __shared__ int s_maxq, s_maxkv;
  __shared__ unsigned long long s_kv_rows;
  const int tid = threadIdx.x;
  const int64_t tpr = (static_cast<int64_t>(T) + cp - 1) / cp;

  if (tid == 0) {
    s_bad = 0;
    s_run[0] = s_run[1] = s_run[2] = s_run[3] = 0;
    s_maxq = s_maxkv = 0;
    s_kv_rows = 0;
  }
  __syncthreads();
  // Inputs: cu-seqlens from 0 to T; seq_lens at least the query lengths, in
  // total within int32 (the KV rows are indexed with int32).
  unsigned long long kv_rows = 0;
  for (int b = tid; b < B; b += kThreads) {
    const int qs = __ldg(qsl + b), qe = __ldg(qsl + b + 1), sl = __ldg(seq_lens + b);
    if (qe < qs || qs < 0 || qe > T) atomicOr(&s_bad, 1);
    else if (sl < qe - qs) atomicOr(&s_bad, 2);
    kv_rows += sl > 0 ? static_cast<unsigned long long>(sl) : 0ull;
  }
  atomicAdd(&s_kv_rows, kv_rows);
  if (tid == 0 && (__ldg(qsl) != 0 || __ldg(qsl + B) != T)) atomicOr(&s_bad, 1);
  __syncthreads();
  if (tid == 0 && s_kv_rows > static_cast<unsigned long long>(INT32_MAX)) s_bad |= 2;
  __syncthreads();
  const int bad = s_bad;
  if (bad && tid == 0) record_error(err, (bad & 1) ? DSA_ERR_DEVICE_BOUNDS : DSA_ERR_DEVICE_SEQ_LENS, 46, bad);

  // local slot -> flat token row
  const int64_t lo_inseq = static_cast<int64_t>(rank) * tpr;
  const int64_t hi_inseq = lo_inseq + tpr < T ? lo_inseq + tpr : T;
  // head-tail: the head chunk [lo_h, hi_h) and the tail chunk [lo_t, hi_t), clipped to T
  const int64_t ch = (tpr + 1) / 2, ct = tpr / 2;
  const int64_t lo_h = static_cast<int64_t>(rank) * ch, lo_t = cp * ch + (cp - 1 - rank) * ct;
  const int64_t hi_h = lo_h + ch < T ? lo_h + ch : T, hi_t = lo_t + ct < T ? lo_t + ct : T;
  for (int64_t i = tid; i < tpr; i += kThreads) {
    const int64_t g = cp_row_of_slot(rank, i, tpr, cp, mode);
    md.local_token_pos[i] = (!bad && g < T) ? static_cast<int32_t>(g) : -1;
  }
  if (tid == 0) {
    md.local_query_start_loc[0] = 0;
    md.local_kv_start_loc[0] = 0;
  }

  if (!bad) {
    for (int base = 0; base < B; base += kThreads) {
      const int b = base + tid;
      Quad v = {0, 0, 0, 0};
      int qs = 0, prefix = 0;
      if (b < B) {
        qs = __ldg(qsl + b);
        const int qe = __ldg(qsl + b + 1);
        const int sl = __ldg(seq_lens + b);
        prefix = sl - (qe - qs);
        v.d = sl / ratio;  // compressed entries of the request (all of it, c = 1)
        int64_t q_len = 0, last = -1;
        if (mode == DSA_CP_IN_SEQ_SPLIT) {
          const int64_t lo = qs > lo_inseq ? qs : lo_inseq;
          const int64_t hi = qe < hi_inseq ? qe : hi_inseq;
          if (hi > lo) {
            q_len = hi - lo;
            last = hi - 1;
          }
        } else if (mode == DSA_CP_HEAD_TAIL) {
          const int64_t lo1 = qs > lo_h ? qs : lo_h, hi1 = qe < hi_h ? qe : hi_h;
          const int64_t lo2 = qs > lo_t ? qs : lo_t, hi2 = qe < hi_t ? qe : hi_t;
          if (hi1 > lo1) {
            q_len += hi1 - lo1;
            last = hi1 - 1;
          }
          if (hi2 > lo2) {  // the tail chunk lies after the head chunk
            q_len += hi2 - lo2;
            last = hi2 - 1;
          }
        } else {
          // first g >= qs with g % cp == rank
          const int64_t g0 = qs + ((rank - qs % cp) % cp + cp) % cp;
          if (g0 < qe) {
            q_len = (qe - 1 - g0) / cp + 1;
            last = g0 + (q_len - 1) * cp;
          }
        }
        // KV extent: the prefix plus the positions up to the last local query,
        // in entries of `ratio` tokens
        if (q_len > 0) v = {1, static_cast<int>(q_len), static_cast<int>((prefix + last - qs + 1) / ratio), v.d};
      }
      Quad tot;
      Quad ex = block_exclusive_scan(v, tot);
      if (v.a) {
        const int j = s_run[0] + ex.a;
        md.local_query_start_loc[j + 1] = s_run[1] + ex.b + v.b;
        md.local_kv_start_loc[j + 1] = s_run[2] + ex.c + v.c;
        md.local_seq_lens[j] = v.c;
        md.local_req_id[j] = b;
        md.local_req_kv_base[j] = s_run[3] + ex.d;  // KV row of position 0
        md.local_req_pos_base[j] = qs - prefix;     // position of flat row g = g - pos_base
        atomicMax(&s_maxq, v.b);
        atomicMax(&s_maxkv, v.c);
      }
      __syncthreads();
      if (tid == 0) {
        s_run[0] += tot.a;
        s_run[1] += tot.b;
        s_run[2] += tot.c;
        s_run[3] += tot.d;
      }
      __syncthreads();
    }
  }

  if (tid == 0) {
    int32_t *s = md.scalars;
    s[DSA_MD_NUM_TOKENS_PAD] = static_cast<int32_t>(tpr * cp);
    s[DSA_MD_TOKENS_PER_RANK] = static_cast<int32_t>(tpr);
    if (mode == DSA_CP_IN_SEQ_SPLIT) {
      s[DSA_MD_LOCAL_START] = static_cast<int32_t>(lo_inseq < T ? lo_inseq : T);
      s[DSA_MD_LOCAL_END] = static_cast<int32_t>(hi_inseq > lo_inseq ? hi_inseq : (lo_inseq < T ? lo_inseq : T));
    } else if (mode == DSA_CP_HEAD_TAIL) {  // from the head chunk's start to the tail chunk's end
      const int64_t st = lo_h < T ? lo_h : T;
      const int64_t en = lo_t + ct < T ? lo_t + ct : T;
      s[DSA_MD_LOCAL_START] = static_cast<int32_t>(st);
      s[DSA_MD_LOCAL_END] = static_cast<int32_t>(en > st ? en : st);
    } else {
      s[DSA_MD_LOCAL_START] = rank < T ? rank : T;
      s[DSA_MD_LOCAL_END] = T;
    }
    s[DSA_MD_LOCAL_BATCH] = s_run[0];
    s[DSA_MD_LOCAL_NUM_TOKENS] = s_run[1];
    s[DSA_MD_LOCAL_MAX_SEQLEN_Q] = s_maxq;
    s[DSA_MD_LOCAL_MAX_SEQLEN_KV] = s_maxkv;
    s[DSA_MD_NUM_TOKENS] = T;
    s[DSA_MD_NUM_KV_ROWS] = bad ? 0 : s_run[3];  // sum of the requests' entries
    s[DSA_MD_COMPRESS_RATIO] = ratio;
  }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_cp_build_local_metadata_compressed(const int32_t *query_start_loc,
                                                             const int32_t *seq_lens, int32_t batch,
                                                             int32_t num_tokens, int32_t cp_size, int32_t cp_rank,
                                                             dsa_cp_mode mode, int32_t compress_ratio,
                                                             const dsa_cp_local_metadata *out, dsa_stream_t stream) {
  if (!query_start_loc || !seq_lens || !out) return DSA_ERR_INVALID_ARG;
  if (compress_ratio < 1) return DSA_ERR_INVALID_ARG;
  if (cp_size < 1 || cp_rank < 0 || cp_rank >= cp_size) return DSA_ERR_INVALID_ARG;
  if (mode != DSA_CP_IN_SEQ_SPLIT && mode != DSA_CP_ROUND_ROBIN && mode != DSA_CP_HEAD_TAIL)
    return DSA_ERR_INVALID_ARG;
  if (!out->scalars || !out->local_query_start_loc || !out->local_seq_lens || !out->local_kv_start_loc ||
      !out->local_req_id || !out->local_req_kv_base || !out->local_token_pos || !out->local_req_pos_base)
    return DSA_ERR_INVALID_ARG;
  if (batch < 0 || num_tokens < 0) return DSA_ERR_SHAPE;
  int32_t pad = 0, tpr = 0;
  dsa_status st = dsa_cp_geometry(num_tokens, cp_size, &pad, &tpr);
  if (st != DSA_OK) return st;
  int *err = device_error_word();
  if (!err) return DSA_ERR_CUDA;
  cp_metadata_kernel<<<1, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      query_start_loc, seq_lens, batch, num_tokens, cp_size, cp_rank, static_cast<int>(mode), compress_ratio, *out,
      err);
  return check_launch();
}

extern "C" dsa_status dsa_cp_build_local_metadata(const int32_t *query_start_loc, const int32_t *seq_lens,
                                                  int32_t batch, int32_t num_tokens, int32_t cp_size,
                                                  int32_t cp_rank, dsa_cp_mode mode,
                                                  const dsa_cp_local_metadata *out, dsa_stream_t stream) {
  return dsa_cp_build_local_metadata_compressed(query_start_loc, seq_lens, batch, num_tokens, cp_size, cp_rank, mode,
                                                1, out, stream);
}
