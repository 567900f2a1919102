// Sliding-window rows for the sparse attention ("feat: DeepSeek-V4 DSA
// context-parallel on NPU", section 背景 names SWA beside the compressed KV;
// 单层前向数据流 (4) gives the attention the original KV's geometry besides
// the sparse selection).  Reading taken: a query at in-request position p
// also attends to the original latent rows of its own request at positions
// max(0, p - W + 1) .. p, under one softmax with its selected entries; at
// compress ratio 1 the entries are those same rows and a row that is both
// selected and in the window counts once.
//
// swa_index_kernel (one warp per local slot) writes the slot's extended
// index row: its selected rows as the top-k left them, then its window rows
// (at ratio 1 only those not selected; at ratio c > 1 every window row,
// numbered after the num_kv_rows compressed rows so that the attention reads
// it from the original KV), then -1; and the row's entry count.  Integer
// work: the result is exact.
//
// At ratio 1 the window rows are consecutive and the selection ascending, so
// the selected rows inside the window form one run of the selection: a
// 32-way search finds where it starts, and each 32-row piece of the window
// then takes the next (at most 32) entries of the run as a bit mask of the
// rows it holds.  Rows are copied 16 bytes at a time when the row lengths
// and pointers allow it.
#include "dsa_common.cuh"
#include "internal.h"

namespace dsa {
namespace {

struct SwaParams {
  dsa_cp_local_metadata md;
  const int32_t *ori_base;  // [local batch] original row of each local request's position 0
  const int32_t *topk_idx;  // [tpr][topk]
  int32_t *ext;             // [tpr][stride]
  int32_t *counts;          // [tpr]
  int32_t tpr, topk, window, stride, num_kv_rows;
  int *err;
};

constexpr int kSwaWarps = 4;

// first index in sel[0, n) whose entry is >= x, for an ascending sel; warp-wide
// (every lane returns it), ceil(log32(n)) + 1 rounds of one load per lane
__device__ __forceinline__ int warp_lower_bound(const int32_t *sel, int n, int x, int lane) {
  int lo = 0, hi = n;
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) >> 5;
    const int at = lo + lane * step;
    const unsigned below = __ballot_sync(0xffffffffu, at < hi && sel[at] < x);
    const int c = __popc(below);  // probes 0 .. c-1 lie below x
    if (c == 0) return lo;
    const int nlo = lo + (c - 1) * step + 1;
    hi = min(lo + c * step, hi);
    lo = nlo;
  }
  const unsigned below = __ballot_sync(0xffffffffu, lo + lane < hi && sel[lo + lane] < x);
  return lo + __popc(below);
}

__global__ void __launch_bounds__(32 * kSwaWarps) swa_index_kernel(const SwaParams P) {
  const int lane = threadIdx.x & 31;
  const int slot = blockIdx.x * kSwaWarps + (threadIdx.x >> 5);
  if (slot >= P.tpr) return;
  const int32_t *sel = P.topk_idx + static_cast<int64_t>(slot) * P.topk;
  int32_t *row = P.ext + static_cast<int64_t>(slot) * P.stride;
  const bool vec = ((P.topk | P.stride) & 3) == 0 && ((reinterpret_cast<uintptr_t>(P.topk_idx) |
                                                       reinterpret_cast<uintptr_t>(P.ext)) & 15) == 0;
  // the selection first (it needs no metadata, so its loads overlap the
  // lookups below): its valid entries come first, then -1
  int mine = 0;
  if (vec) {  // eight 16-byte loads per lane in flight before the stores
    const int4 *s4 = reinterpret_cast<const int4 *>(sel);
    int4 *r4 = reinterpret_cast<int4 *>(row);
    const int n4 = P.topk >> 2;
    for (int k0 = lane; k0 < n4; k0 += 8 * 32) {
      int4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (k0 + 32 * u < n4) v[u] = __ldg(s4 + k0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (k0 + 32 * u < n4) {
          r4[k0 + 32 * u] = v[u];
          mine += (v[u].x >= 0) + (v[u].y >= 0) + (v[u].z >= 0) + (v[u].w >= 0);
        }
    }
  } else {
    for (int k = lane; k < P.topk; k += 32) {
      const int32_t v = sel[k];
      row[k] = v;
      mine += v >= 0;
    }
  }
  const int g = P.md.local_token_pos[slot];
  const int nb = P.md.scalars[DSA_MD_LOCAL_BATCH];
  int n_sel = 0, n_out = 0;
  if (g >= 0 && nb > 0) {
    const int j = find_local_request(P.md.local_query_start_loc, nb, slot);
    const int ratio = max(1, P.md.scalars[DSA_MD_COMPRESS_RATIO]);
    const int pos = g - P.md.local_req_pos_base[j];
    n_sel = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(mine)));
    const int lo = max(0, pos - P.window + 1), nw = pos >= 0 ? pos - lo + 1 : 0;
    const int64_t first = ratio == 1 ? static_cast<int64_t>(P.md.local_req_kv_base[j]) + lo
                                     : static_cast<int64_t>(P.num_kv_rows) + P.ori_base[j] + lo;
    if (pos < 0 || first < 0 || first + nw > INT32_MAX) {
      if (lane == 0) record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 61, slot);
    } else {
      n_out = n_sel;
      // at ratio 1: entries sel[ptr ..] are the selected rows at or past the
      // current piece of the window
      int ptr = ratio == 1 ? warp_lower_bound(sel, n_sel, static_cast<int>(first), lane) : n_sel;
      for (int k0 = 0; k0 < nw; k0 += 32) {
        const int r0 = static_cast<int>(first) + k0;
        unsigned held = 0;  // bit b: row r0 + b is selected
        if (ratio == 1) {
          const int32_t v = ptr + lane < n_sel ? sel[ptr + lane] : INT32_MAX;
          const bool in = v >= r0 && v - r0 < 32;
          held = __reduce_or_sync(0xffffffffu, in ? 1u << (v - r0) : 0u);
          ptr += __popc(__ballot_sync(0xffffffffu, in));
        }
        const bool keep = k0 + lane < nw && !((held >> lane) & 1u);
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          const int at = n_out + __popc(bal & ((1u << lane) - 1u));
          if (at < P.stride) row[at] = r0 + lane;
          else record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 62, slot);
        }
        n_out += __popc(bal);
      }
      n_out = min(n_out, P.stride);
    }
  }
  for (int k = n_out + lane; k < P.stride; k += 32) row[k] = -1;
  if (lane == 0) P.counts[slot] = n_out;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_swa_index(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                    const int32_t *ori_req_kv_base, int32_t num_kv_rows, const int32_t *topk_idx,
                                    int32_t topk, int32_t window, int32_t ext_stride, int32_t *ext_idx,
                                    int32_t *counts, dsa_stream_t stream) {
  if (!md || !ori_req_kv_base || !topk_idx || !ext_idx || !counts) return DSA_ERR_INVALID_ARG;
  if (!md->scalars || !md->local_query_start_loc || !md->local_req_kv_base || !md->local_token_pos ||
      !md->local_req_pos_base)
    return DSA_ERR_INVALID_ARG;
  if (batch < 0 || tpr < 0 || num_kv_rows < 0 || topk < 1 || window < 1) return DSA_ERR_SHAPE;
  if (static_cast<int64_t>(ext_stride) < static_cast<int64_t>(topk) + window) return DSA_ERR_SHAPE;
  if (tpr == 0) return DSA_OK;
  int *err = device_error_word();
  if (!err) return DSA_ERR_CUDA;
  SwaParams P{*md, ori_req_kv_base, topk_idx, ext_idx, counts, tpr, topk, window, ext_stride, num_kv_rows, err};
  const int blocks = (tpr + kSwaWarps - 1) / kSwaWarps;
  swa_index_kernel<<<blocks, 32 * kSwaWarps, 0, reinterpret_cast<cudaStream_t>(stream)>>>(P);
  return check_launch();
}
