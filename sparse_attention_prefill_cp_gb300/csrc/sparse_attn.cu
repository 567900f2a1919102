// MLA sparse attention prefill for one CP view ("feat: DeepSeek-V4 DSA
// context-parallel on NPU", section 单层前向数据流 (4): local queries, the
// full shared latent KV, output [T_local, num_heads_FULL, Dv]).
//
// Per local query token: S = scale * Q K^T over its selected latent rows
// (Q: [128 heads, D], K = the gathered rows [n, D]), softmax over the rows
// with an optional per-head sink in the denominator, O = P V with V the
// first Dv columns of the same rows.
//
// GB300 layout (DeepSeek-V3.2 shapes, D = 576, Dv = 512): one fp32 O
// accumulator of 128 heads x 512 values fills an SM's whole tensor memory,
// so each token runs on a 2-CTA cluster.  CTA c owns value columns
// [256c, 256c + 256) and computes the partial QK over latent dims
// [256c, 256c + 256) + [512 + 32c, 512 + 32c + 32): the gathered rows split
// evenly (576 bytes per CTA per row, no row read twice) and the value
// columns are exactly the CTA's main QK chunks, so one smem tile serves as
// QK's K-major B and PV's MN-major B.
//
// Tensor memory per CTA (512 columns): O (256), two S buffers (2 x 64) and
// the CTA's 256 main Q dims as bf16 (128), so the QK MMA reads A from TMEM
// and only the 64-row key block from shared memory.
//
// Per CTA, 16 warps: 0-7 softmax in two warpgroups (one head row = one TMEM
// lane per thread; warpgroup w owns columns [32w, 32w + 32) of each block),
// 8 TMA for Q then event-driven MMA issue (TMEM owner), 9
// the exchange agent, 10-15 gather of the selected rows with 16-byte cp.async
// straight into the 128B / 64B swizzled tiles (two warps per stage, eight
// threads per 128-byte chunk so that loads coalesce into whole lines).  Key blocks of
// 64 rows, 4 smem stages.  S leaves TMEM as raw q.k sums; the softmax scale
// (times log2 e) is applied in the exponent's FMA.  The partial S tiles are
// exchanged in fp16 (11 significant bits; the logits are far inside its
// range, and the conversion saturates rather than overflow): the softmax threads stage their
// rows locally and warp 9 ships each tile to the peer's double-buffered
// receive tiles with one bulk copy that completes the peer's mbarrier
// transaction count, one block ahead of the softmax that needs it.  Each CTA
// softmaxes its own fp32 partial plus the peer's fp16 one and normalises its
// own O half.  P (bf16) goes to a shared-memory tile, so an S buffer is free
// as soon as it has been read and QK runs two blocks ahead of PV; the
// denominator sums the fp32 exponentials whose bf16 roundings PV uses.  The
// running max is rescaled lazily: O and l change only when some row of a warp
// sees its block max exceed the max in use by more than 2^8.
//
// The tiny shapes (H = 8, D = 64, Dv = 48) run the same kernel on one CTA
// with Q rows 8..127 zero-filled by the TMA.
//
// Over the FP8 latent cache ("[DeepSeek v3.2] 上下文并行详解", 1 核心改动总结:
// round-robin-split lets CP prefill use an FP8 KV cache) the gather warps read
// each selected row's E4M3 codes, tile scales and bf16 rope columns (328
// bytes per row and CTA instead of 576) and dequantise into the same bf16
// tiles, exactly as the cache's dequantiser does; the rest of the kernel is
// unchanged, so the result equals the attention over the dequantised rows.
//
// Output layouts: the view's [tpr][H][Dv] (pad rows zero), or, fused into the
// epilogue's stores, the head-sharded layout that the head/token all-to-all
// after the attention produces (单层前向数据流 (6)): [cp][T][H / cp][Dv], rank
// rd holding heads rd * H / cp .. of every real token (pad slots write
// nothing).  Flat layout: q [T][H][D] and out [T][H][Dv] in token order, the
// view's rows reached through local_token_pos -- the split of q before the
// attention and the rerange after it ([blog] 第三部分) done by the loads and
// stores themselves.
//
// A query's selected rows are KV rows of its own request, whose position 0
// is KV row local_req_kv_base; with chunked prefill the KV holds the prefix
// too and the query's position is g - local_req_pos_base.
#include "dsa_common.cuh"
#include "internal.h"

namespace dsa {
namespace {

template <int NMAIN_, bool TAIL_, int DVC_, bool SPLIT_, bool FP8KV_ = false>
struct AttnCfg {
  static constexpr int NMAIN = NMAIN_;  // 64-wide latent chunks per CTA (128B swizzle)
  static constexpr bool TAIL = TAIL_;   // plus one 32-wide chunk (64B swizzle)
  static constexpr int DVC = DVC_;      // value columns per CTA
  static constexpr bool SPLIT = SPLIT_; // 2-CTA cluster per token
  static constexpr bool FP8KV = FP8KV_; // the rows come from the FP8 latent cache (dequantised by the gather)
  static constexpr int kBN = 64;        // selected rows per block
  static constexpr int kHalf = kBN / 2; // columns per softmax warpgroup
  static constexpr int kStages = 4;
  // warps: 0-7 softmax (two warpgroups); 8 TMEM owner, TMA (Q) then MMA issue;
  // 9 exchange agent; 10-15 row gather, warps 10 + 2g and 11 + 2g taking blocks j = g (mod 3)
  static constexpr int kThreads = 512;
  static constexpr int kQMain = NMAIN * 128 * 128;
  static constexpr int kQTail = TAIL ? 128 * 64 : 0;
  static constexpr int kStageMain = NMAIN * kBN * 128;
  static constexpr int kStageBytes = kStageMain + (TAIL ? kBN * 64 : 0);
  static constexpr int kUnitsPerRow = NMAIN * 8 + (TAIL ? 4 : 0);  // 16-byte pieces per gathered row
  static constexpr int kQKMainSteps = NMAIN * 4;
  static constexpr int kQKSteps = kQKMainSteps + (TAIL ? 2 : 0);
  static constexpr int kPVSteps = kBN / 16;
  // tensor memory columns
  static constexpr int kOCols = (DVC + 63) / 64 * 64;
  static constexpr int kSCol = kOCols;              // two S buffers
  static constexpr int kQCol = kSCol + 2 * kBN;     // Q main dims, bf16 pairs
  static constexpr int kTmemCols = (kQCol + NMAIN * 32) <= 256 ? 256 : 512;
  // shared memory
  static constexpr int kRecvBytes = SPLIT ? 128 * kBN * 2 : 0;  // one partial-S tile (fp16), rows swizzled
  // P [128 heads][64 keys] bf16, SW128: for the pair it overwrites the peer's
  // partial-S tile of the same block (same row layout), so P is double
  // buffered by the two receive tiles; the single CTA keeps its own tile
  static constexpr int kPBytes = SPLIT ? 0 : 128 * 128;
  static constexpr int kOffStage = 0;
  static constexpr int kOffQStage = kOffStage + kStageBytes;  // Q main staged in stages 1..2 at start
  static constexpr int kOffQTail = kOffStage + kStages * kStageBytes;
  static constexpr int kOffRecv = kOffQTail + kQTail;
  static constexpr int kOffStg = kOffRecv + 2 * kRecvBytes;   // our partial-S tiles on their way out (two)
  static constexpr int kOffP = kOffStg + 2 * kRecvBytes;
  static constexpr int kOffRed = kOffP + kPBytes;             // [3][2 warpgroups][128] floats
  static constexpr int kOffBar = kOffRed + 3 * 2 * 128 * 4;
  static constexpr int kNumBars = 2 + 2 * kStages + 2 * 9 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 32 + 1024;
  // the tiny variant asks for enough smem that at most two CTAs share an SM's TMEM
  static constexpr int kSmemBytes = kSmemUsed < 100 * 1024 && !SPLIT ? 100 * 1024 : kSmemUsed;
  static constexpr uint32_t kIdescQK = idesc_bf16(128, kBN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, DVC, false, true);
  static constexpr uint32_t kRecvTx = 128 * kBN * 2;
  static_assert(kQCol + NMAIN * 32 <= kTmemCols, "TMEM budget");
  static_assert(DVC % 16 == 0 && DVC <= NMAIN * 64, "value columns inside the main chunks");
  static_assert(kQMain <= 2 * kStageBytes, "Q staging fits in stages 1..2");
  static_assert(kBN % 8 == 0, "gather covers rows in groups of 8");
  static_assert(kStageBytes % 1024 == 0 && kOffQTail % 1024 == 0 && kOffP % 1024 == 0, "alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

using BigAttn = AttnCfg<4, true, 256, true>;
using TinyAttn = AttnCfg<1, false, 48, false>;
using BigAttnFp8 = AttnCfg<4, true, 256, true, true>;

struct AttnParams {
  dsa_cp_local_metadata md;
  const __nv_bfloat16 *kv;   // [num_kv_rows][D]
  const __nv_bfloat16 *kv2;  // second row source (rows num_kv_rows ..), or nullptr
  const uint8_t *kv8;        // FP8 latent cache [num_kv_rows][kv8_row_bytes] (FP8KV configurations)
  int32_t kv8_row_bytes, kv8_rope;  // its row stride, and the byte offset of the bf16 rope columns
  const int32_t *topk_idx;   // [tpr][idx_stride]
  const int32_t *counts;     // [tpr] valid entries per row (then the rows are not causal-clamped), or nullptr
  const float *sink;         // [H] or nullptr
  __nv_bfloat16 *out;        // [tpr][H][Dv], [cp][T][hc][Dv] when hc > 0, [T][H][Dv] when flat
  float scale_log2;          // softmax_scale * log2(e)
  int32_t topk, H, D, Dv, num_kv_rows;
  int32_t idx_stride;        // entries per index row (topk, or topk + window)
  int32_t num_rows2;         // rows of kv2
  int32_t hc;                // heads per rank of the head-sharded output, 0 = view layout
  int32_t flat;              // 1: q and out in flat token order (rows by local_token_pos)
  int32_t q_rows;            // rows of q: tpr, or T when flat
  int32_t slot_begin;        // slot of CTA pair 0 (and of row 0 of the index rows, and of q / out in the view layout)
  int32_t q_row0;            // flat layout: token of q / out row 0
  int *err;
};

// One arrival per warp: the warp's threads synchronise (ordering their prior
// memory and fenced tcgen05 operations) and lane 0 arrives for all of them.
__device__ __forceinline__ void warp_arrive(uint64_t *bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Zero one output row of the CTA's value columns: head h of the view-layout or
// flat row at out_row, or of token g in the head-sharded layout.  Kept out of
// line: it runs only for pad slots and for queries without keys, and inlined
// its address arithmetic costs the pipelined part of the kernel registers.
__device__ __noinline__ void zero_row(const AttnParams &P, __nv_bfloat16 *out_row, int h, int g, int T, int col0,
                                      int cols) {
  __nv_bfloat16 *o = out_row + static_cast<int64_t>(h) * P.Dv;
  if (P.hc > 0) {  // head-sharded: rank h / hc, token g, head h % hc
    const int rd = h / P.hc;
    o = P.out + ((static_cast<int64_t>(rd) * T + g) * P.hc + (h - rd * P.hc)) * P.Dv + col0;
  }
  for (int c = 0; c < cols; c += 8) *reinterpret_cast<uint4 *>(o + c) = make_uint4(0, 0, 0, 0);
}

// Multiply TMEM columns [c0, c1) of the warp's lanes by alpha (the lazy
// rescale of O).  Out of line: it runs only when a row's max grows by more
// than 2^8.  Warp-collective (tcgen05.ld/st .sync.aligned): the whole warp calls it.
__device__ __noinline__ void scale_o_cols(uint32_t lane_base, int c0, int c1, float alpha) {
#pragma unroll 1
  for (int c = c0; c < c1; c += 32) {
    uint32_t r[32];
    tmem_ld32(lane_base + c, r);
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
    tmem_st32(lane_base + c, r);
  }
  tmem_st_wait();
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The FP8 cache's share of one gather thread (2-CTA configuration): for rows
// r0, r0 + 8, ... of the block, the codes [32 v, 32 v + 32) of the CTA's 256
// value dims and their tile's scale are read with 16-byte loads (four rows in
// flight), dequantised exactly as the cache's dequantiser does
// (bf16(fp32(decode(code)) * scale)) and stored into the 128B-swizzled main
// tiles; the rope columns are bf16 in the cache and go to the tail tile by
// cp.async as they are.  An entry outside the rows is zero-filled (and
// reported if it is a valid entry).
template <class C>
__device__ __forceinline__ void gather_fp8(const AttnParams &P, uint32_t sb, int (&rows)[C::kBN / 8], int k0,
                                           int n_valid, int v, int r0, int crank) {
  static_assert(C::SPLIT && C::NMAIN == 4 && C::TAIL, "the 2-CTA latent split");
  const int cb = C::NMAIN * 64 * crank + 32 * v;   // code byte of the thread's first dim
  const int sbyte = P.Dv + 4 * (cb / 128);          // its tile's scale
  const int chunk = v >> 1;                         // 64-dim chunk of the stage
#pragma unroll
  for (int rr = 0; rr < C::kBN / 8; ++rr) {
    const int row = rows[rr];
    if (k0 + r0 + 8 * rr < n_valid && (row < 0 || row >= P.num_kv_rows)) {
      record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 45, k0 + r0 + 8 * rr);
      rows[rr] = -1;
    } else if (row >= P.num_kv_rows) {
      rows[rr] = -1;
    }
  }
#pragma unroll
  for (int h4 = 0; h4 < C::kBN / 32; ++h4) {  // four rows at a time
    uint4 c0[4], c1[4];
    float scl[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int row = rows[h4 * 4 + q];
      if (row >= 0) {
        const uint8_t *src = P.kv8 + static_cast<int64_t>(row) * P.kv8_row_bytes;
        c0[q] = __ldg(reinterpret_cast<const uint4 *>(src + cb));
        c1[q] = __ldg(reinterpret_cast<const uint4 *>(src + cb + 16));
        scl[q] = __ldg(reinterpret_cast<const float *>(src + sbyte));
      } else {
        c0[q] = c1[q] = make_uint4(0u, 0u, 0u, 0u);
        scl[q] = 0.f;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + 8 * (h4 * 4 + q);
      const uint32_t w8[8] = {c0[q].x, c0[q].y, c0[q].z, c0[q].w, c1[q].x, c1[q].y, c1[q].z, c1[q].w};
      const float sc = scl[q];
#pragma unroll
      for (int u = 0; u < 4; ++u) {  // 8 codes -> one 16-byte unit of bf16
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a, b;
          unpack_f16x2(e4m3x2_to_f16x2((w8[2 * u + (e >> 1)] >> (16 * (e & 1))) & 0xffffu), a, b);
          o[e] = pack_bf16x2(__fmul_rn(a, sc), __fmul_rn(b, sc));
        }
        const int unit = (v & 1) * 4 + u;
        st_shared_v4(sb + chunk * (C::kBN * 128) + r * 128 + ((unit ^ (r & 7)) << 4), o[0], o[1], o[2], o[3]);
      }
    }
  }
  // the rope columns (bf16 in the cache): four threads per row, 16 bytes each
  if (v < 4) {
#pragma unroll
    for (int rr = 0; rr < C::kBN / 8; ++rr) {
      const int r = r0 + 8 * rr, row = rows[rr];
      const uint8_t *src = P.kv8 + static_cast<int64_t>(row < 0 ? 0 : row) * P.kv8_row_bytes + P.kv8_rope + 64 * crank;
      cp_async_16(sb + C::kStageMain + r * 64 + ((v ^ ((r >> 1) & 3)) << 4), src + 16 * v, row < 0 ? 0u : 16u);
    }
  }
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap qmain_map, const __grid_constant__ CUtensorMap qtail_map,
                       const AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *q_full = bars;                     // Q staged + tail landed (TMA)
  uint64_t *q_ready = bars + 1;                // Q main copied into TMEM, staging free (8 softmax warps)
  uint64_t *kv_full = bars + 2;                // [kStages] gathered rows landed (64 gather threads)
  uint64_t *kv_empty = kv_full + C::kStages;   // [kStages] PV done with the stage (MMA commit)
  uint64_t *s_full = kv_empty + C::kStages;    // [2] QK done (MMA commit)
  uint64_t *s_free = s_full + 2;               // [2] S read out of TMEM (8 softmax warps)
  uint64_t *p_full = s_free + 2;               // [2] P tile written (8 softmax warps)
  uint64_t *pv_done = p_full + 2;              // [2] PV done, its P tile free (MMA commit)
  uint64_t *recv_full = pv_done + 2;           // [2] the peer's partial S landed (st.async tx)
  uint64_t *recv_empty = recv_full + 2;        // [2] the peer is done with what we sent (peer's agent)
  uint64_t *red_full = recv_empty + 2;         // [2] both warpgroups' block maxima written (8 warps)
  uint64_t *staged = red_full + 2;             // [2] our partial-S tile written (8 softmax warps)
  uint64_t *stg_free = staged + 2;             // [2] the bulk copy has read our tile (sender)
  uint64_t *fin_full = stg_free + 2;           // both warpgroups' denominators written (8 warps)
  uint64_t *o_staged = fin_full + 1;           // normalised O rows staged in smem (8 warps)
  // [0] tmem, [1] base, [2] keys the query sees (-1: pad or error), [3] g, [4] T
  int32_t *misc = reinterpret_cast<int32_t *>(smem + C::kOffMisc);
  float *red = reinterpret_cast<float *>(smem + C::kOffRed);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = C::SPLIT ? cluster_ctarank() : 0u;
  const uint32_t peer = crank ^ 1u;
  const int slot = P.slot_begin + (C::SPLIT ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x));
  const int main_dim0 = C::SPLIT ? static_cast<int>(crank) * C::NMAIN * 64 : 0;
  const int tail_dim0 = C::NMAIN * 64 * (C::SPLIT ? 2 : 1) + 32 * static_cast<int>(crank);

  // Q's TMA first (warp 8, lane 0): it needs only the token's row, so its
  // latency overlaps the metadata lookup, the barrier set-up and the cluster
  // barrier.  An out-of-range row reads the fill value (the lookup below
  // reports it); a token that turns out to see no key drains the load before
  // it exits.
  bool q_issued = false;
  if (warp == 8 && lane == 0) {
    const int g0 = P.md.local_token_pos[slot];
    mbar_init(q_full, 1);
    fence_mbar_init();
    if (g0 >= 0) {
      const int qrow0 = P.flat ? g0 - P.q_row0 : slot - P.slot_begin;
      tma_prefetch_desc(&qmain_map);
      mbar_arrive_expect_tx(q_full, C::kQMain + C::kQTail);
      for (int i = 0; i < C::NMAIN; ++i)
        tma_load_3d(smem + C::kOffQStage + i * 16384, &qmain_map, main_dim0 + 64 * i, 0, qrow0, q_full);
      if (C::TAIL) tma_load_3d(smem + C::kOffQTail, &qtail_map, tail_dim0, 0, qrow0, q_full);
      q_issued = true;
    }
  }
  if (tid == 0) {
    int base = 0, p = -1;
    const int g = P.md.local_token_pos[slot];
    const int nbatch = P.md.scalars[DSA_MD_LOCAL_BATCH];
    if (g >= 0 && nbatch > 0) {
      const int j = find_local_request(P.md.local_query_start_loc, nbatch, slot);
      base = P.md.local_req_kv_base[j];
      const int pos = g - P.md.local_req_pos_base[j];
      const int ratio = max(1, P.md.scalars[DSA_MD_COMPRESS_RATIO]);
      p = pos >= 0 ? (pos + 1) / ratio : -1;  // keys (entries) the query sees
      if (pos < 0 || base < 0 || base + p > P.num_kv_rows || (P.flat && (g < P.q_row0 || g - P.q_row0 >= P.q_rows))) {
        record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 44, slot);
        p = -1;
      } else if (P.counts) {  // an extended index row: its own entry count
        p = P.counts[slot];
        if (p < 0 || p > P.idx_stride) {
          record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 46, slot);
          p = -1;
        }
      }
    }
    misc[1] = base;
    misc[2] = p;
    misc[3] = g;
    misc[4] = P.md.scalars[DSA_MD_NUM_TOKENS];
    mbar_init(q_ready, 8);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&kv_full[s], 64);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 8);
      mbar_init(&p_full[b], 8);
      mbar_init(&pv_done[b], 1);
      mbar_init(&recv_full[b], 1);
      mbar_init(&recv_empty[b], 1);
      mbar_init(&red_full[b], 8);
      mbar_init(&staged[b], 8);
      mbar_init(&stg_free[b], 1);
    }
    mbar_init(fin_full, 8);
    mbar_init(o_staged, 8);
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(reinterpret_cast<uint32_t *>(&misc[0]), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  if (C::SPLIT) cluster_sync();
  else __syncthreads();
  tc_fence_after();

  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int p = misc[2];
  const int n_valid = p >= 0 ? (P.counts ? p : min(p, P.topk)) : 0;
  const int nb = (n_valid + C::kBN - 1) / C::kBN;
  const int qrow = P.flat ? misc[3] - P.q_row0 : slot - P.slot_begin;  // the row of q and of the output
  __nv_bfloat16 *out_row = P.out + (static_cast<int64_t>(qrow) * P.H) * P.Dv + main_dim0;

  if (nb == 0) {
    // a pad slot (zero rows in the view layout; the other layouts have none),
    // or a token that sees no compressed entry (zero rows in every layout)
    if (warp < 4 && tid < P.H && ((misc[3] >= 0 && p == 0) || (P.hc == 0 && !P.flat)))
      zero_row(P, out_row, tid, misc[3], misc[4], main_dim0, C::DVC);
    if (q_issued) mbar_wait(q_full, 0, P.err, 24);  // the Q load issued at the start has landed
  } else if (warp == 8) {
    if (lane == 0) {
      // ---------------- MMA issuer: QK runs two blocks ahead of PV (Q was
      // loaded by TMA at the start: main dims to a staging tile, tail dims in place)
      const uint32_t st_addr = smem_u32(smem + C::kOffStage);
      const uint32_t qt_addr = smem_u32(smem + C::kOffQTail);
      const uint32_t p_addr = smem_u32(smem + C::kOffP);
      const uint32_t recv_addr = smem_u32(smem + C::kOffRecv);
      // Descriptors are built once here and advanced by constant offsets (in
      // 16-byte units; every shared address is below 256 KB, so the 14-bit
      // address field never carries): rebuilding them per MMA made issue,
      // not the tensor pipe, the limit of the 64-wide QK steps.
      const uint64_t qk_b0 = smem_desc(st_addr, 16, 1024, kLayoutSW128);
      const uint64_t qk_t0 = smem_desc(st_addr + C::kStageMain, 16, 512, kLayoutSW64);
      const uint64_t qt_a0 = smem_desc(qt_addr, 16, 512, kLayoutSW64);
      const uint64_t pv_a0 = smem_desc(C::SPLIT ? recv_addr : p_addr, 16, 1024, kLayoutSW128);
      const uint64_t pv_b0 = smem_desc(st_addr, C::kBN * 128, 1024, kLayoutSW128);
      const uint32_t s_tm = tmem + C::kSCol, q_tm = tmem + C::kQCol;
      bool ok = mbar_wait(q_full, 0, P.err, 23) && mbar_wait(q_ready, 0, P.err, 23);
      tc_fence_after();
      // event-driven issue: QK(j) as soon as its rows have landed, its S buffer
      // is free and PV(j - 3) has been issued, PV(i) as soon as P(i) is
      // written; each stream in order.  S(j) is first read when the softmax
      // starts block j - 1, one block after P(j - 3) is written, so the gate
      // costs QK nothing, and it keeps a QK that became ready early from
      // holding the issuing thread (and the tensor pipe) when P(j - 3) arrives.
      int qk = 0, pv = 0;
      long long t_prog = clock64(), t_check = t_prog;
      while (ok && pv < nb) {
        bool progressed = false;
        if (qk < nb && qk < pv + 3 && mbar_test(&kv_full[qk % C::kStages], (qk / C::kStages) & 1) &&
            (qk < 2 || mbar_test(&s_free[qk & 1], ((qk - 2) >> 1) & 1))) {
          tc_fence_after();
          const uint32_t d = s_tm + (qk & 1) * C::kBN;
          const uint32_t so = static_cast<uint32_t>((qk % C::kStages) * C::kStageBytes) >> 4;
          const uint64_t kb = desc_add(qk_b0, so), kt = desc_add(qk_t0, so);
#pragma unroll
          for (int k = 0; k < C::kQKSteps; ++k) {
            if (k < C::kQKMainSteps) {
              const int i = k >> 2, sub = k & 3;
              mma_ts(d, q_tm + k * 8, desc_add(kb, (i * (C::kBN * 128) + sub * 32) >> 4), C::kIdescQK,
                     k > 0 ? 1u : 0u);
            } else {
              const int t = k - C::kQKMainSteps;
              mma_ss(d, desc_add(qt_a0, t * 2), desc_add(kt, t * 2), C::kIdescQK, 1u);
            }
          }
          mma_commit(&s_full[qk & 1]);
          ++qk;
          progressed = true;
        }
        if (pv < qk && mbar_test(&p_full[pv & 1], (pv >> 1) & 1)) {
          tc_fence_after();
          const int bi = pv & 1, si = pv % C::kStages;
          const uint64_t vb = desc_add(pv_b0, static_cast<uint32_t>(si * C::kStageBytes) >> 4);
          const uint64_t pb = desc_add(pv_a0, C::SPLIT ? static_cast<uint32_t>(bi * C::kRecvBytes) >> 4 : 0u);
#pragma unroll
          for (int k = 0; k < C::kPVSteps; ++k)
            mma_ss(tmem, desc_add(pb, k * 2), desc_add(vb, k * 128), C::kIdescPV, (pv > 0 || k > 0) ? 1u : 0u);
          mma_commit(&pv_done[bi]);
          mma_commit(&kv_empty[si]);
          ++pv;
          progressed = true;
        }
        const long long now = clock64();
        if (progressed) {
          t_prog = now;
        } else if (now - t_check > 100000) {
          t_check = now;
          if (error_set(P.err)) {
            ok = false;
          } else if (now - t_prog > kWaitLimitCycles) {
            record_error(P.err, DSA_ERR_DEVICE_TIMEOUT, 37, qk * 10000 + pv);
            ok = false;
          }
        }
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, P.err, 21);
      if (C::SPLIT) {
        // ---------------- exchange agent: ships each staged partial-S tile to the
        // peer with one bulk copy, and tells the peer when its tiles have been read
        const uint32_t peer_recv = map_to_cta(smem_u32(smem + C::kOffRecv), peer);
        const uint32_t peer_full = map_to_cta(smem_u32(recv_full), peer);
        for (int t = 0; ok && t <= nb; ++t) {
          if (t < nb) {
            const int b = t & 1;
            if (!(ok = mbar_wait(&staged[b], (t >> 1) & 1, P.err, 35, t))) break;
            if (t >= 2 && !(ok = mbar_wait<true>(&recv_empty[b], ((t >> 1) & 1) ^ 1, P.err, 28, t))) break;
            bulk_copy_to_peer(peer_recv + b * C::kRecvBytes, smem + C::kOffStg + b * C::kRecvBytes, C::kRecvBytes,
                              peer_full + b * 8);
            bulk_commit();
            bulk_wait_read0();
            mbar_arrive(&stg_free[b]);
          }
          if (t >= 1) {
            const int b = (t - 1) & 1;
            // PV(t-1) has read P(t-1), which sits in the tile the peer filled
            if (!(ok = mbar_wait(&pv_done[b], ((t - 1) >> 1) & 1, P.err, 36, t - 1))) break;
            mbar_arrive_remote_relaxed(&recv_empty[b], peer);
          }
        }
        bulk_wait_read0();
      }
    }
  } else if (warp >= 10) {
    // ---------------- gather of the selected rows: warps 10 + 2g and 11 + 2g
    // take the blocks j = g (mod 3), block j going to stage j % 4.  Eight
    // consecutive threads copy one 128-byte chunk of a row (one 16-byte
    // cp.async each, the 128B swizzle applied on the destination), so each warp
    // instruction reads four whole lines; a thread covers rows r0, r0 + 8, ...
    // The row indices of the group's next block are fetched while this one lands.
    constexpr int kGroups = 3, kRowsPerThread = C::kBN / 8;
    const int g = (warp - 10) >> 1, t = ((warp - 10) & 1) * 32 + lane;
    const int v = t & 7, r0 = t >> 3;
    const int32_t *idx_row = P.topk_idx + static_cast<int64_t>(slot - P.slot_begin) * P.idx_stride;
    int rows[kRowsPerThread];
    auto fetch = [&](int j) {
#pragma unroll
      for (int rr = 0; rr < kRowsPerThread; ++rr) {
        const int k = j * C::kBN + r0 + 8 * rr;
        rows[rr] = k < n_valid ? __ldg(idx_row + k) : -1;
      }
    };
    if (g < nb) fetch(g);
    for (int j = g; j < nb; j += kGroups) {
      const int s = j % C::kStages;
      if (!mbar_wait(&kv_empty[s], ((j / C::kStages) & 1) ^ 1, P.err, 22, j)) break;
      // stages 1 and 2 held the staged Q until the softmax warps moved it to TMEM
      if ((j == 1 || j == 2) && !mbar_wait(q_ready, 0, P.err, 20, j)) break;
      const uint32_t sb = smem_u32(smem + C::kOffStage + s * C::kStageBytes);
      if constexpr (C::FP8KV) {
        gather_fp8<C>(P, sb, rows, j * C::kBN, n_valid, v, r0, static_cast<int>(crank));
      } else {
#pragma unroll
      for (int rr = 0; rr < kRowsPerThread; ++rr) {
        const int r = r0 + 8 * rr;
        int row = rows[rr];
        if (j * C::kBN + r < n_valid && (row < 0 || row >= P.num_kv_rows + P.num_rows2)) {
          record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 45, j * C::kBN + r);
          row = -1;
        }
        // rows past num_kv_rows come from the second source (window rows of the original KV)
        const __nv_bfloat16 *src = row < P.num_kv_rows ? P.kv + static_cast<int64_t>(row < 0 ? 0 : row) * P.D
                                                      : P.kv2 + static_cast<int64_t>(row - P.num_kv_rows) * P.D;
        const uint32_t nbytes = row < 0 ? 0u : 16u;
#pragma unroll
        for (int i = 0; i < C::NMAIN; ++i)
          cp_async_16(sb + i * (C::kBN * 128) + r * 128 + ((v ^ (r & 7)) << 4), src + main_dim0 + i * 64 + v * 8,
                      nbytes);
        if (C::TAIL && v < 4)
          cp_async_16(sb + C::kStageMain + r * 64 + ((v ^ ((r >> 1) & 3)) << 4), src + tail_dim0 + v * 8, nbytes);
      }
      }
      cp_async_commit();
      if (j + kGroups < nb) fetch(j + kGroups);
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(&kv_full[s]);
    }
    cp_async_wait<0>();
  } else {
    // ---------------- softmax: two warpgroups; thread = head row h = TMEM lane,
    // warpgroup w owns columns [32w, 32w + 32) of every 64-row block.
    // tcgen05.ld/st are warp-collective (.sync.aligned): every decision that
    // guards one is made warp-uniform, including the error path.
    const int h = tid & 127, w = tid >> 7;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, P.err, 27, -1));
    if (ok) {
      // Q main dims: staged rows (128B swizzle) -> TMEM as bf16 pairs, chunks split by warpgroup
      const uint8_t *qs = smem + C::kOffQStage;
#pragma unroll 1
      for (int i = w; i < C::NMAIN; i += 2) {
        uint32_t r[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = *reinterpret_cast<const uint4 *>(qs + i * 16384 + h * 128 + ((u ^ (h & 7)) << 4));
          r[4 * u + 0] = v.x;
          r[4 * u + 1] = v.y;
          r[4 * u + 2] = v.z;
          r[4 * u + 3] = v.w;
        }
        tmem_st32(lane_base + C::kQCol + 32 * i, r);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    warp_arrive(q_ready, lane);

    // partial-S tile rows: 64 fp16 (128 bytes), 16-byte unit u stored at u ^ (h & 7)
    uint8_t *recv0 = smem + C::kOffRecv;
    // stage our 32 columns of a partial S row (fp32 registers, log2 units),
    // rounded to fp16, for the exchange agent (SPLIT only).  Each CTA
    // softmaxes its own fp32 partial plus the peer's fp16 partial and
    // normalises its own O half with its own sum, so the two CTAs need not
    // agree bitwise.
    auto stage = [&](int j, const float (&v)[32]) {
      const int b = j & 1;
      uint8_t *row = smem + C::kOffStg + (j & 1) * C::kRecvBytes + h * 128;
#pragma unroll
      for (int k = 0; k < 32; k += 8) {
        const int u = (w * C::kHalf + k) >> 3;
        *reinterpret_cast<uint4 *>(row + ((u ^ (h & 7)) << 4)) =
            make_uint4(pack_f16x2_sat(v[k], v[k + 1]), pack_f16x2_sat(v[k + 2], v[k + 3]),
                       pack_f16x2_sat(v[k + 4], v[k + 5]), pack_f16x2_sat(v[k + 6], v[k + 7]));
      }
      fence_proxy_async_smem();  // the bulk copy reads the tile through the async proxy
      warp_arrive(&staged[b], lane);
    };
    // load our 32 columns of S(j) from TMEM once (raw q.k units: the softmax
    // scale is applied in the exponent); the buffer is then free for QK(j+2)
    const uint64_t sc2 = f2_pack(P.scale_log2, P.scale_log2);
    auto load_s = [&](int j, float (&v)[32]) {
      uint32_t r[32];
      tmem_ld32(lane_base + C::kSCol + (j & 1) * C::kBN + w * C::kHalf, r);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
      tc_fence_before();
      warp_arrive(&s_free[j & 1], lane);
    };

    float m_used = -__builtin_huge_valf(), l = 0.f;  // m in log2 units; l over this warpgroup's columns
    // S of block i in one register array and block i + 1 loaded into the other;
    // the loop takes two blocks per turn with the arrays' roles swapped, so no
    // copy of S between blocks
    float s_a[32], s_b[32];
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[0], 0, P.err, 27, 0));
      if (ok) {
        tc_fence_after();
        load_s(0, s_a);
        if (C::SPLIT) stage(0, s_a);
      }
    }
    auto block = [&](int i, float (&x)[32], float (&nxt)[32]) -> bool {
      const int b = i & 1;
      if (i + 1 < nb) {
        // fetch (and for the pair, ship) block i+1 ahead: the peer has it by the
        // time it starts block i+1
        const int b1 = (i + 1) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b1], ((i + 1) >> 1) & 1, P.err, 27, i + 1) &&
                                         (!C::SPLIT || i < 1 ||
                                          mbar_wait(&stg_free[(i + 1) & 1], ((i - 1) >> 1) & 1, P.err, 28, i + 1)));
        if (!ok) return false;
        tc_fence_after();
        load_s(i + 1, nxt);
        if (C::SPLIT) stage(i + 1, nxt);
      }
      if (C::SPLIT) {
        if (tid == 0) mbar_arrive_expect_tx(&recv_full[b], C::kRecvTx);
        ok = __all_sync(0xffffffffu, mbar_wait<true>(&recv_full[b], (i >> 1) & 1, P.err, 29, i));
        if (!ok) return false;
        const uint8_t *my_recv = recv0 + b * C::kRecvBytes + h * 128;
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          const int u = (w * C::kHalf + k) >> 3;
          const uint4 v = *reinterpret_cast<const uint4 *>(my_recv + ((u ^ (h & 7)) << 4));
          const uint32_t pv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float lo, hi;
            unpack_f16x2(pv[e], lo, hi);
            f2_unpack(f2_add(f2_pack(x[k + 2 * e], x[k + 2 * e + 1]), f2_pack(lo, hi)), x[k + 2 * e], x[k + 2 * e + 1]);
          }
        }
      }
      // row max over the whole block: this warpgroup's half, then the other's through smem
      const bool full = (i + 1) * C::kBN <= n_valid;
      if (!full) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (i * C::kBN + w * C::kHalf + k >= n_valid) x[k] = -__builtin_huge_valf();
      }
      float m3[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        m3[q] = fmax3(fmax3(x[8 * q], x[8 * q + 1], x[8 * q + 2]), fmax3(x[8 * q + 3], x[8 * q + 4], x[8 * q + 5]),
                      fmaxf(x[8 * q + 6], x[8 * q + 7]));
      red[(b * 2 + w) * 128 + h] = fmaxf(fmax3(m3[0], m3[1], m3[2]), m3[3]);
      warp_arrive(&red_full[b], lane);
      ok = __all_sync(0xffffffffu, mbar_wait(&red_full[b], (i >> 1) & 1, P.err, 33, i));
      if (!ok) return false;
      const float mblk = fmaxf(red[(b * 2) * 128 + h], red[(b * 2 + 1) * 128 + h]) * P.scale_log2;  // log2 units
      // lazy rescale: only when some row of the warp saw its max grow by more
      // than 2^8; rows whose max did not grow get alpha = 1 (exact).  Both
      // warpgroups see the same row maxima, so they decide alike.
      if (__any_sync(0xffffffffu, mblk > m_used + 8.f)) {
        const float m_new = fmaxf(m_used, mblk);
        const float alpha = ex2(m_used - m_new);
        if (i >= 1) {
          // O holds PV(i-1): rescale this warpgroup's half of it before PV(i) accumulates
          ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, P.err, 30, i));
          if (!ok) return false;
          tc_fence_after();
          scale_o_cols(lane_base, w * (C::kOCols / 2), (w + 1) * (C::kOCols / 2), alpha);
        }
        l *= alpha;
        m_used = m_new;
      }
      // the single CTA's P tile: wait until PV(i-1) has consumed it (the pair
      // writes P over the peer's tile of this block, which nothing else reads)
      if (!C::SPLIT && i >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, P.err, 32, i));
        if (!ok) return false;
      }
      uint32_t packed[16];
      const uint64_t nm2 = f2_pack(-m_used, -m_used);
      uint64_t acc[2] = {0, 0};  // +0.0f pairs
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        float t0, t1;
        f2_unpack(f2_fma(f2_pack(x[k], x[k + 1]), sc2, nm2), t0, t1);
        const float e0 = ex2(t0), e1 = ex2(t1);
        packed[k >> 1] = pack_bf16x2(e0, e1);
        // the denominator sums the fp32 exponentials (PV multiplies their bf16
        // roundings: the weights then sum to 1 within ~1e-5)
        acc[(k >> 1) & 1] = f2_add(acc[(k >> 1) & 1], f2_pack(e0, e1));
      }
      float s0, s1, s2, s3;
      f2_unpack(acc[0], s0, s1);
      f2_unpack(acc[1], s2, s3);
      l += (s0 + s1) + (s2 + s3);
      uint8_t *prow = smem + (C::SPLIT ? C::kOffRecv + b * C::kRecvBytes : C::kOffP) + h * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int uu = w * 4 + u;
        *reinterpret_cast<uint4 *>(prow + ((uu ^ (h & 7)) << 4)) =
            make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
      }
      fence_proxy_async_smem();
      warp_arrive(&p_full[b], lane);
      return true;
    };
    for (int i = 0; ok && i < nb; i += 2) {
      ok = block(i, s_a, s_b);
      if (ok && i + 1 < nb) ok = block(i + 1, s_b, s_a);
    }
    ok = __all_sync(0xffffffffu, ok && mbar_wait(&pv_done[(nb - 1) & 1], ((nb - 1) >> 1) & 1, P.err, 31, nb));
    // the two warpgroups' partial sums of the softmax denominator
    red[(4 + w) * 128 + h] = l;
    warp_arrive(fin_full, lane);
    ok = __all_sync(0xffffffffu, mbar_wait(fin_full, 0, P.err, 34) && ok);
    l = red[4 * 128 + h] + red[5 * 128 + h];
    if (ok) {
      tc_fence_after();
      if (P.sink && h < P.H) l += ex2(P.sink[h] * 1.4426950408889634f - m_used);
    }
    const float inv = 1.f / l;
    // destination of output row hh (this CTA's value columns)
    auto out_of = [&](int hh) -> __nv_bfloat16 * {
      if (P.hc > 0) {  // head-sharded: rank hh / hc, token g, head hh % hc
        const int rd = hh / P.hc;
        return P.out + ((static_cast<int64_t>(rd) * misc[4] + misc[3]) * P.hc + (hh - rd * P.hc)) * P.Dv +
               main_dim0;
      }
      return out_row + static_cast<int64_t>(hh) * P.Dv;
    };
    if constexpr (C::SPLIT) {
      // Normalised rows go through shared memory (stages 0-1, free once every
      // PV is done): thread h writes its row's 16-byte units, unit u of row h
      // at u ^ (h & 31) so that neither the row-wise writes nor the column-wise
      // reads below collide on banks; then each warp stores whole 512-byte rows
      // with one coalesced instruction per row.
      static_assert(C::DVC == 256, "one 512-byte row per CTA");
      uint8_t *ost = smem + C::kOffStage;
      if (ok) {
#pragma unroll 1
        for (int c = w * (C::kOCols / 2); c < (w + 1) * (C::kOCols / 2); c += 32) {
          uint32_t r[32];
          tmem_ld32(lane_base + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            const int u = (c + k) >> 3;
            *reinterpret_cast<uint4 *>(ost + h * 512 + ((u ^ (h & 31)) << 4)) =
                make_uint4(pack_bf16x2(__uint_as_float(r[k + 0]) * inv, __uint_as_float(r[k + 1]) * inv),
                           pack_bf16x2(__uint_as_float(r[k + 2]) * inv, __uint_as_float(r[k + 3]) * inv),
                           pack_bf16x2(__uint_as_float(r[k + 4]) * inv, __uint_as_float(r[k + 5]) * inv),
                           pack_bf16x2(__uint_as_float(r[k + 6]) * inv, __uint_as_float(r[k + 7]) * inv));
          }
        }
      }
      warp_arrive(o_staged, lane);
      ok = __all_sync(0xffffffffu, mbar_wait(o_staged, 0, P.err, 39) && ok);
      if (ok) {
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
          const int hh = warp + 8 * k;
          const uint4 v = *reinterpret_cast<const uint4 *>(ost + hh * 512 + ((lane ^ (hh & 31)) << 4));
          *reinterpret_cast<uint4 *>(out_of(hh) + lane * 8) = v;
        }
      }
    } else if (ok) {  // tiny shapes: rows stored directly
      __nv_bfloat16 *o = out_of(h);
#pragma unroll 1
      for (int c = w * (C::kOCols / 2); c < (w + 1) * (C::kOCols / 2); c += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + c, r);
        tmem_ld_wait();
        if (h < P.H) {
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            if (c + k < C::DVC) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(r[k + 0]) * inv, __uint_as_float(r[k + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(r[k + 2]) * inv, __uint_as_float(r[k + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(r[k + 4]) * inv, __uint_as_float(r[k + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(r[k + 6]) * inv, __uint_as_float(r[k + 7]) * inv);
              *reinterpret_cast<uint4 *>(o + c + k) = v;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (C::SPLIT) cluster_sync();  // no CTA leaves while its peer may still touch its smem
}

template <class C>
dsa_status launch_attn(const void *q, int32_t tpr, const AttnParams &P, cudaStream_t stream) {
  CUtensorMap qmain, qtail;
  uint64_t dims[3] = {static_cast<uint64_t>(P.D), static_cast<uint64_t>(P.H), static_cast<uint64_t>(P.q_rows)};
  uint64_t strides[2] = {static_cast<uint64_t>(P.D) * 2, static_cast<uint64_t>(P.H) * P.D * 2};
  uint32_t box_main[3] = {64, 128, 1};
  dsa_status st = encode_tensor_map(&qmain, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box_main,
                                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != DSA_OK) return st;
  if (C::TAIL) {
    uint32_t box_tail[3] = {32, 128, 1};
    st = encode_tensor_map(&qtail, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box_tail,
                           CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != DSA_OK) return st;
  } else {
    qtail = qmain;
  }
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tpr) * (C::SPLIT ? 2u : 1u));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::SPLIT ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, sparse_attn_kernel<C>, qmain, qtail, P);
  if (e != cudaSuccess) return cuda_fail(e);
  return check_launch();
}

}  // namespace
}  // namespace dsa

using namespace dsa;

// An extended index row (the sliding-window call): `counts` valid entries per
// row of `stride`, rows past num_kv_rows read from kv2.
struct ExtIndex {
  const void *kv2;
  int32_t num_rows2;
  const int32_t *counts;
  int32_t stride;
};

// The latent rows as the FP8 cache (E4M3 value columns, fp32 tile scales,
// bf16 rope columns per row).
struct Fp8Rows {
  int32_t row_bytes, rope;
};

static dsa_status sparse_attn_impl(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr, const void *q,
                                   const void *kv, int32_t num_kv_rows, const int32_t *topk_idx, int32_t topk,
                                   const float *attn_sink, float softmax_scale, int32_t H, int32_t D, int32_t Dv,
                                   int32_t cp_size, void *out, int32_t flat_tokens, dsa_stream_t stream,
                                   const ExtIndex *ext = nullptr, int32_t slot_begin = 0, int32_t slot_count = -1,
                                   int32_t q_row0 = 0, const Fp8Rows *fp8 = nullptr) {
  if (!md || !q || !kv || !topk_idx || !out) return DSA_ERR_INVALID_ARG;
  if (!md->scalars || !md->local_query_start_loc || !md->local_req_kv_base || !md->local_token_pos ||
      !md->local_req_pos_base)
    return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out) || !aligned16(topk_idx)) return DSA_ERR_INVALID_ARG;
  if (batch < 0 || tpr < 0 || num_kv_rows < 1 || topk < 1) return DSA_ERR_SHAPE;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return DSA_ERR_INVALID_ARG;
  if (cp_size < 0) return DSA_ERR_INVALID_ARG;
  if (cp_size > 0 && (H < 1 || H % cp_size != 0)) return DSA_ERR_SHAPE;
  if (flat_tokens < 0) return DSA_ERR_SHAPE;
  if (slot_count < 0) slot_count = tpr - slot_begin;
  if (slot_begin < 0 || slot_count < 0 || static_cast<int64_t>(slot_begin) + slot_count > tpr || q_row0 < 0)
    return DSA_ERR_SHAPE;
  if (ext) {
    if (!ext->counts || (ext->num_rows2 > 0 && (!ext->kv2 || !aligned16(ext->kv2)))) return DSA_ERR_INVALID_ARG;
    if (ext->num_rows2 < 0 || ext->stride < topk) return DSA_ERR_SHAPE;
    if (static_cast<int64_t>(num_kv_rows) + ext->num_rows2 > INT32_MAX) return DSA_ERR_SHAPE;
  }
  if (slot_count == 0) return DSA_OK;
  if (static_cast<int64_t>(slot_count) * 2 > INT32_MAX) return DSA_ERR_SHAPE;
  const bool big = H == 128 && D == 576 && Dv == 512 && topk == 2048;
  const bool tiny = H == 8 && D == 64 && Dv == 48 && topk == 64;
  if (!big && !tiny) return DSA_ERR_UNSUPPORTED;
  if (fp8 && (!big || ext)) return DSA_ERR_UNSUPPORTED;
  int *err = device_error_word();
  if (!err) return DSA_ERR_CUDA;
  AttnParams P{*md,
               fp8 ? nullptr : static_cast<const __nv_bfloat16 *>(kv),
               ext ? static_cast<const __nv_bfloat16 *>(ext->kv2) : nullptr,
               fp8 ? static_cast<const uint8_t *>(kv) : nullptr,
               fp8 ? fp8->row_bytes : 0,
               fp8 ? fp8->rope : 0,
               topk_idx,
               ext ? ext->counts : nullptr,
               attn_sink,
               static_cast<__nv_bfloat16 *>(out),
               static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634),
               topk,
               H,
               D,
               Dv,
               num_kv_rows,
               ext ? ext->stride : topk,
               ext ? ext->num_rows2 : 0,
               cp_size > 0 ? H / cp_size : 0,
               flat_tokens > 0 ? 1 : 0,
               flat_tokens > 0 ? flat_tokens : slot_count,
               slot_begin,
               flat_tokens > 0 ? q_row0 : 0,
               err};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fp8) return launch_attn<BigAttnFp8>(q, slot_count, P, s);
  return big ? launch_attn<BigAttn>(q, slot_count, P, s) : launch_attn<TinyAttn>(q, slot_count, P, s);
}

extern "C" dsa_status dsa_sparse_attn_prefill(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                              const void *q, const void *kv, int32_t num_kv_rows,
                                              const int32_t *topk_idx, int32_t topk, const float *attn_sink,
                                              float softmax_scale, int32_t H, int32_t D, int32_t Dv, void *out,
                                              dsa_stream_t stream) {
  return sparse_attn_impl(md, batch, tpr, q, kv, num_kv_rows, topk_idx, topk, attn_sink, softmax_scale, H, D, Dv, 0,
                          out, 0, stream);
}

extern "C" dsa_status dsa_sparse_attn_prefill_flat(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                                   const void *q, int32_t num_tokens, const void *kv,
                                                   int32_t num_kv_rows, const int32_t *topk_idx, int32_t topk,
                                                   const float *attn_sink, float softmax_scale, int32_t H, int32_t D,
                                                   int32_t Dv, void *out, dsa_stream_t stream) {
  if (num_tokens < 1) return num_tokens == 0 ? DSA_OK : DSA_ERR_SHAPE;
  return sparse_attn_impl(md, batch, tpr, q, kv, num_kv_rows, topk_idx, topk, attn_sink, softmax_scale, H, D, Dv, 0,
                          out, num_tokens, stream);
}

extern "C" dsa_status dsa_sparse_attn_prefill_headsharded(const dsa_cp_local_metadata *md, int32_t batch,
                                                          int32_t tpr, const void *q, const void *kv,
                                                          int32_t num_kv_rows, const int32_t *topk_idx, int32_t topk,
                                                          const float *attn_sink, float softmax_scale, int32_t H,
                                                          int32_t D, int32_t Dv, int32_t cp_size, void *out,
                                                          dsa_stream_t stream) {
  if (cp_size < 1) return DSA_ERR_INVALID_ARG;
  return sparse_attn_impl(md, batch, tpr, q, kv, num_kv_rows, topk_idx, topk, attn_sink, softmax_scale, H, D, Dv,
                          cp_size, out, 0, stream);
}

extern "C" dsa_status dsa_sparse_attn_prefill_swa(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                                  const void *q, const void *kv, int32_t num_kv_rows,
                                                  const void *kv_ori, int32_t num_ori_rows, const int32_t *ext_idx,
                                                  int32_t ext_stride, const int32_t *counts, int32_t topk,
                                                  const float *attn_sink, float softmax_scale, int32_t H, int32_t D,
                                                  int32_t Dv, void *out, dsa_stream_t stream) {
  const ExtIndex ext{kv_ori, kv_ori ? num_ori_rows : 0, counts, ext_stride};
  return sparse_attn_impl(md, batch, tpr, q, kv, num_kv_rows, ext_idx, topk, attn_sink, softmax_scale, H, D, Dv, 0,
                          out, 0, stream, &ext);
}

extern "C" dsa_status dsa_sparse_attn_prefill_rows(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                                   int32_t slot_begin, int32_t slot_count, const void *q_rows,
                                                   int32_t q_row0, int32_t num_q_rows, const void *kv,
                                                   int32_t num_kv_rows, const int32_t *topk_rows, int32_t topk,
                                                   const float *attn_sink, float softmax_scale, int32_t H, int32_t D,
                                                   int32_t Dv, void *out_rows, dsa_stream_t stream) {
  if (num_q_rows < 1 || slot_count < 0) return num_q_rows == 0 && slot_count == 0 ? DSA_OK : DSA_ERR_SHAPE;
  return sparse_attn_impl(md, batch, tpr, q_rows, kv, num_kv_rows, topk_rows, topk, attn_sink, softmax_scale, H, D,
                          Dv, 0, out_rows, num_q_rows, stream, nullptr, slot_begin, slot_count, q_row0);
}

extern "C" dsa_status dsa_sparse_attn_prefill_fp8kv(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                                    const void *q, int32_t num_tokens, const void *kv_cache,
                                                    int32_t num_kv_rows, const int32_t *topk_idx, int32_t topk,
                                                    const float *attn_sink, float softmax_scale, int32_t H, int32_t D,
                                                    int32_t Dv, void *out, dsa_stream_t stream) {
  if (num_tokens < 0 || D < 1 || Dv < 1 || Dv > D || Dv % 8 != 0 || (D - Dv) % 8 != 0) return DSA_ERR_SHAPE;
  // the cache row: Dv codes, one fp32 scale per 128 columns, the D - Dv rope columns as bf16, 16-byte padded
  const int32_t tiles = (Dv + 127) / 128;
  const Fp8Rows fp8{(Dv + 4 * tiles + 2 * (D - Dv) + 15) / 16 * 16, Dv + 4 * tiles};
  return sparse_attn_impl(md, batch, tpr, q, kv_cache, num_kv_rows, topk_idx, topk, attn_sink, softmax_scale, H, D,
                          Dv, 0, out, num_tokens, stream, nullptr, 0, -1, 0, &fp8);
}
