// Lightning indexer + causal top-k for one CP view.
//
// DeepSeek Sparse Attention (named in "feat: DeepSeek-V4 DSA context-parallel
// on NPU", section 背景): I[t,s] = sum_j w[t,j] * ReLU(q_I[t,j] . k_I[s]) for
// the view's local queries t against the full index keys s (same page,
// 单层前向数据流 (2)(3) and 4. Indexer full/local 分离), then the topk
// largest I[t,s] over s <= t with ties to the lower s.
//
// indexer_kernel (tcgen05, one CTA per 2 x (256/HI) local queries and a chunk
// of 2048, 4096 or 8192 keys chosen per launch): the key block (128 keys) is
// the MMA's M side, the query tile's (token, head) rows are N = 256, the
// indexer dim is K.  Each TMEM lane is
// then one key holding every head of a token in its own columns, so the
// weighted-ReLU head sum is a per-thread loop.  Two TMEM accumulators of
// 256 columns alternate between the two token groups so the epilogue of one
// overlaps the MMA of the other.  K tiles arrive by TMA (128B swizzle).
// Scores (fp32) go to a workspace row per query, indexed by in-request key
// position.  FP8 operands (IdxCfg<..., true>): E4M3 index rows with one fp32
// scale each, tcgen05.mma kind::f8f6f4; the query rows' scales fold into the
// head weights and each key's scale multiplies its head sums.
//
// topk_kernel (one CTA per query row): radix select of the topk-th largest
// score in three digits (11, 11, 10 bits of order-preserving uint32 keys, -0
// folded into +0), the last two over the short list of keys that share the
// threshold's first digit, then a block-scan compaction in ascending key
// order that takes every score above the threshold and the lowest-index ties.
#include <mutex>

#include "dsa_common.cuh"
#include "internal.h"

namespace dsa {
namespace {

template <int HI_, int DI_, bool FP8_ = false>
struct IdxCfg {
  static constexpr int HI = HI_, DI = DI_;
  // FP8: q_I and k_I are E4M3 rows with one fp32 scale each (the FP8 cache row
  // with D = Dv = DI: DI codes, the scale, zero bytes to a multiple of 16)
  static constexpr bool FP8 = FP8_;
  static constexpr int kEB = FP8 ? 1 : 2;                // bytes per element
  static constexpr int kRowBytes = FP8 ? (DI + 4 + 15) / 16 * 16 : DI * 2;  // global row stride
  static constexpr int kTokPerGroup = 256 / HI;          // tokens in one N = 256 MMA
  static constexpr int kTileTok = 2 * kTokPerGroup;      // two TMEM accumulators
  static constexpr int kRowsQ = kTileTok * HI;           // 512 B-operand rows
  static constexpr int kCW = DI * kEB >= 128 ? 128 / kEB : DI;  // elements per swizzle row
  static constexpr int kCWB = kCW * kEB;                 // 128 B (SW128) or 64 B (SW64)
  static constexpr int kNCh = DI / kCW;
  static constexpr uint32_t kLayout = kCWB == 128 ? kLayoutSW128 : kLayoutSW64;
  static constexpr uint32_t kSBO = 8 * kCWB;             // 8-row swizzle atom
  static constexpr int kBK = 128;                        // keys per block (M)
  static constexpr int kStages = FP8 || DI < 128 ? 4 : 2;
  static constexpr int kQBytes = kNCh * kRowsQ * kCWB;
  static constexpr int kKStageBytes = kNCh * kBK * kCWB;
  static constexpr int kKSteps = DI * kEB / 32;          // MMA K steps of 32 bytes (16 bf16 or 32 E4M3)
  static constexpr int kStepsPerChunk = kCWB / 32;
  static constexpr int kKeyChunk = 2048;                 // keys per CTA (smallest; see key_chunk)
  // epilogue: kEpiParts warps per TMEM lane quarter, each taking 256 / kEpiParts
  // columns (kTokPerPart tokens) of an accumulator
  static constexpr int kEpiParts = 4;
  static constexpr int kEpiWarps = 4 * kEpiParts;
  static constexpr int kColsPerPart = 256 / kEpiParts;
  static constexpr int kTokPerPart = kTokPerGroup / kEpiParts;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;   // warp 0 TMA, 1 MMA, 2.. epilogue
  static constexpr uint32_t kIdesc = FP8 ? idesc_e4m3(128, 256) : idesc_bf16(128, 256, false, false);
  // shared memory carve-up (offsets from a 1024-aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffW = kOffK + kStages * kKStageBytes;
  static constexpr int kOffSlot = kOffW + kTileTok * HI * 4;
  // key segments of the tile: one per local request with a slot to score
  // (base row, keys, first chunk index), kTileTok + 1 entries each
  static constexpr int kOffSeg = kOffSlot + kTileTok * 8;
  static constexpr int kOffBar = kOffSeg + (3 * (kTileTok + 1) * 4 + 7) / 8 * 8;
  static constexpr int kNumBars = 1 + 2 * kStages + 4 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 64 + 1024;  // + alignment slack
  // every CTA allocates all 512 TMEM columns: ask for enough smem to keep one CTA per SM
  static constexpr int kSmemBytes = kSmemUsed < 120 * 1024 ? 120 * 1024 : kSmemUsed;
  static_assert(HI * kTokPerGroup == 256, "HI must divide 256");
  static_assert(kTokPerGroup % kEpiParts == 0 && kTokPerPart * HI == kColsPerPart, "whole tokens per part");
  static_assert(kColsPerPart % 32 == 0, "32-column TMEM loads");
  static_assert(!FP8 || DI == 128, "FP8 rows: one 128-code scale tile");
};

struct IdxParams {
  dsa_cp_local_metadata md;
  const float *w;      // [tpr][HI]
  const uint8_t *q8;   // FP8 only: q_I rows [tpr * HI][kRowBytes] (their scales)
  const uint8_t *k8;   // FP8 only: k_I rows [num_kv_rows][kRowBytes]
  float *scores;       // [rows][ld]
  int64_t ld;          // score row stride (floats)
  int32_t tpr, row_begin, row_end, max_kv_len, num_kv_rows;
  int32_t op_slot0;    // the slot of operand row 0 (q_I, w; 0 when they hold every slot of the view)
  int32_t key_chunk;   // keys per chunk: a multiple of kKeyChunk, set at launch
  int32_t min_keys;    // slots that see at most this many keys are not scored (the top-k takes them all)
  int *err;
};

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const IdxParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *w_s = reinterpret_cast<float *>(smem + C::kOffW);
  int32_t *s_base = reinterpret_cast<int32_t *>(smem + C::kOffSlot);
  int32_t *s_p = s_base + C::kTileTok;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + C::kStages;
  uint64_t *t_full = k_empty + C::kStages;
  uint64_t *t_empty = t_full + 2;
  uint64_t *mma_done = t_empty + 2;
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);  // [0] tmem base, [1] segments, [2] chunks
  int32_t *seg_base = reinterpret_cast<int32_t *>(smem + C::kOffSeg);  // [kTileTok + 1]
  int32_t *seg_len = seg_base + (C::kTileTok + 1);
  int32_t *seg_chunk0 = seg_len + (C::kTileTok + 1);                  // first chunk index; [nseg] = total

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slot0 = P.row_begin + blockIdx.x * C::kTileTok;
  const int local_batch = P.md.scalars[DSA_MD_LOCAL_BATCH];
  const int ratio = max(1, P.md.scalars[DSA_MD_COMPRESS_RATIO]);  // compressed KV: tokens per entry

  // per-slot causal extent: key rows [base, base + last] (base = KV row of the
  // request's position 0 or first entry, last = the query's in-request
  // position, or its last visible entry (p + 1) / ratio - 1 for compressed KV;
  // -1: no key)
  for (int t = tid; t < C::kTileTok; t += C::kThreads) {
    const int slot = slot0 + t;
    int base = 0, p = -1;
    if (slot < P.row_end) {
      const int g = P.md.local_token_pos[slot];
      if (g >= 0 && local_batch > 0) {
        const int j = find_local_request(P.md.local_query_start_loc, local_batch, slot);
        base = P.md.local_req_kv_base[j];
        const int pos = g - P.md.local_req_pos_base[j];
        p = pos >= 0 ? (pos + 1) / ratio - 1 : -1;
        if (pos < 0 || p >= P.max_kv_len || base < 0 || base + p >= P.num_kv_rows) {
          record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 41, slot);
          p = -1;
        }
      }
    }
    s_base[t] = base;
    s_p[t] = p;
  }
  // head weights; with FP8 operands each carries its query row's scale
  // (ReLU(a * x) = a * ReLU(x) for a scale a > 0)
  for (int i = tid; i < C::kTileTok * C::HI; i += C::kThreads) {
    const int slot = slot0 + i / C::HI;
    float wv = 0.f;
    if (slot < P.row_end) {
      const int64_t r = static_cast<int64_t>(slot - P.op_slot0) * C::HI + (i % C::HI);
      wv = P.w[r];
      if constexpr (C::FP8) wv *= *reinterpret_cast<const float *>(P.q8 + r * C::kRowBytes + C::DI);
    }
    w_s[i] = wv;
  }
  __syncthreads();
  if (tid == 0) {
    // The tile's slots may belong to several local requests whose key rows lie
    // far apart (a head-tail view's head and tail chunks, a request with a long
    // prefix after a short one).  Each request with a slot to score is one
    // segment [base, base + most keys of its slots); slots of one request are
    // consecutive, so one pass builds the list.  The segments are cut into
    // chunks of key_chunk keys, numbered across segments.
    int nseg = 0;
    for (int t = 0; t < C::kTileTok; ++t) {
      const int keys = s_p[t] + 1;
      if (keys <= P.min_keys || keys <= 0) continue;
      if (nseg > 0 && seg_base[nseg - 1] == s_base[t]) {
        seg_len[nseg - 1] = max(seg_len[nseg - 1], keys);
      } else {
        seg_base[nseg] = s_base[t];
        seg_len[nseg] = keys;
        ++nseg;
      }
    }
    int chunks = 0;
    for (int sg = 0; sg < nseg; ++sg) {
      seg_chunk0[sg] = chunks;
      chunks += (seg_len[sg] + P.key_chunk - 1) / P.key_chunk;
    }
    seg_chunk0[nseg] = chunks;
    misc[1] = static_cast<uint32_t>(nseg);
    misc[2] = static_cast<uint32_t>(chunks);
    mbar_init(q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&t_full[b], 1);
      mbar_init(&t_empty[b], 32 * C::kEpiWarps);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int nseg = static_cast<int>(misc[1]), nchunks = static_cast<int>(misc[2]);
  // this CTA's chunks: blockIdx.y, blockIdx.y + gridDim.y, ...
  if (static_cast<int>(blockIdx.y) >= nchunks) return;  // nothing to score (before any TMEM is held)
  // key rows [kstart, kend) of chunk c
  auto chunk_range = [&](int c, int &kstart, int &kend) {
    int sg = 0;
    while (sg + 1 < nseg && seg_chunk0[sg + 1] <= c) ++sg;
    kstart = seg_base[sg] + (c - seg_chunk0[sg]) * P.key_chunk;
    kend = min(seg_base[sg] + seg_len[sg], kstart + P.key_chunk);
  };
  if (warp == 1) {
    tmem_alloc(&misc[0], 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // key blocks of this CTA, over all its chunks (the pipeline's block count)
  int nblk = 0;
  for (int c = blockIdx.y; c < nchunks; c += gridDim.y) {
    int ks, ke;
    chunk_range(c, ks, ke);
    nblk += (ke - ks + C::kBK - 1) / C::kBK;
  }
  // first key row of each block in turn: the blocks of chunk blockIdx.y, then
  // of chunk blockIdx.y + gridDim.y, ...
  struct BlockCursor {
    int c, ks, ke;
  };
  auto cursor_begin = [&](BlockCursor &cur) {
    cur.c = blockIdx.y;
    chunk_range(cur.c, cur.ks, cur.ke);
  };
  auto cursor_next = [&](BlockCursor &cur) {
    cur.ks += C::kBK;
    if (cur.ks >= cur.ke) {
      cur.c += gridDim.y;
      if (cur.c < nchunks) chunk_range(cur.c, cur.ks, cur.ke);
    }
  };

  {
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      mbar_arrive_expect_tx(q_full, C::kQBytes);
      for (int c = 0; c < C::kNCh; ++c)
        for (int h = 0; h < C::kRowsQ / 256; ++h)
          tma_load_2d(smem + C::kOffQ + (c * C::kRowsQ + h * 256) * C::kCWB, &qmap, c * C::kCW,
                      (slot0 - P.op_slot0) * C::HI + h * 256, q_full);
      int issued = 0;
      BlockCursor cur;
      cursor_begin(cur);
      for (int j = 0; j < nblk; ++j, cursor_next(cur)) {
        const int s = j % C::kStages;
        if (!mbar_wait(&k_empty[s], ((j / C::kStages) & 1) ^ 1, P.err, 11, j)) break;
        mbar_arrive_expect_tx(&k_full[s], C::kKStageBytes);
        uint8_t *dst = smem + C::kOffK + s * C::kKStageBytes;
        for (int c = 0; c < C::kNCh; ++c)
          tma_load_2d(dst + c * C::kBK * C::kCWB, &kmap, c * C::kCW, cur.ks, &k_full[s]);
        issued = j + 1;
      }
      // drain: every armed load has landed before the CTA can exit
      mbar_wait(q_full, 0, P.err, 12);
      for (int j = issued > C::kStages ? issued - C::kStages : 0; j < issued; ++j)
        mbar_wait(&k_full[j % C::kStages], (j / C::kStages) & 1, P.err, 13, j);
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer
      // descriptors built once, advanced by constant offsets (16-byte units)
      const uint64_t a0 = smem_desc(smem_u32(smem + C::kOffK), 16, C::kSBO, C::kLayout);
      const uint64_t b0 = smem_desc(smem_u32(smem + C::kOffQ), 16, C::kSBO, C::kLayout);
      bool ok = mbar_wait(q_full, 0, P.err, 14);
      for (int j = 0; ok && j < nblk; ++j) {
        const int s = j % C::kStages;
        if (!(ok = mbar_wait(&k_full[s], (j / C::kStages) & 1, P.err, 15, j))) break;
        tc_fence_after();
        for (int g = 0; g < 2; ++g) {
          if (!(ok = mbar_wait(&t_empty[g], (j & 1) ^ 1, P.err, 16, j))) break;
          tc_fence_after();
          const uint64_t as = desc_add(a0, static_cast<uint32_t>(s * C::kKStageBytes) >> 4);
          const uint64_t bg = desc_add(b0, static_cast<uint32_t>(g * 256 * C::kCWB) >> 4);
#pragma unroll
          for (int k = 0; k < C::kKSteps; ++k) {
            const int ch = k / C::kStepsPerChunk, sub = k % C::kStepsPerChunk;
            const uint64_t a = desc_add(as, (ch * C::kBK * C::kCWB + sub * 32) >> 4);
            const uint64_t b = desc_add(bg, (ch * C::kRowsQ * C::kCWB + sub * 32) >> 4);
            if constexpr (C::FP8) mma_ss_f8(tmem + g * 256, a, b, C::kIdesc, k > 0 ? 1u : 0u);
            else mma_ss(tmem + g * 256, a, b, C::kIdesc, k > 0 ? 1u : 0u);
          }
          mma_commit(&t_full[g]);
        }
        mma_commit(&k_empty[s]);
      }
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, P.err, 17);
    } else if (warp >= 2) {
      // ---------------- epilogue: one TMEM lane (= one key) per thread
      const int quad = warp & 3, part = (warp - 2) >> 2;
      const int row_in_blk = quad * 32 + lane;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      BlockCursor cur;
      cursor_begin(cur);
      for (int j = 0; j < nblk; ++j, cursor_next(cur)) {
        const int key = cur.ks + row_in_blk;
        // FP8: the key row's scale multiplies the whole head sum
        float kscale = 1.f;
        if constexpr (C::FP8)
          kscale = key < P.num_kv_rows ? *reinterpret_cast<const float *>(P.k8 + static_cast<int64_t>(key) * C::kRowBytes + C::DI)
                                       : 0.f;
        bool ok = true;
        for (int g = 0; g < 2; ++g) {
          // tcgen05.ld is warp-collective: keep the exit decision warp-uniform
          ok = __all_sync(0xffffffffu, mbar_wait(&t_full[g], j & 1, P.err, 18, j));
          if (!ok) break;
          tc_fence_after();
          // per token, even and odd heads accumulate in the two halves of a
          // packed fp32 pair (fma.rn.f32x2), summed at the end
          uint64_t acc2[C::kTokPerPart];
#pragma unroll
          for (int u = 0; u < C::kTokPerPart; ++u) acc2[u] = 0;  // +0.0f pairs
          const int tok0 = g * C::kTokPerGroup + part * C::kTokPerPart;
          // the weights of 4 consecutive columns per 16-byte shared-memory load (a broadcast)
          const float4 *wrow4 = reinterpret_cast<const float4 *>(w_s + tok0 * C::HI);
#pragma unroll
          for (int c4 = 0; c4 < C::kColsPerPart / 32; ++c4) {
            uint32_t r[32];
            tmem_ld32(lane_base + g * 256 + part * C::kColsPerPart + c4 * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const int col = c4 * 32 + c;
              const float4 wv = wrow4[col >> 2];
              acc2[col / C::HI] = f2_fma(f2_pack(fmaxf(__uint_as_float(r[c]), 0.f), fmaxf(__uint_as_float(r[c + 1]), 0.f)),
                                         f2_pack(wv.x, wv.y), acc2[col / C::HI]);
              acc2[col / C::HI] = f2_fma(f2_pack(fmaxf(__uint_as_float(r[c + 2]), 0.f), fmaxf(__uint_as_float(r[c + 3]), 0.f)),
                                         f2_pack(wv.z, wv.w), acc2[col / C::HI]);
            }
          }
          float acc[C::kTokPerPart];
#pragma unroll
          for (int u = 0; u < C::kTokPerPart; ++u) {
            float lo, hi;
            f2_unpack(acc2[u], lo, hi);
            acc[u] = lo + hi;
            if constexpr (C::FP8) acc[u] *= kscale;
          }
          tc_fence_before();
          mbar_arrive(&t_empty[g]);
#pragma unroll
          for (int u = 0; u < C::kTokPerPart; ++u) {
            const int t = tok0 + u;
            const int ks = key - s_base[t];
            if (ks >= 0 && ks <= s_p[t])
              P.scores[static_cast<int64_t>(slot0 - P.row_begin + t) * P.ld + ks] = acc[u];
          }
        }
        if (!ok) break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ top-k
constexpr int kTopkThreads = 512;

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t b = __float_as_uint(x == 0.f ? 0.f : x);  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive block scan of two counters (512 threads).
__device__ __forceinline__ void scan2(int a, int b, int &ea, int &eb, int &ta, int &tb, int2 *warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int xa = __shfl_up_sync(0xffffffffu, ia, off), xb = __shfl_up_sync(0xffffffffu, ib, off);
    if (lane >= off) {
      ia += xa;
      ib += xb;
    }
  }
  if (lane == 31) warp_tot[warp] = make_int2(ia, ib);
  __syncthreads();
  int pa = 0, pb = 0;
  ta = 0;
  tb = 0;
#pragma unroll
  for (int w = 0; w < kTopkThreads / 32; ++w) {
    const int2 v = warp_tot[w];
    if (w < warp) {
      pa += v.x;
      pb += v.y;
    }
    ta += v.x;
    tb += v.y;
  }
  __syncthreads();
  ea = pa + ia - a;
  eb = pb + ib - b;
}

// Exclusive prefix over the warp's lanes, and the warp total, of a per-lane
// count in [0, 7] (three ballots; the whole warp calls it).
__device__ __forceinline__ void warp_count_scan(int c, int lane, int &excl, int &total) {
  const unsigned lt = (1u << lane) - 1u;
  const unsigned b0 = __ballot_sync(0xffffffffu, c & 1), b1 = __ballot_sync(0xffffffffu, c & 2),
                 b2 = __ballot_sync(0xffffffffu, c & 4);
  excl = __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
  total = __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2);
}

// Radix select in three digits of the order key: bits 31..21 (2048 bins),
// 20..10 (2048) and 9..0 (1024).  The first digit is counted while the row
// is read; when the bin that holds the topk-th largest key has at most
// kCandMax keys, they are collected and the last two digits are counted over
// that short list only, otherwise over the whole row (keys whose higher
// digits match; a warp appends its candidates with one shared atomic).  Then
// one compaction pass in ascending key order takes every key above the
// threshold and the lowest-index keys equal to it (one block scan per chunk
// when every equal key is taken, the common case for float scores; two
// otherwise; 4096 keys per chunk).  The first cache_words keys of the row stay in
// shared memory after the first pass; the rest of a longer row is read again
// from global memory by the later passes.
constexpr int kBins = 2048;
constexpr int kCandMax = 4096;
constexpr int kTopkFixedWords = kBins + kCandMax;  // dynamic shared memory before the key cache

template <int TOPK>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const dsa_cp_local_metadata md, int32_t row_begin,
                                                            int32_t max_kv_len, const float *__restrict__ scores,
                                                            int64_t ld, int32_t *__restrict__ topk_idx,
                                                            int32_t out_slot0, int32_t cache_words, int *err) {
  extern __shared__ uint32_t dyn_smem[];
  uint32_t *hist = dyn_smem;               // [kBins]
  uint32_t *cand = dyn_smem + kBins;       // [kCandMax]
  uint32_t *s_keys = cand + kCandMax;      // [cache_words]
  __shared__ int2 warp_tot[kTopkThreads / 32];
  __shared__ int s_base, s_p, s_digit, s_krem, s_cnt, s_ncand;
  const int tid = threadIdx.x;
  const int slot = row_begin + blockIdx.x;
  int32_t *out = topk_idx + static_cast<int64_t>(slot - out_slot0) * TOPK;
  if (tid == 0) {
    int base = 0, p = -1;
    const int g = md.local_token_pos[slot];
    const int nb = md.scalars[DSA_MD_LOCAL_BATCH];
    if (g >= 0 && nb > 0) {
      const int j = find_local_request(md.local_query_start_loc, nb, slot);
      base = md.local_req_kv_base[j];
      const int pos = g - md.local_req_pos_base[j];
      const int ratio = max(1, md.scalars[DSA_MD_COMPRESS_RATIO]);
      p = pos >= 0 ? (pos + 1) / ratio - 1 : -1;  // last visible key / entry, -1: none
      if (pos < 0 || p >= max_kv_len) {
        record_error(err, DSA_ERR_DEVICE_BOUNDS, 42, slot);
        p = -1;
      }
    }
    s_base = base;
    s_p = p;
    s_ncand = 0;
  }
  for (int i = tid; i < kBins; i += kTopkThreads) hist[i] = 0;
  __syncthreads();
  const int base = s_base, n = s_p + 1;
  if (n <= TOPK) {  // pad slot or short row: every causal key, then -1
    for (int i = tid; i < TOPK; i += kTopkThreads) out[i] = i < n ? base + i : -1;
    return;
  }
  const float *row = scores + static_cast<int64_t>(blockIdx.x) * ld;
  // cached: a multiple of 4 (cache_words is), so a 4-key group is wholly
  // cached or wholly in global memory; rows start 16-byte aligned
  const int cached = min(n, cache_words) & ~3;
  // keys i .. i + 3 (i a multiple of 4); keys at or past n read as 0
  auto keys4_at = [&](int i, uint32_t (&k4)[4]) {
    if (i + 3 < cached) {
      const uint4 v = *reinterpret_cast<const uint4 *>(s_keys + i);
      k4[0] = v.x, k4[1] = v.y, k4[2] = v.z, k4[3] = v.w;
    } else if (i + 3 < n) {
      const float4 v = *reinterpret_cast<const float4 *>(row + i);
      k4[0] = order_key(v.x), k4[1] = order_key(v.y), k4[2] = order_key(v.z), k4[3] = order_key(v.w);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) k4[k] = i + k < n ? order_key(row[i + k]) : 0u;
    }
  };

  // pass 1: read the row, cache its first keys, count the first digit; each
  // thread has kLoads 16-byte loads in flight before it uses any
  constexpr int kLoads = 4;
  for (int i0 = tid * 4; i0 < n; i0 += kTopkThreads * 4 * kLoads) {
    float4 v[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int i = i0 + u * kTopkThreads * 4;
      if (i + 3 < n) v[u] = *reinterpret_cast<const float4 *>(row + i);
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int i = i0 + u * kTopkThreads * 4;
      if (i >= n) break;
      uint32_t k4[4];
      if (i + 3 < n) {
        k4[0] = order_key(v[u].x), k4[1] = order_key(v[u].y), k4[2] = order_key(v[u].z), k4[3] = order_key(v[u].w);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) k4[k] = i + k < n ? order_key(row[i + k]) : 0u;
      }
      if (i + 3 < cached) *reinterpret_cast<uint4 *>(s_keys + i) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (i + k < n) atomicAdd(&hist[k4[k] >> 21], 1u);
    }
  }
  __syncthreads();

  // the digit (of nbins, counted in hist) holding the krem-th largest key:
  // each thread sums nbins / 512 consecutive bins from the top, one block scan
  int krem = TOPK;
  auto find_digit = [&](int nbins) {
    const int per = nbins / kTopkThreads;
    int local = 0;
    for (int k = 0; k < per; ++k) local += static_cast<int>(hist[nbins - 1 - (tid * per + k)]);
    int cum, dummy, tot, tot2;
    scan2(local, 0, cum, dummy, tot, tot2, warp_tot);
    for (int k = 0; k < per; ++k) {
      const int c = static_cast<int>(hist[nbins - 1 - (tid * per + k)]);
      if (cum < krem && cum + c >= krem) {
        s_digit = nbins - 1 - (tid * per + k);
        s_krem = krem - cum;
        s_cnt = c;
      }
      cum += c;
    }
    __syncthreads();
    krem = s_krem;
  };
  find_digit(kBins);
  uint32_t prefix = static_cast<uint32_t>(s_digit) << 21, mask = 0xFFE00000u;
  const bool use_cand = s_cnt <= kCandMax;
  const int lane = tid & 31, warp = tid >> 5;
  if (use_cand) {  // pass 2: the keys of that bin (warp-uniform loop: the ballots need every lane)
    for (int i0 = warp * 128; i0 < n; i0 += kTopkThreads * 4) {
      const int i = i0 + lane * 4;
      uint32_t k4[4];
      keys4_at(i < n ? i : n, k4);
      bool m[4];
      int c = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        m[k] = i + k < n && (k4[k] & mask) == prefix;
        c += m[k];
      }
      int ex, tot;
      warp_count_scan(c, lane, ex, tot);
      int at = 0;
      if (lane == 0 && tot > 0) at = atomicAdd(&s_ncand, tot);
      at = __shfl_sync(0xffffffffu, at, 0) + ex;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (m[k]) cand[at++] = k4[k];
    }
  }
  // digits 2 and 3 over the candidates (or the whole row)
#pragma unroll
  for (int d = 0; d < 2; ++d) {
    const int shift = d == 0 ? 10 : 0, nbins = d == 0 ? 2048 : 1024;
    __syncthreads();  // candidates complete, previous digit read
    for (int i = tid; i < nbins; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    if (use_cand) {
      const int nc = s_ncand;
      for (int i = tid; i < nc; i += kTopkThreads) {
        const uint32_t key = cand[i];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (nbins - 1)], 1u);
      }
    } else {
      for (int i = tid * 4; i < n; i += kTopkThreads * 4) {
        uint32_t k4[4];
        keys4_at(i, k4);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (i + k < n && (k4[k] & mask) == prefix) atomicAdd(&hist[(k4[k] >> shift) & (nbins - 1)], 1u);
      }
    }
    __syncthreads();
    find_digit(nbins);
    prefix |= static_cast<uint32_t>(s_digit) << shift;
    mask |= static_cast<uint32_t>(nbins - 1) << shift;
  }
  // prefix is the threshold key; s_cnt keys equal it, krem of them are taken
  const uint32_t thr = prefix;
  const bool take_all_eq = s_cnt == krem;
  int run_sel = 0, run_eq = 0;
  constexpr int kPer = 8;  // keys per thread and chunk
  for (int t0 = 0; t0 < n; t0 += kTopkThreads * kPer) {
    const int i0 = t0 + tid * kPer;
    uint32_t keys[kPer];
    keys4_at(i0 < n ? i0 : n, *reinterpret_cast<uint32_t(*)[4]>(keys));  // past the end: all invalid below
    keys4_at(i0 + 4 < n ? i0 + 4 : n, *reinterpret_cast<uint32_t(*)[4]>(keys + 4));
    int sel[kPer], c_sel = 0;
    int e_sel, t_sel, e_dummy, t_dummy;
    if (take_all_eq) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        sel[k] = i0 + k < n && keys[k] >= thr;
        c_sel += sel[k];
      }
    } else {
      int c_eq = 0;
#pragma unroll
      for (int k = 0; k < kPer; ++k) c_eq += (i0 + k < n && keys[k] == thr);
      int e_eq, t_eq;
      scan2(c_eq, 0, e_eq, e_dummy, t_eq, t_dummy, warp_tot);
      int r_eq = run_eq + e_eq;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const bool valid = i0 + k < n;
        const bool eq = valid && keys[k] == thr;
        sel[k] = valid && (keys[k] > thr || (eq && r_eq < krem));
        r_eq += eq;
        c_sel += sel[k];
      }
      run_eq += t_eq;
    }
    scan2(c_sel, 0, e_sel, e_dummy, t_sel, t_dummy, warp_tot);
    int pos = run_sel + e_sel;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (sel[k]) {
        if (pos < TOPK) out[pos] = base + i0 + k;
        else record_error(err, DSA_ERR_DEVICE_BOUNDS, 43, slot);
        ++pos;
      }
    }
    run_sel += t_sel;
  }
}

__global__ void fill_kernel(float *p, int64_t n, float v) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    p[i] = v;
}

// ------------------------------------------------------------------ host side
template <class C>
dsa_status make_maps(const void *q_idx, const void *k_idx, int32_t tpr, int32_t num_kv_rows, CUtensorMap *qmap,
                     CUtensorMap *kmap) {
  const CUtensorMapSwizzle sw = C::kCWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUtensorMapDataType dt = C::FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // the rows' DI elements; the FP8 row's scale and padding lie beyond them in the stride
  uint64_t qdims[2] = {static_cast<uint64_t>(C::DI), static_cast<uint64_t>(tpr) * C::HI};
  uint64_t qstr[1] = {static_cast<uint64_t>(C::kRowBytes)};
  uint32_t qbox[2] = {static_cast<uint32_t>(C::kCW), 256};
  dsa_status st = encode_tensor_map(qmap, dt, 2, q_idx, qdims, qstr, qbox, sw);
  if (st != DSA_OK) return st;
  uint64_t kdims[2] = {static_cast<uint64_t>(C::DI), static_cast<uint64_t>(num_kv_rows)};
  uint32_t kbox[2] = {static_cast<uint32_t>(C::kCW), 128};
  return encode_tensor_map(kmap, dt, 2, k_idx, kdims, qstr, kbox, sw);
}

template <class C>
dsa_status launch_indexer(const CUtensorMap &qmap, const CUtensorMap &kmap, IdxParams P, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(indexer_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e);
  const int rows = P.row_end - P.row_begin;
  const int tiles = (rows + C::kTileTok - 1) / C::kTileTok;
  // Keys per CTA: the largest of 1, 2, 4 x kKeyChunk that still leaves about
  // eight waves of CTAs with work (about half of a causal grid has none).
  // Longer chunks spread each CTA's set-up (TMEM, barriers, its 8-query Q
  // tile) over more key blocks; fewer CTAs balance worse.  Measured: 7 %
  // less indexer + top-k time at 64K tokens per request, none lost at 8K.
  const int64_t waves8 = 8LL * num_sms();
  int chunk = C::kKeyChunk;
  while (chunk < 4 * C::kKeyChunk &&
         static_cast<int64_t>(tiles) * ((P.max_kv_len + 2 * chunk - 1) / (2 * chunk)) / 2 >= waves8)
    chunk *= 2;
  P.key_chunk = chunk;
  dim3 grid(tiles, (P.max_kv_len + chunk - 1) / chunk);
  indexer_kernel<C><<<grid, C::kThreads, C::kSmemBytes, stream>>>(qmap, kmap, P);
  return check_launch();
}

struct Args {
  const dsa_cp_local_metadata *md;
  int32_t batch, tpr, max_kv_len, num_kv_rows, HI, DI;
  const void *q_idx, *k_idx;
  const float *w;
  // the slots [slot0, slot0 + nslots) that q_idx, w and the top-k rows hold
  // (nslots < 0: every slot of the view, from slot 0)
  int32_t slot0 = 0, nslots = -1;
  int32_t count() const { return nslots < 0 ? tpr : nslots; }
};

dsa_status validate(const Args &a) {
  if (!a.md || !a.q_idx || !a.k_idx || !a.w) return DSA_ERR_INVALID_ARG;
  if (!a.md->scalars || !a.md->local_query_start_loc || !a.md->local_req_kv_base || !a.md->local_token_pos ||
      !a.md->local_req_pos_base)
    return DSA_ERR_INVALID_ARG;
  if (!aligned16(a.q_idx) || !aligned16(a.k_idx)) return DSA_ERR_INVALID_ARG;
  if (a.batch < 0 || a.tpr < 0 || a.max_kv_len < 1 || a.num_kv_rows < 1) return DSA_ERR_SHAPE;
  if (static_cast<int64_t>(a.tpr) * a.HI > INT32_MAX) return DSA_ERR_SHAPE;
  if (a.nslots >= 0 && (a.slot0 < 0 || static_cast<int64_t>(a.slot0) + a.nslots > a.tpr)) return DSA_ERR_SHAPE;
  return DSA_OK;
}

using BigIdx = IdxCfg<64, 128>;
using TinyIdx = IdxCfg<4, 32>;
using BigIdx8 = IdxCfg<64, 128, true>;

template <class C>
dsa_status run_scores(const Args &a, int32_t row_begin, int32_t row_end, float *out, int64_t ld,
                      cudaStream_t stream) {
  CUtensorMap qmap, kmap;
  dsa_status st = make_maps<C>(a.q_idx, a.k_idx, a.count(), a.num_kv_rows, &qmap, &kmap);
  if (st != DSA_OK) return st;
  int *err = device_error_word();
  if (!err) return DSA_ERR_CUDA;
  IdxParams P{*a.md, a.w, static_cast<const uint8_t *>(a.q_idx), static_cast<const uint8_t *>(a.k_idx), out, ld,
              a.tpr, row_begin, row_end, a.max_kv_len, a.num_kv_rows, a.slot0, C::kKeyChunk, 0, err};
  return launch_indexer<C>(qmap, kmap, P, stream);
}

// Dynamic shared memory of one top-k CTA at most: the histogram, the
// candidate list and up to 12,800 cached keys of the row, so that three CTAs
// (the most their registers allow) fit on an SM whatever the row length; a
// longer row reads its tail from global memory in the later passes.
// Measured: against a 22,016-key cache (two CTAs per SM on long rows) the
// indexer + top-k of a 16-request view takes 2.2 % less time, and against one
// CTA caching 45K keys two CTAs with the shorter cache had been 8 % faster.
constexpr int64_t kTopkSmemMax = 74 * 1024;

template <int TOPK>
dsa_status launch_topk(const dsa_cp_local_metadata &md, int32_t row_begin, int32_t rows, int32_t max_kv_len,
                       const float *scores, int64_t ld, int32_t *topk_idx, int32_t out_slot0, int *err,
                       cudaStream_t stream) {
  const int64_t cap = kTopkSmemMax / 4 - kTopkFixedWords;
  const int32_t cache_words = static_cast<int32_t>(ld < cap ? ld : cap);
  const int smem = (kTopkFixedWords + cache_words) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel<TOPK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  topk_kernel<TOPK><<<static_cast<unsigned>(rows), kTopkThreads, static_cast<size_t>(smem), stream>>>(
      md, row_begin, max_kv_len, scores, ld, topk_idx, out_slot0, cache_words, err);
  return check_launch();
}

template <class C, int TOPK>
dsa_status run_topk(const Args &a, int32_t *topk_idx, void *ws, size_t ws_bytes, cudaStream_t stream) {
  const int64_t ld = (static_cast<int64_t>(a.max_kv_len) + 3) / 4 * 4;
  int64_t rows_fit = static_cast<int64_t>(ws_bytes / (static_cast<size_t>(ld) * 4));
  rows_fit = rows_fit / C::kTileTok * C::kTileTok;
  if (rows_fit < C::kTileTok) return DSA_ERR_WORKSPACE;
  CUtensorMap qmap, kmap;
  dsa_status st = make_maps<C>(a.q_idx, a.k_idx, a.count(), a.num_kv_rows, &qmap, &kmap);
  if (st != DSA_OK) return st;
  int *err = device_error_word();
  if (!err) return DSA_ERR_CUDA;
  float *scores = static_cast<float *>(ws);
  const int64_t end = static_cast<int64_t>(a.slot0) + a.count();
  for (int64_t r0 = a.slot0; r0 < end; r0 += rows_fit) {
    const int32_t r1 = static_cast<int32_t>(r0 + rows_fit < end ? r0 + rows_fit : end);
    IdxParams P{*a.md, a.w, static_cast<const uint8_t *>(a.q_idx), static_cast<const uint8_t *>(a.k_idx), scores,
                ld, a.tpr, static_cast<int32_t>(r0), r1, a.max_kv_len, a.num_kv_rows, a.slot0, C::kKeyChunk, TOPK,
                err};
    st = launch_indexer<C>(qmap, kmap, P, stream);
    if (st != DSA_OK) return st;
    st = launch_topk<TOPK>(*a.md, static_cast<int32_t>(r0), r1 - static_cast<int32_t>(r0), a.max_kv_len, scores, ld,
                           topk_idx, a.slot0, err, stream);
    if (st != DSA_OK) return st;
  }
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_indexer_topk_workspace_size(int32_t tokens_per_rank, int32_t max_kv_len, int32_t topk,
                                                      size_t *bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARG;
  if (tokens_per_rank < 0 || max_kv_len < 1 || topk < 1) return DSA_ERR_SHAPE;
  const size_t row = static_cast<size_t>((static_cast<int64_t>(max_kv_len) + 3) / 4 * 4) * 4;
  const size_t tile = topk <= 64 ? TinyIdx::kTileTok : BigIdx::kTileTok;
  size_t rows = (static_cast<size_t>(tokens_per_rank) + tile - 1) / tile * tile;
  const size_t cap = (size_t(1) << 30) / row / tile * tile;
  if (rows > cap) rows = cap;
  if (rows < tile) rows = tile;
  *bytes = rows * row;
  return DSA_OK;
}

namespace dsa {
namespace {

// The bf16 and FP8 entry points share validation and dispatch.
dsa_status indexer_topk_entry(bool fp8, const Args &a, int32_t topk, int32_t *topk_idx, void *workspace,
                              size_t ws_bytes, cudaStream_t s) {
  dsa_status st = validate(a);
  if (st != DSA_OK) return st;
  if (!topk_idx || !workspace || !aligned16(workspace)) return DSA_ERR_INVALID_ARG;
  if (a.count() == 0) return DSA_OK;
  const bool big = a.HI == 64 && a.DI == 128 && topk == 2048, tiny = a.HI == 4 && a.DI == 32 && topk == 64;
  if (fp8) return big ? run_topk<BigIdx8, 2048>(a, topk_idx, workspace, ws_bytes, s) : DSA_ERR_UNSUPPORTED;
  if (big) return run_topk<BigIdx, 2048>(a, topk_idx, workspace, ws_bytes, s);
  if (tiny) return run_topk<TinyIdx, 64>(a, topk_idx, workspace, ws_bytes, s);
  return DSA_ERR_UNSUPPORTED;
}

dsa_status indexer_scores_entry(bool fp8, const Args &a, int32_t row_begin, int32_t row_count, float *scores,
                                cudaStream_t s) {
  dsa_status st = validate(a);
  if (st != DSA_OK) return st;
  if (!scores) return DSA_ERR_INVALID_ARG;
  if (row_begin < 0 || row_count < 0 || static_cast<int64_t>(row_begin) + row_count > a.tpr) return DSA_ERR_SHAPE;
  if (row_count == 0) return DSA_OK;
  const bool big = a.HI == 64 && a.DI == 128, tiny = a.HI == 4 && a.DI == 32;
  if (fp8 ? !big : !(big || tiny)) return DSA_ERR_UNSUPPORTED;
  const int64_t n = static_cast<int64_t>(row_count) * a.max_kv_len;
  fill_kernel<<<static_cast<unsigned>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, s>>>(
      scores, n, -__builtin_huge_valf());
  st = check_launch();
  if (st != DSA_OK) return st;
  const int32_t row_end = row_begin + row_count;
  if (fp8) return run_scores<BigIdx8>(a, row_begin, row_end, scores, a.max_kv_len, s);
  return big ? run_scores<BigIdx>(a, row_begin, row_end, scores, a.max_kv_len, s)
             : run_scores<TinyIdx>(a, row_begin, row_end, scores, a.max_kv_len, s);
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_indexer_topk(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                       int32_t max_kv_len, const void *q_idx, const void *k_idx, const float *w,
                                       int32_t num_kv_rows, int32_t HI, int32_t DI, int32_t topk,
                                       int32_t *topk_idx, void *workspace, size_t ws_bytes,
                                       dsa_stream_t stream) {
  Args a{md, batch, tpr, max_kv_len, num_kv_rows, HI, DI, q_idx, k_idx, w};
  return indexer_topk_entry(false, a, topk, topk_idx, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_indexer_topk_rows(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                            int32_t max_kv_len, int32_t slot_begin, int32_t slot_count,
                                            const void *q_idx_rows, const void *k_idx, const float *w_rows,
                                            int32_t num_kv_rows, int32_t HI, int32_t DI, int32_t topk,
                                            int32_t *topk_rows, void *workspace, size_t ws_bytes,
                                            dsa_stream_t stream) {
  Args a{md, batch, tpr, max_kv_len, num_kv_rows, HI, DI, q_idx_rows, k_idx, w_rows, slot_begin, slot_count};
  if (slot_count < 0) return DSA_ERR_SHAPE;
  return indexer_topk_entry(false, a, topk, topk_rows, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_indexer_topk_fp8(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                           int32_t max_kv_len, const void *q_idx8, const void *k_idx8,
                                           const float *w, int32_t num_kv_rows, int32_t HI, int32_t DI,
                                           int32_t topk, int32_t *topk_idx, void *workspace, size_t ws_bytes,
                                           dsa_stream_t stream) {
  Args a{md, batch, tpr, max_kv_len, num_kv_rows, HI, DI, q_idx8, k_idx8, w};
  return indexer_topk_entry(true, a, topk, topk_idx, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_indexer_scores(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                         int32_t max_kv_len, const void *q_idx, const void *k_idx, const float *w,
                                         int32_t num_kv_rows, int32_t HI, int32_t DI, int32_t row_begin,
                                         int32_t row_count, float *scores, dsa_stream_t stream) {
  Args a{md, batch, tpr, max_kv_len, num_kv_rows, HI, DI, q_idx, k_idx, w};
  return indexer_scores_entry(false, a, row_begin, row_count, scores, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_indexer_scores_fp8(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                             int32_t max_kv_len, const void *q_idx8, const void *k_idx8,
                                             const float *w, int32_t num_kv_rows, int32_t HI, int32_t DI,
                                             int32_t row_begin, int32_t row_count, float *scores,
                                             dsa_stream_t stream) {
  Args a{md, batch, tpr, max_kv_len, num_kv_rows, HI, DI, q_idx8, k_idx8, w};
  return indexer_scores_entry(true, a, row_begin, row_count, scores, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ no-allocation variant
// Some callers cannot allocate device memory at the point where they run the
// indexer: code inside a custom allocator or memory-pool callback, a runtime
// that has already handed all its memory to a pool, or a framework hook that
// must not call cudaMalloc.  For them dsa_indexer_topk_noalloc takes its score
// workspace from this fixed array instead of a caller buffer.  The array is
// part of the library image: every GPU that loads the library holds these
// 32 MiB until the process exits.
namespace dsa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
static void *s_scratch_ptr[kMaxScratchDevices];
static std::mutex s_scratch_mutex;

// Device address of g_static_scratch on the current device.  In host code the
// symbol's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached; no memory is allocated.
dsa_status static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxScratchDevices) return cuda_fail_msg("device index beyond the scratch table");
  std::lock_guard<std::mutex> lock(s_scratch_mutex);
  if (!s_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    s_scratch_ptr[dev] = p;
  }
  *out = s_scratch_ptr[dev];
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_indexer_topk_noalloc(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                               int32_t max_kv_len, const void *q_idx, const void *k_idx,
                                               const float *w, int32_t num_kv_rows, int32_t HI, int32_t DI,
                                               int32_t topk, int32_t *topk_idx, dsa_stream_t stream) {
  Args a{md, batch, tpr, max_kv_len, num_kv_rows, HI, DI, q_idx, k_idx, w};
  dsa_status st = validate(a);
  if (st != DSA_OK) return st;
  if (!topk_idx) return DSA_ERR_INVALID_ARG;
  const bool big = HI == 64 && DI == 128 && topk == 2048, tiny = HI == 4 && DI == 32 && topk == 64;
  if (!big && !tiny) return DSA_ERR_UNSUPPORTED;
  // the fixed array must hold the scores of at least one query tile
  const size_t row_bytes = static_cast<size_t>((static_cast<int64_t>(max_kv_len) + 3) / 4 * 4) * 4;
  const size_t tile = big ? BigIdx::kTileTok : TinyIdx::kTileTok;
  if (row_bytes * tile > kStaticScratchBytes) return DSA_ERR_WORKSPACE;
  if (tpr == 0) return DSA_OK;
  void *scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return big ? run_topk<BigIdx, 2048>(a, topk_idx, scratch, kStaticScratchBytes, s)
             : run_topk<TinyIdx, 64>(a, topk_idx, scratch, kStaticScratchBytes, s);
}
