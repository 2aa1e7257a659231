// Paged decode / verify attention for a ragged continuous batch (sm_103a).
//
// What it computes ("Continuous Batching and Speculative Decoding: How Modern LLM
// Serving Engines Actually Work", sections "PagedAttention: making the KV cache
// schedulable" and "The core idea"; "llm-inference-optimization-batching", section
// "Anatomy of the KV Cache"): for every query row, softmax attention over the
// sequence's KV positions 0..pos, read through the block table, pos = L - ql + j.
//
// How (split-KV, flash-decoding style; the pages give no kernel design):
//   1. plan_kernel      one CTA: validates lengths, packs query rows, chooses a split
//                       length in pages, writes the work list (sequence, page range,
//                       split, row block), zeroes the split counters and NaN-fills the
//                       rows of sequences with inconsistent lengths.
//   2. attn_bf16_kernel persistent, one CTA per SM, launched as a programmatic
//                       dependent of the plan.  A producer warp takes work units (work
//                       item x KV head) from an atomic counter and streams the unit's
//                       K/V pages into an 8-slot ring of 32-token stages with TMA (one
//                       box per page and operand, landing as [half][token][64] with the
//                       128-byte swizzle), tracked by mbarriers; it prefetches the next
//                       unit's descriptor and block-table entries while streaming.
//                       Four consumer warps compute:
//                         narrow units (<= 16 query rows per KV head: decode, small
//                         verify groups) on warp MMA (mma.sync m16n8k16, bf16 -> fp32),
//                         as S^T = K Q^T with the KV tokens as the 16-row M side and the
//                         GQA rows as N, so 8 rows fill an n8 tile; P^T reaches the PV
//                         operand through movmatrix.  Each warp owns whole stages (round
//                         robin) and keeps its own online softmax; the four are merged
//                         at the end of the unit.
//                         wide units (17..64 rows): S = Q K^T with the rows as M on warp
//                         MMA, two stages per step, softmax in registers, P as bf16 into
//                         a shared tile; an MMA warp accumulates O += P V with tcgen05
//                         (O in tensor memory, V read from the stage as the MN-major
//                         operand), rescaled in place when a row's maximum moves.
//                       A unit covering its whole sequence writes out/lse; otherwise it
//                       writes a normalised fp32 partial and its lse, and the last split
//                       to finish (atomic counter, no waiting) merges them by lse:
//                       O = sum_s e^{lse_s - m} O_s / sum_s e^{lse_s - m},
//                       lse = m + ln sum_s e^{lse_s - m}.
//      attn_f32_kernel  fp32 storage: CUDA-core FMA, one warp per query row, no split.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "../../include/vas.h"
#include "device_util.cuh"
#include "vas_internal.h"

namespace vas {
namespace attn {

constexpr int kStageTokens = 32;   // KV tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;      // TMA loads
constexpr int kMmaWarp = kConsumerWarps + 1;       // tcgen05 issue for wide units
constexpr int kThreads = kConsumerThreads + 64;    // + producer warp + MMA warp
// Quantised KV pages (FP8 E4M3 or INT8 codes with fp32 scales per token and KV head):
// the producer lands a stage's codes in the upper half of its 16-bit slot and its
// scales beside the ring; a converter warp expands the codes in place into f16 in the
// bf16 stage layout and marks the stage ready.  Every product of such a call runs in
// f16 (codes exact; Q scaled into f16 range by a power of two per unit; P in f16, whose
// 11 bits make the two-part P of precise row blocks unnecessary).
constexpr int kKvBf16 = 0, kKvFp8 = 1, kKvInt8 = 2;
constexpr int kConvWarps = 2;
constexpr int kConvWarp0 = kMmaWarp + 1;
constexpr int kThreadsQ = kThreads + 32 * kConvWarps;
constexpr int kTmemCols = 256;
constexpr int kTmemS = 0;    // S of a prompt-chunk stage, two 32-column buffers
constexpr int kTmemO = 64;   // O: 128 lanes x D fp32
constexpr int kRowBlock = 64;      // query rows per unit (four m16 tiles) ...
constexpr int kRowBlockTc = 128;   // ... or, for sequences with more rows (prompt chunks),
                                   // 128: S and PV on tcgen05 with the rows in TMEM lanes
// Rows per unit of a sequence with R query rows (G x query length).
__host__ __device__ __forceinline__ int row_block(int R) {
  return R > kRowBlock ? kRowBlockTc : kRowBlock;
}
constexpr int kNarrowRows = 16;    // units with at most this many rows take the K Q^T form
constexpr int kRing = 4;           // unit descriptors the producer may run ahead
constexpr int kRbBits = 12;        // row-block index bits in Item::split_rb
constexpr int kUnitsPerSm = 16;    // work-list room per SM in the recommended workspace
constexpr int kSplitTargetPerSm = 4;  // split target: work units per SM (the longest-first
                                      // order keeps the tail short with units this long)
// Row blocks in which some row sees fewer KV positions than this are "precise": with
// few tokens each softmax weight is large, and one bf16 rounding of P (relative 2^-8)
// would show in the output at the 1e-2 level.  The plan marks their items with
// kItemPrecise in Item::split_rb; they run on the tcgen05 row-block path (whatever their
// row count) with P in two bf16 parts, hi + lo, about 16 bits.  Such row blocks span at
// most 64 + 128 positions (7 stages), so the extra product is cheap.
constexpr int kPreciseTokens = 64;
constexpr int32_t kItemPrecise = 1 << 30;
constexpr int kPlanThreads = 256;
constexpr int kOrderBuckets = 64;  // page-count classes of the work order
constexpr int kWideOrderWeight = 2;  // a wide unit's page counts twice in the work order
constexpr int kPlanSmemSeqs = 4096;
constexpr int kSeqInvalid = 1;

struct SeqPlan {
  int32_t qrow0;         // first row of q / out / lse
  int32_t nsplit;        // KV splits; 0 = nothing to compute (invalid or no query)
  int32_t partial_base;  // first partial row (nsplit > 1)
  int32_t len;           // L
  int32_t qlen;          // ql
  int32_t flags;         // kSeqInvalid
  int32_t nrb;           // row blocks
  int32_t item0;         // first work item (split 0, row block 0)
};

struct Item {
  int32_t seq, page_begin, page_end, split_rb;  // split << kRbBits | row block (| kItemPrecise)
};

struct PlanHeader {
  int32_t n_items;
  int32_t work_counter;
  int32_t chunk_pages;
  int32_t n_partial_rows;
};

// What the producer hands the consumers for one unit (u < 0: no more work).
struct RingEntry {
  int32_t u, head;
  Item item;
  SeqPlan sp;
  int32_t pad[2];
};

struct Layout {
  size_t seqplan, token_seq, items, order, counters, part_lse, part_o, total;
  int64_t items_cap, partial_cap;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------------------------
// Plan
// ------------------------------------------------------------------------------------
struct PlanArgs {
  const int32_t* seq_lens;
  const int32_t* query_lens;
  SeqPlan* seqplan;
  int32_t* token_seq;
  Item* items;
  int32_t* order;  // work order: item indices, longest first
  PlanHeader* header;
  int32_t* counters;
  void* out;
  float* lse;
  int32_t B, T, G, Hkv, Hq, D, P, maxp, pps, min_chunk, no_split, target_units, is_bf16;
  const uint64_t* tree_mask;  // draft-tree masks, or null
  int64_t items_cap, partial_cap;
  int32_t* err;
};

struct SeqShape {
  bool valid;
  int32_t L, ql, npages, R, nrb;
};

__device__ __forceinline__ SeqShape seq_shape(const PlanArgs& a, int32_t L, int32_t ql) {
  SeqShape s;
  s.L = L;
  s.ql = ql;
  s.valid = ql >= 0 && ql <= a.T && L >= ql && (int64_t)L <= (int64_t)a.maxp * a.P;
  s.npages = s.valid ? (L + a.P - 1) / a.P : 0;
  s.R = s.valid ? a.G * ql : 0;
  s.nrb = (s.R + row_block(s.R) - 1) / row_block(s.R);
  return s;
}

__device__ __forceinline__ int32_t splits_for(const SeqShape& s, int64_t chunk) {
  if (s.R == 0 || s.npages == 0) return 0;
  return (int32_t)((s.npages + chunk - 1) / chunk);
}

// A sequence's split length: the call's c, at least twice the minimum for sequences
// whose units take the narrow path (at most kNarrowRows rows per KV head).  A narrow
// unit's fixed costs (query staging, the merge of its warps, the split's partial) weigh
// more against its short per-stage time than a wide unit's do.
__device__ __forceinline__ int64_t seq_chunk(const PlanArgs& a, const SeqShape& s, int64_t c) {
  return s.R <= kNarrowRows && c < 2 * (int64_t)a.min_chunk ? 2 * (int64_t)a.min_chunk : c;
}

// Block-wide sums of N counters at once.
template <int N>
__device__ __forceinline__ void block_sum(int64_t (&v)[N], int64_t (*red)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1)
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < N; ++k) red[warp][k] = v[k];
  __syncthreads();
  const int nw = (int)(blockDim.x >> 5);
  if (warp == 0) {  // one warp combines the per-warp partials, the block reads the result
    int64_t pv[N];
#pragma unroll
    for (int k = 0; k < N; ++k) pv[k] = lane < nw ? red[lane][k] : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
      for (int k = 0; k < N; ++k) pv[k] += __shfl_xor_sync(0xffffffffu, pv[k], o);
    if (lane == 0)
#pragma unroll
      for (int k = 0; k < N; ++k) red[32][k] = pv[k];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) v[k] = red[32][k];
}

// Exclusive scans of N counters at once (threads in order); totals returned in t.
template <int N>
__device__ __forceinline__ void block_scan(int64_t (&v)[N], int64_t (*red)[4], int64_t (&t)[N]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t inc[N];
#pragma unroll
  for (int k = 0; k < N; ++k) inc[k] = v[k];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int64_t n = __shfl_up_sync(0xffffffffu, inc[k], o);
      if (lane >= o) inc[k] += n;
    }
  __syncthreads();
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < N; ++k) red[warp][k] = inc[k];
  __syncthreads();
  int64_t base[N];
#pragma unroll
  for (int k = 0; k < N; ++k) base[k] = t[k] = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
#pragma unroll
    for (int k = 0; k < N; ++k) {
      if (w < warp) base[k] += red[w][k];
      t[k] += red[w][k];
    }
#pragma unroll
  for (int k = 0; k < N; ++k) v[k] = base[k] + inc[k] - v[k];
  __syncthreads();
}

// Whether row block rb of a sequence (query rows from qrow0) is precise: some row of it
// sees fewer than kPreciseTokens positions.  A row of token j sees the context and, in
// the causal window, tokens 0..j; in a draft tree its ancestors (mask bits below j) and
// itself.  So a chain tree is classified exactly as the causal window.
__device__ __forceinline__ bool rb_precise(const PlanArgs& a, const SeqShape& s, int64_t qrow0,
                                           int rb) {
  const int ctx = s.L - s.ql;
  const int RB = row_block(s.R);
  const int j0 = rb * RB / a.G;
  if (a.tree_mask && s.ql > 1 && s.ql <= 64) {
    const int j1 = min((rb + 1) * RB, s.R) - 1;
    for (int j = j0; j <= j1 / a.G; ++j) {
      const uint64_t below = j ? a.tree_mask[qrow0 + j] & (~0ull >> (64 - j)) : 0ull;
      if (ctx + __popcll(below) + 1 < kPreciseTokens) return true;
    }
    return false;
  }
  return ctx + j0 + 1 < kPreciseTokens;
}


__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanArgs a) {
  pdl_wait_prior_grid();    // the previous kernel in the stream has released the workspace
  pdl_launch_dependents();  // the attention grid may start its prologue
  __shared__ int32_t s_L[kPlanSmemSeqs], s_ql[kPlanSmemSeqs];
  __shared__ int64_t red[33][4];  // per-warp partials + the combined value
  const int tid = threadIdx.x;
  const bool cached = a.B <= kPlanSmemSeqs;
  if (cached)
    for (int i = tid; i < a.B; i += kPlanThreads) {
      s_L[i] = a.seq_lens[i];
      s_ql[i] = a.query_lens[i];
    }
  __syncthreads();
  auto shape = [&](int i) {
    return cached ? seq_shape(a, s_L[i], s_ql[i]) : seq_shape(a, a.seq_lens[i], a.query_lens[i]);
  };

  // Totals: work in page-row-blocks per KV head, packed query rows, invalid sequences.
  int64_t tot[3] = {0, 0, 0};  // cost, rows, bad
  for (int i = tid; i < a.B; i += kPlanThreads) {
    const SeqShape s = shape(i);
    tot[2] += !s.valid;
    tot[0] += (int64_t)s.npages * s.nrb;
    tot[1] += s.ql > 0 ? s.ql : 0;
  }
  block_sum<3>(tot, red);
  const int64_t cost = tot[0], rows = tot[1], bad = tot[2];
  const bool lengths_ok = rows == a.T && bad == 0;
  if (tid == 0 && !lengths_ok) atomicOr(a.err, VAS_DEV_BAD_LENGTHS);

  // Split length: about kSplitTargetPerSm units per SM, at least min_chunk pages, a whole
  // number of stages; doubled until the work list and the partials fit the workspace.
  int64_t c;
  if (a.no_split) {
    c = INT_MAX;
  } else {
    const int64_t want = (cost * a.Hkv + a.target_units - 1) / a.target_units;
    c = want > a.min_chunk ? want : a.min_chunk;
    c = (c + a.pps - 1) / a.pps * a.pps;
  }
  for (int iter = 0; iter < 40; ++iter) {
    int64_t v[2] = {0, 0};  // items, partial rows
    for (int i = tid; i < a.B; i += kPlanThreads) {
      const SeqShape s = shape(i);
      const int32_t ns = splits_for(s, seq_chunk(a, s, c));
      v[0] += (int64_t)ns * s.nrb;
      if (ns > 1) v[1] += (int64_t)ns * a.Hkv * s.R;
    }
    block_sum<2>(v, red);
    if ((v[0] <= a.items_cap && v[1] <= a.partial_cap) || c >= INT_MAX / 2) break;
    c = c * 2 < INT_MAX ? c * 2 : INT_MAX;
  }
  if (!lengths_ok)  // the row -> sequence map is only needed to find rows to NaN-fill
    for (int r = tid; r < a.T; r += kPlanThreads) a.token_seq[r] = -1;
  __syncthreads();

  // Scans in batch order, kPlanThreads sequences at a time.  A sequence's items are
  // (split, row block) pairs, split-major, from item0 on; its merge counters sit there
  // too.
  int64_t carry[3] = {0, 0, 0};  // rows, items, partial rows
  for (int base = 0; base < a.B; base += kPlanThreads) {
    const int i = base + tid;
    SeqShape s;
    s.valid = false;
    s.L = s.ql = s.npages = s.R = s.nrb = 0;
    int32_t ns = 0, qrows = 0;
    if (i < a.B) {
      s = shape(i);
      qrows = s.ql > 0 ? s.ql : 0;
      ns = splits_for(s, seq_chunk(a, s, c));
    }
    int64_t v[3] = {qrows, (int64_t)ns * s.nrb, ns > 1 ? (int64_t)ns * a.Hkv * s.R : 0};
    int64_t t[3];
    block_scan<3>(v, red, t);
    const int64_t my_row0 = v[0] + carry[0];
    const int64_t my_item0 = v[1] + carry[1];
    const int64_t my_part0 = v[2] + carry[2];
    if (i < a.B) {
      SeqPlan sp;
      sp.qrow0 = (int32_t)my_row0;
      sp.len = s.L;
      sp.qlen = s.ql;
      sp.flags = s.valid ? 0 : kSeqInvalid;
      // Rows that do not fit in T cannot be written, and a work list that would
      // overflow its workspace slot cannot be stored (both only when the lengths are
      // inconsistent): skip the sequence.
      const int64_t n_my_items = (int64_t)ns * s.nrb;
      const bool fits = my_row0 + qrows <= a.T && my_item0 + n_my_items <= a.items_cap;
      if (!fits) sp.flags |= kSeqInvalid;
      sp.nsplit = (s.valid && fits) ? ns : 0;
      sp.nrb = s.nrb;
      sp.partial_base = (int32_t)my_part0;
      sp.item0 = (int32_t)(my_item0 < a.items_cap ? my_item0 : 0);
      a.seqplan[i] = sp;
      if (!lengths_ok)
        for (int j = 0; j < qrows && my_row0 + j < a.T; ++j) a.token_seq[my_row0 + j] = i;
      if (ns > 0) {
        // A skipped sequence keeps its slots below the capacity as null items.  The
        // tree masks of a skipped sequence's rows may not exist (rows past T).
        int64_t it = my_item0;
        for (int sp_i = 0; sp_i < ns; ++sp_i) {
          const int64_t cs = seq_chunk(a, s, c);
          const int32_t pb = (int32_t)(sp_i * cs);
          const int32_t pe = (int32_t)((sp_i + 1) * cs < s.npages ? (sp_i + 1) * cs : s.npages);
          for (int rb = 0; rb < s.nrb && it < a.items_cap; ++rb) {
            const bool prec = a.is_bf16 && sp.nsplit > 0 && rb_precise(a, s, my_row0, rb);
            Item item;
            item.seq = sp.nsplit > 0 ? i : -1;
            item.page_begin = pb;
            item.page_end = pe;
            item.split_rb = (sp_i << kRbBits) | rb | (prec ? kItemPrecise : 0);
            a.items[it++] = item;
          }
        }
      }
      if (sp.nsplit > 1)  // arrival counters of the last-split merge
        for (int k = 0; k < s.nrb * a.Hkv; ++k) a.counters[(size_t)sp.item0 * a.Hkv + k] = 0;
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) carry[k] += t[k];
  }
  // Work order: the items by decreasing estimated time (kOrderBuckets buckets up to the
  // longest), so that the longest units start first and the grid ends on short ones (a
  // unit's place in the order changes only which CTA runs it and when).  The estimate is
  // the page count, doubled for wide units (17..64 rows per KV head), which stream at
  // about half the rate of narrow ones.
  {
    __shared__ int32_t hist[kOrderBuckets];
    const int64_t n_items = carry[1] < a.items_cap ? carry[1] : a.items_cap;
    const int64_t cmax = c > 2 * (int64_t)a.min_chunk ? c : 2 * (int64_t)a.min_chunk;
    const int64_t span = cmax < (int64_t)a.maxp ? cmax : (int64_t)a.maxp;  // longest item
    auto bucket = [&](int64_t i) {
      const Item& t = a.items[i];
      int w = 1;
      if (t.seq >= 0) {
        const int R = a.G * (cached ? s_ql[t.seq] : a.query_lens[t.seq]);
        if (R > kNarrowRows && R <= kRowBlock) w = kWideOrderWeight;
      }
      const int64_t b = (int64_t)(t.page_end - t.page_begin) * w * kOrderBuckets /
                        (kWideOrderWeight * span + 1);
      return (int)(b < 0 ? 0 : (b < kOrderBuckets ? b : kOrderBuckets - 1));
    };
    for (int b = tid; b < kOrderBuckets; b += kPlanThreads) hist[b] = 0;
    __syncthreads();  // every item is written, the histogram is clear
    for (int64_t i = tid; i < n_items; i += kPlanThreads) atomicAdd(&hist[bucket(i)], 1);
    __syncthreads();
    if (tid == 0) {
      int32_t run = 0;
      for (int b = kOrderBuckets - 1; b >= 0; --b) {
        const int32_t h = hist[b];
        hist[b] = run;
        run += h;
      }
    }
    __syncthreads();
    for (int64_t i = tid; i < n_items; i += kPlanThreads)
      a.order[atomicAdd(&hist[bucket(i)], 1)] = (int32_t)i;
  }
  if (tid == 0) {
    a.header->n_items = (int32_t)(carry[1] < a.items_cap ? carry[1] : a.items_cap);
    a.header->work_counter = 0;
    a.header->chunk_pages = (int32_t)(c < INT_MAX ? c : INT_MAX);
    a.header->n_partial_rows = (int32_t)carry[2];
  }
  if (lengths_ok) return;
  __syncthreads();

  // Rows owned by no sequence, or by one with inconsistent lengths, are NaN.
  for (int r = tid; r < a.T; r += kPlanThreads) {
    const int seq = a.token_seq[r];
    if (seq >= 0 && !(a.seqplan[seq].flags & kSeqInvalid)) continue;
    for (int h = 0; h < a.Hq; ++h) {
      const size_t row = (size_t)r * a.Hq + h;
      a.lse[row] = NAN;
      if (a.is_bf16) {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + row * a.D;
        for (int d = 0; d < a.D; ++d) o[d] = __float2bfloat16(NAN);
      } else {
        float* o = static_cast<float*>(a.out) + row * a.D;
        for (int d = 0; d < a.D; ++d) o[d] = NAN;
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// Attention, bf16 storage
// ------------------------------------------------------------------------------------
struct AttnArgs {
  const void* q;
  void* out;
  float* lse;
  const int32_t* block_table;
  const SeqPlan* seqplan;
  const Item* items;
  const int32_t* order;  // work order: item indices, longest first
  PlanHeader* header;
  int32_t* counters;
  float* part_o;
  float* part_lse;
  const void* k_pages;  // fp32 path only
  const void* v_pages;  // fp32 path only
  int32_t T, Hq, Hkv, G, maxp, num_pages, P;
  float scale_log2;  // softmax scale * log2(e)
  float scale;
  int32_t* err;
  const uint64_t* tree_mask;  // draft-tree visibility per query token, or null (causal)
  const float* k_scale;       // quantised pools: [num_pages, Hkv, P] fp32
  const float* v_scale;
};

template <int D, int KQ = kKvBf16>
struct Smem {
  // Stages in the 16-bit ring.  In a decode unit warp w consumes the stages s with
  // s % kConsumerWarps == w and waits on slot s % kSlots by phase parity.  The parity
  // test is only sound if the slot's previous fill was consumed by the same warp, i.e.
  // if kSlots is a multiple of the number of consumer warps; otherwise a warp could pass
  // the parity test while the slot's previous fill is still in flight.  The same holds
  // for the converters of quantised pools (stage s goes to converter s % kConvWarps).
  static constexpr int kSlots = 8;
  static_assert(kSlots % kConsumerWarps == 0 && kSlots % kConvWarps == 0,
                "stage slots must be a multiple of the consumer warps and of the converters");
  static constexpr int NH = D / 64;                        // 128-byte halves per token row
  static constexpr int kRowBytes = D * 2;
  static constexpr int kOperandBytes = kStageTokens * kRowBytes;  // K or V of one stage
  static constexpr int kStageBytes = 2 * kOperandBytes;
  static constexpr int kQStride = D * 2 + 16;               // padded Q row
  static constexpr int kQBytes = kRowBlock * kQStride;
  static constexpr int kNarrowStride = D + 4;               // floats per merge row
  static constexpr int kNarrowWarpFloats = kNarrowRows * kNarrowStride + 2 * kNarrowRows;
  static constexpr int kNarrowBytes = kConsumerWarps * kNarrowWarpFloats * 4;
  // Wide units: two P tiles of the tcgen05 PV product (by step parity), each 128 rows
  // (TMEM lanes) of 128 bytes -- the 64 tokens of a two-stage step -- in the K-major
  // 128-byte-swizzled layout.  They reuse the query staging, which is dead once the
  // warps hold their query fragments.
  static constexpr int kPTileOff = 0;
  static constexpr int kPTileBytes = 128 * 128;
  // Prompt-chunk units: their query tile (128 rows, K-major 128-byte swizzle,
  // [D/64][row][64]) after the P tiles.
  static constexpr int kQTileOff = kPTileOff + 2 * kPTileBytes;
  // Precise units: the rounding error of each P tile as a second bf16 tile (bf16 calls
  // only).
  static constexpr int kPLoOff = kQTileOff + 128 * D * 2;
  static constexpr int kWideBytes = kPLoOff + (KQ == kKvBf16 ? 2 * kPTileBytes : 0);
  static constexpr int kMergeBytes = kNarrowBytes > kWideBytes ? kNarrowBytes : kWideBytes;
  static constexpr int kScratchBytes = kQBytes > kMergeBytes ? kQBytes : kMergeBytes;
  static constexpr int kScratchOff = kSlots * kStageBytes;
  static constexpr int kRingOff = kScratchOff + ((kScratchBytes + 127) / 128) * 128;
  // Quantised pools: a stage's codes land in the upper half of its slot, K codes
  // [32][D] bytes at kCodeOff, V codes after them; its scales (32 K, 32 V) in the
  // scale array.
  static constexpr bool kQ = KQ != kKvBf16;
  static constexpr int kCodeOff = kOperandBytes;
  static constexpr int kScaleOff = kRingOff + kRing * (int)sizeof(RingEntry);
  static constexpr int kBarOff = kScaleOff + (kQ ? kSlots * 2 * kStageTokens * 4 : 0);
  // full[kSlots], empty[kSlots], ufull[kRing], uempty[kRing], tensor-memory unit
  // barriers bp[2], bo[2], bs[2], bq, bfin, ready[kSlots] (quantised pools) |
  // meta[kSlots], flag[4], tmem base, qmax[4]
  static constexpr int kWideBars = 8;
  static constexpr int kBarBytes = (2 * kSlots + 2 * kRing + kWideBars + (kQ ? kSlots : 0)) * 8 +
                                   (kSlots + 4 + 1 + 4) * 4;
  // Draft-tree masks of the unit's rows (row r: its token's mask, own bit set).
  static constexpr int kTmaskOff = ((kBarOff + kBarBytes + 7) / 8) * 8;
  static constexpr int kBytes = kTmaskOff + kRowBlockTc * 8;
  static constexpr int kDynBytes = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kDynBytes <= 227 * 1024, "shared memory of one CTA");
  static_assert(kPLoOff % 1024 == 0 && kQTileOff % 1024 == 0, "swizzle atoms of the tiles");
  static_assert(kScaleOff % 16 == 0, "scale arrays take bulk copies");
};

// Byte offset of 16-byte column chunk gc of token row t inside one operand of a stage.
// A stage operand is its pages in order, each page one TMA box laid out as
// [D/64 halves][P tokens][64] with the 128-byte swizzle (the chunk index XOR-ed with the
// token row modulo 8).  A page half is the canonical K-major (for K) and MN-major (for V)
// 128-byte-swizzled operand layout of tcgen05.
template <int D, int P>
__device__ __forceinline__ uint32_t kv_off(int t, int gc) {
  return (uint32_t)((t / P) * (P * D * 2) + (gc >> 3) * (P * 128) + (t % P) * 128 +
                    (((gc & 7) ^ (t & 7)) << 4));
}
// Byte offset of token row t (a multiple of 8) in every column half: added to an offset
// from kv_off for row t0 % 8, it gives row t0 + t.
template <int D, int P>
__host__ __device__ constexpr uint32_t tok_off(int t) {
  return (uint32_t)((t / P) * (P * D * 2) + (t % P) * 128);
}

// Conditional rescaling.  Probabilities are taken against a per-row reference maximum
// that may trail the true running maximum by up to kRebase (log2 units, so p <= 2^8);
// the accumulators are rescaled only when a new maximum exceeds the reference by more
// than that.  Sum and output share the reference, so the normalised result is exact.
constexpr float kRebase = 8.f;

// Per-lane ldmatrix byte offsets (relative to a stage operand) for the narrow path:
// koff[ks % 4]: K A-fragment of token tile 0, k-step ks; voff[dt % 4]: V^T A-fragment of
// token tile 0, d-tile dt.  Steps 4 apart are the same chunks of the next 64-column
// half (half_off), and token tile 1 adds 16 rows: both are immediates.
template <int P>
__host__ __device__ constexpr uint32_t half_off(int i) {
  return (uint32_t)(i >> 2) * (P * 128);
}
template <int D, int P>
__device__ __forceinline__ void narrow_offsets(int lane, uint32_t (&koff)[4], uint32_t (&voff)[4]) {
  const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    koff[i] = kv_off<D, P>((mi & 1) * 8 + r8, 2 * i + (mi >> 1));
    voff[i] = kv_off<D, P>((mi >> 1) * 8 + r8, 2 * i + (mi & 1));
  }
}

// ---- the 16-bit element type of a call: bf16, or f16 for quantised pools -------------
template <int KQ>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (KQ == kKvBf16) mma_bf16_16816(d, a, b0, b1);
  else mma_f16_16816(d, a, b0, b1);
}
template <int KQ>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (KQ == kKvBf16) return pack_bf16x2(lo, hi);
  else return pack_f16x2(lo, hi);
}
template <int KQ>
__device__ __forceinline__ void unpack2(uint32_t v, float& lo, float& hi) {
  if constexpr (KQ == kKvBf16) {
    lo = bf16_lo_f32(v);
    hi = bf16_hi_f32(v);
  } else {
    f16x2_to_f32(v, lo, hi);
  }
}

// ---- narrow units: S^T = K Q^T, one warp per stage -------------------------------
// Quantised pools (KQ): the stage holds the codes as f16; the scores are multiplied by
// the K scale of their token (ks) and P by the V scale of its token (vs) before the
// PV product, which then sums scale * code * p.
template <int D, int P, int NN, bool MASKED, int KQ>
__device__ __forceinline__ void narrow_stage(uint32_t kbase, uint32_t vbase, int loaded,
                                             const uint32_t (&qb)[D / 16][NN][2],
                                             const uint32_t (&koff)[4],
                                             const uint32_t (&voff)[4],
                                             float (&oT)[D / 16][NN][4], float (&mref)[NN][2],
                                             float (&l)[NN][2], int t_abs0,
                                             const int (&lim)[NN][2], float c, int lane,
                                             const uint64_t* tm, int ctx_end, const float* ks,
                                             const float* vs) {
  constexpr uint32_t kTile = tok_off<D, P>(16);  // 16 token rows
  const int g = lane >> 2;
  float s[2][NN][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    float acc[2][NN][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int nn = 0; nn < NN; ++nn) acc[h][nn][0] = acc[h][nn][1] = acc[h][nn][2] = acc[h][nn][3] = 0.f;
    if (!MASKED || 16 * mt < loaded) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(kbase + koff[ks & 3] + half_off<P>(ks) + mt * kTile, a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int nn = 0; nn < NN; ++nn) mma16816<KQ>(acc[ks & 1][nn], a, qb[ks][nn][0], qb[ks][nn][1]);
      }
    }
    float ksc[2] = {1.f, 1.f};
    if constexpr (KQ != kKvBf16) {
      ksc[0] = ks[16 * mt + g];
      ksc[1] = ks[16 * mt + g + 8];
    }
#pragma unroll
    for (int nn = 0; nn < NN; ++nn)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[mt][nn][e] = acc[0][nn][e] + acc[1][nn][e];
        if constexpr (KQ != kKvBf16) s[mt][nn][e] *= ksc[e >> 1];
      }
  }
  if (MASKED) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nn = 0; nn < NN; ++nn)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tt = 16 * mt + g + 8 * (e >> 1);
          if (tt >= loaded || t_abs0 + tt > lim[nn][e & 1]) s[mt][nn][e] = -INFINITY;
        }
    // Draft tree: in the draft window (positions from ctx_end on) a row keeps only its
    // ancestors and itself.  Scores already past the causal limit stay dropped.
    if (tm != nullptr) {
#pragma unroll
      for (int nn = 0; nn < NN; ++nn)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t mk = tm[8 * nn + 2 * (lane & 3) + h];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hi = 0; hi < 2; ++hi) {
              const int dt = t_abs0 + 16 * mt + g + 8 * hi - ctx_end;
              if (dt >= 0 && !((mk >> (dt & 63)) & 1)) s[mt][nn][2 * hi + h] = -INFINITY;
            }
        }
    }
  }

  // Rebase the rows whose maximum outgrew the reference.
  float mx[NN][2];
  bool up = false;
#pragma unroll
  for (int nn = 0; nn < NN; ++nn)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[nn][h] = fmaxf(fmaxf(s[0][nn][h], s[0][nn][h + 2]), fmaxf(s[1][nn][h], s[1][nn][h + 2]));
      up |= mx[nn][h] * c > mref[nn][h] + kRebase;
    }
  if (__any_sync(0xffffffffu, up)) {
#pragma unroll
    for (int nn = 0; nn < NN; ++nn)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v = mx[nn][h];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        const float vs = v * c;
        if (vs > mref[nn][h] + kRebase) {  // same decision on all 8 lanes of the row
          const float alpha = exp2f(mref[nn][h] - vs);
          l[nn][h] *= alpha;
#pragma unroll
          for (int dt = 0; dt < D / 16; ++dt) {
            oT[dt][nn][h] *= alpha;
            oT[dt][nn][h + 2] *= alpha;
          }
          mref[nn][h] = vs;
        }
      }
  }
#pragma unroll
  for (int nn = 0; nn < NN; ++nn) {
    const float nm0 = mref[nn][0] == -INFINITY ? 0.f : -mref[nn][0];
    const float nm1 = mref[nn][1] == -INFINITY ? 0.f : -mref[nn][1];
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = exp2f(fmaf(s[mt][nn][e], c, (e & 1) ? nm1 : nm0));
        s[mt][nn][e] = p;
        if (e & 1) rs1 += p;
        else rs0 += p;
      }
    l[nn][0] += rs0;
    l[nn][1] += rs1;
  }

  // O^T += V^T P^T: the P^T operand is the transpose of the S^T accumulator tile.
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    if (!MASKED || 16 * kk < loaded) {
      uint32_t pb[NN][2];
      float vsc[2] = {1.f, 1.f};
      if constexpr (KQ != kKvBf16) {
        vsc[0] = vs[16 * kk + g];
        vsc[1] = vs[16 * kk + g + 8];
      }
#pragma unroll
      for (int nn = 0; nn < NN; ++nn) {
        pb[nn][0] = movmatrix_trans(pack2<KQ>(s[kk][nn][0] * vsc[0], s[kk][nn][1] * vsc[0]));
        pb[nn][1] = movmatrix_trans(pack2<KQ>(s[kk][nn][2] * vsc[1], s[kk][nn][3] * vsc[1]));
      }
#pragma unroll
      for (int dt = 0; dt < D / 16; ++dt) {
        uint32_t a[4];
        ldsm_x4_trans(vbase + voff[dt & 3] + half_off<P>(dt) + kk * kTile, a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int nn = 0; nn < NN; ++nn) mma16816<KQ>(oT[dt][nn], a, pb[nn][0], pb[nn][1]);
      }
    }
  }
}

// Per-lane ldmatrix byte offsets of the K B-fragments of the wide path: token tile 0
// (8 rows), d-chunks 4 qd .. 4 qd + 3 at kw[qd % 2] + half_off(2 qd).
template <int D, int P>
__device__ __forceinline__ void wide_offsets(int lane, uint32_t (&kw)[2]) {
  const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int i = 0; i < 2; ++i) kw[i] = kv_off<D, P>(r8, 4 * i + mi);
}

// ---- wide units: S = Q K^T of one m16 row tile over a step, in registers -------------
// A step is NST (1 or 2) consecutive 32-token stages of the unit: token tt of the step
// lies in stage tt / 32 (K tile kb[tt / 32]).  Warp MMA for the scores (rows g and g + 8
// of the tile, tokens 8 nt + 2 tq + {0, 1}), online softmax with the conditional
// rescaling, and P as bf16 into this warp's 16 rows of the step's P tile (prow: the tile
// row of row g; byte 2 tt of a row before the swizzle).  alpha / rescale report a moved
// reference maximum: O, held in TMEM, is rescaled by the caller.
template <int D, int P, int NST, int KQ>
__device__ __forceinline__ void wide_s_step(const uint32_t (&kb)[2], int tvalid, bool masked,
                                            const uint32_t (&qa)[D / 16][4],
                                            const uint32_t (&kw)[2], float (&mref)[2],
                                            float (&l)[2], float (&alpha)[2], bool& rescale,
                                            int t_abs0, int limA, int limB, float c, int lane,
                                            uint8_t* prow, const uint64_t* tmw, int ctx_end,
                                            const float* ks0, const float* ks1,
                                            const float* vs0, const float* vs1) {
  constexpr int NT = 4 * NST;
  const int g = lane >> 2, tq = lane & 3;
  float s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
  // k-steps outside, token tiles inside: independent accumulation chains in flight.
  // Every tile is computed (rows of a stage past its loaded tokens are stale but inside
  // the tile, and masked below), so the products carry no branches.
#pragma unroll
  for (int qd = 0; qd < D / 32; ++qd)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb[nt >> 2] + kw[qd & 1] + half_off<P>(2 * qd) + tok_off<D, P>(8 * (nt & 3)), b0,
              b1, b2, b3);
      mma16816<KQ>(s[nt], qa[2 * qd], b0, b1);
      mma16816<KQ>(s[nt], qa[2 * qd + 1], b2, b3);
    }
  // Quantised pools: token tt's scores times its K scale (stage tt / 32).
  if constexpr (KQ != kKvBf16) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 k2 = *reinterpret_cast<const float2*>((nt < 4 ? ks0 : ks1) + 8 * (nt & 3) + 2 * tq);
      s[nt][0] *= k2.x;
      s[nt][1] *= k2.y;
      s[nt][2] *= k2.x;
      s[nt][3] *= k2.y;
    }
  }
  if (masked) {
    // Draft tree: rows g and g + 8 keep only their ancestors (and themselves) among the
    // draft tokens (positions from ctx_end on).
    const uint64_t mA = tmw ? tmw[0] : ~0ull, mB = tmw ? tmw[8] : ~0ull;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tt = 8 * nt + 2 * tq + (e & 1);
        const int dt = t_abs0 + tt - ctx_end;
        const bool in_tree = dt < 0 || (((e < 2) ? mA : mB) >> (dt & 63)) & 1;
        if (tt >= tvalid || t_abs0 + tt > ((e < 2) ? limA : limB) || !in_tree) s[nt][e] = -INFINITY;
      }
  }
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
  alpha[0] = alpha[1] = 1.f;
  rescale = false;
  const bool up = mx[0] * c > mref[0] + kRebase || mx[1] * c > mref[1] + kRebase;
  if (__any_sync(0xffffffffu, up)) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v = mx[h];
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
      const float vs = v * c;
      if (vs > mref[h] + kRebase) {  // same decision on the quad sharing the row
        if (mref[h] != -INFINITY) rescale = true;
        alpha[h] = exp2f(mref[h] - vs);
        l[h] *= alpha[h];
        mref[h] = vs;
      }
    }
  }
  const float nm[2] = {mref[0] == -INFINITY ? 0.f : -mref[0], mref[1] == -INFINITY ? 0.f : -mref[1]};
  // Rows g and g + 8 share the swizzle (tile rows 32 w + g, 32 w + g + 8).
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[e] = ex2_approx(fmaf(s[nt][e], c, nm[e >> 1]));
      l[e >> 1] += p[e];
    }
    if constexpr (KQ != kKvBf16) {  // P times the V scale of its token
      const float2 v2 = *reinterpret_cast<const float2*>((nt < 4 ? vs0 : vs1) + 8 * (nt & 3) + 2 * tq);
      p[0] *= v2.x;
      p[1] *= v2.y;
      p[2] *= v2.x;
      p[3] *= v2.y;
    }
    const int off = ((nt ^ g) << 4) + 4 * tq;
    *reinterpret_cast<uint32_t*>(prow + off) = pack2<KQ>(p[0], p[1]);
    *reinterpret_cast<uint32_t*>(prow + 8 * 128 + off) = pack2<KQ>(p[2], p[3]);
  }
}

// ---- prompt-chunk units: one row of P ---------------------------------------------------
// Row r's 32 scores sr (fp32 bits, raw Q K^T) of one stage to probabilities against the
// reference maximum mu (scaled by c), written as bf16 into its 128-byte row of the P
// tile (K-major, 128-byte swizzle); tokens outside `valid` get 0.  Returns the row's sum
// of P.  A precise unit also writes each value's bf16 rounding error into the low tile
// (O += P_lo V follows O += P V).
// Quantised pools: the scores sr are already scaled by their tokens' K scales, and P
// is multiplied by the V scale of its token (vs) before it is written (the sum is of P
// itself).
template <int D, bool PRECISE, int KQ>
__device__ __forceinline__ float chunk_p_row(const uint32_t (&sr)[32], uint32_t valid, float c,
                                             float mu, uint8_t* prow, int r, const float* vs) {
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t hw[16];
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float e0 = ex2_approx(fmaf(__uint_as_float(sr[i]), c, -mu));
    const float e1 = ex2_approx(fmaf(__uint_as_float(sr[i + 1]), c, -mu));
    float p0 = (valid >> i) & 1 ? e0 : 0.f;
    float p1 = (valid >> (i + 1)) & 1 ? e1 : 0.f;
    s4[(i >> 1) & 3] += p0 + p1;
    if constexpr (KQ != kKvBf16) {
      p0 *= vs[i];
      p1 *= vs[i + 1];
    }
    const uint32_t h = pack2<KQ>(p0, p1);
    hw[i >> 1] = h;
    if constexpr (PRECISE) {
      // The low part goes out at once: its 16 words are never live together.
      float h0, h1;
      unpack2<KQ>(h, h0, h1);
      const uint32_t lo = pack2<KQ>(p0 - h0, p1 - h1);
      *reinterpret_cast<uint32_t*>(prow + (Smem<D>::kPLoOff - Smem<D>::kPTileOff) +
                                   (((i >> 3) ^ (r & 7)) << 4) + (i & 7) * 2) = lo;
    }
  }
#pragma unroll
  for (int ch = 0; ch < 4; ++ch)
    *reinterpret_cast<uint4*>(prow + ((ch ^ (r & 7)) << 4)) =
        make_uint4(hw[4 * ch], hw[4 * ch + 1], hw[4 * ch + 2], hw[4 * ch + 3]);
  return (s4[0] + s4[1]) + (s4[2] + s4[3]);
}

// ---- quantised pools: the unit's Q in f16 ----------------------------------------------
// Largest magnitude of eight bf16 values.
__device__ __forceinline__ float absmax_bf16x8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo_f32(w[i])), fabsf(bf16_hi_f32(w[i]))));
  return m;
}
// Eight bf16 values times mul (a power of two), as f16 (exact unless below the f16
// normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, float mul) {
  uint4 r;
  r.x = pack_f16x2(bf16_lo_f32(v.x) * mul, bf16_hi_f32(v.x) * mul);
  r.y = pack_f16x2(bf16_lo_f32(v.y) * mul, bf16_hi_f32(v.y) * mul);
  r.z = pack_f16x2(bf16_lo_f32(v.z) * mul, bf16_hi_f32(v.z) * mul);
  r.w = pack_f16x2(bf16_lo_f32(v.w) * mul, bf16_hi_f32(v.w) * mul);
  return r;
}

// ---- unit classification ------------------------------------------------------------
// Draft-tree units: sequences with 2..64 query tokens when a tree is given; longer
// query windows (prompt chunks) and decode rows keep the causal window.
__device__ __forceinline__ bool tree_unit(const AttnArgs& a, int ql) {
  return a.tree_mask != nullptr && ql > 1 && ql <= 64;
}
// The smallest position limit over the rows of a row block starting at row r0: the
// causal limit of its first token, or for a tree the last context position (any draft
// token may be hidden from a row).
__device__ __forceinline__ int unit_min_lim(const AttnArgs& a, int L, int ql, int r0) {
  return tree_unit(a, ql) ? L - ql - 1 : L - ql + r0 / a.G;
}

// ---- output helpers ----------------------------------------------------------------
__device__ __forceinline__ size_t out_row(const AttnArgs& a, const SeqPlan& sp, int head, int r) {
  const int j = r / a.G, hh = r % a.G;
  return (size_t)(sp.qrow0 + j) * a.Hq + (size_t)head * a.G + hh;
}

__device__ __forceinline__ size_t partial_row(const AttnArgs& a, const SeqPlan& sp, int split,
                                              int head, int r) {
  return (size_t)sp.partial_base + ((size_t)split * a.Hkv + head) * ((size_t)a.G * sp.qlen) + r;
}

// Merge the partials of every split of rows r0 .. r0+Rb-1 of one KV head (the caller is
// the last split to finish: all partials are in memory).  Four consumer warps.
template <int D>
__device__ void merge_splits(const AttnArgs& a, const SeqPlan& sp, int head, int r0, int Rb,
                             int warp, int lane) {
  constexpr int E = D / 32;
  const float kLn2 = 0.6931471805599453f;
  for (int rr = warp; rr < Rb; rr += kConsumerWarps) {
    const int r = r0 + rr;
    float mx = -INFINITY;
    bool bad = false;
    for (int s = lane; s < sp.nsplit; s += 32) {
      const float v = __ldcg(a.part_lse + partial_row(a, sp, s, head, r));
      bad |= isnan(v);
      mx = fmaxf(mx, v);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    bad = __any_sync(0xffffffffu, bad);
    const float mu = mx == -INFINITY ? 0.f : mx;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    for (int s = 0; s < sp.nsplit; ++s) {
      const size_t pr = partial_row(a, sp, s, head, r);
      const float w = exp2f((__ldcg(a.part_lse + pr) - mu) * 1.4426950408889634f);
      wsum += w;
      const float* po = a.part_o + pr * D + lane * E;
      if constexpr (E == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(po));
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(po));
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
    const float inv = 1.f / wsum;
    const size_t orow = out_row(a, sp, head, r);
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + orow * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float x0 = bad ? NAN : acc[e] * inv, x1 = bad ? NAN : acc[e + 1] * inv;
      *reinterpret_cast<uint32_t*>(og + e) = pack_bf16x2(x0, x1);
    }
    if (lane == 0) a.lse[orow] = bad ? NAN : mu + log2f(wsum) * kLn2;
  }
}

// A split unit whose arrival was counted; the CTA that counted last merges the rows.
// The count's result is only examined at the start of the CTA's next unit, so the
// atomic's round trip overlaps the hand-over to that unit.
struct PendingMerge {
  SeqPlan sp;
  int32_t head, r0, Rb, valid;
  int32_t old;   // thread 0 only: the counter's value before this CTA's arrival
  int32_t* ctr;  // thread 0 only: the counter
};

// A 32-bit load with acquire semantics at GPU scope.
__device__ __forceinline__ int32_t load_acquire_gpu(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// All consumer threads: the CTA's partial rows have been written.
__device__ __forceinline__ void count_split_arrival(const AttnArgs& a, const SeqPlan& sp,
                                                    const Item& it, int head, int r0, int Rb,
                                                    PendingMerge& pm) {
  named_bar_sync(1, kConsumerThreads);  // every partial store of the CTA is issued
  if (threadIdx.x == 0) {
    const int rb = it.split_rb & ((1 << kRbBits) - 1);
    pm.ctr = a.counters + ((size_t)sp.item0 + rb) * a.Hkv + head;
    __threadfence();  // orders the CTA's partials before the count (cumulative via the barrier)
    pm.old = atomicAdd(pm.ctr, 1);
  }
  pm.sp = sp;
  pm.head = head;
  pm.r0 = r0;
  pm.Rb = Rb;
  pm.valid = 1;
}

// Thread 0, before the named barrier that precedes finish_pending: whether this CTA
// counted the last split of its previous unit.  If so, an acquire read of the counter
// (which holds every split's released count) orders the other CTAs' partials before
// the barrier, and so before every consumer's reads of them.
__device__ __forceinline__ int32_t last_split_seen(const PendingMerge& pm) {
  const bool last = pm.valid && pm.old == pm.sp.nsplit - 1;
  if (last) (void)load_acquire_gpu(pm.ctr);
  return last;
}

// All consumer threads; `flag` was set by thread 0 (last_split_seen) before the last
// named barrier.
template <int D>
__device__ __forceinline__ void finish_pending(const AttnArgs& a, PendingMerge& pm,
                                               const int32_t* flag, int warp, int lane) {
  if (pm.valid && *flag) merge_splits<D>(a, pm.sp, pm.head, pm.r0, pm.Rb, warp, lane);
  pm.valid = 0;
}

// KQ: kKvBf16 (bf16 pages, tm_k / tm_v over the pool) or kKvFp8 / kKvInt8 (8-bit codes,
// tm_k / tm_v over the code pools, scales in a.k_scale / a.v_scale).
template <int D, int P, int KQ>
__global__ void __launch_bounds__(KQ == kKvBf16 ? kThreads : kThreadsQ, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using S = Smem<D, KQ>;
  constexpr bool kQuant = KQ != kKvBf16;
  constexpr int kSlots = S::kSlots;
  constexpr int PPS = kStageTokens / P;  // pages per stage
  constexpr int kPageBytes = P * D * 2;  // one page of one head, one operand (16-bit)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint8_t* scratch = smem + S::kScratchOff;
  RingEntry* ring = reinterpret_cast<RingEntry*>(smem + S::kRingOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* empty = full + kSlots;
  uint64_t* ufull = empty + kSlots;
  uint64_t* uempty = ufull + kRing;
  // Wide and prompt-chunk units: bp[b] P of the step with parity b is in shared memory;
  // bo[b] the PV product of that step is done; bs[b] S of that step is in TMEM (prompt
  // chunks); bq the query tile is staged (prompt chunks); bfin every tcgen05.mma of the
  // CTA has completed.
  uint64_t* bp = uempty + kRing;
  uint64_t* bo = bp + 2;
  uint64_t* bs = bo + 2;
  uint64_t* bq = bs + 2;
  uint64_t* bfin = bq + 1;
  uint64_t* ready = bfin + 1;  // quantised pools: the stage's codes are converted
  int32_t* meta = reinterpret_cast<int32_t*>(ready + (kQuant ? kSlots : 0));
  int32_t* flag = meta + kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(flag + 4);
  float* qmax = reinterpret_cast<float*>(tmem_slot + 1);
  float* stage_scales = reinterpret_cast<float*>(smem + S::kScaleOff);  // [kSlots][K 32 | V 32]
  // What the consumers and the MMA warp wait on before reading a stage: its copies
  // (bf16), or its conversion (quantised pools; the converter waits on the copies).
  uint64_t* stage_ready = kQuant ? ready : full;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&ufull[r], 1);
      // consumers, the MMA warp and (quantised pools) the converters
      mbar_init(&uempty[r], kConsumerWarps + 1 + (kQuant ? kConvWarps : 0));
    }
    if (kQuant)
      for (int s = 0; s < kSlots; ++s) mbar_init(&ready[s], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bp[b], kConsumerWarps);
      mbar_init(&bo[b], 1);
      mbar_init(&bs[b], 1);
    }
    mbar_init(bq, kConsumerWarps);
    mbar_init(bfin, 1);
    mbar_fence_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensor_map(&tm_k);
    prefetch_tensor_map(&tm_v);
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);  // one CTA per SM: never contended
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_prior_grid();  // the plan of this call is complete and visible

  const int32_t n_units = a.header->n_items * a.Hkv;
  int32_t* const work_counter = &a.header->work_counter;

  if (warp == kProducerWarp) {
    // ------------------------------ producer ------------------------------
    // KV of decode and verify units is read once per call; a prompt chunk's pages are
    // read by each of its row blocks, so they are kept in L2 as long as other data.
    const uint64_t pol_once = l2_policy_evict_first();
    const uint64_t pol_shared = l2_policy_evict_normal();
    uint32_t stage_it = 0, unit_it = 0;
    bool ok = true;
    // Descriptor pipeline: unit u is streamed while the next unit's descriptor and
    // first block-table chunk are in flight, and the atomic for the one after.
    int32_t u = 0, u1 = 0, u2_lane0 = 0;
    if (lane == 0) {
      u = atomicAdd(work_counter, 1);
      u1 = atomicAdd(work_counter, 1);
    }
    u = __shfl_sync(0xffffffffu, u, 0);
    u1 = __shfl_sync(0xffffffffu, u1, 0);
    Item it{}, it1{};
    SeqPlan sp{}, sp1{};
    if (u < n_units) {
      it = a.items[a.order[u / a.Hkv]];
      if (it.seq >= 0) sp = a.seqplan[it.seq];
    }
    if (u1 < n_units) {
      it1 = a.items[a.order[u1 / a.Hkv]];
      if (it1.seq >= 0) sp1 = a.seqplan[it1.seq];
    }
    if (lane == 0) u2_lane0 = atomicAdd(work_counter, 1);
    int32_t bt_cur = 0;  // this lane's block-table entry of the unit's first 32 pages
    if (u < n_units && it.seq >= 0 && it.page_begin + lane < it.page_end)
      bt_cur = a.block_table[(size_t)it.seq * a.maxp + it.page_begin + lane];
    for (;;) {
      const int slot = unit_it % kRing;
      ok = mbar_wait(&uempty[slot], ((unit_it / kRing) & 1) ^ 1);
      if (!ok) break;
      if (u >= n_units) {
        if (lane == 0) {
          ring[slot].u = -1;
          mbar_arrive(&ufull[slot]);
        }
        break;
      }
      if (lane == 0) {
        RingEntry e;
        e.u = u;
        e.head = u % a.Hkv;
        e.item = it;
        e.sp = sp;
        e.pad[0] = e.pad[1] = 0;
        ring[slot] = e;
        mbar_arrive(&ufull[slot]);
      }
      ++unit_it;
      // Prefetch the next unit's first block-table chunk and the descriptor after it.
      int32_t bt_next = 0;
      if (u1 < n_units && it1.seq >= 0 && it1.page_begin + lane < it1.page_end)
        bt_next = a.block_table[(size_t)it1.seq * a.maxp + it1.page_begin + lane];
      const int32_t u2 = __shfl_sync(0xffffffffu, u2_lane0, 0);
      Item it2{};
      SeqPlan sp2{};
      if (u2 < n_units) it2 = a.items[a.order[u2 / a.Hkv]];
      if (lane == 0) u2_lane0 = atomicAdd(work_counter, 1);

      if (it.seq >= 0) {
        const int head = u % a.Hkv;
        const int32_t* bt_row = a.block_table + (size_t)it.seq * a.maxp;
        const uint64_t pol = a.G * sp.qlen > kRowBlock ? pol_shared : pol_once;
        for (int pg0 = it.page_begin; pg0 < it.page_end && ok; pg0 += 32) {
          const int npg = min(32, it.page_end - pg0);
          const int32_t my_id =
              pg0 == it.page_begin ? bt_cur : (lane < npg ? bt_row[pg0 + lane] : 0);
          for (int s0 = 0; s0 < npg; s0 += PPS) {
            const int slot_s = stage_it % kSlots;
            ok = mbar_wait(&empty[slot_s], ((stage_it / kSlots) & 1) ^ 1);
            if (!ok) break;
            const int n_in = min(PPS, npg - s0);
            int ids[PPS];
            uint32_t bytes = 0;
            int bad = 0;
#pragma unroll
            for (int e = 0; e < PPS; ++e) {
              ids[e] = __shfl_sync(0xffffffffu, my_id, (s0 + e) & 31);
              if (e < n_in) {
                if (ids[e] < 0 || ids[e] >= a.num_pages) bad = 1;
                else bytes += kQuant ? 2u * (P * D + P * 4) : 2u * kPageBytes;
              }
            }
            if (kQuant && lane == 0) {
              // Codes: one box per page and operand, [P tokens][D bytes], into the upper
              // half of the slot (K codes, then V codes); scales: P floats per page, head
              // and operand, contiguous in [page][head][slot].
              meta[slot_s] = bad;
              mbar_arrive_expect_tx(&full[slot_s], bytes);
              uint8_t* kdst = stages + slot_s * S::kStageBytes + S::kCodeOff;
              uint8_t* vdst = kdst + kStageTokens * D;
              float* ksd = stage_scales + slot_s * 2 * kStageTokens;
              float* vsd = ksd + kStageTokens;
#pragma unroll
              for (int e = 0; e < PPS; ++e) {
                if (e < n_in && ids[e] >= 0 && ids[e] < a.num_pages) {
                  tma_load_3d(kdst + e * P * D, &tm_k, &full[slot_s], 0, ids[e] * P, head, pol);
                  tma_load_3d(vdst + e * P * D, &tm_v, &full[slot_s], 0, ids[e] * P, head, pol);
                  const size_t so = ((size_t)ids[e] * a.Hkv + head) * P;
                  bulk_load(ksd + e * P, a.k_scale + so, P * 4, &full[slot_s], pol);
                  bulk_load(vsd + e * P, a.v_scale + so, P * 4, &full[slot_s], pol);
                }
              }
            }
            if (!kQuant && lane == 0) {
              meta[slot_s] = bad;
              mbar_arrive_expect_tx(&full[slot_s], bytes);
              uint8_t* kdst = stages + slot_s * S::kStageBytes;
              uint8_t* vdst = kdst + S::kOperandBytes;
#pragma unroll
              for (int e = 0; e < PPS; ++e) {
                if (e < n_in && ids[e] >= 0 && ids[e] < a.num_pages) {
                  // One box per page and operand: [D/64 halves][P tokens][64].
                  tma_load_4d(kdst + e * kPageBytes, &tm_k, &full[slot_s], 0, ids[e] * P, 0, head, pol);
                  tma_load_4d(vdst + e * kPageBytes, &tm_v, &full[slot_s], 0, ids[e] * P, 0, head, pol);
                }
              }
            }
            __syncwarp();
            ++stage_it;
          }
        }
      }
      if (!ok) break;
      if (u2 < n_units && it2.seq >= 0) sp2 = a.seqplan[it2.seq];
      u = u1;
      it = it1;
      sp = sp1;
      bt_cur = bt_next;
      u1 = u2;
      it1 = it2;
      sp1 = sp2;
    }
    if (!ok && lane == 0) atomicOr(a.err, VAS_DEV_TIMEOUT);
    pdl_launch_dependents();  // no more work for this CTA: the next kernel may launch
    // Let every copy this warp issued land before the CTA can exit.
    for (uint32_t d = stage_it > kSlots ? stage_it - kSlots : 0; d < stage_it; ++d)
      mbar_wait(&full[d % kSlots], (d / kSlots) & 1);
    return;
  }

  if (kQuant && warp >= kConvWarp0) {
    // ------------------------------ converters ------------------------------
    // Follow the unit ring.  Converter c takes the stages s with s % kConvWarps == c:
    // once the stage's copies have landed (full) it expands the codes in place -- K codes
    // from the upper half of the slot into the K operand, then V codes, all read before
    // any is overwritten, into the V operand -- zeroes the scales past the loaded tokens
    // and past the sequence end (the pool may hold anything there), and marks the stage
    // ready.  kSlots is a multiple of kConvWarps, so each converter waits only on slots
    // it handled last.
    const int cw = warp - kConvWarp0;
    constexpr int kC = D / 16;                           // 16-code chunks per token row
    constexpr int kPer = kStageTokens * kC / 32;  // chunks per lane per operand
    static_assert(32 % kC == 0, "a lane keeps one code chunk of its token rows");
    uint32_t stage_it = 0, unit_it = 0;
    bool ok = true;
    for (;;) {
      const int slot = unit_it % kRing;
      if (!mbar_wait(&ufull[slot], (unit_it / kRing) & 1)) {
        ok = false;
        break;
      }
      const RingEntry re = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&uempty[slot]);
      ++unit_it;
      if (re.u < 0) break;
      const Item it = re.item;
      if (it.seq < 0) continue;
      const int L = re.sp.len;
      const int n_stages = (it.page_end - it.page_begin + PPS - 1) / PPS;
      for (int si = 0; si < n_stages; ++si, ++stage_it) {
        if ((int)(stage_it % kConvWarps) != cw) continue;
        const int slot_s = stage_it % kSlots;
        if (!mbar_wait(&full[slot_s], (stage_it / kSlots) & 1)) {
          ok = false;
          break;
        }
        const int pg = it.page_begin + si * PPS;
        const int loaded = min(PPS, it.page_end - pg) * P;
        const int t_abs0 = pg * P;
        uint8_t* kt = stages + slot_s * S::kStageBytes;
        uint8_t* vt = kt + S::kOperandBytes;
        const uint8_t* kc = kt + S::kCodeOff;
        const uint8_t* vc = kc + kStageTokens * D;
        auto expand = [&](uint4 x, uint4& y0, uint4& y1) {
          if constexpr (KQ == kKvFp8) {
            e4m3x4_to_f16x4(x.x, y0.x, y0.y);
            e4m3x4_to_f16x4(x.y, y0.z, y0.w);
            e4m3x4_to_f16x4(x.z, y1.x, y1.y);
            e4m3x4_to_f16x4(x.w, y1.z, y1.w);
          } else {
            s8x4_to_f16x4(x.x, y0.x, y0.y);
            s8x4_to_f16x4(x.y, y0.z, y0.w);
            s8x4_to_f16x4(x.z, y1.x, y1.y);
            s8x4_to_f16x4(x.w, y1.z, y1.w);
          }
        };
        // Chunk i of this lane: token t0 + (32 / kC) i, code chunk ch (fixed per lane),
        // so every offset below is a per-lane constant plus an immediate.
        const int t0 = lane / kC, ch = lane % kC;
        // K: its codes lie above the K operand, so each chunk goes straight out.
        uint4 xk[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int t = t0 + (32 / kC) * i;
          xk[i] = t < loaded ? *reinterpret_cast<const uint4*>(kc + t * D + ch * 16)
                             : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int t = t0 + (32 / kC) * i;
          if (t < loaded) {
            uint4 y0, y1;
            expand(xk[i], y0, y1);
            *reinterpret_cast<uint4*>(kt + kv_off<D, P>(t, 2 * ch)) = y0;
            *reinterpret_cast<uint4*>(kt + kv_off<D, P>(t, 2 * ch + 1)) = y1;
          }
        }
        // V: its f16 rows cover the K and V codes; read them all first.
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int t = t0 + (32 / kC) * i;
          xk[i] = t < loaded ? *reinterpret_cast<const uint4*>(vc + t * D + ch * 16)
                             : make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int t = t0 + (32 / kC) * i;
          if (t < loaded) {
            uint4 y0, y1;
            expand(xk[i], y0, y1);
            *reinterpret_cast<uint4*>(vt + kv_off<D, P>(t, 2 * ch)) = y0;
            *reinterpret_cast<uint4*>(vt + kv_off<D, P>(t, 2 * ch + 1)) = y1;
          }
        }
        {
          const bool live = lane < loaded && t_abs0 + lane < L;
          float* sc = stage_scales + slot_s * 2 * kStageTokens;
          if (!live) {
            sc[lane] = 0.f;
            sc[kStageTokens + lane] = 0.f;
          }
        }
        fence_proxy_async_smem();  // tcgen05 reads these stages as operands
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[slot_s]);
      }
      if (!ok) break;
    }
    if (!ok && lane == 0) atomicOr(a.err, VAS_DEV_TIMEOUT);
    return;
  }

  if (warp == kMmaWarp) {
    // ------------------------------ MMA warp ------------------------------
    // Follows the unit ring like the consumers.  A wide unit is taken in steps of two
    // 32-token stages (one at an odd end).  For step k (parity b = k & 1), once the
    // consumer warps have written P tile b (bp[b]), it issues O += P_b V in TMEM (M 128
    // lanes, N = D, 16 tokens per product over the step's loaded tokens) and commits
    // to the stages' empty barriers (they may be refilled) and to bo[b].  Lane 0
    // issues; the warp waits together.
    // wk: steps of wide and prompt-chunk units (bp, bo); wc: stages of prompt-chunk units
    // (bs, the S buffers); wq: prompt-chunk units (bq).
    uint32_t stage_it = 0, unit_it = 0, wk = 0, wc = 0, wq = 0;
    bool ok = true;
    constexpr uint32_t kIdO = umma_idesc_bf16(128, D, false, true, kQuant);
    constexpr uint32_t kIdS = umma_idesc_bf16(128, P == 32 ? 32 : 16, false, false, kQuant);
    // All operands are 128-byte swizzled with 1024-byte 8-row groups: the high descriptor
    // word is shared, the low word carries the start address.
    constexpr uint32_t kDescHi = umma_desc_hi_sw128(1024);
    const uint32_t p_lo = umma_desc_lo(smem_u32(scratch + S::kPTileOff), 16);  // P tile 0
    const uint32_t q_lo = umma_desc_lo(smem_u32(scratch + S::kQTileOff), 16);
    constexpr uint32_t kPLoDesc = (S::kPLoOff - S::kPTileOff) >> 4;  // descriptor units
    for (;;) {
      const int slot = unit_it % kRing;
      if (!mbar_wait(&ufull[slot], (unit_it / kRing) & 1)) {
        ok = false;
        break;
      }
      const RingEntry re = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&uempty[slot]);
      ++unit_it;
      if (re.u < 0) break;
      const Item it = re.item;
      if (it.seq < 0) continue;
      const int n_stages = (it.page_end - it.page_begin + PPS - 1) / PPS;
      const int R = a.G * re.sp.qlen;
      const int RB = row_block(R);
      const int r0 = (it.split_rb & ((1 << kRbBits) - 1)) * RB;
      const int Rb = min(RB, R - r0);
      const bool precise = (it.split_rb & kItemPrecise) != 0;
      if (n_stages == 0 || (!precise && RB == kRowBlock && Rb <= kNarrowRows)) {  // consumers alone
        stage_it += n_stages;
        continue;
      }
      if (RB == kRowBlockTc || precise) {
        // A prompt-chunk unit, one step per stage.  S_k = Q K_k^T into S buffer k & 1
        // (M 128 lanes; N the stage's 32 tokens, as two 16-token products with 16-token
        // pages) once the query tile is staged and the stage has landed; O += P_k V_k
        // after bp.  S of stage k + 2 is issued after O of stage k, so its completion also
        // covers that product, the last reader of the P tile stage k + 2 rewrites.
        if (!mbar_wait(bq, wq & 1)) {
          ok = false;
          break;
        }
        ++wq;
        // S_j = Q K_j^T into S buffer (wc + j) & 1, issued by lane 0 once stage j has landed.
        auto s_products = [&](int j) {
          const int slot_s = (stage_it + j) % kSlots;
          const uint32_t k_lo = umma_desc_lo(smem_u32(stages + slot_s * S::kStageBytes), 16);
          const uint32_t dt = tmem + kTmemS + ((wc + j) & 1) * 32;
          // Straight-line issue (a branch between products costs more than a product):
          // every page of the slot, loaded or not -- scores of tokens past the loaded
          // ones are masked by the consumers.
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t qstep = ((ks >> 2) * (128 * 128) + (ks & 3) * 32) >> 4;
#pragma unroll
            for (int e = 0; e < PPS; ++e) {
              const uint32_t kstep = (e * kPageBytes + (ks >> 2) * (P * 128) + (ks & 3) * 32) >> 4;
              umma_bf16_lh(dt + e * P, q_lo + qstep, k_lo + kstep, kDescHi, kIdS, ks > 0);
            }
          }
          umma_commit(&bs[(wc + j) & 1]);
        };
        auto stage_landed = [&](int j) {
          const uint32_t st = stage_it + j;
          return mbar_wait(&stage_ready[st % kSlots], (st / kSlots) & 1);
        };
        // The stage loop comes in two copies: a precise unit adds O += P_lo V after each
        // O += P V (this loop is the issue-bound part of prompt chunks, and a branch in
        // it costs them).  Per stage j: both barriers (P_j written, stage j + 2 landed)
        // are probed first, so that their latencies overlap, then one straight-line
        // issue of O += P_j V_j and S_{j+2}.
        auto stages_pv = [&](auto prec) {
          bool good = stage_landed(0) && (n_stages < 2 || stage_landed(1));
          if (good && lane == 0) {
            tc_fence_after();
            s_products(0);
            if (n_stages > 1) s_products(1);
          }
          __syncwarp();
          for (int j = 0; good && j < n_stages; ++j) {
            const uint32_t k = wk + j, b = k & 1;
            const bool more = j + 2 < n_stages;
            const uint32_t st2 = stage_it + j + 2;
            bool gp = mbar_test_wait(&bp[b], (k >> 1) & 1);
            bool g2 = !more || mbar_test_wait(&stage_ready[st2 % kSlots], (st2 / kSlots) & 1);
            if (!gp) gp = mbar_wait(&bp[b], (k >> 1) & 1);
            if (!g2) g2 = stage_landed(j + 2);
            if (!gp || !g2) {
              good = false;
              break;
            }
            if (lane == 0) {
              tc_fence_after();
              const uint32_t st = stage_it + j;
              const int slot_s = st % kSlots;
              const int pg = it.page_begin + j * PPS;
              const int loaded = min(PPS, it.page_end - pg) * P;
              const uint32_t pb_lo = p_lo + ((b * S::kPTileBytes) >> 4);
              const uint32_t v_lo = umma_desc_lo(
                  smem_u32(stages + slot_s * S::kStageBytes + S::kOperandBytes), P * 128);
              // 16 or 32 loaded tokens (a 32-token page is always whole): the second
              // 16-token product only when its V rows were loaded.
              const bool two = P == 32 || loaded > 16;
              constexpr uint32_t kV1 = tok_off<D, P>(16) >> 4;
              umma_bf16_lh(tmem + kTmemO, pb_lo, v_lo, kDescHi, kIdO, j > 0);
              if (two) umma_bf16_lh(tmem + kTmemO, pb_lo + 2, v_lo + kV1, kDescHi, kIdO, true);
              if constexpr (decltype(prec)::value) {
                umma_bf16_lh(tmem + kTmemO, pb_lo + kPLoDesc, v_lo, kDescHi, kIdO, true);
                if (two) umma_bf16_lh(tmem + kTmemO, pb_lo + kPLoDesc + 2, v_lo + kV1, kDescHi, kIdO, true);
              }
              umma_commit(&empty[slot_s]);
              umma_commit(&bo[b]);
              // S of stage j + 2 after O of stage j: its completion also covers that
              // product, the last reader of the P tile stage j + 2 rewrites.
              if (more) s_products(j + 2);
            }
            __syncwarp();
          }
          return good;
        };
        if constexpr (kQuant) ok = stages_pv(std::false_type{});  // f16 P needs no low part
        else ok = precise ? stages_pv(std::true_type{}) : stages_pv(std::false_type{});
        wk += n_stages;
        wc += n_stages;
        stage_it += n_stages;
        if (!ok) break;
        continue;
      }
      const int n_steps = (n_stages + 1) >> 1;
      for (int j = 0; j < n_steps; ++j) {
        const uint32_t k = wk + j, b = k & 1;
        if (!mbar_wait(&bp[b], (k >> 1) & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t pb_lo = p_lo + ((b * S::kPTileBytes) >> 4);
          // Straight-line issue per stage: 16 or 32 loaded tokens (a 32-token page is
          // always whole).  V (MN-major): 64-column blocks a page half apart, 8-token
          // groups 1024 B.
          constexpr uint32_t kV1 = tok_off<D, P>(16) >> 4;
          auto stage_pv = [&](int h, bool first) {
            const uint32_t st = stage_it + 2 * j + h;
            const int slot_s = st % kSlots;
            const int pg = it.page_begin + (2 * j + h) * PPS;
            const bool two = P == 32 || min(PPS, it.page_end - pg) * P > 16;
            const uint32_t v_lo = umma_desc_lo(
                smem_u32(stages + slot_s * S::kStageBytes + S::kOperandBytes), P * 128);
            const uint32_t pa = pb_lo + ((h * 64) >> 4);
            umma_bf16_lh(tmem + kTmemO, pa, v_lo, kDescHi, kIdO, !first);
            if (two) umma_bf16_lh(tmem + kTmemO, pa + 2, v_lo + kV1, kDescHi, kIdO, true);
            umma_commit(&empty[slot_s]);
          };
          stage_pv(0, j == 0);
          if (2 * j + 1 < n_stages) stage_pv(1, false);
          umma_commit(&bo[b]);
        }
        __syncwarp();
      }
      wk += n_steps;
      stage_it += n_stages;
      if (!ok) break;
    }
    // Tensor memory is freed only after every product this warp issued has completed.
    if (lane == 0) umma_commit(bfin);
    __syncwarp();
    if (!mbar_wait(bfin, 0)) ok = false;
    if (!ok && lane == 0) atomicOr(a.err, VAS_DEV_TIMEOUT);
    tc_fence_before();
    named_bar_sync(2, kConsumerThreads + 32);
    return;
  }

  // -------------------------------- consumers --------------------------------
  const int tid = threadIdx.x;  // 0 .. kConsumerThreads-1
  const int g = lane >> 2, tq = lane & 3;
  const float kLn2 = 0.6931471805599453f;
  uint32_t stage_it = 0, unit_it = 0;
  uint32_t wk = 0;  // steps of wide and prompt-chunk units (the MMA warp counts the same)
  uint32_t wc = 0;  // stages of prompt-chunk units (S buffers, bs)
  bool timed_out = false;
  PendingMerge pm;
  pm.valid = 0;
  pm.old = 0;
  for (;;) {
    const int slot = unit_it % kRing;
    const bool got = mbar_wait(&ufull[slot], (unit_it / kRing) & 1);
    if (tid == 0) *flag = last_split_seen(pm);
    RingEntry re;
    re.u = -1;
    if (got) re = ring[slot];
    // The slot goes back to the producer at once: holding it to the end of the unit caps
    // the producer at kRing units ahead of the oldest unit in flight, which measured
    // slower on long mixed batches.
    __syncwarp();
    if (lane == 0 && got) mbar_arrive(&uempty[slot]);
    ++unit_it;
    // Every consumer warp takes the same decision (a warp that left alone would strand
    // the others at a named barrier); this barrier also frees the scratch area of the
    // previous unit's merge for the next query rows.
    const bool stop = named_bar_or(1, kConsumerThreads, !got);
    finish_pending<D>(a, pm, flag, warp, lane);  // the previous unit's merge, if this CTA was last
    if (stop) {
      timed_out = true;
      break;
    }
    if (re.u < 0) break;
    const Item it = re.item;
    if (it.seq < 0) continue;
    const SeqPlan sp = re.sp;
    const int head = re.head;
    const int split = (it.split_rb & ~kItemPrecise) >> kRbBits;
    const int rb = it.split_rb & ((1 << kRbBits) - 1);
    const bool precise = (it.split_rb & kItemPrecise) != 0;
    const int L = sp.len, ql = sp.qlen;
    const int R = a.G * ql;
    const int RB = row_block(R);
    const int r0 = rb * RB;
    const int Rb = min(RB, R - r0);
    const int n_stages = (it.page_end - it.page_begin + PPS - 1) / PPS;
    const uint32_t stage0 = stage_it;  // first stage of this unit in the CTA's stream
    // Draft tree (at most 64 query tokens; longer chunks keep the causal window): its
    // rows' masks go to shared memory, own bit set, and no stage that reaches the draft
    // window counts as interior.
    const int ctx_end = L - ql;
    const bool tree = tree_unit(a, ql);
    uint64_t* tm = tree ? reinterpret_cast<uint64_t*>(smem + S::kTmaskOff) : nullptr;
    if (tree) {
      const int j = (r0 + tid) / a.G;
      tm[tid] = tid < Rb ? a.tree_mask[sp.qrow0 + j] | (1ull << j) : ~0ull;
    }
    const int min_lim = unit_min_lim(a, L, ql, r0);

    // Prompt-chunk and precise row blocks: tcgen05 S and PV, rows in TMEM lanes.
    const bool chunk = (RB == kRowBlockTc || precise) && n_stages > 0;
    const bool wide = !chunk && Rb > kNarrowRows && n_stages > 0;
    // Quantised pools: Q goes to f16 times qmul = 2^-e, the power of two that brings
    // the unit's largest |q| under 2^15 (1 for any ordinary Q), and the scores are
    // scaled back through cunit.
    float qmul = 1.f, cunit = a.scale_log2;
    if constexpr (kQuant) {
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
      float mx = 0.f;
      for (int c = tid; c < Rb * (D / 8); c += kConsumerThreads)
        mx = fmaxf(mx, absmax_bf16x8(*reinterpret_cast<const uint4*>(
                           qg + out_row(a, sp, head, r0 + c / (D / 8)) * D + (c % (D / 8)) * 8)));
#pragma unroll
      for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) qmax[warp] = mx;
      named_bar_sync(1, kConsumerThreads);
      const float m = fmaxf(fmaxf(qmax[0], qmax[1]), fmaxf(qmax[2], qmax[3]));
      if (m > 32768.f && m <= 3.0e38f) {
        int e;
        frexpf(m, &e);  // m < 2^e
        qmul = ldexpf(1.f, 15 - e);
        cunit = ldexpf(a.scale_log2, e - 15);
      }
    }
    if (chunk) {
      // The query tile for tcgen05 S: rows 0 .. Rb-1 (row r: token r / G, head
      // head * G + r % G) in the K-major 128-byte-swizzled layout.  Rows past Rb keep
      // whatever they held: they only feed accumulator rows that are never read.
      constexpr int kChunks = D / 8;
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
      uint8_t* qt = scratch + S::kQTileOff;
      for (int c = tid; c < Rb * kChunks; c += kConsumerThreads) {
        const int row = c / kChunks, gc = c % kChunks;
        uint4 v = *reinterpret_cast<const uint4*>(qg + out_row(a, sp, head, r0 + row) * D + gc * 8);
        if constexpr (kQuant) v = bf16x8_to_f16x8(v, qmul);
        *reinterpret_cast<uint4*>(qt + (gc >> 3) * (128 * 128) + row * 128 +
                                  (((gc & 7) ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bq);
    } else {
      // Stage the unit's query rows (row r: token r / G, head head * G + r % G); rows
      // past Rb up to the MMA tile are zero.
      constexpr int kChunks = D / 8;
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
      const int rows_pad = Rb <= 8 ? 8 : ((Rb + 15) & ~15);
      for (int c = tid; c < rows_pad * kChunks; c += kConsumerThreads) {
        const int row = c / kChunks, ch = c % kChunks;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < Rb) {
          v = *reinterpret_cast<const uint4*>(qg + out_row(a, sp, head, r0 + row) * D + ch * 8);
          if constexpr (kQuant) v = bf16x8_to_f16x8(v, qmul);
        }
        *reinterpret_cast<uint4*>(scratch + row * S::kQStride + ch * 16) = v;
      }
      named_bar_sync(1, kConsumerThreads);
    }

    bool poison = false;
    if (chunk) {
      // ========================= prompt-chunk unit (tcgen05) =========================
      // Thread r of the consumer warps owns row r of the 128-row block (TMEM lane r).  Per
      // stage it reads its 32 scores from TMEM, applies the causal limit and the online
      // softmax, and writes its probabilities as bf16 into the stage's P tile; the MMA
      // warp accumulates O = P V in TMEM, rescaled here in place when the reference
      // maximum moves.
      const int r = tid;
      const bool row_ok = r < Rb;
      const bool warp_ok = 32 * warp < Rb;
      const int lim = row_ok ? L - ql + (r0 + r) / a.G : -1;
      const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
      const float c = cunit;
      float mref = -INFINITY, l = 0.f;
      for (int si = 0; si < n_stages; ++si, ++stage_it) {
        const uint32_t k = wk + si, b = k & 1, kc = wc + si;
        const int slot_s = stage_it % kSlots;
        // S of this stage is in TMEM; its commit also covers the product that last read
        // P tile b.
        const bool got = mbar_wait_fast(&bs[kc & 1], (kc >> 1) & 1) &&
                         mbar_wait_fast(&stage_ready[slot_s], (stage_it / kSlots) & 1);
        if (!__all_sync(0xffffffffu, got)) {  // the warp leaves together
          timed_out = true;
          stage_it += n_stages - si;
          break;
        }
        tc_fence_after();
        if (meta[slot_s]) poison = true;
        const int pg = it.page_begin + si * PPS;
        const int loaded = min(PPS, it.page_end - pg) * P;
        const int t_abs0 = pg * P;
        if (t_abs0 + loaded > L) {
          // Slots past the sequence end may hold anything (NaN included); their V rows
          // meet P = 0 in the product, so they are zeroed first.
          uint8_t* vt = stages + slot_s * S::kStageBytes + S::kOperandBytes;
          const int z0 = max(0, L - t_abs0);
          for (int cc = z0 * (D / 8) + tid; cc < loaded * (D / 8); cc += kConsumerThreads)
            *reinterpret_cast<uint4*>(vt + kv_off<D, P>(cc / (D / 8), cc % (D / 8))) =
                make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
        }
        if (warp_ok) {
          uint32_t sr[32];
          tmem_ld32(tmem + lane_base + kTmemS + (kc & 1) * 32, sr);
          const float* kss = stage_scales + slot_s * 2 * kStageTokens;  // quantised pools
          if constexpr (kQuant) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 k4 = *reinterpret_cast<const float4*>(kss + i);
              sr[i] = __float_as_uint(__uint_as_float(sr[i]) * k4.x);
              sr[i + 1] = __float_as_uint(__uint_as_float(sr[i + 1]) * k4.y);
              sr[i + 2] = __float_as_uint(__uint_as_float(sr[i + 2]) * k4.z);
              sr[i + 3] = __float_as_uint(__uint_as_float(sr[i + 3]) * k4.w);
            }
          }
          // Valid tokens of this row form a prefix of the stage: i < loaded, t <= lim.
          const int nv = row_ok ? max(0, min(loaded, lim - t_abs0 + 1)) : 0;
          uint32_t valid = nv >= 32 ? 0xffffffffu : (1u << nv) - 1u;
          // Draft tree: token i of the stage is draft token i - d0 when i >= d0.
          const int d0 = ctx_end - t_abs0;
          if (tree && d0 < 32) {
            const uint64_t mr = tm[r];
            valid &= d0 > 0 ? (uint32_t)(mr << d0) | ((1u << d0) - 1u)
                            : (-d0 < 64 ? (uint32_t)(mr >> -d0) : 0u);
          }
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < 32; ++i)
            m4[i & 3] = fmaxf(m4[i & 3], (valid >> i) & 1 ? __uint_as_float(sr[i]) : -INFINITY);
          const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c;  // c > 0
          const bool rebase = mx > mref + kRebase;
          const bool rescale = rebase && si > 0 && mref != -INFINITY;
          const float alpha = rebase ? exp2f(mref - mx) : 1.f;
          if (rebase) {
            l *= alpha;
            mref = mx;
          }
          if (__any_sync(0xffffffffu, rescale)) {
            // O holds the products up to the previous stage: wait for the last of them.
            const uint32_t kp = k - 1;
            if (!mbar_wait(&bo[kp & 1], (kp >> 1) & 1)) timed_out = true;
            tc_fence_after();
            const float f = rescale ? alpha : 1.f;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t ov[32];
              tmem_ld32(tmem + lane_base + kTmemO + cc * 32, ov);
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
              tmem_st32(tmem + lane_base + kTmemO + cc * 32, ov);
            }
          }
          const float mu = mref == -INFINITY ? 0.f : mref;
          uint8_t* prow = scratch + S::kPTileOff + b * S::kPTileBytes + r * 128;
          if constexpr (kQuant)  // f16 P needs no low part
            l += chunk_p_row<D, false, KQ>(sr, valid, c, mu, prow, r, kss + kStageTokens);
          else
            l += precise ? chunk_p_row<D, true, KQ>(sr, valid, c, mu, prow, r, kss + kStageTokens)
                         : chunk_p_row<D, false, KQ>(sr, valid, c, mu, prow, r, kss + kStageTokens);
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bp[b]);
      }
      // The unit's last product (it covers every earlier one).
      if (!timed_out) {
        const uint32_t kl = wk + n_stages - 1;
        if (!mbar_wait(&bo[kl & 1], (kl >> 1) & 1)) timed_out = true;
      }
      wk += n_stages;
      wc += n_stages;
      tc_fence_after();
      poison = named_bar_or(1, kConsumerThreads, poison);
      if (named_bar_or(1, kConsumerThreads, timed_out)) {
        timed_out = true;
        break;
      }
      if (warp_ok) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float row_lse = l > 0.f ? (mref + log2f(l)) * kLn2 : -INFINITY;
        if (poison) row_lse = NAN;
        const bool whole = sp.nsplit == 1;
        const size_t orow = row_ok ? (whole ? out_row(a, sp, head, r0 + r)
                                            : partial_row(a, sp, split, head, r0 + r))
                                   : 0;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kTmemO + cc * 32, ov);
          if (!row_ok) continue;
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = poison ? NAN : __uint_as_float(ov[i]) * inv;
          if (whole) {
            uint4* og = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow * D +
                                                 cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              og[q4] = make_uint4(pack_bf16x2(x[8 * q4], x[8 * q4 + 1]),
                                  pack_bf16x2(x[8 * q4 + 2], x[8 * q4 + 3]),
                                  pack_bf16x2(x[8 * q4 + 4], x[8 * q4 + 5]),
                                  pack_bf16x2(x[8 * q4 + 6], x[8 * q4 + 7]));
          } else {
            float4* po = reinterpret_cast<float4*>(a.part_o + orow * D + cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              po[q4] = make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
          }
        }
        if (row_ok) {
          if (whole) a.lse[orow] = row_lse;
          else a.part_lse[orow] = row_lse;
        }
      }
      tc_fence_before();
    } else if (!wide) {
      // ============================ narrow unit ============================
      auto run = [&](auto nn_tag) {
        constexpr int NN = decltype(nn_tag)::value;
        uint32_t qb[D / 16][NN][2];
#pragma unroll
        for (int kp = 0; kp < D / 32; ++kp)
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) {
            const int row = 8 * nn + (lane & 7);
            const int ch = 4 * kp + (lane >> 3);
            ldsm_x4(smem_u32(scratch + row * S::kQStride + ch * 16), qb[2 * kp][nn][0],
                    qb[2 * kp][nn][1], qb[2 * kp + 1][nn][0],
                    qb[2 * kp + 1][nn][1]);
          }
        uint32_t koff[4], voff[4];
        narrow_offsets<D, P>(lane, koff, voff);
        float oT[D / 16][NN][4];
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
          for (int nn = 0; nn < NN; ++nn) oT[dt][nn][0] = oT[dt][nn][1] = oT[dt][nn][2] = oT[dt][nn][3] = 0.f;
        float m[NN][2], l[NN][2];
        int lim[NN][2];
#pragma unroll
        for (int nn = 0; nn < NN; ++nn)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            m[nn][e] = -INFINITY;
            l[nn][e] = 0.f;
            const int row = 8 * nn + 2 * tq + e;
            lim[nn][e] = row < Rb ? L - ql + (r0 + row) / a.G : L - 1;
          }
        for (int si = 0; si < n_stages; ++si, ++stage_it) {
          if ((int)(stage_it % kConsumerWarps) != warp) continue;
          const int slot_s = stage_it % kSlots;
          if (!mbar_wait(&stage_ready[slot_s], (stage_it / kSlots) & 1)) {
            timed_out = true;
            stage_it += n_stages - si;
            break;
          }
          if (meta[slot_s]) poison = true;
          const int pg = it.page_begin + si * PPS;
          const int loaded = min(PPS, it.page_end - pg) * P;
          const int t_abs0 = pg * P;
          const uint32_t kbase = smem_u32(stages + slot_s * S::kStageBytes);
          const uint32_t vbase = kbase + S::kOperandBytes;
          if (t_abs0 + loaded > L) {
            // Pool slots past the end of the sequence may hold anything: zero their V
            // rows so that a zero attention weight cannot meet a NaN.
            uint8_t* vrow = stages + slot_s * S::kStageBytes + S::kOperandBytes;
            const int z0 = max(0, L - t_abs0);
            for (int c = z0 * (D / 8) + lane; c < loaded * (D / 8); c += 32)
              *reinterpret_cast<uint4*>(vrow + kv_off<D, P>(c / (D / 8), c % (D / 8))) =
                  make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            __syncwarp();
          }
          const float* kss = kQuant ? stage_scales + slot_s * 2 * kStageTokens : nullptr;
          const float* vss = kQuant ? kss + kStageTokens : nullptr;
          if (loaded == kStageTokens && t_abs0 + kStageTokens - 1 <= min_lim)
            narrow_stage<D, P, NN, false, KQ>(kbase, vbase, loaded, qb, koff, voff, oT, m, l,
                                              t_abs0, lim, cunit, lane, tm, ctx_end, kss, vss);
          else
            narrow_stage<D, P, NN, true, KQ>(kbase, vbase, loaded, qb, koff, voff, oT, m, l,
                                             t_abs0, lim, cunit, lane, tm, ctx_end, kss, vss);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot_s]);
        }
#pragma unroll
        for (int nn = 0; nn < NN; ++nn)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            l[nn][e] += __shfl_xor_sync(0xffffffffu, l[nn][e], 4);
            l[nn][e] += __shfl_xor_sync(0xffffffffu, l[nn][e], 8);
            l[nn][e] += __shfl_xor_sync(0xffffffffu, l[nn][e], 16);
          }
        // Merge the four warps' states through shared memory.
        named_bar_sync(1, kConsumerThreads);  // all warps are done with the Q rows
        float* wb = reinterpret_cast<float*>(scratch) + (size_t)warp * S::kNarrowWarpFloats;
        // Rows a warp never touched keep m = -inf, l = 0 and contribute nothing.
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
          for (int nn = 0; nn < NN; ++nn)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wb[(8 * nn + 2 * tq + (e & 1)) * S::kNarrowStride + 16 * dt + g + 8 * (e >> 1)] =
                  oT[dt][nn][e];
        if (g == 0)
#pragma unroll
          for (int nn = 0; nn < NN; ++nn)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              wb[kNarrowRows * S::kNarrowStride + 8 * nn + 2 * tq + e] = m[nn][e];
              wb[kNarrowRows * S::kNarrowStride + kNarrowRows + 8 * nn + 2 * tq + e] = l[nn][e];
            }
      };
      if (Rb <= 8) run(std::integral_constant<int, 1>{});
      else run(std::integral_constant<int, 2>{});
      // Bad pages and timeouts seen by any warp's stages concern the whole unit.
      poison = named_bar_or(1, kConsumerThreads, poison);
      if (named_bar_or(1, kConsumerThreads, timed_out)) {
        timed_out = true;
        break;
      }
      const float* buf = reinterpret_cast<const float*>(scratch);
      // Per row: the weight of each warp's partition and 1 / l, one thread per row; then
      // every lane writes its column of each row.
      // Warp w took the stages with (stage0 + si) % 4 == w.  Summing the partitions in
      // the order of si % 4, not of w, makes the result independent of stage0, i.e. of
      // which units this CTA happened to run before: reruns are bit-identical.
      float* coef = reinterpret_cast<float*>(scratch + S::kNarrowBytes);  // [row][8]
      if (tid < Rb) {
        const int r = tid;
        float mw[kConsumerWarps], M = -INFINITY;
#pragma unroll
        for (int pt = 0; pt < kConsumerWarps; ++pt) {
          const int w = (stage0 + pt) % kConsumerWarps;
          mw[pt] = buf[w * S::kNarrowWarpFloats + kNarrowRows * S::kNarrowStride + r];
          M = fmaxf(M, mw[pt]);
        }
        const float mu = M == -INFINITY ? 0.f : M;
        float Lsum = 0.f;
#pragma unroll
        for (int pt = 0; pt < kConsumerWarps; ++pt) {
          const int w = (stage0 + pt) % kConsumerWarps;
          const float f = exp2f(mw[pt] - mu);
          Lsum += f * buf[w * S::kNarrowWarpFloats + kNarrowRows * S::kNarrowStride + kNarrowRows + r];
          coef[r * 8 + pt] = f;
        }
        coef[r * 8 + 4] = Lsum > 0.f ? 1.f / Lsum : 0.f;
        float row_lse = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
        if (poison) row_lse = NAN;
        if (sp.nsplit == 1) a.lse[out_row(a, sp, head, r0 + r)] = row_lse;
        else a.part_lse[partial_row(a, sp, split, head, r0 + r)] = row_lse;
      }
      named_bar_sync(1, kConsumerThreads);
      const int d = warp * 32 + lane;  // this lane's output column
      if (d < D) {
#pragma unroll 1
        for (int r = 0; r < Rb; ++r) {
          const float4 f = *reinterpret_cast<const float4*>(coef + r * 8);
          const float fw[kConsumerWarps] = {f.x, f.y, f.z, f.w};
          float acc = 0.f;
#pragma unroll
          for (int pt = 0; pt < kConsumerWarps; ++pt) {
            const int w = (stage0 + pt) % kConsumerWarps;
            acc = fmaf(fw[pt], buf[w * S::kNarrowWarpFloats + r * S::kNarrowStride + d], acc);
          }
          const float x = poison ? NAN : acc * coef[r * 8 + 4];
          if (sp.nsplit == 1)
            static_cast<__nv_bfloat16*>(a.out)[out_row(a, sp, head, r0 + r) * D + d] = __float2bfloat16(x);
          else
            a.part_o[partial_row(a, sp, split, head, r0 + r) * D + d] = x;
        }
      }
    } else {
      // ============================= wide unit =============================
      // Warp w < nM owns m16 row tile w (rows 16 w .. 16 w + 15): S = Q K^T by warp MMA
      // and the softmax in registers, P into tile rows 32 w + (0 .. 15) (TMEM lanes of
      // this warp).  The MMA warp accumulates O = P V in TMEM with tcgen05; thread t < 16
      // of warp w reads, rescales and finally writes O row 16 w + t.
      const int nM = (Rb + 15) >> 4;
      const bool active = warp < nM;
      const int g = lane >> 2;
      uint32_t qa[D / 16][4];
      if (active) {
        const int mi = lane >> 3;
        const int row = 16 * warp + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int ch = 2 * ks + (mi >> 1);
          ldsm_x4(smem_u32(scratch + row * S::kQStride + ch * 16), qa[ks][0], qa[ks][1],
                  qa[ks][2], qa[ks][3]);
        }
      }
      uint32_t kw[2];
      wide_offsets<D, P>(lane, kw);
      named_bar_sync(1, kConsumerThreads);  // the query staging becomes the P tiles
      const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
      float mref[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
      const int rA = r0 + 16 * warp + g, rB = rA + 8;
      const int limA = rA < R ? L - ql + rA / a.G : L - 1;
      const int limB = rB < R ? L - ql + rB / a.G : L - 1;
      const uint64_t* tmw = tm ? tm + 16 * warp + g : nullptr;
      const int n_steps = (n_stages + 1) >> 1;
      for (int sj = 0; sj < n_steps; ++sj) {
        const uint32_t k = wk + sj, b = k & 1;
        const int nst = min(2, n_stages - 2 * sj);
        // Both stages of the step are loaded (and their V rows past the sequence end
        // zeroed: those slots may hold anything, NaN included, and meet P = 0).
        uint32_t kb[2];
        const float* ksp[2] = {nullptr, nullptr};  // quantised pools: the stages' scales
        int loaded = 0;
        bool got = true;
        const int t_abs0 = (it.page_begin + 2 * sj * PPS) * P;
        for (int h = 0; h < nst; ++h) {
          const uint32_t st = stage_it + h;
          const int slot_s = st % kSlots;
          got = got && mbar_wait_fast(&stage_ready[slot_s], (st / kSlots) & 1);
          if (meta[slot_s]) poison = true;
          const int pg = it.page_begin + (2 * sj + h) * PPS;
          const int ld = min(PPS, it.page_end - pg) * P;
          kb[h] = smem_u32(stages + slot_s * S::kStageBytes);
          ksp[h] = stage_scales + slot_s * 2 * kStageTokens;
          const int ta = pg * P;
          if (ta + ld > L) {
            uint8_t* vt = stages + slot_s * S::kStageBytes + S::kOperandBytes;
            const int z0 = max(0, L - ta);
            for (int cc = z0 * (D / 8) + tid; cc < ld * (D / 8); cc += kConsumerThreads)
              *reinterpret_cast<uint4*>(vt + kv_off<D, P>(cc / (D / 8), cc % (D / 8))) =
                  make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
          loaded += ld;
        }
        if (nst == 1) {
          kb[1] = kb[0];
          ksp[1] = ksp[0];
        }
        if (!__all_sync(0xffffffffu, got)) {  // the warp leaves together
          timed_out = true;
          stage_it += n_stages - 2 * sj;
          break;
        }
        stage_it += nst;
        // P tile b was last read by the product two steps back.  Every warp waits for
        // it, idle ones included: a warp that arrived on bp[b] for step k before that
        // product was issued would be counted in the phase of step k - 2.
        if (k >= 2 && !mbar_wait_fast(&bo[b], ((k - 2) >> 1) & 1)) timed_out = true;
        if (active) {
          tc_fence_after();
          uint8_t* prow = scratch + S::kPTileOff + b * S::kPTileBytes + (32 * warp + g) * 128;
          // Masking is a runtime switch: a separate unmasked instantiation would cost the
          // whole kernel register spills.
          const bool masked = loaded < 2 * kStageTokens || t_abs0 + 2 * kStageTokens - 1 > min_lim;
          float alpha[2];
          bool rescale;
          if (nst == 2)
            wide_s_step<D, P, 2, KQ>(kb, loaded, masked, qa, kw, mref, l, alpha, rescale, t_abs0,
                                     limA, limB, cunit, lane, prow, tmw, ctx_end, ksp[0], ksp[1],
                                     ksp[0] + kStageTokens, ksp[1] + kStageTokens);
          else
            wide_s_step<D, P, 1, KQ>(kb, loaded, true, qa, kw, mref, l, alpha, rescale, t_abs0,
                                     limA, limB, cunit, lane, prow, tmw, ctx_end, ksp[0], ksp[1],
                                     ksp[0] + kStageTokens, ksp[1] + kStageTokens);
          if (__any_sync(0xffffffffu, rescale && sj > 0)) {
            // O holds the products up to the previous step: wait for the last of them,
            // then scale row 16 w + t (lane t < 16) by its factor (held by lane 4 (t % 8)).
            const uint32_t kp = k - 1;
            if (!mbar_wait(&bo[kp & 1], (kp >> 1) & 1)) timed_out = true;
            tc_fence_after();
            const float f0 = __shfl_sync(0xffffffffu, alpha[0], 4 * (lane & 7));
            const float f1 = __shfl_sync(0xffffffffu, alpha[1], 4 * (lane & 7));
            const float f = lane < 8 ? f0 : (lane < 16 ? f1 : 1.f);
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t ov[32];
              tmem_ld32(tmem + lane_base + kTmemO + cc * 32, ov);
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
              tmem_st32(tmem + lane_base + kTmemO + cc * 32, ov);
            }
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bp[b]);
      }
      // The unit's last product (it covers every earlier one).
      if (!timed_out) {
        const uint32_t kl = wk + n_steps - 1;
        if (!mbar_wait(&bo[kl & 1], (kl >> 1) & 1)) timed_out = true;
      }
      wk += n_steps;
      tc_fence_after();
      poison = named_bar_or(1, kConsumerThreads, poison);
      if (named_bar_or(1, kConsumerThreads, timed_out)) {
        timed_out = true;
        break;
      }
      if (active) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
          l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
        }
        // Lane t < 16 writes row 16 w + t: its (m, l) from lane 4 (t % 8), half t / 8.
        const float mA = __shfl_sync(0xffffffffu, mref[0], 4 * (lane & 7));
        const float mB = __shfl_sync(0xffffffffu, mref[1], 4 * (lane & 7));
        const float lA = __shfl_sync(0xffffffffu, l[0], 4 * (lane & 7));
        const float lB = __shfl_sync(0xffffffffu, l[1], 4 * (lane & 7));
        const float mm = lane < 8 ? mA : mB, ll = lane < 8 ? lA : lB;
        const int rr = 16 * warp + lane;
        const bool row_ok = lane < 16 && rr < Rb;
        const float inv = ll > 0.f ? 1.f / ll : 0.f;
        float row_lse = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
        if (poison) row_lse = NAN;
        const bool whole = sp.nsplit == 1;
        const size_t orow = row_ok ? (whole ? out_row(a, sp, head, r0 + rr)
                                            : partial_row(a, sp, split, head, r0 + rr))
                                   : 0;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kTmemO + cc * 32, ov);
          if (!row_ok) continue;
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = poison ? NAN : __uint_as_float(ov[i]) * inv;
          if (whole) {
            uint4* og = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow * D +
                                                 cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              og[q4] = make_uint4(pack_bf16x2(x[8 * q4], x[8 * q4 + 1]),
                                  pack_bf16x2(x[8 * q4 + 2], x[8 * q4 + 3]),
                                  pack_bf16x2(x[8 * q4 + 4], x[8 * q4 + 5]),
                                  pack_bf16x2(x[8 * q4 + 6], x[8 * q4 + 7]));
          } else {
            float4* po = reinterpret_cast<float4*>(a.part_o + orow * D + cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              po[q4] = make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
          }
        }
        if (row_ok) {
          if (whole) a.lse[orow] = row_lse;
          else a.part_lse[orow] = row_lse;
        }
      }
      tc_fence_before();
    }
    if (poison && tid == 0) atomicOr(a.err, VAS_DEV_BAD_PAGE);
    if (sp.nsplit > 1) count_split_arrival(a, sp, it, head, r0, Rb, pm);
  }
  if (timed_out && lane == 0) atomicOr(a.err, VAS_DEV_TIMEOUT);
  // Tensor memory goes back once the MMA warp has seen its last product complete.
  tc_fence_before();
  named_bar_sync(2, kConsumerThreads + 32);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------
// Attention, fp32 storage: one warp per query row on the CUDA cores (no split)
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) attn_f32_kernel(const AttnArgs a) {
  constexpr int E = D / 32;  // elements per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* qg = static_cast<const float*>(a.q);
  const float* kp = static_cast<const float*>(a.k_pages);
  const float* vp = static_cast<const float*>(a.v_pages);
  float* og = static_cast<float*>(a.out);
  __shared__ float qs[4][D];
  pdl_wait_prior_grid();
  const int32_t n_units = a.header->n_items * a.Hkv;
  for (int32_t u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Item it = a.items[a.order[u / a.Hkv]];
    if (it.seq < 0) continue;
    const int head = u % a.Hkv;
    const SeqPlan sp = a.seqplan[it.seq];
    const int rb = it.split_rb & ((1 << kRbBits) - 1);
    const int L = sp.len, ql = sp.qlen, R = a.G * ql;
    const int32_t* bt_row = a.block_table + (size_t)it.seq * a.maxp;
    const int RB = row_block(R);
    for (int r = rb * RB + warp; r < min(R, rb * RB + RB); r += 4) {
      const int j = r / a.G;
      const int pos = L - ql + j;
      const size_t orow = out_row(a, sp, head, r);
      // Draft tree: among the draft tokens (positions from L - ql on) only the ancestors
      // and the token itself are visible.
      const bool tree = tree_unit(a, ql);
      const uint64_t vis = tree ? a.tree_mask[sp.qrow0 + j] | (1ull << j) : ~0ull;
      __syncwarp();
#pragma unroll
      for (int e = 0; e < E; ++e) qs[warp][lane + 32 * e] = qg[orow * D + lane + 32 * e];
      __syncwarp();
      float acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.f;
      float mrun = -INFINITY, lrun = 0.f;
      bool bad = false;
      for (int t0 = 0; t0 <= pos; t0 += 32) {
        const int t = t0 + lane;
        int page = -1;
        float sc = -INFINITY;
        if (t <= pos) {
          page = bt_row[t / a.P];
          if (page < 0 || page >= a.num_pages) {
            bad = true;
            page = -1;
          } else if (t >= L - ql && !((vis >> ((t - (L - ql)) & 63)) & 1)) {
            page = -1;  // outside the tree: no score, no value row
          } else {
            const float* krow = kp + (((size_t)page * a.P + t % a.P) * a.Hkv + head) * D;
            float dot = 0.f;
            for (int d = 0; d < D; ++d) dot = fmaf(qs[warp][d], krow[d], dot);
            sc = dot * a.scale;
          }
        }
        float bm = sc;
#pragma unroll
        for (int off = 16; off; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
        const float mnew = fmaxf(mrun, bm);
        const float mu = mnew == -INFINITY ? 0.f : mnew;
        const float alpha = expf(mrun - mu);
        const float p = expf(sc - mu);
        float ps = p;
#pragma unroll
        for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        lrun = lrun * alpha + ps;
        mrun = mnew;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= alpha;
        const int nt = min(32, pos + 1 - t0);
        for (int tt = 0; tt < nt; ++tt) {
          const float pt = __shfl_sync(0xffffffffu, p, tt);
          const int pg = __shfl_sync(0xffffffffu, page, tt);
          if (pg < 0) continue;
          const int ta = t0 + tt;
          const float* vrow = vp + (((size_t)pg * a.P + ta % a.P) * a.Hkv + head) * D;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(pt, vrow[lane + 32 * e], acc[e]);
        }
      }
      bad = __any_sync(0xffffffffu, bad);
      const float inv = 1.f / lrun;
#pragma unroll
      for (int e = 0; e < E; ++e) og[orow * D + lane + 32 * e] = bad ? NAN : acc[e] * inv;
      if (lane == 0) {
        a.lse[orow] = bad ? NAN : mrun + logf(lrun);
        if (bad) atomicOr(a.err, VAS_DEV_BAD_PAGE);
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------
bool dims_ok(const vas_attn_dims* d) {
  if (!d) return false;
  if (d->num_seqs < 0 || d->total_q_tokens < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0)
    return false;
  if (d->num_q_heads % d->num_kv_heads) return false;
  if (d->num_pages < 0 || d->max_pages_per_seq < 0) return false;
  if (!(d->scale >= 0.f) || std::isinf(d->scale)) return false;
  if ((int64_t)d->total_q_tokens * d->num_q_heads > INT32_MAX) return false;
  return true;
}

bool dims_supported(const vas_attn_dims* d) {
  return (d->head_dim == 64 || d->head_dim == 128) && (d->page_size == 16 || d->page_size == 32) &&
         (d->kv_dtype == VAS_BF16 || d->kv_dtype == VAS_F32 || d->kv_dtype == VAS_FP8_E4M3 ||
          d->kv_dtype == VAS_INT8);
}

bool kv_quantized(const vas_attn_dims* d) {
  return d->kv_dtype == VAS_FP8_E4M3 || d->kv_dtype == VAS_INT8;
}

int64_t items_min(const vas_attn_dims* d) {
  const int64_t G = d->num_q_heads / d->num_kv_heads;
  return (int64_t)d->num_seqs + (G * d->total_q_tokens + kRowBlock - 1) / kRowBlock + 1;
}

int64_t items_extra(int sms) { return 4LL * kUnitsPerSm * (sms > 0 ? sms : 160); }

Layout make_layout(const vas_attn_dims* d, int64_t items_cap, int64_t partial_cap) {
  Layout L;
  size_t off = align_up(sizeof(PlanHeader), 256);
  L.seqplan = off;
  off = align_up(off + (size_t)d->num_seqs * sizeof(SeqPlan), 256);
  L.token_seq = off;
  off = align_up(off + (size_t)d->total_q_tokens * 4, 256);
  L.items = off;
  off = align_up(off + (size_t)items_cap * sizeof(Item), 256);
  L.order = off;
  off = align_up(off + (size_t)items_cap * 4, 256);
  L.counters = off;
  off = align_up(off + (size_t)items_cap * d->num_kv_heads * 4, 256);
  L.part_lse = off;
  off = align_up(off + (size_t)partial_cap * 4, 256);
  L.part_o = off;
  off = align_up(off + (size_t)partial_cap * d->head_dim * 4, 256);
  L.total = off;
  L.items_cap = items_cap;
  L.partial_cap = partial_cap;
  return L;
}

// Largest layout that fits ws_bytes (partial capacity grows with the workspace).
bool fit_layout(const vas_attn_dims* d, size_t ws_bytes, Layout* out) {
  const int64_t imin = items_min(d);
  const int64_t icap_pref = imin + items_extra(num_sms());
  for (int64_t icap : {icap_pref, imin}) {
    const Layout base = make_layout(d, icap, 0);
    if (base.total > ws_bytes) continue;
    const size_t per_row = (size_t)(d->head_dim + 1) * 4;
    int64_t pcap = (int64_t)((ws_bytes - base.total) / per_row);
    while (pcap > 0 && make_layout(d, icap, pcap).total > ws_bytes) pcap -= 64;
    if (pcap < 0) pcap = 0;
    if (pcap > INT32_MAX) pcap = INT32_MAX;
    *out = make_layout(d, icap, pcap);
    return true;
  }
  return false;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D view of a page pool with the token before the column half:
// (64, num_pages * P, D/64, Hkv), strides (Hkv*D*2, 128, D*2) bytes, 128-byte swizzle.
// A box of (64, P, D/64, 1) -- one page of one KV head -- then lands as
// [half][token][64].
bool encode_pool_map(CUtensorMap* map, const void* base, const vas_attn_dims* d) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {64, (cuuint64_t)d->num_pages * d->page_size,
                              (cuuint64_t)d->head_dim / 64, (cuuint64_t)d->num_kv_heads};
  const cuuint64_t strides[3] = {(cuuint64_t)d->num_kv_heads * d->head_dim * 2, 128,
                                 (cuuint64_t)d->head_dim * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)d->page_size, (cuuint32_t)d->head_dim / 64, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of an 8-bit code pool: (D bytes, num_pages * P tokens, Hkv), strides
// (Hkv*D, D) bytes, no swizzle.  A box of (D, P, 1) -- one page of one KV head -- lands
// as [P tokens][D bytes].
bool encode_code_map(CUtensorMap* map, const void* base, const vas_attn_dims* d) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d->head_dim, (cuuint64_t)d->num_pages * d->page_size,
                              (cuuint64_t)d->num_kv_heads};
  const cuuint64_t strides[2] = {(cuuint64_t)d->num_kv_heads * d->head_dim,
                                 (cuuint64_t)d->head_dim};
  const cuuint32_t box[3] = {(cuuint32_t)d->head_dim, (cuuint32_t)d->page_size, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            // a token row of one head is D <= 128 bytes: 256-byte promotion would fetch
            // the next head's row too (measured: 5.8 GB of DRAM reads for 4.3 GB of codes)
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int P, int KQ>
int launch_bf16(const CUtensorMap& mk, const CUtensorMap& mv, const AttnArgs& args, int grid,
                cudaStream_t stream) {
  using S = Smem<D, KQ>;
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VAS_E_CUDA;
  std::call_once(once[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(attn_bf16_kernel<D, P, KQ>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              S::kDynBytes);
  });
  if (attr_err[dev & 63] != cudaSuccess) return VAS_E_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(KQ == kKvBf16 ? kThreads : kThreadsQ);
  cfg.dynamicSmemBytes = S::kDynBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, attn_bf16_kernel<D, P, KQ>, mk, mv, args) != cudaSuccess) {
    cudaGetLastError();
    return VAS_E_CUDA;
  }
  return VAS_OK;
}

}  // namespace attn
}  // namespace vas

using namespace vas::attn;

extern "C" {

size_t paged_attn_workspace_min(const vas_attn_dims* dims) {
  if (!dims_ok(dims) || !dims_supported(dims)) return 0;
  return make_layout(dims, items_min(dims), 0).total;
}

size_t paged_attn_workspace_size(const vas_attn_dims* dims) {
  if (!dims_ok(dims) || !dims_supported(dims)) return 0;
  // Room for every output row to be split 8 ways on average.
  const int64_t pcap = (int64_t)dims->total_q_tokens * dims->num_q_heads * 8;
  return make_layout(dims, items_min(dims) + items_extra(vas::num_sms()),
                     pcap < INT32_MAX ? pcap : INT32_MAX)
      .total;
}

}  // extern "C"

namespace {

int attn_launch(const void* q, const void* k_pages, const void* v_pages, const float* k_scale,
                const float* v_scale, const int32_t* block_table, const int32_t* seq_lens,
                const int32_t* query_lens, const uint64_t* tree_mask, void* out, float* lse,
                const vas_attn_dims* dims, void* workspace, size_t workspace_bytes,
                vas_stream_t stream_) {
  if (!dims_ok(dims)) return VAS_E_INVALID_ARG;
  if (!dims_supported(dims)) return VAS_E_UNSUPPORTED;
  const vas_attn_dims& d = *dims;
  const bool quant = kv_quantized(dims);
  // Quantised pools need their scales; the other storage types take none.
  if (quant != (k_scale != nullptr) || quant != (v_scale != nullptr)) return VAS_E_INVALID_ARG;
  if (d.num_seqs == 0 || d.total_q_tokens == 0) return VAS_OK;
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !query_lens || !out || !lse ||
      !workspace)
    return VAS_E_INVALID_ARG;
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k_pages, 16) || mis(v_pages, 16) || mis(out, 16) || mis(lse, 4) ||
      mis(block_table, 4) || mis(seq_lens, 4) || mis(query_lens, 4) || mis(workspace, 256) ||
      mis(tree_mask, 8) || mis(k_scale, 16) || mis(v_scale, 16))
    return VAS_E_INVALID_ARG;
  if (d.num_pages == 0 || d.max_pages_per_seq == 0) return VAS_E_INVALID_ARG;
  if ((int64_t)d.num_pages * d.page_size > INT32_MAX) return VAS_E_INVALID_ARG;

  Layout lay;
  if (!fit_layout(dims, workspace_bytes, &lay)) return VAS_E_WORKSPACE;
  int32_t* err = vas::device_error_word();
  const int sms = vas::num_sms();
  if (!err || !sms) return VAS_E_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  const int G = d.num_q_heads / d.num_kv_heads;
  const bool bf16 = d.kv_dtype != VAS_F32;  // the tensor-core kernel; out and q are bf16
  PlanArgs pa;
  pa.seq_lens = seq_lens;
  pa.query_lens = query_lens;
  pa.seqplan = reinterpret_cast<SeqPlan*>(ws + lay.seqplan);
  pa.token_seq = reinterpret_cast<int32_t*>(ws + lay.token_seq);
  pa.items = reinterpret_cast<Item*>(ws + lay.items);
  pa.order = reinterpret_cast<int32_t*>(ws + lay.order);
  pa.header = reinterpret_cast<PlanHeader*>(ws);
  pa.counters = reinterpret_cast<int32_t*>(ws + lay.counters);
  pa.out = out;
  pa.lse = lse;
  pa.B = d.num_seqs;
  pa.T = d.total_q_tokens;
  pa.G = G;
  pa.Hkv = d.num_kv_heads;
  pa.Hq = d.num_q_heads;
  pa.D = d.head_dim;
  pa.P = d.page_size;
  pa.maxp = d.max_pages_per_seq;
  pa.pps = kStageTokens / d.page_size;
  // A split of fewer than 32 stages (1024 tokens) costs more in per-unit latency (query
  // staging, the partial written and merged) than it returns in balance across SMs.
  pa.min_chunk = 32 * pa.pps;
  pa.no_split = bf16 ? 0 : 1;
  pa.target_units = kSplitTargetPerSm * sms;
  pa.is_bf16 = bf16 ? 1 : 0;
  pa.tree_mask = tree_mask;
  pa.items_cap = lay.items_cap;
  pa.partial_cap = lay.partial_cap;
  pa.err = err;
  // Tensor maps first, so that the plan and the attention grid are launched back to back.
  CUtensorMap mk, mv;
  if (quant && (!encode_code_map(&mk, k_pages, dims) || !encode_code_map(&mv, v_pages, dims)))
    return VAS_E_CUDA;
  if (!quant && bf16 &&
      (!encode_pool_map(&mk, k_pages, dims) || !encode_pool_map(&mv, v_pages, dims)))
    return VAS_E_CUDA;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, plan_kernel, pa) != cudaSuccess) {
      cudaGetLastError();
      return VAS_E_CUDA;
    }
  }

  const float scale = d.scale > 0.f ? d.scale : 1.0f / std::sqrt((float)d.head_dim);
  AttnArgs aa;
  aa.q = q;
  aa.out = out;
  aa.lse = lse;
  aa.block_table = block_table;
  aa.seqplan = pa.seqplan;
  aa.items = pa.items;
  aa.order = pa.order;
  aa.header = pa.header;
  aa.counters = pa.counters;
  aa.part_o = reinterpret_cast<float*>(ws + lay.part_o);
  aa.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  aa.k_pages = k_pages;
  aa.v_pages = v_pages;
  aa.T = d.total_q_tokens;
  aa.Hq = d.num_q_heads;
  aa.Hkv = d.num_kv_heads;
  aa.G = G;
  aa.maxp = d.max_pages_per_seq;
  aa.num_pages = d.num_pages;
  aa.P = d.page_size;
  aa.scale = scale;
  aa.scale_log2 = scale * 1.4426950408889634f;
  aa.err = err;
  aa.tree_mask = tree_mask;
  aa.k_scale = k_scale;
  aa.v_scale = v_scale;

  if (quant) {
    const int grid = sms;
    const bool fp8 = d.kv_dtype == VAS_FP8_E4M3;
    if (d.head_dim == 128 && d.page_size == 16)
      return fp8 ? launch_bf16<128, 16, kKvFp8>(mk, mv, aa, grid, stream)
                 : launch_bf16<128, 16, kKvInt8>(mk, mv, aa, grid, stream);
    if (d.head_dim == 128)
      return fp8 ? launch_bf16<128, 32, kKvFp8>(mk, mv, aa, grid, stream)
                 : launch_bf16<128, 32, kKvInt8>(mk, mv, aa, grid, stream);
    if (d.page_size == 16)
      return fp8 ? launch_bf16<64, 16, kKvFp8>(mk, mv, aa, grid, stream)
                 : launch_bf16<64, 16, kKvInt8>(mk, mv, aa, grid, stream);
    return fp8 ? launch_bf16<64, 32, kKvFp8>(mk, mv, aa, grid, stream)
               : launch_bf16<64, 32, kKvInt8>(mk, mv, aa, grid, stream);
  }
  if (bf16) {
    const int grid = sms;
    if (d.head_dim == 128 && d.page_size == 16)
      return launch_bf16<128, 16, kKvBf16>(mk, mv, aa, grid, stream);
    if (d.head_dim == 128) return launch_bf16<128, 32, kKvBf16>(mk, mv, aa, grid, stream);
    if (d.page_size == 16) return launch_bf16<64, 16, kKvBf16>(mk, mv, aa, grid, stream);
    return launch_bf16<64, 32, kKvBf16>(mk, mv, aa, grid, stream);
  }
  const int grid = 4 * sms;
  if (d.head_dim == 128) attn_f32_kernel<128><<<grid, 128, 0, stream>>>(aa);
  else attn_f32_kernel<64><<<grid, 128, 0, stream>>>(aa);
  return cudaGetLastError() == cudaSuccess ? VAS_OK : VAS_E_CUDA;
}

}  // namespace

extern "C" {

int paged_attn_fwd(const void* q, const void* k_pages, const void* v_pages,
                   const int32_t* block_table, const int32_t* seq_lens,
                   const int32_t* query_lens, void* out, float* lse,
                   const vas_attn_dims* dims, void* workspace, size_t workspace_bytes,
                   vas_stream_t stream) {
  return attn_launch(q, k_pages, v_pages, nullptr, nullptr, block_table, seq_lens, query_lens,
                     nullptr, out, lse, dims, workspace, workspace_bytes, stream);
}

int paged_attn_fwd_tree(const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, const int32_t* seq_lens,
                        const int32_t* query_lens, const uint64_t* tree_mask, void* out,
                        float* lse, const vas_attn_dims* dims, void* workspace,
                        size_t workspace_bytes, vas_stream_t stream) {
  if (!tree_mask) return VAS_E_INVALID_ARG;
  return attn_launch(q, k_pages, v_pages, nullptr, nullptr, block_table, seq_lens, query_lens,
                     tree_mask, out, lse, dims, workspace, workspace_bytes, stream);
}

int paged_attn_fwd_quant(const void* q, const void* k_pages, const void* v_pages,
                         const float* k_scale, const float* v_scale, const int32_t* block_table,
                         const int32_t* seq_lens, const int32_t* query_lens,
                         const uint64_t* tree_mask, void* out, float* lse,
                         const vas_attn_dims* dims, void* workspace, size_t workspace_bytes,
                         vas_stream_t stream) {
  if (!dims || !kv_quantized(dims) || !k_scale || !v_scale) return VAS_E_INVALID_ARG;
  return attn_launch(q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, query_lens,
                     tree_mask, out, lse, dims, workspace, workspace_bytes, stream);
}

}  // extern "C"
