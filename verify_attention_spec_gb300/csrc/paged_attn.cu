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
//                       length in pages and writes the work list (sequence, page range,
//                       split, row block) to the workspace.
//   2. attn_bf16_kernel persistent, one CTA per SM.  A producer warp takes work units
//                       (work item x KV head) from an atomic counter and streams the
//                       unit's K/V page slices into a 4-stage shared-memory ring with
//                       TMA (one 3-D box per 128-byte column half of a page), tracked by
//                       mbarriers.  Four consumer warps run QK^T and PV on the tensor
//                       cores (mma.sync m16n8k16 bf16 -> fp32) with an online softmax;
//                       the GQA group x query tokens of one KV head form the MMA rows.
//                       A unit that covers its whole sequence writes out/lse directly;
//                       otherwise it writes a normalised fp32 partial and its lse.
//      attn_f32_kernel  fp32 storage: CUDA-core FMA, one warp per query row.
//   3. combine_kernel   merges the partials of split sequences by their lse
//                       (O = sum_s e^{lse_s - m} O_s / sum_s e^{lse_s - m},
//                       lse = m + ln sum_s e^{lse_s - m}) and NaN-fills rows that a
//                       device-detected error left undefined.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/vas.h"
#include "device_util.cuh"
#include "vas_internal.h"

namespace vas {
namespace attn {

constexpr int kStageTokens = 64;   // KV tokens per pipeline stage
constexpr int kStages = 4;         // stages in the shared-memory ring
constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kRowBlock = 64;      // MMA rows per unit (four m16 tiles)
constexpr int kRing = 4;           // work units the producer may run ahead
constexpr int kRbBits = 12;        // row-block index bits in Item::split_rb
constexpr int kUnitsPerSm = 16;    // split target: work units per SM
constexpr int kPlanThreads = 1024;
constexpr int kSeqInvalid = 1;

struct SeqPlan {
  int32_t qrow0;         // first row of q / out / lse
  int32_t nsplit;        // KV splits; 0 = nothing to compute (invalid or no query)
  int32_t partial_base;  // first partial row (nsplit > 1)
  int32_t len;           // L
  int32_t qlen;          // ql
  int32_t flags;         // kSeqInvalid
  int32_t nrb;           // row blocks
  int32_t pad;
};

struct Item {
  int32_t seq, page_begin, page_end, split_rb;  // split << kRbBits | row block
};

struct PlanHeader {
  int32_t n_items;
  int32_t work_counter;
  int32_t chunk_pages;
  int32_t n_partial_rows;
};

struct Layout {
  size_t seqplan, token_seq, items, part_lse, part_o, total;
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
  PlanHeader* header;
  int32_t B, T, G, Hkv, P, maxp, pps, min_chunk, no_split, target_units;
  int64_t items_cap, partial_cap;
  int32_t* err;
};

__device__ __forceinline__ int64_t block_sum_i64(int64_t v, int64_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int64_t t = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

// Exclusive scan of v over the block (threads in order); returns the prefix, stores the
// block total in *total.
__device__ __forceinline__ int64_t block_excl_scan_i64(int64_t v, int64_t* red,
                                                       int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  __syncthreads();
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  int64_t before = 0, all = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (w < warp) before += red[w];
    all += red[w];
  }
  *total = all;
  return before + inc - v;
}

struct SeqShape {
  bool valid;
  int32_t L, ql, npages, R, nrb;
};

__device__ __forceinline__ SeqShape seq_shape(const PlanArgs& a, int i) {
  SeqShape s;
  s.L = a.seq_lens[i];
  s.ql = a.query_lens[i];
  s.valid = s.ql >= 0 && s.ql <= a.T && s.L >= s.ql && (int64_t)s.L <= (int64_t)a.maxp * a.P;
  s.npages = s.valid ? (s.L + a.P - 1) / a.P : 0;
  s.R = s.valid ? a.G * s.ql : 0;
  s.nrb = (s.R + kRowBlock - 1) / kRowBlock;
  return s;
}

__device__ __forceinline__ int32_t splits_for(const SeqShape& s, int64_t chunk) {
  if (s.R == 0 || s.npages == 0) return 0;
  return (int32_t)((s.npages + chunk - 1) / chunk);
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanArgs a) {
  __shared__ int64_t red[kPlanThreads / 32];
  __shared__ int64_t s_chunk;
  __shared__ int32_t s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // Totals: work in page-row-blocks per KV head, and the packed query rows.
  int64_t cost = 0, rows = 0;
  for (int i = tid; i < a.B; i += kPlanThreads) {
    const SeqShape s = seq_shape(a, i);
    if (!s.valid) s_bad = 1;
    cost += (int64_t)s.npages * s.nrb;
    rows += s.ql > 0 ? s.ql : 0;
  }
  const int64_t total_cost = block_sum_i64(cost, red);
  const int64_t total_rows = block_sum_i64(rows, red);
  if (tid == 0 && (total_rows != a.T || s_bad)) atomicOr(a.err, VAS_DEV_BAD_LENGTHS);

  // Split length: about kUnitsPerSm units per SM, at least min_chunk pages, a whole
  // number of stages; doubled until the work list and the partials fit the workspace.
  if (tid == 0) {
    int64_t c = (int64_t)a.pps;
    if (a.no_split) {
      c = INT_MAX;
    } else {
      const int64_t want = (total_cost * a.Hkv + a.target_units - 1) / a.target_units;
      c = want > a.min_chunk ? want : a.min_chunk;
      c = (c + a.pps - 1) / a.pps * a.pps;
    }
    s_chunk = c;
  }
  __syncthreads();
  for (int iter = 0; iter < 40; ++iter) {
    const int64_t c = s_chunk;
    int64_t n_items = 0, n_part = 0;
    for (int i = tid; i < a.B; i += kPlanThreads) {
      const SeqShape s = seq_shape(a, i);
      const int32_t ns = splits_for(s, c);
      n_items += (int64_t)ns * s.nrb;
      if (ns > 1) n_part += (int64_t)ns * a.Hkv * s.R;
    }
    const int64_t tot_items = block_sum_i64(n_items, red);
    const int64_t tot_part = block_sum_i64(n_part, red);
    __syncthreads();
    if ((tot_items <= a.items_cap && tot_part <= a.partial_cap) || c >= INT_MAX / 2) break;
    if (tid == 0) s_chunk = c * 2 < INT_MAX ? c * 2 : INT_MAX;
    __syncthreads();
  }
  const int64_t c = s_chunk;

  for (int r = tid; r < a.T; r += kPlanThreads) a.token_seq[r] = -1;
  __syncthreads();

  // Scans in batch order, kPlanThreads sequences at a time.
  int64_t carry_rows = 0, carry_items = 0, carry_part = 0;
  for (int base = 0; base < a.B; base += kPlanThreads) {
    const int i = base + tid;
    SeqShape s;
    s.valid = false;
    s.L = s.ql = s.npages = s.R = s.nrb = 0;
    int32_t ns = 0, qrows = 0;
    if (i < a.B) {
      s = seq_shape(a, i);
      qrows = s.ql > 0 ? s.ql : 0;
      ns = splits_for(s, c);
    }
    int64_t t_rows, t_items, t_part;
    const int64_t my_row0 = carry_rows + block_excl_scan_i64(qrows, red, &t_rows);
    const int64_t my_item0 = carry_items + block_excl_scan_i64((int64_t)ns * s.nrb, red, &t_items);
    const int64_t my_part0 =
        carry_part + block_excl_scan_i64(ns > 1 ? (int64_t)ns * a.Hkv * s.R : 0, red, &t_part);
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
      sp.pad = 0;
      a.seqplan[i] = sp;
      for (int j = 0; j < qrows && my_row0 + j < a.T; ++j) a.token_seq[my_row0 + j] = i;
      if (ns > 0) {
        // A skipped sequence keeps its slots below the capacity as null items.
        int64_t it = my_item0;
        for (int sp_i = 0; sp_i < ns; ++sp_i) {
          const int32_t pb = (int32_t)(sp_i * c);
          const int32_t pe = (int32_t)((sp_i + 1) * c < s.npages ? (sp_i + 1) * c : s.npages);
          for (int rb = 0; rb < s.nrb && it < a.items_cap; ++rb) {
            Item item;
            item.seq = sp.nsplit > 0 ? i : -1;
            item.page_begin = pb;
            item.page_end = pe;
            item.split_rb = (sp_i << kRbBits) | rb;
            a.items[it++] = item;
          }
        }
      }
    }
    carry_rows += t_rows;
    carry_items += t_items;
    carry_part += t_part;
  }
  if (tid == 0) {
    a.header->n_items = (int32_t)(carry_items < a.items_cap ? carry_items : a.items_cap);
    a.header->work_counter = 0;
    a.header->chunk_pages = (int32_t)(c < INT_MAX ? c : INT_MAX);
    a.header->n_partial_rows = (int32_t)carry_part;
  }
}

// ------------------------------------------------------------------------------------
// Attention, bf16 storage: TMA page staging + mma.sync
// ------------------------------------------------------------------------------------
struct AttnArgs {
  const void* q;
  void* out;
  float* lse;
  const int32_t* block_table;
  const SeqPlan* seqplan;
  const Item* items;
  PlanHeader* header;
  float* part_o;
  float* part_lse;
  const void* k_pages;  // fp32 path only
  const void* v_pages;  // fp32 path only
  int32_t T, Hq, Hkv, G, maxp, num_pages, P;
  float scale_log2;  // softmax scale * log2(e)
  float scale;
  int32_t* err;
};

template <int D>
struct Smem {
  static constexpr int NH = D / 64;                  // 128-byte column halves per row
  static constexpr int kHalfBytes = kStageTokens * 128;
  static constexpr int kOperandBytes = NH * kHalfBytes;  // K or V of one stage
  static constexpr int kStageBytes = 2 * kOperandBytes;
  static constexpr int kQStride = D * 2 + 16;            // padded Q row
  static constexpr int kQBytes = kRowBlock * kQStride;
  static constexpr int kCombineFloats = (D / 8) * 4 + 4; // per thread: O frags + m,l x2
  static constexpr int kCombineBytes = kConsumerWarps * 32 * kCombineFloats * 4;
  static constexpr int kScratchBytes = kQBytes > kCombineBytes ? kQBytes : kCombineBytes;
  static constexpr int kStagesOff = 0;
  static constexpr int kScratchOff = kStages * kStageBytes;
  static constexpr int kBarOff = kScratchOff + ((kScratchBytes + 127) / 128) * 128;
  // full[kStages], empty[kStages], ufull[kRing], uempty[kRing], ring_u[kRing], meta[kStages]
  static constexpr int kBarBytes = (2 * kStages + 2 * kRing) * 8 + kRing * 4 + kStages * 4;
  static constexpr int kBytes = kBarOff + kBarBytes;
  static constexpr int kDynBytes = kBytes + 1024;  // slack for 1024-byte alignment
};

// QK^T, online softmax and PV for one warp's token slice of one stage.
// kbase / vbase: shared addresses of the stage's K and V (swizzled 128-byte rows).
template <int D, int TS>
__device__ __forceinline__ void stage_compute(uint32_t kbase, uint32_t vbase, int ts0,
                                              int tvalid, const uint32_t (&qa)[D / 16][4],
                                              float (&o)[D / 8][4], float (&m)[2],
                                              float (&l)[2], int t_abs0, int limA, int limB,
                                              bool need_mask, float scale_log2, int lane) {
  constexpr int NT = TS / 8;
  constexpr int kHalfBytes = Smem<D>::kHalfBytes;
  const int g = lane >> 2, tq = lane & 3, mi = lane >> 3, r8 = lane & 7;
  (void)g;

  float s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    if (8 * nt < tvalid) {
      const int t = ts0 + 8 * nt + r8;  // stage row this lane addresses
#pragma unroll
      for (int qd = 0; qd < D / 32; ++qd) {
        const int gc = 4 * qd + mi;  // 16-byte column chunk 0 .. D/8-1
        const uint32_t addr =
            kbase + (gc >> 3) * kHalfBytes + t * 128 + ((((gc & 7) ^ (t & 7))) << 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        mma_bf16_16816(s[nt], qa[2 * qd], b0, b1);
        mma_bf16_16816(s[nt], qa[2 * qd + 1], b2, b3);
      }
    }
  }

  // Scale to log2 units, mask, running max.
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tt = 8 * nt + 2 * tq + (e & 1);  // token within the slice
      const int lim = (e < 2) ? limA : limB;
      const bool off = tt >= tvalid || (need_mask && t_abs0 + ts0 + tt > lim);
      const float v = off ? -INFINITY : s[nt][e] * scale_log2;
      s[nt][e] = v;
      mx[e >> 1] = fmaxf(mx[e >> 1], v);
    }
  }
  float alpha[2], muse[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    const float mnew = fmaxf(m[h], mx[h]);
    muse[h] = mnew == -INFINITY ? 0.f : mnew;
    alpha[h] = exp2f(m[h] - muse[h]);
    m[h] = mnew;
  }
  float rs[2] = {0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float p = exp2f(s[nt][e] - muse[e >> 1]);
      s[nt][e] = p;
      rs[e >> 1] += p;
    }
  }
  l[0] = l[0] * alpha[0] + rs[0];
  l[1] = l[1] * alpha[1] + rs[1];
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    o[dt][0] *= alpha[0];
    o[dt][1] *= alpha[0];
    o[dt][2] *= alpha[1];
    o[dt][3] *= alpha[1];
  }

  // O += P V over 16-token k-steps.
#pragma unroll
  for (int kk = 0; kk < TS / 16; ++kk) {
    if (16 * kk < tvalid) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      const int t = ts0 + 16 * kk + (mi & 1) * 8 + r8;
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int gc = 2 * dp + (mi >> 1);
        const uint32_t addr =
            vbase + (gc >> 3) * kHalfBytes + t * 128 + ((((gc & 7) ^ (t & 7))) << 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(addr, b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
      }
    }
  }
}

template <int D, int P>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using S = Smem<D>;
  constexpr int PPS = kStageTokens / P;  // pages per stage
  constexpr int kPageBytes = P * 128;    // one column half of one page of one head
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem + S::kStagesOff;
  uint8_t* scratch = smem + S::kScratchOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* ufull = empty + kStages;
  uint64_t* uempty = ufull + kRing;
  int32_t* ring_u = reinterpret_cast<int32_t*>(uempty + kRing);
  int32_t* meta = ring_u + kRing;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&ufull[r], 1);
      mbar_init(&uempty[r], kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const int32_t n_units = a.header->n_items * a.Hkv;

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      prefetch_tensor_map(&tm_k);
      prefetch_tensor_map(&tm_v);
    }
    const uint64_t pol = l2_policy_evict_first();
    uint32_t stage_it = 0, unit_it = 0;
    int32_t u_next = 0;
    if (lane == 0) u_next = atomicAdd(&a.header->work_counter, 1);
    bool ok = true;
    for (;;) {
      const int32_t u = __shfl_sync(0xffffffffu, u_next, 0);
      const int slot = unit_it % kRing;
      ok = mbar_wait(&uempty[slot], ((unit_it / kRing) & 1) ^ 1);
      if (!ok) break;
      if (u >= n_units) {
        if (lane == 0) {
          ring_u[slot] = -1;
          mbar_arrive(&ufull[slot]);
        }
        break;
      }
      if (lane == 0) {
        u_next = atomicAdd(&a.header->work_counter, 1);  // next unit, consumed next pass
        ring_u[slot] = u;
        mbar_arrive(&ufull[slot]);
      }
      ++unit_it;
      const Item it = a.items[u / a.Hkv];
      const int head = u % a.Hkv;
      if (it.seq < 0) continue;
      const int32_t* bt_row = a.block_table + (size_t)it.seq * a.maxp;
      for (int pg0 = it.page_begin; pg0 < it.page_end && ok; pg0 += 32) {
        const int npg = min(32, it.page_end - pg0);
        const int32_t my_id = lane < npg ? bt_row[pg0 + lane] : 0;
        for (int s0 = 0; s0 < npg; s0 += PPS) {
          const int stage = stage_it % kStages;
          ok = mbar_wait(&empty[stage], ((stage_it / kStages) & 1) ^ 1);
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
              else bytes += 2u * S::NH * kPageBytes;
            }
          }
          if (lane == 0) {
            meta[stage] = bad;
            mbar_arrive_expect_tx(&full[stage], bytes);
            uint8_t* kdst = stages + stage * S::kStageBytes;
            uint8_t* vdst = kdst + S::kOperandBytes;
#pragma unroll
            for (int e = 0; e < PPS; ++e) {
              if (e < n_in && ids[e] >= 0 && ids[e] < a.num_pages) {
#pragma unroll
                for (int h = 0; h < S::NH; ++h) {
                  const int off = h * S::kHalfBytes + e * kPageBytes;
                  tma_load_3d(kdst + off, &tm_k, &full[stage], h * 64, head, ids[e] * P, pol);
                  tma_load_3d(vdst + off, &tm_v, &full[stage], h * 64, head, ids[e] * P, pol);
                }
              }
            }
          }
          __syncwarp();
          ++stage_it;
        }
      }
      if (!ok) break;
    }
    if (!ok && lane == 0) atomicOr(a.err, VAS_DEV_TIMEOUT);
    // Let every copy this warp issued land before the CTA can exit.
    for (uint32_t d = stage_it > kStages ? stage_it - kStages : 0; d < stage_it; ++d)
      mbar_wait(&full[d % kStages], (d / kStages) & 1);
    return;
  }

  // -------------------------------- consumers --------------------------------
  const int tid = threadIdx.x;  // 0 .. kConsumerThreads-1
  const int g = lane >> 2, tq = lane & 3;
  uint32_t stage_it = 0, unit_it = 0;
  for (;;) {
    const int slot = unit_it % kRing;
    if (!mbar_wait(&ufull[slot], (unit_it / kRing) & 1)) {
      if (lane == 0) atomicOr(a.err, VAS_DEV_TIMEOUT);
      break;
    }
    const int32_t u = ring_u[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&uempty[slot]);
    ++unit_it;
    if (u < 0) break;

    const Item it = a.items[u / a.Hkv];
    if (it.seq < 0) continue;
    const int head = u % a.Hkv;
    const SeqPlan sp = a.seqplan[it.seq];
    const int split = it.split_rb >> kRbBits, rb = it.split_rb & ((1 << kRbBits) - 1);
    const int L = sp.len, ql = sp.qlen;
    const int R = a.G * ql;
    const int r0 = rb * kRowBlock;
    const int Rb = min(kRowBlock, R - r0);
    const int nM = (Rb + 15) >> 4;
    const int nW = nM == 1 ? 4 : (nM == 2 ? 2 : 1);
    const bool active = warp < nM * nW;
    const int mt = warp % nM;
    const int slice = warp / nM;
    const int TS = kStageTokens / nW;

    // Stage the unit's query rows (row r: token r / G, head head * G + r % G).
    named_bar_sync(1, kConsumerThreads);
    {
      constexpr int kChunks = D / 8;
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
      for (int c = tid; c < kRowBlock * kChunks; c += kConsumerThreads) {
        const int row = c / kChunks, ch = c % kChunks;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < Rb) {
          const int r = r0 + row;
          const int j = r / a.G, hh = r % a.G;
          const size_t src = ((size_t)(sp.qrow0 + j) * a.Hq + (size_t)head * a.G + hh) * D + ch * 8;
          v = *reinterpret_cast<const uint4*>(qg + src);
        }
        *reinterpret_cast<uint4*>(scratch + row * S::kQStride + ch * 16) = v;
      }
    }
    named_bar_sync(1, kConsumerThreads);
    uint32_t qa[D / 16][4];
    if (active) {
      const int mi = lane >> 3;
      const int row = 16 * mt + (mi & 1) * 8 + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int ch = 2 * ks + (mi >> 1);
        ldsm_x4(smem_u32(scratch + row * S::kQStride + ch * 16), qa[ks][0], qa[ks][1], qa[ks][2],
                qa[ks][3]);
      }
    }

    float o[D / 8][4];
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    const int rA = r0 + 16 * mt + g, rB = rA + 8;
    const int limA = rA < R ? L - ql + rA / a.G : L - 1;
    const int limB = rB < R ? L - ql + rB / a.G : L - 1;
    const int min_lim = L - ql + r0 / a.G;  // smallest causal limit of this row block
    bool poison = false, timed_out = false;

    for (int pg = it.page_begin; pg < it.page_end; pg += PPS) {
      const int stage = stage_it % kStages;
      if (!mbar_wait(&full[stage], (stage_it / kStages) & 1)) {
        timed_out = true;
        break;
      }
      ++stage_it;
      if (meta[stage]) poison = true;
      const int loaded = min(PPS, it.page_end - pg) * P;
      const int t_abs0 = pg * P;
      const uint32_t kbase = smem_u32(stages + stage * S::kStageBytes);
      const uint32_t vbase = kbase + S::kOperandBytes;
      if (active) {
        const int ts0 = slice * TS;
        const int tvalid = min(TS, loaded - ts0);
        if (tvalid > 0) {
          // Pool slots past the end of the sequence may hold anything: zero their V
          // rows so that a zero attention weight cannot meet a NaN.
          if (t_abs0 + ts0 + tvalid > L) {
            const int z0 = max(0, L - t_abs0 - ts0);
            uint8_t* vrow = stages + stage * S::kStageBytes + S::kOperandBytes;
            for (int c = z0 * 8 * S::NH + lane; c < tvalid * 8 * S::NH; c += 32) {
              const int t = ts0 + c / (8 * S::NH), rem = c % (8 * S::NH);
              *reinterpret_cast<uint4*>(vrow + (rem >> 3) * S::kHalfBytes + t * 128 +
                                        (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          const bool need_mask = t_abs0 + ts0 + tvalid - 1 > min_lim;
          if (TS == 16)
            stage_compute<D, 16>(kbase, vbase, ts0, tvalid, qa, o, m, l, t_abs0, limA, limB,
                                 need_mask, a.scale_log2, lane);
          else if (TS == 32)
            stage_compute<D, 32>(kbase, vbase, ts0, tvalid, qa, o, m, l, t_abs0, limA, limB,
                                 need_mask, a.scale_log2, lane);
          else
            stage_compute<D, 64>(kbase, vbase, ts0, tvalid, qa, o, m, l, t_abs0, limA, limB,
                                 need_mask, a.scale_log2, lane);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (timed_out) {
      if (lane == 0) atomicOr(a.err, VAS_DEV_TIMEOUT);
      break;
    }

    // Row sums across the quad that shares a row.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }

    // Merge the token slices of one m-tile (nW warps) through shared memory.
    float* cb = reinterpret_cast<float*>(scratch);
    named_bar_sync(1, kConsumerThreads);  // everyone is done with the Q rows
    if (active && nW > 1 && slice > 0) {
      float* mine = cb + (size_t)warp * 32 * S::kCombineFloats;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) mine[(dt * 4 + e) * 32 + lane] = o[dt][e];
      mine[(D / 2 + 0) * 32 + lane] = m[0];
      mine[(D / 2 + 1) * 32 + lane] = m[1];
      mine[(D / 2 + 2) * 32 + lane] = l[0];
      mine[(D / 2 + 3) * 32 + lane] = l[1];
    }
    named_bar_sync(1, kConsumerThreads);
    if (active && slice == 0) {
      for (int sl = 1; sl < nW; ++sl) {
        const float* other = cb + (size_t)(mt + sl * nM) * 32 * S::kCombineFloats;
        float om[2] = {other[(D / 2 + 0) * 32 + lane], other[(D / 2 + 1) * 32 + lane]};
        float ol[2] = {other[(D / 2 + 2) * 32 + lane], other[(D / 2 + 3) * 32 + lane]};
        float fa[2], fb[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float mm = fmaxf(m[h], om[h]);
          const float mu = mm == -INFINITY ? 0.f : mm;
          fa[h] = exp2f(m[h] - mu);
          fb[h] = exp2f(om[h] - mu);
          l[h] = l[h] * fa[h] + ol[h] * fb[h];
          m[h] = mm;
        }
#pragma unroll
        for (int dt = 0; dt < D / 8; ++dt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[dt][e] = o[dt][e] * fa[e >> 1] + other[(dt * 4 + e) * 32 + lane] * fb[e >> 1];
      }

      // Write: the final rows (one split) or this split's normalised partial.
      const float kLn2 = 0.6931471805599453f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = h ? rB : rA;
        if (r >= r0 + Rb) continue;
        const int j = r / a.G, hh = r % a.G;
        const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
        float row_lse = l[h] > 0.f ? (m[h] + log2f(l[h])) * kLn2 : -INFINITY;
        if (poison) row_lse = NAN;
        if (sp.nsplit == 1) {
          const size_t orow = (size_t)(sp.qrow0 + j) * a.Hq + (size_t)head * a.G + hh;
          __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + orow * D;
#pragma unroll
          for (int dt = 0; dt < D / 8; ++dt) {
            float x0 = o[dt][2 * h] * inv, x1 = o[dt][2 * h + 1] * inv;
            if (poison) x0 = x1 = NAN;
            *reinterpret_cast<uint32_t*>(og + dt * 8 + 2 * tq) = pack_bf16x2(x0, x1);
          }
          if (tq == 0) a.lse[orow] = row_lse;
        } else {
          const size_t prow =
              (size_t)sp.partial_base + ((size_t)split * a.Hkv + head) * R + r;
          float* po = a.part_o + prow * D;
#pragma unroll
          for (int dt = 0; dt < D / 8; ++dt) {
            float x0 = o[dt][2 * h] * inv, x1 = o[dt][2 * h + 1] * inv;
            if (poison) x0 = x1 = NAN;
            *reinterpret_cast<float2*>(po + dt * 8 + 2 * tq) = make_float2(x0, x1);
          }
          if (tq == 0) a.part_lse[prow] = row_lse;
        }
      }
    }
    if (poison && tid == 0) atomicOr(a.err, VAS_DEV_BAD_PAGE);
  }
}

// ------------------------------------------------------------------------------------
// Attention, fp32 storage: one warp per query row on the CUDA cores
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
  const int32_t n_units = a.header->n_items * a.Hkv;
  for (int32_t u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Item it = a.items[u / a.Hkv];
    if (it.seq < 0) continue;
    const int head = u % a.Hkv;
    const SeqPlan sp = a.seqplan[it.seq];
    const int rb = it.split_rb & ((1 << kRbBits) - 1);
    const int L = sp.len, ql = sp.qlen, R = a.G * ql;
    const int32_t* bt_row = a.block_table + (size_t)it.seq * a.maxp;
    for (int r = rb * kRowBlock + warp; r < min(R, rb * kRowBlock + kRowBlock); r += 4) {
      const int j = r / a.G, hh = r % a.G;
      const int pos = L - ql + j;
      const size_t orow = (size_t)(sp.qrow0 + j) * a.Hq + (size_t)head * a.G + hh;
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
// LSE merge of split partials; NaN fill of rows a device-detected error left undefined
// ------------------------------------------------------------------------------------
struct CombineArgs {
  const SeqPlan* seqplan;
  const int32_t* token_seq;
  const float* part_o;
  const float* part_lse;
  void* out;
  float* lse;
  int32_t T, Hq, Hkv, G, D, is_bf16;
};

__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;  // (token, q head)
  if (row >= (int64_t)a.T * a.Hq) return;
  const int token = (int)(row / a.Hq), h = (int)(row % a.Hq);
  const int seq = a.token_seq[token];
  SeqPlan sp;
  bool nan_fill = seq < 0;
  if (!nan_fill) {
    sp = a.seqplan[seq];
    if (sp.flags & kSeqInvalid) nan_fill = true;
    else if (sp.nsplit <= 1) return;  // written by the attention kernel
  }
  float outv[4];
  float row_lse;
  if (nan_fill) {
    outv[0] = outv[1] = outv[2] = outv[3] = NAN;
    row_lse = NAN;
  } else {
    const int j = token - sp.qrow0, g = h / a.G, hh = h % a.G;
    const int R = a.G * sp.qlen, r = j * a.G + hh;
    const int ns = sp.nsplit;
    auto prow = [&](int s) -> size_t {
      return (size_t)sp.partial_base + ((size_t)s * a.Hkv + g) * R + r;
    };
    float mx = -INFINITY;
    bool any_nan = false;
    for (int s = lane; s < ns; s += 32) {
      const float v = a.part_lse[prow(s)];
      any_nan |= isnan(v);
      mx = fmaxf(mx, v);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    any_nan = __any_sync(0xffffffffu, any_nan);
    const float mu = mx == -INFINITY ? 0.f : mx;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    const int E = a.D / 32;  // 2 or 4 elements per lane
    for (int s = 0; s < ns; ++s) {
      const float w = expf(a.part_lse[prow(s)] - mu);
      wsum += w;
      const float* po = a.part_o + prow(s) * a.D + lane * E;
      if (E == 4) {
        const float4 v = *reinterpret_cast<const float4*>(po);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(po);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
    const float inv = 1.f / wsum;
    for (int e = 0; e < 4; ++e) outv[e] = any_nan ? NAN : acc[e] * inv;
    row_lse = any_nan ? NAN : mu + logf(wsum);
  }
  const int E = a.D / 32;
  if (a.is_bf16) {
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out) + row * a.D + lane * E;
    for (int e = 0; e < E; e += 2)
      *reinterpret_cast<uint32_t*>(og + e) = pack_bf16x2(outv[e], outv[e + 1]);
  } else {
    float* og = static_cast<float*>(a.out) + row * a.D + lane * E;
    for (int e = 0; e < E; ++e) og[e] = outv[e];
  }
  if (lane == 0) a.lse[row] = row_lse;
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
         (d->kv_dtype == VAS_BF16 || d->kv_dtype == VAS_F32);
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

// 3-D view of a page pool: (D, Hkv, num_pages * P) with a (64, 1, P) box, 128B swizzle.
bool encode_pool_map(CUtensorMap* map, const void* base, const vas_attn_dims* d) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d->head_dim, (cuuint64_t)d->num_kv_heads,
                              (cuuint64_t)d->num_pages * d->page_size};
  const cuuint64_t strides[2] = {(cuuint64_t)d->head_dim * 2,
                                 (cuuint64_t)d->num_kv_heads * d->head_dim * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)d->page_size};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int P>
int launch_bf16(const CUtensorMap& mk, const CUtensorMap& mv, const AttnArgs& args, int grid,
                cudaStream_t stream) {
  using S = Smem<D>;
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  static cudaError_t attr_err[64];
  std::call_once(once[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(attn_bf16_kernel<D, P>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              S::kDynBytes);
  });
  if (attr_err[dev & 63] != cudaSuccess) return VAS_E_CUDA;
  attn_bf16_kernel<D, P><<<grid, kThreads, S::kDynBytes, stream>>>(mk, mv, args);
  return cudaGetLastError() == cudaSuccess ? VAS_OK : VAS_E_CUDA;
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

int paged_attn_fwd(const void* q, const void* k_pages, const void* v_pages,
                   const int32_t* block_table, const int32_t* seq_lens,
                   const int32_t* query_lens, void* out, float* lse,
                   const vas_attn_dims* dims, void* workspace, size_t workspace_bytes,
                   vas_stream_t stream_) {
  if (!dims_ok(dims)) return VAS_E_INVALID_ARG;
  if (!dims_supported(dims)) return VAS_E_UNSUPPORTED;
  const vas_attn_dims& d = *dims;
  if (d.num_seqs == 0 || d.total_q_tokens == 0) return VAS_OK;
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !query_lens || !out || !lse ||
      !workspace)
    return VAS_E_INVALID_ARG;
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k_pages, 16) || mis(v_pages, 16) || mis(out, 16) || mis(lse, 4) ||
      mis(block_table, 4) || mis(seq_lens, 4) || mis(query_lens, 4) || mis(workspace, 256))
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
  const bool bf16 = d.kv_dtype == VAS_BF16;
  PlanArgs pa;
  pa.seq_lens = seq_lens;
  pa.query_lens = query_lens;
  pa.seqplan = reinterpret_cast<SeqPlan*>(ws + lay.seqplan);
  pa.token_seq = reinterpret_cast<int32_t*>(ws + lay.token_seq);
  pa.items = reinterpret_cast<Item*>(ws + lay.items);
  pa.header = reinterpret_cast<PlanHeader*>(ws);
  pa.B = d.num_seqs;
  pa.T = d.total_q_tokens;
  pa.G = G;
  pa.Hkv = d.num_kv_heads;
  pa.P = d.page_size;
  pa.maxp = d.max_pages_per_seq;
  pa.pps = kStageTokens / d.page_size;
  pa.min_chunk = 2 * pa.pps;
  pa.no_split = bf16 ? 0 : 1;
  pa.target_units = kUnitsPerSm * sms;
  pa.items_cap = lay.items_cap;
  pa.partial_cap = lay.partial_cap;
  pa.err = err;
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(pa);
  if (cudaGetLastError() != cudaSuccess) return VAS_E_CUDA;

  const float scale = d.scale > 0.f ? d.scale : 1.0f / std::sqrt((float)d.head_dim);
  AttnArgs aa;
  aa.q = q;
  aa.out = out;
  aa.lse = lse;
  aa.block_table = block_table;
  aa.seqplan = pa.seqplan;
  aa.items = pa.items;
  aa.header = pa.header;
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

  int rc = VAS_OK;
  if (bf16) {
    CUtensorMap mk, mv;
    if (!encode_pool_map(&mk, k_pages, dims) || !encode_pool_map(&mv, v_pages, dims))
      return VAS_E_CUDA;
    const int grid = sms;
    if (d.head_dim == 128 && d.page_size == 16) rc = launch_bf16<128, 16>(mk, mv, aa, grid, stream);
    else if (d.head_dim == 128) rc = launch_bf16<128, 32>(mk, mv, aa, grid, stream);
    else if (d.page_size == 16) rc = launch_bf16<64, 16>(mk, mv, aa, grid, stream);
    else rc = launch_bf16<64, 32>(mk, mv, aa, grid, stream);
  } else {
    const int grid = 4 * sms;
    if (d.head_dim == 128) attn_f32_kernel<128><<<grid, 128, 0, stream>>>(aa);
    else attn_f32_kernel<64><<<grid, 128, 0, stream>>>(aa);
    rc = cudaGetLastError() == cudaSuccess ? VAS_OK : VAS_E_CUDA;
  }
  if (rc != VAS_OK) return rc;

  CombineArgs ca;
  ca.seqplan = pa.seqplan;
  ca.token_seq = pa.token_seq;
  ca.part_o = aa.part_o;
  ca.part_lse = aa.part_lse;
  ca.out = out;
  ca.lse = lse;
  ca.T = d.total_q_tokens;
  ca.Hq = d.num_q_heads;
  ca.Hkv = d.num_kv_heads;
  ca.G = G;
  ca.D = d.head_dim;
  ca.is_bf16 = bf16 ? 1 : 0;
  const int64_t rows = (int64_t)d.total_q_tokens * d.num_q_heads;
  combine_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(ca);
  return cudaGetLastError() == cudaSuccess ? VAS_OK : VAS_E_CUDA;
}

}  // extern "C"
