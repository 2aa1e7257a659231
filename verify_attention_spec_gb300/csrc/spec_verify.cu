// Speculative verification: modified rejection sampling (sm_103a).
//
// The rule ("Continuous Batching & Speculative Decoding", section "The Modified
// Rejection Sampling Algorithm"; "Continuous Batching and Speculative Decoding: How
// Modern LLM Serving Engines Actually Work", section "The core idea"):
//   accept x_i while r_i <= min(1, p_i(x_i) / q_i(x_i)) -- tested as r_i q_i <= p_i in
//   double -- halt at the first rejection j, then draw the token at position j from
//   max(0, p_j - q_j) (or from p_k when all k drafts are accepted) by inverse CDF.
//
// Kernel: one thread-block cluster of C CTAs per sequence (C <= 8, fewer for small
// vocabularies); CTA r of the cluster owns slice r of the vocabulary.  Every CTA runs
// the k ratio tests itself (k scattered loads) and finds j; the same threads compute the
// draw's uniform for every position, so it is ready once j is known.  One streaming
// pass over the CTA's slice of row j then builds w = max(0, p_j - q_j): one thread
// streams the slice into a ring of shared-memory stages by bulk copy (cp.async.bulk,
// completion counted on an mbarrier per stage), so the bytes in flight do not depend on
// registers; each warp reduces one 256-element tile of a stage, 8 contiguous elements per
// lane in fp32 and everything above as float-float pairs (about 44 significant bits; this
// part's double-precision rate is far too low for a per-element reduction), and keeps
// the tile and stage totals.  Slice
// totals meet through distributed shared memory after one cluster barrier, so every CTA
// agrees on S and on the slice holding the target s_j * S.  That CTA walks its stage and
// tile totals to the tile holding the target, reads only that tile again (from L2), scans
// its lanes as float-float pairs, and the crossing lane walks its 8 elements.  Rows that are not
// 16-byte aligned (a vocabulary that is not a multiple of 4) are staged by plain loads.
// Uniforms come from Philox4x32-10 keyed by the seed with counter (position, sequence,
// 0, 0).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/vas.h"
#include "device_util.cuh"
#include "philox.cuh"
#include "vas_internal.h"

namespace cg = cooperative_groups;

namespace vas {
namespace verify {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kLaneElems = 8;                  // contiguous elements per lane per tile
constexpr int kTile = 32 * kLaneElems;          // elements per warp tile
constexpr int kStageElems = kWarps * kTile;     // one tile per warp per stage
constexpr int kStages = 3;                      // ring depth (stages in flight)
constexpr int kMaxCluster = 8;
constexpr int kSliceMin = 4096;                 // smallest vocabulary slice per CTA
constexpr int kMaxStagesPerSlice = 64;          // bounds the vocabulary at 8 x 64 x 2048
constexpr int64_t kMaxVocab = (int64_t)kMaxCluster * kMaxStagesPerSlice * kStageElems;
constexpr size_t kRingBytes = (size_t)kStages * 2 * kStageElems * sizeof(float);

struct Args {
  const float* p;
  const float* q;
  const int32_t* draft;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t B, k, V, slice;  // slice: vocabulary elements per CTA (multiple of kTile)
  int32_t bulk;            // every row is 16-byte aligned: stages arrive by bulk copy
  uint32_t key0, key1;
  int32_t* err;
};

// The 8 weights of one lane's group starting at x0 (elements at or past end are zero),
// read from global memory (the rescan of one tile).
__device__ __forceinline__ void load_weights(const float* prow, const float* qrow, int x0,
                                             int end, bool vec, float (&w)[kLaneElems]) {
  if (vec && x0 + kLaneElems <= end) {
    const float4 p0 = __ldg(reinterpret_cast<const float4*>(prow + x0));
    const float4 p1 = __ldg(reinterpret_cast<const float4*>(prow + x0 + 4));
    const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    if (qrow) {
      const float4 q0 = __ldg(reinterpret_cast<const float4*>(qrow + x0));
      const float4 q1 = __ldg(reinterpret_cast<const float4*>(qrow + x0 + 4));
      const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = fmaxf(pv[e] - qv[e], 0.f);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = pv[e];
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < kLaneElems; ++e) {
    const int x = x0 + e;
    float v = 0.f;
    if (x < end) {
      const float pv = __ldg(prow + x);
      v = qrow ? fmaxf(pv - __ldg(qrow + x), 0.f) : pv;
    }
    w[e] = v;
  }
}

__device__ __forceinline__ float group_sum(const float (&w)[kLaneElems]) {
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < kLaneElems; ++e) s += w[e];
  return s;
}

// Shared state of one CTA (the ring of stages is dynamic shared memory).
struct Smem {
  uint64_t full[kStages];                      // stage landed (bulk-copy bytes)
  ff32 tile[kMaxStagesPerSlice][kWarps];       // total of each tile, in x order
  ff32 stage[kMaxStagesPerSlice];              // total of each stage
  ff32 total[2];                               // this CTA's slice total, one per pass
  ff32 peer_total[2][kMaxCluster];             // every rank's slice total (pushed by it)
  ff32 base, target, all;
  ff32 u1[kThreads];                           // draw uniform at each position
  int32_t j, bad, owner, use_p;
};

// Among vals[0 .. n) (n <= 64, non-negative), the first i with vals[i] > 0 whose prefix
// base + vals[0] + ... + vals[i] exceeds target; when rounding leaves none, the last i
// with vals[i] > 0; -1 if no value is positive.  `before` receives base plus the values
// ahead of i.  Called by a whole warp (inclusive scans of two values per lane).
__device__ __forceinline__ int warp_first_crossing(const ff32* vals, int n, ff32 base,
                                                   ff32 target, ff32& before) {
  const int lane = threadIdx.x & 31;
  const ff32 zero = {0.f, 0.f};
  const ff32 a = lane < n ? vals[lane] : zero;
  const ff32 b = lane + 32 < n ? vals[lane + 32] : zero;
  ff32 ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff32 na = ff_shfl_up(ia, o), nb = ff_shfl_up(ib, o);
    if (lane >= o) {
      ia = ff_add(ia, na);
      ib = ff_add(ib, nb);
    }
  }
  const ff32 tot_a = ff_shfl(ia, 31);
  ib = ff_add(tot_a, ib);
  ff32 ea = ff_shfl_up(ia, 1), eb = ff_shfl_up(ib, 1);
  if (lane == 0) {
    ea = zero;
    eb = tot_a;
  }
  const unsigned ma = __ballot_sync(0xffffffffu, a.hi > 0.f && ff_gt(ff_add(base, ia), target));
  const unsigned mb = __ballot_sync(0xffffffffu, b.hi > 0.f && ff_gt(ff_add(base, ib), target));
  int idx = -1;
  bool upper = false;
  if (ma) {
    idx = __ffs(ma) - 1;
  } else if (mb) {
    idx = __ffs(mb) - 1;
    upper = true;
  } else {
    const unsigned la = __ballot_sync(0xffffffffu, a.hi > 0.f);
    const unsigned lb = __ballot_sync(0xffffffffu, b.hi > 0.f);
    if (lb) {
      idx = 31 - __clz(lb);
      upper = true;
    } else if (la) {
      idx = 31 - __clz(la);
    }
  }
  if (idx < 0) {
    before = base;
    return -1;
  }
  before = ff_add(base, ff_shfl(upper ? eb : ea, idx));
  return upper ? idx + 32 : idx;
}

// One pass over this CTA's slice [x_begin, x_end) of the row: w = max(0, p - q) (kHasQ)
// or p.  Stage s holds elements x_begin + s * kStageElems ...; warp w reduces tile w of
// each stage.  `g` counts the stages this CTA has put through the ring so far (mbarrier
// phases continue across passes).  Leaves the tile, stage and slice totals in sm.
template <bool kHasQ>
__device__ __forceinline__ void slice_pass(const Args& a, const float* prow, const float* qrow,
                                           int x_begin, int x_end, float* ring, Smem& sm,
                                           uint32_t& g, int pass) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_stages = (x_end - x_begin + kStageElems - 1) / kStageElems;
  auto issue = [&](int s) {  // thread 0: bulk copies of stage s into its ring slot
    const uint32_t slot = (g + s) % kStages;
    float* sp = ring + (size_t)slot * 2 * kStageElems;
    const int x0 = x_begin + s * kStageElems;
    const uint32_t bytes = (uint32_t)min(kStageElems, x_end - x0) * sizeof(float);
    mbar_arrive_expect_tx(&sm.full[slot], kHasQ ? 2 * bytes : bytes);
    bulk_load_plain(sp, prow + x0, bytes, &sm.full[slot]);
    if (kHasQ) bulk_load_plain(sp + kStageElems, qrow + x0, bytes, &sm.full[slot]);
  };
  if (a.bulk && tid == 0)
    for (int s = 0; s < min(kStages, n_stages); ++s) issue(s);
  for (int s = 0; s < n_stages; ++s) {
    const uint32_t gs = g + s;
    const float* sp = ring + (size_t)(gs % kStages) * 2 * kStageElems;
    const float* sq = sp + kStageElems;
    const int x0 = x_begin + s * kStageElems;
    const int n = min(kStageElems, x_end - x0);
    if (a.bulk) {
      if (!mbar_wait(&sm.full[gs % kStages], (gs / kStages) & 1)) atomicOr(a.err, VAS_DEV_TIMEOUT);
    } else {
      float* dp = ring + (size_t)(gs % kStages) * 2 * kStageElems;
      for (int i = tid; i < n; i += kThreads) {
        dp[i] = __ldg(prow + x0 + i);
        if (kHasQ) dp[kStageElems + i] = __ldg(qrow + x0 + i);
      }
      __syncthreads();
    }
    const int e0 = warp * kTile + lane * kLaneElems;
    float w[kLaneElems];
    if (e0 + kLaneElems <= n) {
      const float4 p0 = *reinterpret_cast<const float4*>(sp + e0);
      const float4 p1 = *reinterpret_cast<const float4*>(sp + e0 + 4);
      const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      if (kHasQ) {
        const float4 q0 = *reinterpret_cast<const float4*>(sq + e0);
        const float4 q1 = *reinterpret_cast<const float4*>(sq + e0 + 4);
        const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = fmaxf(pv[e] - qv[e], 0.f);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pv[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < kLaneElems; ++e) {
        const int i = e0 + e;
        w[e] = i < n ? (kHasQ ? fmaxf(sp[i] - sq[i], 0.f) : sp[i]) : 0.f;
      }
    }
    ff32 v = {group_sum(w), 0.f};
#pragma unroll
    for (int o = 16; o; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
    if (lane == 0) sm.tile[s][warp] = v;
    __syncthreads();  // every warp is done with the slot and has written its tile total
    if (tid == 0) {
      if (a.bulk && s + kStages < n_stages) issue(s + kStages);
      ff32 st = sm.tile[s][0];
#pragma unroll
      for (int t = 1; t < kWarps; ++t) st = ff_add(st, sm.tile[s][t]);
      sm.stage[s] = st;
    }
  }
  g += n_stages;
  if (tid == 0) {
    ff32 run = {0.f, 0.f};
    for (int s = 0; s < n_stages; ++s) run = ff_add(run, sm.stage[s]);
    sm.total[pass] = run;
  }
}

__global__ void __launch_bounds__(kThreads) spec_verify_kernel(const Args a) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / C;
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  float* ring = reinterpret_cast<float*>(dyn_smem);
  __shared__ Smem sm;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, V = a.V;
  if (tid == 0) {
    sm.j = k;
    sm.bad = 0;
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], 1);
    mbar_fence_init();
  }
  pdl_wait_prior_grid();  // inputs written by the previous kernel in the stream are visible
  __syncthreads();

  // 1. Ratio tests (every CTA of the cluster, redundantly): thread i < k tests draft x_i
  //    with r_i = word 0 of Philox(i, b); thread i <= k keeps word 1, the uniform of a
  //    draw at position i.
  if (tid <= k) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)tid, (uint32_t)b, 0u, 0u), a.key0, a.key1);
    sm.u1[tid] = ff_from_double(philox_uniform(w.y));
    if (tid < k) {
      const int x = a.draft[(size_t)b * k + tid];
      if (x < 0 || x >= V) {
        atomicOr(&sm.bad, 1);
      } else {
        const double pi = a.p[((size_t)b * (k + 1) + tid) * V + x];
        const double qi = a.q[((size_t)b * k + tid) * V + x];
        const double r = philox_uniform(w.x);
        if (!(r * qi <= pi)) atomicMin(&sm.j, tid);
      }
    }
  }
  __syncthreads();
  int32_t* out = a.out_tokens + (size_t)b * (k + 1);
  if (sm.bad) {  // the same in every CTA of the cluster: all leave before any barrier
    if (rank == 0) {
      for (int t = tid; t <= k; t += kThreads) out[t] = -1;
      if (tid == 0) {
        a.accepted_len[b] = -1;
        atomicOr(a.err, VAS_DEV_BAD_TOKEN);
      }
    }
    return;
  }
  const int j = sm.j;

  // 2. One pass over this CTA's slice of the row to draw from.
  const int x_begin = rank * a.slice;
  const int x_end = min(V, x_begin + a.slice);
  const float* prow = a.p + ((size_t)b * (k + 1) + j) * V;
  const float* qrow0 = j < k ? a.q + ((size_t)b * k + j) * V : nullptr;
  int use_p = 0;
  float S = 0.f;  // high part of the row total (> 0 exactly when the total is)
  uint32_t g = 0;
  for (int pass = 0; pass < 2; ++pass) {
    const float* qrow = use_p ? nullptr : qrow0;
    if (qrow) slice_pass<true>(a, prow, qrow, x_begin, x_end, ring, sm, g, pass);
    else slice_pass<false>(a, prow, nullptr, x_begin, x_end, ring, sm, g, pass);
    __syncthreads();
    // Publish this slice's total in every CTA of the cluster (remote stores ahead of the
    // barrier, so that no CTA reads another's shared memory after it).
    if (tid < C) *cluster.map_shared_rank(&sm.peer_total[pass][rank], tid) = sm.total[pass];
    cluster_arrive();
    cluster_wait();  // every slice total of this pass is here
    if (tid == 0) {
      const ff32 zero = {0.f, 0.f};
      ff32 all = zero, before = zero, last_pos_base = zero;
      int owner = -1, last = -1;
      for (int r = 0; r < C; ++r) all = ff_add(all, sm.peer_total[pass][r]);
      sm.all = all;
      sm.use_p = 0;
      if (!(all.hi > 0.f) && j < k && pass == 0) {
        sm.use_p = 1;  // zero residual after a rejection: draw from p_j instead
      } else if (all.hi > 0.f) {
        const ff32 target = ff_mul(sm.u1[j], all);
        ff32 run = zero;
        for (int r = 0; r < C; ++r) {
          const ff32 t = sm.peer_total[pass][r];
          if (t.hi > 0.f) {
            if (owner < 0 && ff_gt(ff_add(run, t), target)) {
              owner = r;
              before = run;
            }
            last = r;
            last_pos_base = run;
          }
          run = ff_add(run, t);
        }
        if (owner < 0) {  // rounding put the target past the total: last slice with mass
          owner = last;
          before = last_pos_base;
        }
        sm.target = target;
        sm.base = before;
      }
      sm.owner = owner;
    }
    __syncthreads();
    S = sm.all.hi;
    if (!sm.use_p) break;
    use_p = 1;
    if (rank == 0 && tid == 0) atomicOr(a.err, VAS_DEV_RESIDUAL_FALLBACK);
  }
  const float* qrow = use_p ? nullptr : qrow0;

  // 3. The CTA that holds the target finds the token: stage totals, then the stage's tile
  //    totals locate the tile; one warp rescans from that tile on.
  if (S > 0.f && sm.owner == rank && warp == 0) {
    const int n_stages = (x_end - x_begin + kStageElems - 1) / kStageElems;
    const ff32 target = sm.target;
    ff32 stage_base, tile_base;
    const int hs = warp_first_crossing(sm.stage, n_stages, sm.base, target, stage_base);
    const int ht = hs < 0 ? -1 : warp_first_crossing(sm.tile[hs], kWarps, stage_base, target, tile_base);
    if (ht < 0) {  // no stage or tile with mass (only possible with non-finite inputs)
      if (lane == 0) {
        out[j] = -1;
        atomicOr(a.err, VAS_DEV_EMPTY_ROW);
      }
    } else {
      const bool vec = ((reinterpret_cast<uintptr_t>(prow) | reinterpret_cast<uintptr_t>(qrow)) & 15) == 0;
      ff32 base = tile_base;
      int found = -1, last_pos = -1;
      for (int t0 = x_begin + (hs * kWarps + ht) * kTile; t0 < x_end && found < 0; t0 += kTile) {
        float w[kLaneElems];
        const int x0 = t0 + lane * kLaneElems;
        load_weights(prow, qrow, x0, x_end, vec, w);
        const float gs = group_sum(w);
        ff32 inc = {gs, 0.f};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const ff32 n = ff_shfl_up(inc, o);
          if (lane >= o) inc = ff_add(inc, n);
        }
        ff32 exc = ff_shfl_up(inc, 1);
        if (lane == 0) exc = {0.f, 0.f};
        const unsigned cross = __ballot_sync(0xffffffffu, gs > 0.f && ff_gt(ff_add(base, inc), target));
        int my_last = -1;
#pragma unroll
        for (int e = 0; e < kLaneElems; ++e)
          if (w[e] > 0.f) my_last = x0 + e;
#pragma unroll
        for (int o = 16; o; o >>= 1) my_last = max(my_last, __shfl_xor_sync(0xffffffffu, my_last, o));
        if (my_last >= 0) last_pos = my_last;
        if (cross) {
          const int src = __ffs(cross) - 1;
          int pick = -1;
          if (lane == src) {
            ff32 c = ff_add(base, exc);
            int lastpos_here = -1;
#pragma unroll
            for (int e = 0; e < kLaneElems; ++e) {
              if (w[e] > 0.f) {
                c = ff_add_f(c, w[e]);
                lastpos_here = x0 + e;
                if (pick < 0 && ff_gt(c, target)) pick = x0 + e;
              }
            }
            if (pick < 0) pick = lastpos_here;  // rounding inside the group
          }
          found = __shfl_sync(0xffffffffu, pick, src);
        }
        base = ff_add(base, ff_shfl(inc, 31));
      }
      if (lane == 0) out[j] = found >= 0 ? found : last_pos;
    }
  }

  // 4. The cluster's first CTA writes the accepted drafts, the padding and the length.
  if (rank == 0) {
    for (int t = tid; t <= k; t += kThreads) {
      if (t < j) out[t] = a.draft[(size_t)b * k + t];
      else if (t > j) out[t] = -1;
      else if (!(S > 0.f)) out[t] = -1;
    }
    if (tid == 0) {
      a.accepted_len[b] = j;
      if (!(S > 0.f)) atomicOr(a.err, VAS_DEV_EMPTY_ROW);
    }
  }
}

}  // namespace verify
}  // namespace vas

extern "C" int spec_verify(const float* p, const float* q, const int32_t* draft_tokens,
                           uint64_t seed, int32_t* accepted_len, int32_t* out_tokens, int32_t B,
                           int32_t k, int32_t V, vas_stream_t stream) {
  using namespace vas::verify;
  if (B < 0 || k < 0 || V <= 0) return VAS_E_INVALID_ARG;
  if (B == 0) return VAS_OK;
  if (!p || !accepted_len || !out_tokens || (k > 0 && (!q || !draft_tokens)))
    return VAS_E_INVALID_ARG;
  if ((int64_t)(k + 1) * V > INT32_MAX / 2) return VAS_E_INVALID_ARG;
  if (k >= kThreads) return VAS_E_INVALID_ARG;
  if ((int64_t)B * kMaxCluster > INT32_MAX) return VAS_E_INVALID_ARG;
  if ((int64_t)V > kMaxVocab) return VAS_E_UNSUPPORTED;
  int32_t* err = vas::device_error_word();
  if (!err) return VAS_E_CUDA;
  // The ring needs the dynamic shared-memory opt-in, once per device.
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VAS_E_CUDA;
  std::call_once(once[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(
        spec_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRingBytes);
  });
  if (attr_err[dev & 63] != cudaSuccess) return VAS_E_CUDA;
  int C = (V + kSliceMin - 1) / kSliceMin;
  if (C > kMaxCluster) C = kMaxCluster;
  int slice = (V + C - 1) / C;
  slice = (slice + kTile - 1) / kTile * kTile;
  C = (V + slice - 1) / slice;
  Args a;
  a.p = p;
  a.q = q;
  a.draft = draft_tokens;
  a.accepted_len = accepted_len;
  a.out_tokens = out_tokens;
  a.B = B;
  a.k = k;
  a.V = V;
  a.slice = slice;
  a.bulk = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(q)) & 15) == 0;
  a.key0 = static_cast<uint32_t>(seed);
  a.key1 = static_cast<uint32_t>(seed >> 32);
  a.err = err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kRingBytes;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, spec_verify_kernel, a) != cudaSuccess) {
    cudaGetLastError();
    return VAS_E_CUDA;
  }
  return VAS_OK;
}
