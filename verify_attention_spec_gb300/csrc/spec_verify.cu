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
// the k ratio tests itself (k scattered loads) and finds j.  One streaming pass over
// its slice of row j builds w = max(0, p_j - q_j) in fp32, sums 8 contiguous elements
// per lane in fp32 and everything above in fp64 (tile totals kept in shared memory),
// and publishes the slice total; after a cluster barrier every CTA reads all totals
// through distributed shared memory, so all agree on S and on the slice holding the
// target s_j * S.  In that CTA the stored warp and tile totals locate the tile; only
// that tile is read again, its lanes are scanned in fp64 and the crossing lane walks
// its 8 elements.  Uniforms come from Philox4x32-10 keyed by the seed with
// counter (position, sequence, 0, 0).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

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
constexpr int kMaxCluster = 8;
constexpr int kSliceMin = 4096;                 // smallest vocabulary slice per CTA
constexpr int kMaxTilesPerWarp = 64;            // bounds the vocabulary at 8 x 8 x 64 x 256
constexpr int64_t kMaxVocab = (int64_t)kMaxCluster * kWarps * kMaxTilesPerWarp * kTile;

struct Args {
  const float* p;
  const float* q;
  const int32_t* draft;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t B, k, V, slice;  // slice: vocabulary elements per CTA (multiple of kTile)
  uint32_t key0, key1;
  int32_t* err;
};

// The 8 weights of one lane's group starting at x0 (elements at or past end are zero).
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

__global__ void __launch_bounds__(kThreads) spec_verify_kernel(const Args a) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / C;

  __shared__ int32_t s_j, s_bad;
  __shared__ double s_warp[kWarps];
  __shared__ double s_tile[kWarps][kMaxTilesPerWarp];  // fp64 total of each warp tile
  __shared__ double s_total[2];  // this CTA's slice total, one slot per pass
  __shared__ double s_base, s_target, s_all;
  __shared__ int32_t s_owner, s_use_p, s_draw;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, V = a.V;
  pdl_wait_prior_grid();  // inputs written by the previous kernel in the stream are visible
  if (tid == 0) {
    s_j = k;
    s_bad = 0;
    s_draw = -1;
  }
  __syncthreads();

  // 1. Ratio tests (every CTA of the cluster, redundantly): thread i < k tests draft x_i
  //    with r_i = word 0 of Philox(i, b).
  if (tid < k) {
    const int x = a.draft[(size_t)b * k + tid];
    if (x < 0 || x >= V) {
      atomicOr(&s_bad, 1);
    } else {
      const double pi = a.p[((size_t)b * (k + 1) + tid) * V + x];
      const double qi = a.q[((size_t)b * k + tid) * V + x];
      const uint4 w = philox4x32_10(make_uint4((uint32_t)tid, (uint32_t)b, 0u, 0u), a.key0, a.key1);
      const double r = philox_uniform(w.x);
      if (!(r * qi <= pi)) atomicMin(&s_j, tid);
    }
  }
  __syncthreads();
  int32_t* out = a.out_tokens + (size_t)b * (k + 1);
  if (s_bad) {  // the same in every CTA of the cluster: all leave before any barrier
    if (rank == 0) {
      for (int t = tid; t <= k; t += kThreads) out[t] = -1;
      if (tid == 0) {
        a.accepted_len[b] = -1;
        atomicOr(a.err, VAS_DEV_BAD_TOKEN);
      }
    }
    return;
  }
  const int j = s_j;

  // 2. This CTA's slice of the row to draw from; warps take consecutive tiles.
  const int sl_begin = rank * a.slice;
  const int sl_end = min(V, sl_begin + a.slice);
  const int warp_span = ((a.slice + kWarps * kTile - 1) / (kWarps * kTile)) * kTile;
  const int x_begin = min(sl_end, sl_begin + warp * warp_span);
  const int x_end = min(sl_end, x_begin + warp_span);
  const float* prow = a.p + ((size_t)b * (k + 1) + j) * V;
  const float* qrow0 = j < k ? a.q + ((size_t)b * k + j) * V : nullptr;
  int use_p = 0;
  double S = 0.0;
  for (int pass = 0; pass < 2; ++pass) {
    const float* qrow = use_p ? nullptr : qrow0;
    const bool vec = ((reinterpret_cast<uintptr_t>(prow) | reinterpret_cast<uintptr_t>(qrow)) & 15) == 0;
    // Tile totals: fp32 over each lane's 8 elements, fp64 across the 32 lanes.  Four
    // tiles per iteration keep several loads of each lane in flight.
    const int n_tiles = (x_end - x_begin + kTile - 1) / kTile;
    for (int t = 0; t < n_tiles; t += 4) {
      float gsum[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float w[kLaneElems];
        const int x0 = x_begin + (t + u) * kTile + lane * kLaneElems;
        if (t + u < n_tiles) load_weights(prow, qrow, x0, x_end, vec, w);
        else
#pragma unroll
          for (int e = 0; e < kLaneElems; ++e) w[e] = 0.f;
        gsum[u] = group_sum(w);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        double v = (double)gsum[u];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && t + u < n_tiles) s_tile[warp][t + u] = v;
      }
    }
    __syncwarp();
    if (lane == 0) {
      double acc = 0.0;
      for (int t = 0; t < n_tiles; ++t) acc += s_tile[warp][t];
      s_warp[warp] = acc;
    }
    __syncthreads();
    if (tid == 0) {
      double run = 0.0;
      for (int w = 0; w < kWarps; ++w) run += s_warp[w];
      s_total[pass] = run;
    }
    cluster.sync();  // every slice total of this pass is published
    if (tid == 0) {
      double before = 0.0, all = 0.0, last_pos_base = 0.0;
      int owner = -1, last = -1;
      double tot[kMaxCluster];
      for (int r = 0; r < C; ++r) {
        tot[r] = *cluster.map_shared_rank(&s_total[pass], r);
        all += tot[r];
      }
      s_all = all;
      s_use_p = 0;
      if (all == 0.0 && j < k && pass == 0) {
        s_use_p = 1;  // zero residual after a rejection: draw from p_j instead
      } else if (all > 0.0) {
        const uint4 w = philox4x32_10(make_uint4((uint32_t)j, (uint32_t)b, 0u, 0u), a.key0, a.key1);
        const double target = philox_uniform(w.y) * all;
        double run = 0.0;
        for (int r = 0; r < C; ++r) {
          if (tot[r] > 0.0) {
            if (owner < 0 && run + tot[r] > target) {
              owner = r;
              before = run;
            }
            last = r;
            last_pos_base = run;
          }
          run += tot[r];
        }
        if (owner < 0) {  // rounding put the target past the total: last slice with mass
          owner = last;
          before = last_pos_base;
        }
        s_target = target;
        s_base = before;
      }
      s_owner = owner;
    }
    __syncthreads();
    S = s_all;
    if (!s_use_p) break;
    use_p = 1;
    if (rank == 0 && tid == 0) atomicOr(a.err, VAS_DEV_RESIDUAL_FALLBACK);
  }
  const float* qrow = use_p ? nullptr : qrow0;

  // 3. The CTA that holds the target finds the token: warp totals first, then the
  //    crossing warp rescans its range tile by tile.
  if (S > 0.0 && s_owner == rank) {
    if (tid == 0) {
      double run = s_base;
      int hit = -1, lastw = -1;
      double hit_base = 0.0, last_base = 0.0;
      for (int w = 0; w < kWarps; ++w) {
        if (s_warp[w] > 0.0) {
          if (hit < 0 && run + s_warp[w] > s_target) {
            hit = w;
            hit_base = run;
          }
          lastw = w;
          last_base = run;
        }
        run += s_warp[w];
      }
      if (hit < 0) {
        hit = lastw;
        hit_base = last_base;
      }
      s_owner = hit;  // reused: the warp that rescans
      s_base = hit_base;
    }
    __syncthreads();
    if (warp == s_owner) {
      const bool vec = ((reinterpret_cast<uintptr_t>(prow) | reinterpret_cast<uintptr_t>(qrow)) & 15) == 0;
      const double target = s_target;
      // The tile that holds the target, from the stored tile totals (no memory traffic).
      const int n_tiles = (x_end - x_begin + kTile - 1) / kTile;
      double base = s_base;
      int t_hit = -1, t_last = -1;
      double b_hit = 0.0, b_last = 0.0;
      {
        double run = base;
        for (int t = 0; t < n_tiles; ++t) {
          const double v = s_tile[warp][t];
          if (v > 0.0) {
            if (t_hit < 0 && run + v > target) {
              t_hit = t;
              b_hit = run;
            }
            t_last = t;
            b_last = run;
          }
          run += v;
        }
      }
      if (t_hit < 0) {
        t_hit = t_last;
        b_hit = b_last;
      }
      base = b_hit;
      int found = -1, last_pos = -1;
      for (int t0 = x_begin + t_hit * kTile; t0 < x_end && found < 0; t0 += kTile) {
        float w[kLaneElems];
        const int x0 = t0 + lane * kLaneElems;
        load_weights(prow, qrow, x0, x_end, vec, w);
        const double gs = (double)group_sum(w);
        double inc = gs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double n = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += n;
        }
        const double excl = base + inc - gs;
        const unsigned cross = __ballot_sync(0xffffffffu, gs > 0.0 && base + inc > target);
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
            double c = excl;
            int lastpos_here = -1;
#pragma unroll
            for (int e = 0; e < kLaneElems; ++e) {
              if (w[e] > 0.f) {
                c += (double)w[e];
                lastpos_here = x0 + e;
                if (pick < 0 && c > target) pick = x0 + e;
              }
            }
            if (pick < 0) pick = lastpos_here;  // rounding inside the group
          }
          found = __shfl_sync(0xffffffffu, pick, src);
        }
        base += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (lane == 0) out[j] = found >= 0 ? found : last_pos;
    }
  }

  // 4. The cluster's first CTA writes the accepted drafts, the padding and the length.
  if (rank == 0) {
    for (int t = tid; t <= k; t += kThreads) {
      if (t < j) out[t] = a.draft[(size_t)b * k + t];
      else if (t > j) out[t] = -1;
      else if (S == 0.0) out[t] = -1;
    }
    if (tid == 0) {
      a.accepted_len[b] = j;
      if (S == 0.0) atomicOr(a.err, VAS_DEV_EMPTY_ROW);
    }
  }
  cluster.sync();  // no CTA leaves while a peer may still read its shared memory
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
  a.key0 = static_cast<uint32_t>(seed);
  a.key1 = static_cast<uint32_t>(seed >> 32);
  a.err = err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * C));
  cfg.blockDim = dim3(kThreads);
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
