// Verification of a draft tree (sm_103a).
//
// The pages verify a tree of candidates in one pass ("Continuous Batching & Speculative
// Decoding", section "4. Tree Attention & Medusa Heads") and give the rule for one
// candidate ("The Modified Rejection Sampling Algorithm"); the walk applies that rule to
// a node's children in turn:
//   at node u (the root is node 0, the last context token) the children, in node order,
//   are tested against a residual R with total S (R = p_u and S = 1 at first): child c
//   with token x is accepted iff r_c S q_u(x) <= R(x); a rejection turns R into
//   max(0, R - S q_u) and S into its sum.  An accepted child becomes u.  When a node's
//   children are all rejected, or it has none, one token is drawn from R by inverse CDF
//   and the walk ends.  A zero residual after a rejection draws from p_u instead.
// With q_u >= 0 and every S >= 0 the residual after k rejections has a closed form,
// R_k = max(0, p_u - c_k q_u) with c_k = S_0 + ... + S_{k-1} (by induction: where
// R_{k-1} = 0, p_u <= c_{k-1} q_u <= c_k q_u), so each element costs one product and
// one maximum in any pass.
// For a chain this is spec_verify's rule with its uniforms: r_c is word 0 of
// Philox(c - 1, b), the draw at node u uses word 1 of Philox(u, b).
//
// Kernel: one thread-block cluster of C CTAs per sequence (C <= 8, fewer for small
// vocabularies and for batches that would not fit four CTAs per SM); CTA r owns slice r
// of the vocabulary.  Every CTA takes the same
// decisions (thread 0, from the same values), so the clusters' CTAs walk in step.  A
// pass covers each slice in tiles of 256 consecutive elements, 8 contiguous per lane:
// each lane sums its 8 weights, the warp scans the 32 lane sums (fp32, lane order) and
// the last lane's value is the tile's total, kept in shared memory; tile totals add up
// in fp64 to the slice total, which each CTA stores into every CTA of the cluster before
// the pass's cluster barrier; every CTA then adds the C slice totals in rank order.  A draw finds the slice, then the tile where the inverse CDF
// crosses its target; that CTA repeats the tile's scan and walks the crossing lane's 8
// elements.  Weights are fp32 (R_k from p, q and c_k); totals, c_k and thresholds are
// fp64 (this part's fp64 rate is too low for fp64 per element).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/vas.h"
#include "device_util.cuh"
#include "philox.cuh"
#include "vas_internal.h"

namespace cg = cooperative_groups;

namespace vas {
namespace verify_tree {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNodes = 255;  // draft nodes per sequence (node indices fit in a byte)

struct Args {
  const float* p;  // [B, n + 1, V]
  const float* q;  // [B, n, V]
  const int32_t* draft;    // [B, n]
  const int32_t* parents;  // [B, n]: parent of node i + 1, in 0..i
  int32_t* accepted_len;   // [B]
  int32_t* out_tokens;     // [B, n + 1]
  int32_t* path;           // [B, n]
  int32_t B, n, V, slice;  // slice: vocabulary elements per CTA (multiple of kTile)
  uint32_t key0, key1;
  int32_t* err;
};

// The weight of element y in a pass: max(0, p - c q), the residual for the pass's
// c (c_{k+1} for a rejection's new residual, c_k for a draw from R_k); a draw from p_u
// passes c = 0.
__device__ __forceinline__ float weight(float p, float q, float c) {
  return fmaxf(fmaf(-c, q, p), 0.f);
}

constexpr int kLaneElems = 8;
constexpr int kTile = 32 * kLaneElems;
constexpr int kMaxCluster = 8;
constexpr int kSliceMin = 4096;     // smallest vocabulary slice per CTA
constexpr int kMaxTiles = 160;      // tiles per slice: vocabularies up to 8 x 160 x 256
// One tile per warp in flight keeps the kernel at 64 registers, so four CTAs share an SM
// and a batch of 64 trees still gets eight CTAs per tree: shorter passes, which is what
// the walk's chain of passes waits on (four tiles in flight at two CTAs per SM measured
// 94 us on 64 trees over V = 128256, this 80 us).
constexpr int kTilesPerIter = 1;
constexpr int kCtasPerSm = 4;
constexpr int64_t kMaxVocab = (int64_t)kMaxCluster * kMaxTiles * kTile;

// One lane's 8 inputs from x0 (past V: zero), as two float4 loads per row when the
// rows are 16-byte aligned and the 8 elements lie inside the row.
__device__ __forceinline__ void lane_load(const float* pu, const float* qu, int x0, int V,
                                          bool vec, float (&p8)[kLaneElems],
                                          float (&q8)[kLaneElems]) {
  if (vec && x0 + kLaneElems <= V) {
    const float4 a0 = __ldg(reinterpret_cast<const float4*>(pu + x0));
    const float4 a1 = __ldg(reinterpret_cast<const float4*>(pu + x0 + 4));
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(qu + x0));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(qu + x0 + 4));
    p8[0] = a0.x; p8[1] = a0.y; p8[2] = a0.z; p8[3] = a0.w;
    p8[4] = a1.x; p8[5] = a1.y; p8[6] = a1.z; p8[7] = a1.w;
    q8[0] = b0.x; q8[1] = b0.y; q8[2] = b0.z; q8[3] = b0.w;
    q8[4] = b1.x; q8[5] = b1.y; q8[6] = b1.z; q8[7] = b1.w;
  } else {
#pragma unroll
    for (int e = 0; e < kLaneElems; ++e) {
      p8[e] = x0 + e < V ? __ldg(pu + x0 + e) : 0.f;
      q8[e] = x0 + e < V ? __ldg(qu + x0 + e) : 0.f;
    }
  }
}

// One lane's 8 weights from x0 (past V: zero), and their fp32 sum.
__device__ __forceinline__ float lane_weights(const float* pu, const float* qu, int x0, int V,
                                              bool vec, float c, float (&w)[kLaneElems]) {
  float p8[kLaneElems], q8[kLaneElems];
  lane_load(pu, qu, x0, V, vec, p8, q8);
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < kLaneElems; ++e) {
    w[e] = x0 + e < V ? weight(p8[e], q8[e], c) : 0.f;
    sum += w[e];
  }
  return sum;
}

// Inclusive scan of one fp32 value per lane, in lane order (the tile totals and the
// draw's rescan of a tile run the same code, so they agree to the bit).
__device__ __forceinline__ float warp_inclusive_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// A pass over this CTA's slice [xb, V' = min(V, xb + slice)): every tile's total into
// s_tile[]; returns the slice total (every thread) and leaves the slice's last element
// with positive weight in *s_last.
__device__ double pass_totals(const float* pu, const float* qu, int xb, int V, float c,
                              double* s_tile, int* s_last, double* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_tiles = (V - xb + kTile - 1) / kTile;
  const bool vec = ((reinterpret_cast<uintptr_t>(pu) | reinterpret_cast<uintptr_t>(qu)) & 15) == 0;
  if (threadIdx.x == 0) *s_last = -1;
  __syncthreads();
  int last = -1;
  // kTilesPerIter tiles per iteration: their loads all go out before any is used.
  for (int t0 = warp * kTilesPerIter; t0 < n_tiles; t0 += kWarps * kTilesPerIter) {
    float p8[kTilesPerIter][kLaneElems], q8[kTilesPerIter][kLaneElems];
#pragma unroll
    for (int j = 0; j < kTilesPerIter; ++j) {
      const int x0 = xb + (t0 + j) * kTile + lane * kLaneElems;
      if (t0 + j < n_tiles) lane_load(pu, qu, x0, V, vec, p8[j], q8[j]);
    }
    float v[kTilesPerIter];
#pragma unroll
    for (int j = 0; j < kTilesPerIter; ++j) {
      const int x0 = xb + (t0 + j) * kTile + lane * kLaneElems;
      v[j] = 0.f;
      if (t0 + j < n_tiles)
#pragma unroll
        for (int e = 0; e < kLaneElems; ++e) {
          const float w = x0 + e < V ? weight(p8[j][e], q8[j][e], c) : 0.f;
          v[j] += w;
          if (w > 0.f) last = x0 + e;
        }
    }
#pragma unroll
    for (int j = 0; j < kTilesPerIter; ++j) {
      const float tile = warp_inclusive_scan(v[j]);
      if (lane == 31 && t0 + j < n_tiles) s_tile[t0 + j] = tile;
    }
  }
  if (last >= 0) atomicMax(s_last, last);
  __syncthreads();
  if (warp == 0) {  // the row total, tiles in order
    double v = 0.0;
    for (int t = lane; t < n_tiles; t += 32) v += s_tile[t];
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) *s_total = v;
  }
  __syncthreads();
  return *s_total;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) spec_verify_tree_kernel(const Args a) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.n, V = a.V;
  const int xb = min(V, rank * a.slice), xe = min(V, xb + a.slice);  // this CTA's slice
  __shared__ int32_t s_par[kMaxNodes], s_x[kMaxNodes];
  __shared__ float s_pux[kMaxNodes], s_qux[kMaxNodes];  // p_u, q_u at the child's token
  __shared__ double s_S[kMaxNodes + 1];  // S_0 .. S_k of the current node
  __shared__ double s_tile[kMaxTiles];
  __shared__ double s_total;
  __shared__ int32_t s_last;
  // Every rank's slice total and last element with weight, stored here by that rank
  // before the pass's cluster barrier; two sets, by pass parity.
  __shared__ double s_pub[2][kMaxCluster];
  __shared__ int32_t s_pub_last[2][kMaxCluster];
  __shared__ int32_t s_bad, s_accept, s_tile_hit, s_found;
  __shared__ double s_target, s_before;
  pdl_wait_prior_grid();  // inputs written by the previous kernel in the stream are visible

  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) {
    const int pi = a.parents[(size_t)b * n + i];
    const int xi = a.draft[(size_t)b * n + i];
    s_par[i] = pi;
    s_x[i] = xi;
    if (pi < 0 || pi > i) atomicOr(&s_bad, 2);
    if (xi < 0 || xi >= V) atomicOr(&s_bad, 1);
  }
  __syncthreads();
  int32_t* out = a.out_tokens + (size_t)b * (n + 1);
  int32_t* path = a.path + (size_t)b * n;
  if (rank == 0) {
    for (int t = tid; t <= n; t += kThreads) out[t] = -1;
    for (int t = tid; t < n; t += kThreads) path[t] = -1;
  }
  if (s_bad) {  // the same in every CTA of the cluster: all leave before any barrier
    if (rank == 0 && tid == 0) {
      a.accepted_len[b] = -1;
      atomicOr(a.err, (s_bad & 1 ? VAS_DEV_BAD_TOKEN : 0) | (s_bad & 2 ? VAS_DEV_BAD_TREE : 0));
    }
    return;
  }

  int pp = 0;  // publication slot: passes alternate, one cluster barrier each
  // A pass over the slices; returns the row total, identical in every CTA (slice
  // totals added in rank order), and the row's last element with weight in *last.
  auto cluster_pass = [&](const float* pu, const float* qu, float c, int* last) -> double {
    const double mine = pass_totals(pu, qu, xb, xe, c, s_tile, &s_last, &s_total);
    if (tid < C) {  // this slice's total into every rank of the cluster
      *cluster.map_shared_rank(&s_pub[pp][rank], tid) = mine;
      *cluster.map_shared_rank(&s_pub_last[pp][rank], tid) = s_last;
    }
    cluster.sync();  // every slice total of this pass is here
    double all = 0.0;
    int lst = -1;
    for (int r = 0; r < C; ++r) {
      all += s_pub[pp][r];
      lst = max(lst, s_pub_last[pp][r]);
    }
    pp ^= 1;
    *last = lst;
    return all;
  };

  int u = 0, depth = 0;
  for (;;) {
    const float* pu = a.p + ((size_t)b * (n + 1) + u) * V;
    const float* qu = a.q + ((size_t)b * n + (u < n ? u : 0)) * V;
    int k = 0, next = -1, last = -1;
    bool fallback = false;
    double ck = 0.0;  // c_k = S_0 + ... + S_{k-1} (every thread keeps the same sum)
    if (tid == 0) s_S[0] = 1.0;
    // p_u and q_u at every child's token, loaded at once.
    for (int i = u + tid; i < n; i += kThreads)
      if (s_par[i] == u) {
        s_pux[i] = pu[s_x[i]];
        s_qux[i] = qu[s_x[i]];
      }
    __syncthreads();
    for (int c = u + 1; c <= n; ++c) {
      if (s_par[c - 1] != u) continue;
      if (tid == 0) {
        const float qx = s_qux[c - 1];
        const double rx = fmax((double)s_pux[c - 1] - ck * (double)qx, 0.0);
        const uint4 w = philox4x32_10(make_uint4((uint32_t)(c - 1), (uint32_t)b, 0u, 0u),
                                      a.key0, a.key1);
        s_accept = philox_uniform(w.x) * s_S[k] * (double)qx <= rx;
      }
      __syncthreads();
      const bool accepted = s_accept;
      __syncthreads();  // read by every thread before thread 0 can write the next test
      if (accepted) {
        next = c;
        break;
      }
      // Rejected: the new residual's total.
      ck += s_S[k];
      const double total = cluster_pass(pu, qu, (float)ck, &last);
      ++k;
      if (tid == 0) s_S[k] = total;
      __syncthreads();
      if (total == 0.0) {
        fallback = true;
        break;
      }
    }
    if (next >= 0) {
      if (rank == 0 && tid == 0) {
        out[depth] = s_x[next - 1];
        path[depth] = next;
      }
      ++depth;
      u = next;
      continue;
    }
    // Draw at node u: from R_k, or from p_u (nothing rejected, or the fallback).
    const bool from_p = k == 0 || fallback;
    const double total = cluster_pass(pu, qu, from_p ? 0.f : (float)ck, &last);
    if (tid == 0) {
      s_tile_hit = -1;
      s_found = -1;
      if (total > 0.0) {
        const uint4 w4 = philox4x32_10(make_uint4((uint32_t)u, (uint32_t)b, 0u, 0u), a.key0,
                                       a.key1);
        const double target = philox_uniform(w4.y) * total;
        // The slice (rank order, as the total was formed), then the tile, where the
        // running total passes the target.
        double c = 0.0;
        int owner = -1;
        for (int r = 0; r < C; ++r) {
          const double t = s_pub[pp ^ 1][r];
          if (owner < 0 && c + t > target) owner = r;
          if (owner < 0) c += t;
        }
        if (owner == rank) {
          const int n_tiles = (xe - xb + kTile - 1) / kTile;
          for (int t = 0; t < n_tiles; ++t) {
            if (c + s_tile[t] > target) {
              s_tile_hit = t;
              break;
            }
            c += s_tile[t];
          }
        }
        s_target = target;
        s_before = c;  // the total before the tile
      }
    }
    __syncthreads();
    if (warp == 0 && s_tile_hit >= 0) {
      // Repeat the tile's scan; the lane whose span holds the target walks its elements
      // (its last element with weight when rounding leaves the target past them).
      float w[kLaneElems];
      const int x0 = xb + s_tile_hit * kTile + lane * kLaneElems;
      const bool vec = ((reinterpret_cast<uintptr_t>(pu) | reinterpret_cast<uintptr_t>(qu)) & 15) == 0;
      const float ls = lane_weights(pu, qu, x0, xe, vec, from_p ? 0.f : (float)ck, w);
      const float inc = warp_inclusive_scan(ls);
      const double target = s_target;
      const double hi = s_before + (double)inc;
      const double up = __shfl_up_sync(0xffffffffu, hi, 1);
      const double lo = lane == 0 ? s_before : up;  // the spans tile [before, before + tile)
      if (ls > 0.f && lo <= target && target < hi) {
        double c = lo;
        int pick = -1;
#pragma unroll
        for (int e = 0; e < kLaneElems; ++e) {
          if (w[e] > 0.f) pick = x0 + e;
          c += w[e];
          if (w[e] > 0.f && c > target) break;
        }
        atomicMax(&s_found, pick);  // the lanes' spans do not overlap
      }
    }
    __syncthreads();
    if (tid < C) *cluster.map_shared_rank(&s_pub_last[pp][rank], tid) = s_found;  // for the cluster
    cluster.sync();
    if (rank == 0 && tid == 0) {
      int found = -1;
      for (int r = 0; r < C; ++r) found = max(found, s_pub_last[pp][r]);
      // Rounding can leave the target at or past the last crossing: the last token with
      // mass, as for the plain rule.
      const int drawn = total > 0.0 ? (found >= 0 ? found : last) : -1;
      out[depth] = drawn;
      a.accepted_len[b] = depth;
      if (drawn < 0) atomicOr(a.err, VAS_DEV_EMPTY_ROW);
      if (fallback) atomicOr(a.err, VAS_DEV_RESIDUAL_FALLBACK);
    }
    cluster.sync();  // no CTA leaves while a peer may still read its shared memory
    return;
  }
}

}  // namespace verify_tree
}  // namespace vas

extern "C" int spec_verify_tree(const float* p, const float* q, const int32_t* draft_tokens,
                                const int32_t* parents, uint64_t seed, int32_t* accepted_len,
                                int32_t* out_tokens, int32_t* path, int32_t B, int32_t n,
                                int32_t V, vas_stream_t stream) {
  using namespace vas::verify_tree;
  if (B < 0 || n < 1 || n > kMaxNodes || V <= 0) return VAS_E_INVALID_ARG;
  if (B == 0) return VAS_OK;
  if (!p || !q || !draft_tokens || !parents || !accepted_len || !out_tokens || !path)
    return VAS_E_INVALID_ARG;
  if ((int64_t)(n + 1) * V > INT32_MAX / 2) return VAS_E_INVALID_ARG;
  if ((int64_t)V > kMaxVocab) return VAS_E_UNSUPPORTED;
  if ((int64_t)B * kMaxCluster > INT32_MAX) return VAS_E_INVALID_ARG;
  int32_t* err = vas::device_error_word();
  if (!err) return VAS_E_CUDA;
  Args a;
  a.p = p;
  a.q = q;
  a.draft = draft_tokens;
  a.parents = parents;
  a.accepted_len = accepted_len;
  a.out_tokens = out_tokens;
  a.path = path;
  a.B = B;
  a.n = n;
  a.V = V;
  // Cluster size and slices as for spec_verify: slices of at least kSliceMin elements,
  // whole tiles.
  // Each sequence's walk is long-lived: with many sequences, fewer CTAs per sequence
  // keep the whole grid resident (kCtasPerSm CTAs per SM).
  int C = (V + kSliceMin - 1) / kSliceMin;
  if (C > kMaxCluster) C = kMaxCluster;
  const int sms = vas::num_sms();
  while (C > 1 && (int64_t)B * C > (int64_t)kCtasPerSm * (sms > 0 ? sms : 148)) --C;
  int slice = (V + C - 1) / C;
  slice = (slice + kTile - 1) / kTile * kTile;
  C = (V + slice - 1) / slice;
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
  if (cudaLaunchKernelEx(&cfg, spec_verify_tree_kernel, a) != cudaSuccess) {
    cudaGetLastError();
    return VAS_E_CUDA;
  }
  return VAS_OK;
}
