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
// For a chain this is spec_verify's rule with its uniforms: r_c is word 0 of
// Philox(c - 1, b), the draw at node u uses word 1 of Philox(u, b).
//
// Kernel: one CTA of 512 threads per sequence; thread 0 takes the decisions, the CTA
// makes the passes over the vocabulary.  A pass covers the row in tiles of 256
// consecutive elements, 8 contiguous per lane: each lane sums its 8 weights, the warp
// scans the 32 lane sums (fp32, lane order) and the last lane's value is the tile's
// total, kept in shared memory; tile totals add up in fp64.  The residual's new total
// is the sum of the tile totals; a draw walks the tile totals to the tile where the
// inverse CDF crosses its target, repeats that tile's scan and walks the crossing
// lane's 8 elements.  Weights are fp32 (R_k recomputed per element from p, q and
// S_0..S_{k-1}); totals and thresholds are fp64 (this part's fp64 rate is too low for
// fp64 per element).
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/vas.h"
#include "device_util.cuh"
#include "philox.cuh"
#include "vas_internal.h"

namespace vas {
namespace verify_tree {

constexpr int kThreads = 512;
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
  int32_t B, n, V;
  uint32_t key0, key1;
  int32_t* err;
};

// R_k(y): R_0 = p, R_{i+1} = max(0, R_i - S_i q), with S_0 = 1 (fp32 per element).
__device__ __forceinline__ float residual(float p, float q, const float* S, int k) {
  float r = p;
  for (int i = 0; i < k; ++i) r = fmaxf(r - S[i] * q, 0.f);
  return r;
}

// The weight of element y in a pass: the rejection's new residual (next = true), or
// the row to draw from (p_u, or R_k).
__device__ __forceinline__ float weight(float p, float q, const float* S, int k, bool from_p,
                                        bool next) {
  if (next) return fmaxf(residual(p, q, S, k) - S[k] * q, 0.f);
  return from_p ? p : residual(p, q, S, k);
}

constexpr int kLaneElems = 8;
constexpr int kTile = 32 * kLaneElems;
constexpr int kMaxTiles = (128256 * 2 + kTile - 1) / kTile;  // vocabularies up to 256512

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
                                              bool vec, const float* S, int k, bool from_p,
                                              bool next, float (&w)[kLaneElems]) {
  float p8[kLaneElems], q8[kLaneElems];
  lane_load(pu, qu, x0, V, vec, p8, q8);
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < kLaneElems; ++e) {
    w[e] = x0 + e < V ? weight(p8[e], q8[e], S, k, from_p, next) : 0.f;
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

// A pass: every tile's total into s_tile[]; returns the row total (every thread)
// and the last element with positive weight (thread 0's *last).
__device__ double pass_totals(const float* pu, const float* qu, int V, const float* S, int k,
                              bool from_p, bool next, double* s_tile, int* s_last,
                              double* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_tiles = (V + kTile - 1) / kTile;
  const bool vec = ((reinterpret_cast<uintptr_t>(pu) | reinterpret_cast<uintptr_t>(qu)) & 15) == 0;
  if (threadIdx.x == 0) *s_last = -1;
  __syncthreads();
  int last = -1;
  // Four tiles per iteration keep several loads of each lane in flight.
  for (int t0 = warp * 4; t0 < n_tiles; t0 += kWarps * 4) {
    // All four tiles' loads go out before any of them is used.
    float p8[4][kLaneElems], q8[4][kLaneElems];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int x0 = (t0 + j) * kTile + lane * kLaneElems;
      if (t0 + j < n_tiles) lane_load(pu, qu, x0, V, vec, p8[j], q8[j]);
    }
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int x0 = (t0 + j) * kTile + lane * kLaneElems;
      v[j] = 0.f;
      if (t0 + j < n_tiles)
#pragma unroll
        for (int e = 0; e < kLaneElems; ++e) {
          const float w = x0 + e < V ? weight(p8[j][e], q8[j][e], S, k, from_p, next) : 0.f;
          v[j] += w;
          if (w > 0.f) last = x0 + e;
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
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

__global__ void __launch_bounds__(kThreads, 1) spec_verify_tree_kernel(const Args a) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.n, V = a.V;
  __shared__ int32_t s_par[kMaxNodes], s_x[kMaxNodes];
  __shared__ double s_S[kMaxNodes + 1];
  __shared__ float s_Sf[kMaxNodes + 1];
  __shared__ double s_tile[kMaxTiles];
  __shared__ double s_total;
  __shared__ int32_t s_bad, s_accept, s_tile_hit, s_found, s_last;
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
  for (int t = tid; t <= n; t += kThreads) out[t] = -1;
  for (int t = tid; t < n; t += kThreads) path[t] = -1;
  if (s_bad) {
    if (tid == 0) {
      a.accepted_len[b] = -1;
      atomicOr(a.err, (s_bad & 1 ? VAS_DEV_BAD_TOKEN : 0) | (s_bad & 2 ? VAS_DEV_BAD_TREE : 0));
    }
    return;
  }

  int u = 0, depth = 0;
  for (;;) {
    const float* pu = a.p + ((size_t)b * (n + 1) + u) * V;
    const float* qu = a.q + ((size_t)b * n + (u < n ? u : 0)) * V;
    int k = 0, next = -1;
    bool fallback = false;
    if (tid == 0) {
      s_S[0] = 1.0;
      s_Sf[0] = 1.f;
    }
    for (int c = u + 1; c <= n; ++c) {
      if (s_par[c - 1] != u) continue;
      if (tid == 0) {
        const int x = s_x[c - 1];
        const float qx = qu[x];
        const double rx = residual(pu[x], qx, s_Sf, k);
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
      const double total = pass_totals(pu, qu, V, s_Sf, k, false, true, s_tile, &s_last, &s_total);
      ++k;
      if (tid == 0) {
        s_S[k] = total;
        s_Sf[k] = (float)total;
      }
      __syncthreads();
      if (total == 0.0) {
        fallback = true;
        break;
      }
    }
    if (next >= 0) {
      if (tid == 0) {
        out[depth] = s_x[next - 1];
        path[depth] = next;
      }
      ++depth;
      u = next;
      continue;
    }
    // Draw at node u: from R_k, or from p_u (nothing rejected, or the fallback).
    const bool from_p = k == 0 || fallback;
    const double total = pass_totals(pu, qu, V, s_Sf, k, from_p, false, s_tile, &s_last, &s_total);
    const int n_tiles = (V + kTile - 1) / kTile;
    double target = 0.0;
    if (total > 0.0) {
      const uint4 w4 = philox4x32_10(make_uint4((uint32_t)u, (uint32_t)b, 0u, 0u), a.key0, a.key1);
      target = philox_uniform(w4.y) * total;
    }
    if (tid == 0) {
      // The tile where the running total passes the target (tiles in order).
      s_tile_hit = -1;
      s_found = -1;
      double c = 0.0;
      for (int t = 0; t < n_tiles && total > 0.0; ++t) {
        if (c + s_tile[t] > target) {
          s_tile_hit = t;
          s_total = c;  // the total before the tile
          break;
        }
        c += s_tile[t];
      }
    }
    __syncthreads();
    if (warp == 0 && s_tile_hit >= 0) {
      // Repeat the tile's scan; the lane whose span holds the target walks its elements
      // (its last element with weight when rounding leaves the target past them).
      float w[kLaneElems];
      const int x0 = s_tile_hit * kTile + lane * kLaneElems;
      const bool vec = ((reinterpret_cast<uintptr_t>(pu) | reinterpret_cast<uintptr_t>(qu)) & 15) == 0;
      const float ls = lane_weights(pu, qu, x0, V, vec, s_Sf, k, from_p, false, w);
      const float inc = warp_inclusive_scan(ls);
      const double hi = s_total + (double)inc;
      const double up = __shfl_up_sync(0xffffffffu, hi, 1);
      const double lo = lane == 0 ? s_total : up;  // the spans tile [before, before + tile)
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
    if (tid == 0) {
      // Rounding can leave the target at or past the last crossing: the last token with
      // mass, as for the plain rule.
      const int drawn = total > 0.0 ? (s_found >= 0 ? s_found : s_last) : -1;
      out[depth] = drawn;
      a.accepted_len[b] = depth;
      if (drawn < 0) atomicOr(a.err, VAS_DEV_EMPTY_ROW);
      if (fallback) atomicOr(a.err, VAS_DEV_RESIDUAL_FALLBACK);
    }
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
  if ((int64_t)V > (int64_t)kMaxTiles * kTile) return VAS_E_UNSUPPORTED;
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
  a.key0 = static_cast<uint32_t>(seed);
  a.key1 = static_cast<uint32_t>(seed >> 32);
  a.err = err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, spec_verify_tree_kernel, a) != cudaSuccess) {
    cudaGetLastError();
    return VAS_E_CUDA;
  }
  return VAS_OK;
}
