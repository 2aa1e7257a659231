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
// Kernel: one CTA of 256 threads per sequence.  Thread 0 takes the decisions; the CTA
// makes the passes over the vocabulary: each thread owns a contiguous chunk of it, so
// one block scan of the 256 chunk totals locates the chunk where the inverse CDF
// crosses its target, and its thread walks that chunk.  The residual and every sum are
// in fp64 (the inputs are fp32), R_k recomputed per element from p, q and S_0..S_{k-1}.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/vas.h"
#include "device_util.cuh"
#include "philox.cuh"
#include "vas_internal.h"

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
  int32_t B, n, V;
  uint32_t key0, key1;
  int32_t* err;
};

// R_k(y): R_0 = p, R_{i+1} = max(0, R_i - S_i q), with S_0 = 1.
__device__ __forceinline__ double residual(double p, double q, const double* S, int k) {
  double r = p;
  for (int i = 0; i < k; ++i) r = fmax(r - S[i] * q, 0.0);
  return r;
}

// Block-wide exclusive scan of one double per thread; returns the thread's exclusive
// prefix and writes the block total to *total.
__device__ double block_exclusive_scan(double v, double* s_warp, double* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  __syncthreads();  // s_warp may still be read by a previous scan
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  double base = 0.0, all = 0.0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) base += s_warp[w];
    all += s_warp[w];
  }
  *total = all;
  return base + inc - v;
}

__global__ void __launch_bounds__(kThreads) spec_verify_tree_kernel(const Args a) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = a.n, V = a.V;
  __shared__ int32_t s_par[kMaxNodes], s_x[kMaxNodes];
  __shared__ double s_S[kMaxNodes + 1];
  __shared__ double s_warp[kWarps];
  __shared__ int32_t s_bad, s_accept, s_found, s_last;
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

  const int chunk = (V + kThreads - 1) / kThreads;
  const int y0 = min(V, tid * chunk), y1 = min(V, y0 + chunk);
  int u = 0, depth = 0;
  for (;;) {
    const float* pu = a.p + ((size_t)b * (n + 1) + u) * V;
    const float* qu = a.q + ((size_t)b * n + (u < n ? u : 0)) * V;
    int k = 0, next = -1;
    bool fallback = false;
    if (tid == 0) s_S[0] = 1.0;
    for (int c = u + 1; c <= n; ++c) {
      if (s_par[c - 1] != u) continue;
      if (tid == 0) {
        const int x = s_x[c - 1];
        const double qx = qu[x];
        const double rx = residual(pu[x], qx, s_S, k);
        const uint4 w = philox4x32_10(make_uint4((uint32_t)(c - 1), (uint32_t)b, 0u, 0u),
                                      a.key0, a.key1);
        s_accept = philox_uniform(w.x) * s_S[k] * qx <= rx;
      }
      __syncthreads();
      const bool accepted = s_accept;
      __syncthreads();  // read by every thread before thread 0 can write the next test
      if (accepted) {
        next = c;
        break;
      }
      // Rejected: the new residual's total.
      double part = 0.0;
      for (int y = y0; y < y1; ++y) {
        const double qy = qu[y];
        part += fmax(residual(pu[y], qy, s_S, k) - s_S[k] * qy, 0.0);
      }
      double total;
      block_exclusive_scan(part, s_warp, &total);
      ++k;
      if (tid == 0) s_S[k] = total;
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
    double part = 0.0;
    int last = -1;
    for (int y = y0; y < y1; ++y) {
      const double w = from_p ? (double)pu[y] : residual(pu[y], qu[y], s_S, k);
      part += w;
      if (w > 0.0) last = y;
    }
    double total;
    const double before = block_exclusive_scan(part, s_warp, &total);
    if (tid == 0) {
      s_found = -1;
      s_last = -1;
    }
    __syncthreads();
    if (last >= 0) atomicMax(&s_last, last);
    if (total > 0.0) {
      const uint4 w4 = philox4x32_10(make_uint4((uint32_t)u, (uint32_t)b, 0u, 0u), a.key0, a.key1);
      const double target = philox_uniform(w4.y) * total;
      // The thread whose chunk holds the crossing walks it: smallest y with w(y) > 0 and
      // inclusive prefix > target.
      if (before <= target && target < before + part) {
        double c = before;
        for (int y = y0; y < y1; ++y) {
          const double w = from_p ? (double)pu[y] : residual(pu[y], qu[y], s_S, k);
          c += w;
          if (w > 0.0 && c > target) {
            atomicMax(&s_found, y);  // one thread only: the chunks do not overlap
            break;
          }
        }
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
