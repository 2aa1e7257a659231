// Speculative verification: modified rejection sampling, one CTA per sequence (sm_103a).
//
// The rule ("Continuous Batching & Speculative Decoding", section "The Modified
// Rejection Sampling Algorithm"; "Continuous Batching and Speculative Decoding: How
// Modern LLM Serving Engines Actually Work", section "The core idea"):
//   accept x_i while r_i <= min(1, p_i(x_i) / q_i(x_i)) -- tested as r_i q_i <= p_i in
//   double -- halt at the first rejection j, then draw the token at position j from
//   max(0, p_j - q_j) (or from p_k when all k drafts are accepted) by inverse CDF.
//
// Kernel: the k ratio tests run on k threads; a block-wide min finds j.  One streaming
// pass over row j builds w = max(0, p_j - q_j) (fp32 elementwise), sums it in fp32 over
// 8 contiguous elements per lane and in fp64 above that; the warp totals are scanned in
// fp64.  The warp whose range holds the target s_j * S rescans its range tile by tile
// (fp64 lane scan) and the crossing lane walks its 8 elements.  Uniforms come from
// Philox4x32-10 keyed by the seed with counter (position, sequence, 0, 0).
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/vas.h"
#include "philox.cuh"
#include "vas_internal.h"

namespace vas {
namespace verify {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kLaneElems = 8;                  // contiguous elements per lane per tile
constexpr int kTile = 32 * kLaneElems;          // elements per warp tile

struct Args {
  const float* p;
  const float* q;
  const int32_t* draft;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t B, k, V;
  uint32_t key0, key1;
  int32_t* err;
};

// The 8 weights of one lane's group starting at x0 (elements past V are zero).
__device__ __forceinline__ void load_weights(const float* prow, const float* qrow, int x0, int V,
                                             bool vec, float (&w)[kLaneElems]) {
  if (vec && x0 + kLaneElems <= V) {
    const float4 p0 = __ldg(reinterpret_cast<const float4*>(prow + x0));
    const float4 p1 = __ldg(reinterpret_cast<const float4*>(prow + x0 + 4));
    float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
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
    if (x < V) {
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
  __shared__ int32_t s_j, s_bad, s_draw, s_use_p;
  __shared__ double s_warp[kWarps];
  __shared__ double s_base[kWarps];
  __shared__ double s_total, s_target;
  __shared__ int32_t s_warp_hit;

  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, V = a.V;
  if (tid == 0) {
    s_j = k;
    s_bad = 0;
    s_draw = -1;
    s_use_p = 0;
  }
  __syncthreads();

  // 1. Ratio tests: thread i < k tests draft x_i with r_i = word 0 of Philox(i, b).
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
  if (s_bad) {
    for (int t = tid; t <= k; t += kThreads) out[t] = -1;
    if (tid == 0) {
      a.accepted_len[b] = -1;
      atomicOr(a.err, VAS_DEV_BAD_TOKEN);
    }
    return;
  }
  const int j = s_j;

  // 2. One pass over the row to draw from; per-warp fp64 totals.
  const int warp_span = ((V + kWarps * kTile - 1) / (kWarps * kTile)) * kTile;
  const int x_begin = warp * warp_span;
  const int x_end = min(V, x_begin + warp_span);
  const float* prow = a.p + ((size_t)b * (k + 1) + j) * V;
  const float* qrow0 = j < k ? a.q + ((size_t)b * k + j) * V : nullptr;
  for (int attempt = 0; attempt < 2; ++attempt) {
    const float* qrow = s_use_p ? nullptr : qrow0;
    const bool vec = ((reinterpret_cast<uintptr_t>(prow) | reinterpret_cast<uintptr_t>(qrow)) & 15) == 0;
    double acc = 0.0;
    for (int x0 = x_begin + lane * kLaneElems; x0 < x_end; x0 += kTile) {
      float w[kLaneElems];
      load_weights(prow, qrow, x0, x_end, vec, w);
      acc += (double)group_sum(w);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) s_warp[warp] = acc;
    __syncthreads();
    if (tid == 0) {
      double run = 0.0;
      for (int w = 0; w < kWarps; ++w) {
        s_base[w] = run;
        run += s_warp[w];
      }
      s_total = run;
      if (run == 0.0 && j < k && !s_use_p) {
        s_use_p = 1;  // zero residual: draw from p_j
        atomicOr(a.err, VAS_DEV_RESIDUAL_FALLBACK);
      } else {
        s_use_p |= 2;  // done
      }
    }
    __syncthreads();
    if (s_use_p & 2) break;
  }
  const float* qrow = (s_use_p & 1) ? nullptr : qrow0;

  // 3. Target of the inverse CDF and the warp that holds it.
  if (tid == 0) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)j, (uint32_t)b, 0u, 0u), a.key0, a.key1);
    const double sj = philox_uniform(w.y);
    s_target = sj * s_total;
    int hit = -1, last = -1;
    for (int w2 = 0; w2 < kWarps; ++w2) {
      if (s_warp[w2] > 0.0) {
        last = w2;
        if (hit < 0 && s_base[w2] + s_warp[w2] > s_target) hit = w2;
      }
    }
    s_warp_hit = hit >= 0 ? hit : last;  // rounding past the total: last warp with mass
  }
  __syncthreads();

  // 4. The chosen warp rescans its range tile by tile.
  if (s_total > 0.0 && warp == s_warp_hit) {
    const bool vec = ((reinterpret_cast<uintptr_t>(prow) | reinterpret_cast<uintptr_t>(qrow)) & 15) == 0;
    const double target = s_target;
    double base = s_base[warp];
    int found = -1, last_pos = -1;
    for (int t0 = x_begin; t0 < x_end && found < 0; t0 += kTile) {
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
      // last element with mass seen so far (for the rounding fallback)
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
    if (lane == 0) s_draw = found >= 0 ? found : last_pos;
  }
  __syncthreads();

  // 5. Emit.
  for (int t = tid; t <= k; t += kThreads) {
    int32_t v = -1;
    if (t < j) v = a.draft[(size_t)b * k + t];
    else if (t == j) v = s_draw;
    out[t] = v;
  }
  if (tid == 0) {
    a.accepted_len[b] = j;
    if (s_draw < 0) atomicOr(a.err, VAS_DEV_EMPTY_ROW);
  }
}

}  // namespace verify
}  // namespace vas

extern "C" int spec_verify(const float* p, const float* q, const int32_t* draft_tokens,
                           uint64_t seed, int32_t* accepted_len, int32_t* out_tokens, int32_t B,
                           int32_t k, int32_t V, vas_stream_t stream) {
  if (B < 0 || k < 0 || V <= 0) return VAS_E_INVALID_ARG;
  if (B == 0) return VAS_OK;
  if (!p || !accepted_len || !out_tokens || (k > 0 && (!q || !draft_tokens)))
    return VAS_E_INVALID_ARG;
  if ((int64_t)(k + 1) * V > INT32_MAX / 2) return VAS_E_INVALID_ARG;
  if (k >= vas::verify::kThreads) return VAS_E_INVALID_ARG;
  int32_t* err = vas::device_error_word();
  if (!err) return VAS_E_CUDA;
  vas::verify::Args a;
  a.p = p;
  a.q = q;
  a.draft = draft_tokens;
  a.accepted_len = accepted_len;
  a.out_tokens = out_tokens;
  a.B = B;
  a.k = k;
  a.V = V;
  a.key0 = static_cast<uint32_t>(seed);
  a.key1 = static_cast<uint32_t>(seed >> 32);
  a.err = err;
  vas::verify::spec_verify_kernel<<<B, vas::verify::kThreads, 0,
                                     reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? VAS_OK : VAS_E_CUDA;
}
