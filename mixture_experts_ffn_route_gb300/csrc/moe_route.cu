// Router selection over the fp32 logits of the gating GEMM.
//
// "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例", section 路由与负载 / 路由张量:
//   a = score(l);  I_t = TopK(a + beta);  g = alpha * a / sum_{I_t} a
// (beta selects only; the weights use the raw affinity).  The softmax gate of
// "Megatron 分布式训练全维度并行技术文档" (section 4.2) selects the top-k of
// softmax(l), which is the top-k of l itself.  Section 路由与负载 / Hash 路由:
// the ids are a table row of the token id, the gate formula is unchanged.
//
// One warp per token.  The k winners are found by k+1 rounds of a warp
// arg-max (larger score first, equal scores to the lower id).  The fp32
// selection is final unless two neighbouring scores among the first k+1 are
// closer than a decision band; such a token is re-decided with float64 logits
// recomputed from X and Wg for every expert within the band of the k-th score,
// so that the ids equal those of an exact evaluation except at exact ties.
#include <float.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kWarps = 8;          // tokens per block
constexpr int kMaxK = 16;
// Decision bands.  The fp32 tensor-core logit differs from the exact one by
// at most a few 1e-5 at the workload sizes.  Sigmoid and sqrt-softplus have
// slope <= 1/2, so their scores are within ~2e-5 of exact and a band of 2e-4
// on the score leaves a margin of about 10x.  Softmax selects on the logit
// itself; its band is 1e-3 * max(1, |l|).
constexpr float kBand = 2e-4f;
constexpr float kBandSoftmax = 1e-3f;

__device__ __forceinline__ float band_at(float v, int fn) {
  return fn == 2 ? kBandSoftmax * fmaxf(1.0f, fabsf(v)) : kBand;
}

__device__ __forceinline__ float score_f32(float l, int fn) {
  if (fn == 0) return 1.0f / (1.0f + expf(-l));
  if (fn == 1) return sqrtf(fmaxf(l, 0.0f) + log1pf(expf(-fabsf(l))));
  return l;  // softmax: select on the logit (monotone in the softmax value)
}

__device__ __forceinline__ double score_f64(double l, int fn) {
  if (fn == 0) return 1.0 / (1.0 + exp(-l));
  if (fn == 1) return sqrt(fmax(l, 0.0) + log1p(exp(-fabs(l))));
  return l;
}

// (value, id) arg-max across the warp: larger value, then lower id.
__device__ __forceinline__ void warp_argmax(float& v, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oid = __shfl_xor_sync(0xffffffffu, id, o);
    if (ov > v || (ov == v && oid < id)) { v = ov; id = oid; }
  }
}

__device__ __forceinline__ void warp_argmax_d(double& v, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oid = __shfl_xor_sync(0xffffffffu, id, o);
    if (ov > v || (ov == v && oid < id)) { v = ov; id = oid; }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// float64 logit l[t, e] = sum_h X[t, h] Wg[h, e] (bf16 products are exact).
__device__ double logit_f64(const uint16_t* __restrict__ xrow, const uint16_t* __restrict__ Wg,
                            int H, int E, int e, int lane) {
  double acc = 0.0;
  for (int h = lane; h < H; h += 32) {
    const float x = __uint_as_float(static_cast<uint32_t>(__ldg(xrow + h)) << 16);
    const float w = __uint_as_float(static_cast<uint32_t>(__ldg(Wg + static_cast<long long>(h) * E + e)) << 16);
    acc += static_cast<double>(x) * static_cast<double>(w);
  }
  return warp_sum_d(acc);
}

__global__ void __launch_bounds__(kWarps * 32)
    route_select_kernel(const float* __restrict__ logits, const uint16_t* __restrict__ X,
                        const uint16_t* __restrict__ Wg, const float* __restrict__ bias,
                        const int32_t* __restrict__ token_ids, const int32_t* __restrict__ tid2eid,
                        int V, int T, int H, int E, int k, int fn, float alpha, int renorm,
                        int32_t* __restrict__ E_ids, float* __restrict__ G, int* status) {
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + warp;
  if (t >= T) return;
  float* s = sh + warp * E;  // selection scores of this token
  const float* lrow = logits + static_cast<long long>(t) * E;

  // softmax normaliser (max and sum over all experts)
  float lmax = -FLT_MAX, zsum = 0.0f;
  if (fn == 2) {
    for (int e = lane; e < E; e += 32) lmax = fmaxf(lmax, lrow[e]);
    lmax = warp_max(lmax);
    for (int e = lane; e < E; e += 32) zsum += expf(lrow[e] - lmax);
    zsum = warp_sum(zsum);
  }

  int sel[kMaxK];
  bool tok_ok = true;
  if (token_ids != nullptr) {
    // ---------------------------------------------------------------- hash
    const int tok = token_ids[t];
    tok_ok = tok >= 0 && tok < V;
    if (!tok_ok && lane == 0) set_flag(status, kFlagBadToken);
#pragma unroll 1
    for (int j = 0; j < k; ++j) sel[j] = tok_ok ? tid2eid[static_cast<long long>(tok) * k + j] : -1;
  } else {
    // ---------------------------------------------------------------- top-k
    for (int e = lane; e < E; e += 32) {
      float v = score_f32(lrow[e], fn);
      if (bias != nullptr) v += bias[e];
      s[e] = v;
    }
    __syncwarp();
    const int rounds = (k < E) ? k + 1 : k;
    float top[kMaxK + 1];
#pragma unroll 1
    for (int r = 0; r < rounds; ++r) {
      float best = -FLT_MAX;
      int bid = 0x7fffffff;
      for (int e = lane; e < E; e += 32) {
        const float v = s[e];
        if (v > best || (v == best && e < bid)) { best = v; bid = e; }
      }
      warp_argmax(best, bid);
      top[r] = best;
      if (r < k) sel[r] = bid;
      if (lane == 0) s[bid] = -FLT_MAX;  // taken
      __syncwarp();
    }
    // ambiguity: two neighbouring scores among the first k+1 within the band
    bool close = false;
#pragma unroll 1
    for (int r = 0; r + 1 < rounds; ++r) {
      close |= (top[r] - top[r + 1]) < band_at(top[r], fn);
    }
    if (close) {
      // candidates: the k winners plus every expert within the band below the
      // k-th score; restore the scores, then decide in float64.
      for (int e = lane; e < E; e += 32) {
        float v = score_f32(lrow[e], fn);
        if (bias != nullptr) v += bias[e];
        s[e] = v;
      }
      __syncwarp();
      const float kth = top[k - 1];
      const float lim = kth - 2.0f * band_at(kth, fn);
      const uint16_t* xrow = X + static_cast<long long>(t) * H;
      // candidates are taken one at a time by the whole warp; every lane keeps
      // the same sorted list of the k best float64 scores.
      double best_v[kMaxK];
      int best_id[kMaxK];
#pragma unroll 1
      for (int j = 0; j < k; ++j) { best_v[j] = -DBL_MAX; best_id[j] = 0x7fffffff; }
#pragma unroll 1
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool cand = (e < E) && (s[e] >= lim);
        unsigned m = __ballot_sync(0xffffffffu, cand);
        while (m) {
          const int c = e0 + __ffs(m) - 1;
          m &= m - 1;
          const double l64 = logit_f64(xrow, Wg, H, E, c, lane);
          double v = score_f64(l64, fn);
          if (bias != nullptr) v += static_cast<double>(bias[c]);
          // insert (v, c) into the sorted top-k list (all lanes hold copies)
          int pos = k;
#pragma unroll 1
          for (int j = k - 1; j >= 0; --j) {
            if (v > best_v[j] || (v == best_v[j] && c < best_id[j])) pos = j; else break;
          }
          if (pos < k) {
#pragma unroll 1
            for (int j = k - 1; j > pos; --j) { best_v[j] = best_v[j - 1]; best_id[j] = best_id[j - 1]; }
            best_v[pos] = v;
            best_id[pos] = c;
          }
        }
      }
#pragma unroll 1
      for (int j = 0; j < k; ++j) sel[j] = best_id[j];
    }
  }

  // ------------------------------------------------------------------ gates
  if (lane == 0) {
    float a[kMaxK];
    float den = 0.0f;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      const int e = sel[j];
      float v = 0.0f;
      if (e >= 0 && e < E) {
        const float l = lrow[e];
        v = (fn == 2) ? expf(l - lmax) / zsum : score_f32(l, fn);
      } else if (tok_ok) {
        set_flag(status, kFlagBadExpert);  // a table entry outside [0, E)
      }
      a[j] = v;
      den += v;
    }
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      float g = alpha * a[j];
      if (renorm) g = den > 0.0f ? alpha * a[j] / den : 0.0f;
      E_ids[static_cast<long long>(t) * k + j] = sel[j];
      G[static_cast<long long>(t) * k + j] = g;
    }
  }
}

cudaError_t launch_route_select(const float* logits, const uint16_t* X, const uint16_t* Wg,
                                const float* bias, const int32_t* token_ids,
                                const int32_t* tid2eid, int V, int T, int H, int E, int k,
                                int score_fn, float alpha, int renorm, int32_t* E_ids, float* G,
                                int* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int blocks = (T + kWarps - 1) / kWarps;
  const size_t sh = static_cast<size_t>(kWarps) * E * sizeof(float);
  if (sh > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sh));
    if (e != cudaSuccess) return e;
  }
  route_select_kernel<<<blocks, kWarps * 32, sh, s>>>(logits, X, Wg, bias, token_ids, tid2eid, V,
                                                      T, H, E, k, score_fn, alpha, renorm, E_ids,
                                                      G, status);
  return cudaGetLastError();
}

}  // namespace moe
