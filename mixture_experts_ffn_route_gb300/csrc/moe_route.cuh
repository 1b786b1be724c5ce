// Device helpers of the router kernels (moe_route.cu, moe_route_fused.cu):
// score functions, decision bands and warp arg-max with the lower-id tie rule.
//
// "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例", section 路由与负载 / 路由张量:
//   a = score(l);  I_t = TopK(a + beta);  g = alpha * a / sum_{I_t} a
// (beta selects only; the weights use the raw affinity).  The softmax gate of
// "Megatron 分布式训练全维度并行技术文档" (section 4.2) selects the top-k of
// softmax(l), which is the top-k of l itself.
#pragma once

#include <float.h>

#include "moe_common.cuh"

namespace moe {

constexpr int kMaxK = 16;
// Decision bands.  Sigmoid and sqrt-softplus have slope <= 1/3, so their fp32
// scores are within ~2e-5 of exact; a band of 2e-4 on the score leaves a
// margin of about 10x.  Softmax selects on the logit itself; its band is
// 1e-3 * max(1, |l|).
constexpr float kBand = 2e-4f;
constexpr float kBandSoftmax = 1e-3f;

__device__ __forceinline__ float band_at(float v, int fn) {
  return fn == 2 ? kBandSoftmax * fmaxf(1.0f, fabsf(v)) : kBand;
}

// fp32 scores with the fast exponential and division (relative errors of a
// few 1e-6 for |l| <= 20: a sigmoid error of ~1e-6, far inside the band; a
// logit below -88 gives an infinite denominator and a score of 0); log1p
// stays the accurate one, since sqrt amplifies the error of a softplus near
// zero.
__device__ __forceinline__ float score_f32(float l, int fn) {
  if (fn == 0) return __fdividef(1.0f, 1.0f + __expf(-l));
  if (fn == 1) return sqrtf(fmaxf(l, 0.0f) + log1pf(__expf(-fabsf(l))));
  return l;  // softmax: select on the logit (monotone in the softmax value)
}

__device__ __forceinline__ double score_f64(double l, int fn) {
  if (fn == 0) return 1.0 / (1.0 + exp(-l));
  if (fn == 1) return sqrt(fmax(l, 0.0) + log1p(exp(-fabs(l))));
  return l;
}

// (value, id) order: larger value first, equal values lower id first.
template <typename V>
__device__ __forceinline__ bool before(V v, int id, V ov, int oid) {
  return v > ov || (v == ov && id < oid);
}

template <typename V>
__device__ __forceinline__ void warp_argmax(V& v, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const V ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oid = __shfl_xor_sync(0xffffffffu, id, o);
    if (before(ov, oid, v, id)) { v = ov; id = oid; }
  }
}

// warp_argmax carrying a payload of the winning entry along.
template <typename V>
__device__ __forceinline__ void warp_argmax_payload(V& v, int& id, float& pay) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const V ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oid = __shfl_xor_sync(0xffffffffu, id, o);
    const float op = __shfl_xor_sync(0xffffffffu, pay, o);
    if (before(ov, oid, v, id)) { v = ov; id = oid; pay = op; }
  }
}

template <typename V>
__device__ __forceinline__ V warp_sum(V v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Gate of one selected expert from its fp32 logit: the affinity (softmax:
// exp(l - lmax) / zsum over all experts of the token), scaled by alpha and,
// with renorm, divided by den, the sum of the k affinities.
__device__ __forceinline__ float affinity_f32(float l, int fn, float lmax, float zsum) {
  return fn == 2 ? __expf(l - lmax) / zsum : score_f32(l, fn);
}

}  // namespace moe
