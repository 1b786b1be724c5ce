// Elementwise kernels of the layer backward (the GEMMs are in moe_gemm_bwd.cu):
//   un-permute backward: dYp[r] = g_{t,j} dY_t per assignment row, the
//       mixing-weight gradient dG_{t,j} = <dY_t, Y_e(x_t)>, dYp = dY for the
//       shared rows;
//   the permuted token rows Xp (for the Linear1 weight gradient);
//   router backward: dL/dlogits from dG through the gates and the affinity;
//   the k-way input-gradient sum dX_t = sum_j dXp[row(t, j)] + shared + router.
// Steps of "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例" (section 反向的通信:
// un-permute backward, the k dgrads of a token added, router and input) and
// of the parallelism page's section 4.7 (反向流程, steps 1 and 5).
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kRowThreads = 256;

// The token and the gate of permuted row r; false past the last row.  A
// permutation entry outside the A assignments (debug build) gives t = -1.
__device__ __forceinline__ bool row_source(const int* __restrict__ perm, const int* __restrict__ row_off,
                                           int E, int k, int has_shared, long long A, int r, int* t,
                                           int* f) {
  const int routed = __ldg(row_off + E);
  if (r < routed) {
    *f = __ldg(perm + r);
    *t = *f / k;
    if (!in_bounds(*f, A)) *t = *f = -1;
    return true;
  }
  if (has_shared && r < __ldg(row_off + E + 1)) {
    *f = -1;
    *t = r - routed;
    return true;
  }
  return false;
}

// One block per permuted row (grid-stride).  H is a multiple of 64.
__global__ void __launch_bounds__(kRowThreads)
    unpermute_bwd_kernel(const uint16_t* __restrict__ dY, const float* __restrict__ G,
                         const int* __restrict__ perm, const int* __restrict__ row_off,
                         const float* __restrict__ Yp, int rows_max, int k, int H, int E,
                         int has_shared, uint16_t* __restrict__ dYp, float* __restrict__ dG) {
  __shared__ float red[kRowThreads / 32];
  // rows_max = A (+ T shared-expert rows): the assignments A = T k
  const long long A = has_shared ? static_cast<long long>(rows_max) / (k + 1) * k : rows_max;
  for (int r = blockIdx.x; r < rows_max; r += gridDim.x) {
    int t, f;
    if (!row_source(perm, row_off, E, k, has_shared, A, r, &t, &f)) return;
    if (t < 0) continue;  // block-uniform
    const float g = f >= 0 ? __ldg(G + f) : 1.0f;
    const uint16_t* dy = dY + static_cast<long long>(t) * H;
    const float* yp = Yp + static_cast<long long>(r) * H;
    uint16_t* out = dYp + static_cast<long long>(r) * H;
    float dot = 0.0f;
    for (int c = 8 * threadIdx.x; c < H; c += 8 * kRowThreads) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(dy + c));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
      if (f >= 0) {
        const float4 y0 = __ldcs(reinterpret_cast<const float4*>(yp + c));
        const float4 y1 = __ldcs(reinterpret_cast<const float4*>(yp + c + 4));
        const float ys[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = bf16_lo(w[i]), b = bf16_hi(w[i]);
          dot += a * ys[2 * i] + b * ys[2 * i + 1];
          o[i] = pack_bf16x2(g * a, g * b);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = w[i];
      }
      *reinterpret_cast<uint4*>(out + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (f >= 0) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = dot;
      __syncthreads();
      if (threadIdx.x == 0) {
        float s = 0.0f;
        for (int w = 0; w < kRowThreads / 32; ++w) s += red[w];
        dG[f] = s;
      }
      __syncthreads();
    }
  }
}

// Xp[r] = X[token of r], one block per row.
__global__ void __launch_bounds__(kRowThreads)
    gather_rows_kernel(const uint16_t* __restrict__ X, const int* __restrict__ perm,
                       const int* __restrict__ row_off, int rows_max, int k, int H, int E,
                       int has_shared, uint16_t* __restrict__ Xp) {
  const long long A = has_shared ? static_cast<long long>(rows_max) / (k + 1) * k : rows_max;
  for (int r = blockIdx.x; r < rows_max; r += gridDim.x) {
    int t, f;
    if (!row_source(perm, row_off, E, k, has_shared, A, r, &t, &f)) return;
    if (t < 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<long long>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(Xp + static_cast<long long>(r) * H);
    for (int c = threadIdx.x; c < H / 8; c += kRowThreads) dst[c] = __ldg(src + c);
  }
}

// dX_t = sum_j dXp[inv[t k + j]] (in j order) + dXp[shared row of t] + dXr_t.
__global__ void __launch_bounds__(kRowThreads)
    dx_reduce_kernel(const float* __restrict__ dXp, const int* __restrict__ inv,
                     const int* __restrict__ row_off, const float* __restrict__ dXr, int T, int k,
                     int H, int E, int has_shared, uint16_t* __restrict__ dX) {
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    int rows[17];
    int n = 0;
    const long long A = static_cast<long long>(T) * k;
    for (int j = 0; j < k; ++j) {
      const int r = __ldg(inv + static_cast<long long>(t) * k + j);
      if (r >= 0 && in_bounds(r, A)) rows[n++] = r;
    }
    if (has_shared) {
      const int r = __ldg(row_off + E) + t;
      if (in_bounds(r, A + T)) rows[n++] = r;
    }
    for (int c = 4 * threadIdx.x; c < H; c += 4 * kRowThreads) {
      float4 s = __ldcs(reinterpret_cast<const float4*>(dXr + static_cast<long long>(t) * H + c));
      float a[4] = {s.x, s.y, s.z, s.w};
      for (int i = 0; i < n; ++i) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(dXp + static_cast<long long>(rows[i]) * H + c));
        a[0] += v.x; a[1] += v.y; a[2] += v.z; a[3] += v.w;
      }
      uint2 o;
      o.x = pack_bf16x2(a[0], a[1]);
      o.y = pack_bf16x2(a[2], a[3]);
      *reinterpret_cast<uint2*>(dX + static_cast<long long>(t) * H + c) = o;
    }
  }
}

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + __expf(-z)); }

// Router backward, one warp per token.  Gates g_j = alpha a_j / S (S the sum
// over the selected ids) or alpha a_j; dL/da_j = (alpha / S)(dG_j - sum_i
// dG_i a_i / S) or alpha dG_j; then dL/dl through the affinity: sigmoid
// a (1 - a), sqrt-softplus sigma(l) / (2 a), softmax a (da - sum a da) over
// all experts.  dl is written as bf16 [T, E], zero where it vanishes.
__global__ void __launch_bounds__(256)
    router_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ E_ids,
                      const float* __restrict__ dG, int T, int E, int k, int score_fn,
                      float alpha, int renorm, uint16_t* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps) {
    const float* lt = logits + static_cast<long long>(t) * E;
    uint16_t* out = dl + static_cast<long long>(t) * E;
    // softmax normaliser over all experts
    float mx = -INFINITY, den = 0.0f;
    if (score_fn == 2) {
      for (int e = lane; e < E; e += 32) mx = fmaxf(mx, lt[e]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      for (int e = lane; e < E; e += 32) den += __expf(lt[e] - mx);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    }
    // lane j < k: selected expert j
    int e_j = -1;
    float a_j = 0.0f, l_j = 0.0f, dg_j = 0.0f;
    if (lane < k) {
      e_j = __ldg(E_ids + static_cast<long long>(t) * k + lane);
      if (e_j >= 0 && e_j < E) {
        l_j = lt[e_j];
        dg_j = __ldg(dG + static_cast<long long>(t) * k + lane);
        if (score_fn == 0) a_j = sigmoid_f(l_j);
        else if (score_fn == 1) a_j = sqrtf(fmaxf(l_j, 0.0f) + log1pf(__expf(-fabsf(l_j))));
        else a_j = __expf(l_j - mx) / den;
      } else {
        e_j = -1;
      }
    }
    float S = a_j, SdA = dg_j * a_j;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      S += __shfl_xor_sync(0xffffffffu, S, o);
      SdA += __shfl_xor_sync(0xffffffffu, SdA, o);
    }
    float da_j = 0.0f;
    if (e_j >= 0) da_j = renorm ? (S > 0.0f ? alpha / S * (dg_j - SdA / S) : 0.0f) : alpha * dg_j;
    if (score_fn != 2) {
      for (int e = lane; e < E; e += 32) out[e] = 0;
      __syncwarp();
      if (e_j >= 0) {
        const float d = score_fn == 0 ? da_j * a_j * (1.0f - a_j)
                                      : (a_j > 0.0f ? da_j * sigmoid_f(l_j) / (2.0f * a_j) : 0.0f);
        __nv_bfloat16 b = __float2bfloat16_rn(d);
        out[e_j] = *reinterpret_cast<uint16_t*>(&b);
      }
    } else {
      // dl_e = p_e (da_e - sum_i p_i da_i); da is nonzero at the selected ids
      float pda = a_j * da_j;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pda += __shfl_xor_sync(0xffffffffu, pda, o);
      for (int e = lane; e < E; e += 32) {
        float da_e = 0.0f;
        for (int j = 0; j < k; ++j) {
          const int ej = __shfl_sync(0xffffffffu, e_j, j);
          const float dj = __shfl_sync(0xffffffffu, da_j, j);
          if (ej == e) da_e += dj;
        }
        const float p = __expf(lt[e] - mx) / den;
        __nv_bfloat16 b = __float2bfloat16_rn(p * (da_e - pda));
        out[e] = *reinterpret_cast<uint16_t*>(&b);
      }
    }
  }
}

}  // namespace

cudaError_t launch_unpermute_bwd(const uint16_t* dY, const float* G, const int* perm,
                                 const int* row_off, const float* Yp, int rows_max, int k, int H,
                                 int E, int has_shared, uint16_t* dYp, float* dG, cudaStream_t s) {
  if (rows_max <= 0) return cudaSuccess;
  const int grid = rows_max < 8 * num_sms() ? rows_max : 8 * num_sms();
  unpermute_bwd_kernel<<<grid, kRowThreads, 0, s>>>(dY, G, perm, row_off, Yp, rows_max, k, H, E,
                                                    has_shared, dYp, dG);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const uint16_t* X, const int* perm, const int* row_off, int rows_max,
                               int k, int H, int E, int has_shared, uint16_t* Xp, cudaStream_t s) {
  if (rows_max <= 0) return cudaSuccess;
  const int grid = rows_max < 8 * num_sms() ? rows_max : 8 * num_sms();
  gather_rows_kernel<<<grid, kRowThreads, 0, s>>>(X, perm, row_off, rows_max, k, H, E, has_shared, Xp);
  return cudaGetLastError();
}

cudaError_t launch_dx_reduce(const float* dXp, const int* inv, const int* row_off, const float* dXr,
                             int T, int k, int H, int E, int has_shared, uint16_t* dX, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int grid = T < 8 * num_sms() ? T : 8 * num_sms();
  dx_reduce_kernel<<<grid, kRowThreads, 0, s>>>(dXp, inv, row_off, dXr, T, k, H, E, has_shared, dX);
  return cudaGetLastError();
}

cudaError_t launch_router_bwd(const float* logits, const int32_t* E_ids, const float* dG, int T,
                              int E, int k, int score_fn, float alpha, int renorm, uint16_t* dl,
                              cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int blocks = (T + 7) / 8;
  router_bwd_kernel<<<blocks, 256, 0, s>>>(logits, E_ids, dG, T, E, k, score_fn, alpha, renorm, dl);
  return cudaGetLastError();
}

MOE_DEFINE_BOUNDS_TAKE(backward)

}  // namespace moe
