// Per-row symmetric int8 quantisation, the "mega_moe" page's A8W8 scenario
// (section 计算过程): s_i = max|x_i| / 127 and q_i = round(x_i / s_i), the
// nearest integer with halves away from zero, so |q| <= 127.  A row of zeros
// gets s = 0 and codes 0.  The codes are written as fp16 values (exact for
// |q| <= 127) because the int8 GEMMs run on the fp16 tensor-core path.
// Division and rounding are IEEE float32 (__fdiv_rn, roundf).
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kQuantWarps = 8;

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void load8(const uint16_t* row, int v, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(row) + v);
  x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

__device__ __forceinline__ void load8(const float* row, int v, float (&x)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(row) + 2 * v);
  const float4 b = __ldg(reinterpret_cast<const float4*>(row) + 2 * v + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ uint32_t code_pair(float a, float b, float s) {
  const float qa = s > 0.0f ? roundf(__fdiv_rn(a, s)) : 0.0f;
  const float qb = s > 0.0f ? roundf(__fdiv_rn(b, s)) : 0.0f;
  const __half2 h = __floats2half2_rn(qa, qb);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <typename In>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quant_rows_kernel(const In* __restrict__ x, const int* __restrict__ rows_dev, int rows_max,
                      int cols, uint16_t* __restrict__ codes, float* __restrict__ scales,
                      const int* __restrict__ inv, int k) {
  const int rows = rows_dev != nullptr ? *rows_dev : rows_max;
  const int lane = threadIdx.x & 31;
  const int vecs = cols / 8;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nw) {
    const In* row = x + static_cast<long long>(r) * cols;
    // destination rows: r itself, or with inv the k rows of token r in expert
    // order (dropped assignments, inv = -1, skipped)
    int dst[16];
    int ndst = 1;
    dst[0] = r;
    if (inv != nullptr) {
      ndst = 0;
      for (int j = 0; j < k; ++j) {
        const int d = __ldg(inv + static_cast<long long>(r) * k + j);
        if (d >= 0 && in_bounds(d, static_cast<long long>(rows) * k)) dst[ndst++] = d;
      }
    }
    float amax = 0.0f;
    for (int v = lane; v < vecs; v += 32) {
      float e[8];
      load8(row, v, e);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(e[i]));
    }
    amax = warp_max_f(amax);
    const float s = __fdiv_rn(amax, 127.0f);
    for (int v = lane; v < vecs; v += 32) {
      float e[8];
      load8(row, v, e);
      const uint4 c = make_uint4(code_pair(e[0], e[1], s), code_pair(e[2], e[3], s),
                                 code_pair(e[4], e[5], s), code_pair(e[6], e[7], s));
      for (int d = 0; d < ndst; ++d)
        reinterpret_cast<uint4*>(codes + static_cast<long long>(dst[d]) * cols)[v] = c;
    }
    if (lane == 0)
      for (int d = 0; d < ndst; ++d) scales[dst[d]] = s;
  }
}

static int quant_grid(int rows) {
  int blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  const int cap = 8 * num_sms();
  return blocks < cap ? (blocks > 0 ? blocks : 1) : cap;
}

cudaError_t launch_quant_rows_bf16(const uint16_t* x, int rows, int cols, uint16_t* codes,
                                   float* scales, const int* inv, int k, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (inv != nullptr && (k < 1 || k > 16)) return cudaErrorInvalidValue;
  quant_rows_kernel<uint16_t><<<quant_grid(rows), kQuantWarps * 32, 0, s>>>(x, nullptr, rows, cols,
                                                                             codes, scales, inv, k);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows_f32(const float* x, const int* rows_dev, int rows_max, int cols,
                                  uint16_t* codes, float* scales, cudaStream_t s) {
  if (rows_max <= 0) return cudaSuccess;
  quant_rows_kernel<float><<<quant_grid(rows_max), kQuantWarps * 32, 0, s>>>(
      x, rows_dev, rows_max, cols, codes, scales, nullptr, 0);
  return cudaGetLastError();
}

MOE_DEFINE_BOUNDS_TAKE(quant)

}  // namespace moe
