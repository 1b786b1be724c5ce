// Epilogue of the bf16 grouped GEMMs: the accumulator rows of one warp (its
// TMEM lane quarter, 32 rows from output row wrow0) go TMEM -> registers (one
// row per lane) -> a padded shared staging block -> global memory, with every
// store instruction writing whole 128-byte lines (4 rows of fp32 or 8 rows of
// bf16).  KIND selects SwiGLU (gate columns 0-127 and up columns 128-255 of
// the accumulator, bf16 out), gate-scaled bf16 rows into the tokens' rows of
// Y (the top-1 combine), or fp32 rows.
#pragma once

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

// Row pitch (32-bit words) of the epilogue staging buffer: 32 data words plus
// 4 of padding, so 16-byte accesses by the 8 lanes of one phase touch 8
// distinct bank quads.
constexpr int kStgWords = 36;

// tb: TMEM address of this warp's lane quarter in the tile's accumulator;
// rows at or past row_end are not stored; n is the tile's column tile.
template <int KIND, int BN>
__device__ __forceinline__ void epilogue_store(const GemmParams& p, uint32_t tb, int wrow0,
                                               int row_end, int n, uint32_t* stg, int lane) {
  if (KIND == kGemmSwiGLU) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      float g[32], u[32];
      tmem_ld_32x32(tb + c, g);
      tmem_ld_32x32(tb + 128 + c, u);
      const int col = n * 128 + c;
      if (p.h_out != nullptr && wrow0 + lane < row_end && col < p.n_out) {
        // keep the pre-activations for the backward (bf16, gate | up)
        uint16_t* hrow = p.h_out + static_cast<long long>(wrow0 + lane) * (2 * p.up_off);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          reinterpret_cast<uint4*>(hrow + col)[i] =
              make_uint4(pack_bf16x2(g[8 * i], g[8 * i + 1]), pack_bf16x2(g[8 * i + 2], g[8 * i + 3]),
                         pack_bf16x2(g[8 * i + 4], g[8 * i + 5]), pack_bf16x2(g[8 * i + 6], g[8 * i + 7]));
          reinterpret_cast<uint4*>(hrow + p.up_off + col)[i] =
              make_uint4(pack_bf16x2(u[8 * i], u[8 * i + 1]), pack_bf16x2(u[8 * i + 2], u[8 * i + 3]),
                         pack_bf16x2(u[8 * i + 4], u[8 * i + 5]), pack_bf16x2(u[8 * i + 6], u[8 * i + 7]));
        }
      }
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        // SiLU(g) * u; the fast divide (2 ulp) returns 0 once 1 + e^-g
        // exceeds 2^126, the limit of g / (1 + e^-g) there
        const float a0 = __fdividef(g[2 * i], 1.0f + __expf(-g[2 * i])) * u[2 * i];
        const float a1 = __fdividef(g[2 * i + 1], 1.0f + __expf(-g[2 * i + 1])) * u[2 * i + 1];
        w[i] = pack_bf16x2(a0, a1);
      }
      uint4* srow4 = reinterpret_cast<uint4*>(stg + lane * kStgWords);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        srow4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      __syncwarp();
      if (col < p.n_out) {
        // 8 rows x 64 bytes per instruction: lane -> row rr + lane/4, quad lane%4
        const int qd = lane & 3;
#pragma unroll
        for (int rr = 0; rr < 32; rr += 8) {
          const int r = rr + (lane >> 2);
          const uint4 v = reinterpret_cast<const uint4*>(stg + r * kStgWords)[qd];
          const int grow = wrow0 + r;
          if (grow < row_end)
            *reinterpret_cast<uint4*>(out + static_cast<long long>(grow) * p.ldo + col + 8 * qd) = v;
        }
      }
      __syncwarp();
    }
  } else if (KIND == kGemmCombineK1) {
    // the top-1 combine fused here: each row scaled by its token's gate,
    // rounded once to bf16 (RNE) and stored to that token's row of Y (with
    // k = 1 the permutation entry of an assignment row is its token)
    constexpr bool K1 = true;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    float g = 1.0f;
    if (K1) {
      const int my = wrow0 + lane;
      const int f = my < row_end ? __ldg(p.gather_perm + my) : -1;
      g = f >= 0 && in_bounds(f, p.gather_rows) ? __ldg(p.gate + f) : 0.0f;
    }
    int dst[4];  // output row of each of the four rows this lane stores, or -1
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int grow = wrow0 + 8 * i + (lane >> 2);
      dst[i] = grow < row_end ? (K1 ? __ldg(p.gather_perm + grow) : grow) : -1;
      if (dst[i] >= 0 && !in_bounds(dst[i], p.gather_rows)) dst[i] = -1;
    }
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float v[32];
      tmem_ld_32x32(tb + c, v);
      const int col = n * BN + c;
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(g * v[2 * i], g * v[2 * i + 1]);
      uint4* srow4 = reinterpret_cast<uint4*>(stg + lane * kStgWords);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        srow4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      __syncwarp();
      if (col < p.n_out) {
        // 8 rows x 64 bytes per instruction: lane -> row rr + lane/4, quad lane%4
        const int qd = lane & 3;
#pragma unroll
        for (int rr = 0; rr < 32; rr += 8) {
          const int r = rr + (lane >> 2);
          const uint4 x = reinterpret_cast<const uint4*>(stg + r * kStgWords)[qd];
          const int d = dst[rr >> 3];
          if (d >= 0)
            *reinterpret_cast<uint4*>(out + static_cast<long long>(d) * p.ldo + col + 8 * qd) = x;
        }
      }
      __syncwarp();
    }
  } else {
    // fp32 outputs: router logits and Linear2
    float* out = static_cast<float*>(p.out);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float v[32];
      tmem_ld_32x32(tb + c, v);
      const int col = n * BN + c;
      float4* srow4 = reinterpret_cast<float4*>(stg + lane * kStgWords);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        srow4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      __syncwarp();
      // 4 rows x 128 bytes per instruction: lane -> row rr + lane/8, quad lane%8
      const int qd = lane & 7;
      if (col + 4 * qd < p.n_out) {
#pragma unroll
        for (int rr = 0; rr < 32; rr += 4) {
          const int r = rr + (lane >> 3);
          const float4 x = reinterpret_cast<const float4*>(stg + r * kStgWords)[qd];
          const int grow = wrow0 + r;
          if (grow < row_end)
            *reinterpret_cast<float4*>(out + static_cast<long long>(grow) * p.ldo + col + 4 * qd) = x;
        }
      }
      __syncwarp();
    }
  }
}

}  // namespace moe
