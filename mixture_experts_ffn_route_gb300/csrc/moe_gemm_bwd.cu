// Persistent grouped GEMMs of the layer backward on the tcgen05 tensor cores
// (bf16 operands, fp32 accumulator in TMEM).
//
//   dgrad Linear2 + SwiGLU backward (split M):
//       dA = dYp W2[e]^T                         (K = H, B K-major)
//       dHg = dA * Hu * SiLU'(Hg), dHu = dA * SiLU(Hg)  -> dH [rows, 2I] bf16
//   dgrad Linear1 (split M):  dXp = dH W1[e]^T   (K = 2I)  -> [rows, H] fp32
//   wgrad Linear2 (split K):  dW2[e] = Act_e^T dYp_e       -> [I, H] fp32
//   wgrad Linear1 (split K):  dW1[e] = Xp_e^T dH_e         -> [H, 2I] fp32
//   router:  dWg = X^T dl (split K, one group), dX_r = dl Wg^T (dense)
// These are the expert dgrad / wgrad and router steps of the backward in
// "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例" (section 反向的通信) and the
// parallelism page's section 4.7 (反向流程, steps 3 and 5).
//
// Structure (one CTA per SM, 224 threads):
//   warp 0      TMA producer; tiles 128 x 256, k-block 64, 4 stages of 48 KB.
//               K-major operands come as 128-byte rows of 64 k; MN-major ones
//               (the transposed activations of the weight gradients) as
//               64-wide column blocks of 64 k-rows, both 128-byte swizzled.
//   warp 1      TMEM (two 256-column accumulators); one lane issues
//               tcgen05.mma (M 128, N 256, K 16) and commits.
//   warps 2..5  epilogue: fp32 rows, or the SwiGLU backward with bf16 out.
//   warp 6      split K only: a group's last k-block may hold rows of the next
//               group; the warp waits for the stage's TMA, zeroes those k-rows
//               of A and only then releases the stage to the MMA.
#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_tile.cuh"

namespace moe {
namespace {

constexpr int kBwdBN = 256;
constexpr int kBwdA = kBM * kBK * 2;      // 16 KB
constexpr int kBwdB = kBwdBN * kBK * 2;   // 32 KB
constexpr int kBwdStage = kBwdA + kBwdB;
constexpr int kBwdStages = 4;
constexpr int kBwdRing = kBwdStages * kBwdStage;
constexpr int kBwdBarBytes = 256;
constexpr int kBwdStgWords = 36;
constexpr int kBwdStg = 4 * 32 * kBwdStgWords * 4;
constexpr int kBwdSmem = kBwdRing + 1024 + kBwdBarBytes + kBwdStg;
constexpr int kBwdThreads = 224;
static_assert(8 * (3 * kBwdStages + 4) + 8 <= kBwdBarBytes, "barrier area");
static_assert(kBwdSmem <= 232448, "shared memory");

struct BwdTile {
  int group, m, n;
  int row0, row_end;  // split M: output rows [row0, row_end); split K: output rows m*128 .. M
  int k0, nkb, valid_last;  // split K: first contraction row, k-blocks, rows of the last one
  bool second;
};

template <bool SPLIT_K>
__device__ __forceinline__ BwdTile decode_bwd(const BwdParams& p, int tile) {
  BwdTile b;
  if (SPLIT_K) {
    const int tpg = p.m_tiles * p.n_tiles;
    b.group = tile / tpg;
    const int r = tile - b.group * tpg;
    b.n = r / p.m_tiles;
    b.m = r - b.n * p.m_tiles;
    b.row0 = b.m * kBM;
    b.row_end = p.M;
    b.k0 = __ldg(p.row_off + b.group);
    const int rows = __ldg(p.row_off + b.group + 1) - b.k0;
    b.nkb = (rows + kBK - 1) / kBK;
    b.valid_last = rows - (b.nkb - 1) * kBK;
    b.second = (b.group == p.shared_group);
  } else {
    GemmParams q;
    q.row_off = p.row_off;
    q.tile_off = p.tile_off;
    q.num_groups = p.num_groups;
    q.dense_rows = p.dense_rows;
    q.shared_group = p.shared_group;
    q.a2_shared = 0;
    q.n_tiles = p.n_tiles;
    q.tile_doff = nullptr;  // plain group order
    q.tile_soff = nullptr;
    const TileInfo t = decode_tile(q, tile);
    b.group = t.group;
    b.m = t.m;
    b.n = t.n;
    b.row0 = t.row0;
    b.row_end = t.row_end;
    b.k0 = 0;
    b.nkb = p.num_kb;
    b.valid_last = kBK;
    b.second = t.second;
  }
  return b;
}

template <bool A_MN, bool B_MN, int EPI, bool SPLIT_K>
__global__ void __launch_bounds__(kBwdThreads, 1)
    gemm_bwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bar_area = smem + kBwdRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * (3 * kBwdStages + 4));
  uint32_t* stg_area = reinterpret_cast<uint32_t*>(bar_area + kBwdBarBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tiles0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bar_area);         // stage ready for the MMA
  const uint32_t empty0 = full0 + 8 * kBwdStages;    // stage free for the producer
  const uint32_t landed0 = empty0 + 8 * kBwdStages;  // split K: TMA bytes landed
  const uint32_t tfull0 = landed0 + 8 * kBwdStages;
  const uint32_t tempty0 = tfull0 + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kBwdStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
      mbar_init(landed0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (!SPLIT_K && p.shared_group >= 0) tma_prefetch_desc(&tmB2);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 2 * kBwdBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int total;
  if (SPLIT_K)
    total = p.num_groups * p.m_tiles * p.n_tiles;
  else
    total = ((p.row_off == nullptr) ? (p.dense_rows + kBM - 1) / kBM
                                    : __ldg(p.tile_off + p.num_groups)) * p.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
        const BwdTile t = decode_bwd<SPLIT_K>(p, tile);
        const CUtensorMap* mB = (!SPLIT_K && t.second) ? &tmB2 : &tmB;
        const int bz = t.second ? 0 : t.group;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, p.status, abort_flag)) break;
          // split K: the fix-up warp checks the rows before the MMA sees them
          const uint32_t fb = (SPLIT_K ? landed0 : full0) + 8 * stage;
          const uint32_t sa = tiles0 + stage * kBwdStage;
          const uint32_t sb = sa + kBwdA;
          const int krow = t.k0 + kb * kBK;
          mbar_arrive_expect_tx(fb, kBwdStage);
          if (A_MN) {
            tma_load_2d(sa, &tmA, fb, t.m * kBM, krow);
            tma_load_2d(sa + 64 * 128, &tmA, fb, t.m * kBM + 64, krow);
          } else {
            tma_load_2d(sa, &tmA, fb, kb * kBK, t.row0);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < kBwdBN / 64; ++j)
              tma_load_2d(sb + j * (64 * 128), &tmB, fb, t.n * kBwdBN + 64 * j, krow);
          } else {
            tma_load_3d(sb, mB, fb, kb * kBK, t.n * kBwdBN, bz);
          }
          if (++stage == kBwdStages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ split-K fix-up
    // Zero the k-rows past the group's end in the last k-block's A tile (two
    // 64-row blocks of 128-byte rows); the B rows there then multiply zeros.
    if (SPLIT_K) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        if (__shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0)) break;
        const BwdTile t = decode_bwd<SPLIT_K>(p, tile);
        bool ok = true;
        for (int kb = 0; kb < t.nkb; ++kb) {
          bool w = true;
          if (lane == 0) w = mbar_wait(landed0 + 8 * stage, phase, p.status, abort_flag);
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
          if (kb == t.nkb - 1 && t.valid_last < kBK) {
            uint8_t* sa = smem + stage * kBwdStage;
            const int chunks = (kBK - t.valid_last) * 16;  // 16-byte chunks to clear
            for (int i = lane; i < chunks; i += 32) {
              const int kr = t.valid_last + (i >> 4);
              const int blk = (i >> 3) & 1;
              *reinterpret_cast<uint4*>(sa + blk * (64 * 128) + kr * 128 + (i & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(full0 + 8 * stage);
          if (++stage == kBwdStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f32acc(kBM, kBwdBN, kFmtBF16, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++local) {
        const BwdTile t = decode_bwd<SPLIT_K>(p, tile);
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kBwdBN;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, p.status, abort_flag)) break;
          if (SPLIT_K) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = tiles0 + stage * kBwdStage;
          const uint32_t sb = sa + kBwdA;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // K-major: 128-byte rows of 64 k, a 16-wide k step is 32 bytes.
            // MN-major: 128-byte rows hold 64 m (or n) of one k; 8-row groups
            // 1024 B apart, 64-wide blocks 8 KB apart, a k step is 16 rows.
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 16 * 128, 64 * 128, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 16 * 128, 64 * 128, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 16, 1024);
            mma_f16(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == kBwdStages) { stage = 0; phase ^= 1; }
        }
        mma_commit(tfull0 + 8 * acc);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint32_t* stg = stg_area + q * 32 * kBwdStgWords;
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const BwdTile t = decode_bwd<SPLIT_K>(p, tile);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const bool got = mbar_wait(tfull0 + 8 * acc, acc_phase, p.status, abort_flag);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBwdBN;
      const int wrow0 = t.row0 + q * 32;
      if (wrow0 >= t.row_end) {
        tc_fence_before();
        mbar_arrive(tempty0 + 8 * acc);
        continue;
      }
      const bool zero = SPLIT_K && t.nkb == 0;  // a group without rows: zero gradient
      const int row = wrow0 + lane;
      if (EPI == kBwdF32) {
        float* out = static_cast<float*>(p.out);
        if (SPLIT_K)
          out = t.second ? static_cast<float*>(p.out2) : out + t.group * p.out_group_stride;
#pragma unroll 1
        for (int c = 0; c < kBwdBN; c += 32) {
          float v[32];
          if (zero) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
          } else {
            tmem_ld_32x32(tb + c, v);
          }
          if (c + 32 == kBwdBN) {
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * acc);
          }
          const int col = t.n * kBwdBN + c;
          float4* srow4 = reinterpret_cast<float4*>(stg + lane * kBwdStgWords);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            srow4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          __syncwarp();
          const int qd = lane & 7;
          if (col + 4 * qd < p.N) {
#pragma unroll
            for (int rr = 0; rr < 32; rr += 4) {
              const int r = rr + (lane >> 3);
              const float4 x = reinterpret_cast<const float4*>(stg + r * kBwdStgWords)[qd];
              const int grow = wrow0 + r;
              if (grow < t.row_end)
                *reinterpret_cast<float4*>(out + static_cast<long long>(grow) * p.ldo + col + 4 * qd) = x;
            }
          }
          __syncwarp();
        }
      } else {
        // SwiGLU backward: accumulator column i is dA[:, i]; with the kept
        // pre-activations Hg = H[:, i], Hu = H[:, I + i] this thread's row gets
        // dH[:, i] = dA Hu SiLU'(Hg) and dH[:, I + i] = dA SiLU(Hg), bf16.
        uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll 1
        for (int c = 0; c < kBwdBN; c += 32) {
          float da[32];
          tmem_ld_32x32(tb + c, da);
          if (c + 32 == kBwdBN) {
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * acc);
          }
          const int col = t.n * kBwdBN + c;
          uint32_t wg[16], wu[16];
          if (row < t.row_end && col < p.N) {
            const uint4* hg4 = reinterpret_cast<const uint4*>(p.h_in + static_cast<long long>(row) * p.ldo + col);
            const uint4* hu4 = reinterpret_cast<const uint4*>(p.h_in + static_cast<long long>(row) * p.ldo + p.up_off + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 g4 = __ldg(hg4 + j);
              const uint4 u4 = __ldg(hu4 + j);
              const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
              const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float o_g[2], o_u[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const float g = h ? bf16_hi(gw[i]) : bf16_lo(gw[i]);
                  const float u = h ? bf16_hi(uw[i]) : bf16_lo(uw[i]);
                  const float s = __fdividef(1.0f, 1.0f + __expf(-g));
                  const float d = da[8 * j + 2 * i + h];
                  o_g[h] = d * u * (s * (1.0f + g * (1.0f - s)));
                  o_u[h] = d * g * s;
                }
                wg[4 * j + i] = pack_bf16x2(o_g[0], o_g[1]);
                wu[4 * j + i] = pack_bf16x2(o_u[0], o_u[1]);
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) wg[i] = wu[i] = 0u;
          }
          uint4* srow4 = reinterpret_cast<uint4*>(stg + lane * kBwdStgWords);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            srow4[i] = make_uint4(wg[4 * i], wg[4 * i + 1], wg[4 * i + 2], wg[4 * i + 3]);
            srow4[4 + i] = make_uint4(wu[4 * i], wu[4 * i + 1], wu[4 * i + 2], wu[4 * i + 3]);
          }
          __syncwarp();
          if (col < p.N) {
            // 8 rows x 64 bytes per store instruction, gate half then up half
            const int qd = lane & 3;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
              for (int rr = 0; rr < 32; rr += 8) {
                const int r = rr + (lane >> 2);
                const uint4 v = reinterpret_cast<const uint4*>(stg + r * kBwdStgWords)[4 * half + qd];
                const int grow = wrow0 + r;
                if (grow < t.row_end)
                  *reinterpret_cast<uint4*>(out + static_cast<long long>(grow) * p.ldo +
                                            half * p.up_off + col + 8 * qd) = v;
              }
            }
          }
          __syncwarp();
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * kBwdBN);
  }
}

template <bool A_MN, bool B_MN, int EPI, bool SPLIT_K>
cudaError_t launch_bwd(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                       const BwdParams& p, int grid, cudaStream_t s) {
  auto kern = gemm_bwd_kernel<A_MN, B_MN, EPI, SPLIT_K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kBwdThreads, kBwdSmem, s>>>(a, b, b2, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_bwd(bool a_mn, bool b_mn, int epi, bool split_k, const CUtensorMap& a,
                            const CUtensorMap& b, const CUtensorMap& b2, const BwdParams& p,
                            int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  // the combinations the backward uses
  if (!a_mn && !b_mn && epi == kBwdSwiGLU && !split_k) return launch_bwd<false, false, kBwdSwiGLU, false>(a, b, b2, p, grid, s);
  if (!a_mn && !b_mn && epi == kBwdF32 && !split_k) return launch_bwd<false, false, kBwdF32, false>(a, b, b2, p, grid, s);
  if (a_mn && b_mn && epi == kBwdF32 && split_k) return launch_bwd<true, true, kBwdF32, true>(a, b, b2, p, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
