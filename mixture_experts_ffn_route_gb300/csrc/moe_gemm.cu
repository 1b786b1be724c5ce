// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05).
//
// Serves the contractions of the layer:
//   router     : logits[T, E] = X[T, H] Wg[H, E]                          (fp32 out)
//   Linear1    : Act[rows, I] = SiLU(X_e W1[e][:, :I]) * (X_e W1[e][:, I:])   (bf16 out)
//   Linear2    : Yp[rows, H]  = Act W2[e]                     (fp32 out;
//                top-1: the gate-scaled rows straight into Y)
// The expert FFN is the "Expert Compute" step of the "mega_moe" page
// (section 计算公式: Linear1 projection, SwiGLU activation, Linear2
// projection); the router product is the
// gating linear of "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例" (section 路由张量).
//
// Structure (one CTA per SM):
//   warp 0      TMA producer: A tile [128 rows x 64 k] K-major and B tile
//               [64 k x BN cols] MN-major (the weights keep their [K][N] row-major
//               layout), both with 128-byte swizzle, into a STAGES-deep ring.
//   warp 1      allocates TMEM; one lane issues tcgen05.mma (M=128, or M=64
//               for a tile of at most 64 rows; N=BN, K=16) into one of two
//               TMEM accumulators and commits to mbarriers.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one row per thread),
//               fuse SwiGLU (or the top-1 combine), stage through shared
//               memory for full-line stores, free the accumulator so the next
//               tile's MMAs overlap this epilogue.
//   warps 6..9  Linear1 only: copy the A rows straight from the token rows X
//               by the dispatch permutation (cp.async), so the permuted rows are
//               never written to memory.
// Tiles are walked in (group, column tile, 128-row tile) order, or with the
// dense groups' tiles interleaved into the others' (moe_tile.cuh), striding by
// gridDim.x.  Group row ranges come from device memory.
#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_gemm_epi.cuh"
#include "moe_tile.cuh"

namespace moe {

template <int KIND>
struct KindInfo {
  static constexpr bool SWIGLU = (KIND == kGemmSwiGLU);
  static constexpr int BN = (KIND == kGemmRouter) ? 128 : 256;
  static constexpr int THREADS = 320;
};

template <int BN>
struct GemmCfg {
  static constexpr int A_BYTES = kBM * kBK * 2;   // 16 KB
  static constexpr int B_BYTES = BN * kBK * 2;    // 8 KB per 64 columns
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_BYTES = 256;
  // epilogue staging: per epilogue warp 32 rows x kStgWords 32-bit words
  static constexpr int STG_BYTES = 4 * 32 * kStgWords * 4;
  static constexpr int SMEM_BYTES = RING_BYTES + 1024 + BAR_BYTES + STG_BYTES;
  static_assert(8 * (2 * STAGES + 4) + 8 <= BAR_BYTES, "barrier area");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// First weight column of 64-wide B box j of column tile n.  SwiGLU tiles hold
// 128 gate columns followed by the matching 128 up columns.
template <int KIND>
__device__ __forceinline__ int b_box_col(const GemmParams& p, int n, int j) {
  if (KIND == kGemmSwiGLU) return (j < 2) ? n * 128 + j * 64 : p.up_off + n * 128 + (j - 2) * 64;
  return n * KindInfo<KIND>::BN + j * 64;
}

template <int KIND>
__global__ void __launch_bounds__(KindInfo<KIND>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                   const GemmParams p) {
  constexpr bool SWIGLU = KindInfo<KIND>::SWIGLU;
  constexpr int BN = KindInfo<KIND>::BN;
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bar_area = smem + C::RING_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * (2 * C::STAGES + 4));
  uint32_t* stg_area = reinterpret_cast<uint32_t*>(bar_area + C::BAR_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tiles0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bar_area);
  const uint32_t empty0 = full0 + 8 * C::STAGES;
  const uint32_t tfull0 = empty0 + 8 * C::STAGES;
  const uint32_t tempty0 = tfull0 + 16;

  const bool gather = SWIGLU && (p.gather_src != nullptr);
  if (threadIdx.x == 0) {
    // arrivals completing a stage: the TMA producer's and one per gather thread
    const int full_count = 1 + (gather ? 128 : 0);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full0 + 8 * s, full_count);
      mbar_init(empty0 + 8 * s, 1);
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
    if (p.shared_group >= 0) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_mt = (p.row_off == nullptr) ? (p.dense_rows + kBM - 1) / kBM
                                              : __ldg(p.tile_off + p.num_groups);
  const int total = total_mt * p.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 waits for a free stage, posts the byte count and loads B, and A
    // too unless the gather warps copy the A rows.
    if (lane == 0) {
      const uint64_t evict_first = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
        const TileInfo t = decode_tile(p, tile);
        const CUtensorMap* mA = (t.second && p.a2_shared) ? &tmA2 : &tmA;
        const CUtensorMap* mB = t.second ? &tmB2 : &tmB;
        const int bz = t.second ? 0 : t.group;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, p.status, abort_flag)) break;
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t sa = tiles0 + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          if (!gather) {
            mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
            tma_load_2d(sa, mA, fb, kb * kBK, t.a_row0);
          } else {
            mbar_arrive_expect_tx(fb, C::B_BYTES);
          }
          if (p.l2_hint && t.stream) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_3d_hint(sb + j * (64 * kBK * 2), mB, fb, b_box_col<KIND>(p, t.n, j), kb * kBK,
                               bz, evict_first);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_3d(sb + j * (64 * kBK * 2), mB, fb, b_box_col<KIND>(p, t.n, j), kb * kBK, bz);
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp >= 6 && warp < 10) {
    // ------------------------------------------------------------ row gather
    // Linear1 only: the four gather warps copy each A tile's 128 token rows
    // (assignment row r -> token perm[r] / k) into the 128-byte-swizzled
    // K-major layout the MMA reads: 16-byte chunk c of tile row r lands at
    // chunk c ^ (r % 8).  Eight lanes cover one 128-byte row segment, so one
    // instruction moves four whole rows.  Every thread then arrives on the
    // stage's barrier when its copies have landed (cp.async.mbarrier.arrive),
    // which lets the warps run the full ring ahead of the MMA.  Rows past the
    // group's end are not copied: their stale products only reach accumulator
    // rows the epilogue never stores.
    if (gather) {
      const int gw = warp - 6;       // 0..3: rows 32*gw .. 32*gw + 31
      const int c = lane & 7;        // 16-byte chunk of the row segment
      const int rq = lane >> 3;      // row within a group of four
      const long long ld = static_cast<long long>(p.num_kb) * kBK;  // X row stride
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        if (__shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0)) break;
        const TileInfo t = decode_tile(p, tile);
        int tok[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 32 * gw + 4 * i + rq;
          if (t.second) {
            const int x = t.m * kBM + r;
            tok[i] = x < p.gather_rows ? x : -1;
          } else {
            const int row = t.row0 + r;
            const int f = row < t.row_end ? __ldg(p.gather_perm + row) : -1;
            tok[i] = f >= 0 && in_bounds(f, static_cast<long long>(p.gather_rows) * p.gather_k)
                         ? f / p.gather_k
                         : -1;
          }
        }
        bool ok = true;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          bool w = true;
          if (lane == 0) w = mbar_wait(empty0 + 8 * stage, phase ^ 1, p.status, abort_flag);
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
          const uint32_t sa = tiles0 + stage * C::STAGE_BYTES;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 32 * gw + 4 * i + rq;
            if (tok[i] >= 0)
              cp_async16(sa + r * 128 + ((c ^ (r & 7)) << 4),
                         p.gather_src + tok[i] * ld + kb * kBK + c * 8);
          }
          cp_async_arrive(full0 + 8 * stage);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f32acc(kBM, BN, kFmtBF16, false, true);
      // tiles of at most 64 rows (short experts) run M = 64 MMAs: half the
      // tensor work on rows that are padding
      constexpr uint32_t idesc64 = idesc_f32acc(64, BN, kFmtBF16, false, true);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++local) {
        const TileInfo t = decode_tile(p, tile);
        const uint32_t id = (t.row_end - t.row0 <= 64) ? idesc64 : idesc;
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, p.status, abort_flag)) break;
          // rows copied by the gather warps went through the generic proxy;
          // order them before the tensor cores read the stage
          if (gather) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = tiles0 + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // A: K-major rows of 128 B; a 16-wide k step is 32 B along the row.
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            // B: MN-major; rows of 128 B hold 64 n-values of one k; 8-row groups
            // are 1024 B apart (SBO) and 64-column blocks 8 KB apart (LBO).
            const uint64_t bd = smem_desc_sw128(sb + kk * 16 * 128, 64 * kBK * 2, 1024);
            mma_f16(d, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        mma_commit(tfull0 + 8 * acc);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Each warp owns 32 accumulator rows (its TMEM lane quarter), or 16 after
    // an M = 64 MMA, which leaves row 16q + l in lane l < 16 of quarter q (the
    // tcgen05 data-path layout of an M = 64, one-CTA MMA: the first 16 lanes
    // of each 32-lane quarter hold all N columns; groups of 63, 64 and 65 rows
    // are parity cases of their own).  A
    // chunk of 32 columns goes TMEM -> registers (one row per lane) -> a
    // padded shared staging block -> global memory with every store
    // instruction writing whole 128-byte lines (4 rows of fp32 or 8 rows of
    // bf16 per instruction).
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t* stg = stg_area + q * 32 * kStgWords;
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const TileInfo t = decode_tile(p, tile);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const bool got = mbar_wait(tfull0 + 8 * acc, acc_phase, p.status, abort_flag);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const bool m64 = t.row_end - t.row0 <= 64;
      const int wrow0 = t.row0 + q * (m64 ? 16 : 32);  // first output row of this warp
      const int wend = m64 ? min(t.row_end, wrow0 + 16) : t.row_end;
      if (wrow0 >= wend) {
        // all rows of this warp lie past the group's end: nothing to store
        tc_fence_before();
        mbar_arrive(tempty0 + 8 * acc);
        continue;
      }
      epilogue_store<KIND, BN>(p, tb, wrow0, wend, t.n, stg, lane);
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [rows, cols] 16-bit row-major, box = 64 columns x 128 rows, 128-byte swizzle.
bool make_map_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows < 1 ? 1 : rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBM)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [groups, K, N] bf16 row-major (N contiguous), box = 64 n x 64 k x 1.
bool make_map_weights(CUtensorMap* m, const void* base, int64_t groups, int64_t K, int64_t N) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K),
                        static_cast<cuuint64_t>(groups)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 2, static_cast<cuuint64_t>(N * K) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBK), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MX codes, [rows, cols] (cols contiguous): one 128-byte row segment per box
// row, 128 rows, 128-byte swizzle.  kMxFp8: bytes; kMxFp4Spread: packed E2M1
// spread by the map type to 16 codes per 16 bytes of shared memory (the box
// counts codes); kMxFp4Packed: the packed bytes as they are.
static CUtensorMapDataType mx_map_type(int layout) {
  return layout == kMxFp4Spread ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
}

bool make_map_mx_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int layout) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const bool packed = layout == kMxFp4Packed;
  const int64_t row_bytes = layout == kMxFp8 ? cols : cols / 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(packed ? row_bytes : cols),
                        static_cast<cuuint64_t>(rows < 1 ? 1 : rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(packed ? 128 : kMxBK), static_cast<cuuint32_t>(kBM)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, mx_map_type(layout), 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MX weight codes [groups, N, K] (K contiguous), box = one 128-byte row
// segment x box_rows n x 1, 128-byte swizzle: the K-major B tiles.
bool make_map_mx_weights(CUtensorMap* m, const void* base, int64_t groups, int64_t N, int64_t K,
                         int box_rows, int layout) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const bool packed = layout == kMxFp4Packed;
  const int64_t rb = layout == kMxFp8 ? K : K / 2;  // bytes per weight row
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(packed ? rb : K), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(groups)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(rb), static_cast<cuuint64_t>(N * rb)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(packed ? 128 : kMxBK), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, mx_map_type(layout), 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, cols] bf16 row-major, box = box_cols x box_rows, 128-byte swizzle.
bool make_map_bf16_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols,
                      int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows < 1 ? 1 : rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [groups, N, K] bf16 (K contiguous): the K-major B tiles of the backward's
// input gradients (W2 [E, I, H] read as N = I, K = H; W1 [E, H, 2I] as N = H,
// K = 2I; Wg [H, E] as N = H, K = E), box = 64 k x 256 n x 1.
bool make_map_bf16_kmajor_b(CUtensorMap* m, const void* base, int64_t groups, int64_t N, int64_t K) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(groups)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(N * K) * 2};
  cuuint32_t box[3] = {64, 256, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [groups, N, K] int8 row-major (K contiguous: one row per output channel),
// box = 64 k x 128 rows x 1, 64-byte swizzle.
bool make_map_i8_rows(CUtensorMap* m, const void* base, int64_t groups, int64_t N, int64_t K) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(groups)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N * K)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_block_n(GemmKind kind) { return kind == kGemmRouter ? 128 : 256; }

template <int KIND>
static cudaError_t launch_one(const GemmMaps& m, const GemmParams& p, int grid, cudaStream_t s) {
  using I = KindInfo<KIND>;
  using C = GemmCfg<I::BN>;
  auto kern = gemm_tc_kernel<KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, I::THREADS, C::SMEM_BYTES, s>>>(m.a, m.a2, m.b, m.b2, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm(GemmKind kind, const GemmMaps& maps, const GemmParams& p, int grid,
                        cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  switch (kind) {
    case kGemmRouter: return launch_one<kGemmRouter>(maps, p, grid, s);
    case kGemmSwiGLU: return launch_one<kGemmSwiGLU>(maps, p, grid, s);
    case kGemmPlain: return launch_one<kGemmPlain>(maps, p, grid, s);
    case kGemmCombineK1: return launch_one<kGemmCombineK1>(maps, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

MOE_DEFINE_BOUNDS_TAKE(gemm)

}  // namespace moe
