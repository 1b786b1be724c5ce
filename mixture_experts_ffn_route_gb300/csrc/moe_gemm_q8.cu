// Persistent grouped GEMM of the A8W8-INT form with the weights as the tensor
// cores' A operand in TMEM: the output channels are the MMA's M, the tokens
// its N ("mega_moe" page, section 计算过程, A8W8 scenario).
//
//   Linear1: D[c][m] = sum_k W1q[e][c][k] q[m][k] for the gate channels c and
//            the matching up channels I + c; epilogue Act[m][c] = SiLU(Hg) * Hu
//            with H = (D * s1[c]) * sx[m] (fp32 out, re-quantised per row later)
//   Linear2: D[h][m] = sum_k W2q[e][h][k] a8[m][k]; Yp[m][h] = (D * s2[h]) * sa[m]
//            (bf16 or fp32 out)
//
// GB300's tensor cores have no int8 form for sm_103a, so the int8 codes are
// multiplied as fp16: |code| <= 127 is exact in fp16, a product is exact in
// fp32, and the fp32 accumulator holds the int32 sum exactly while every
// partial sum stays below 2^24 in magnitude.  Converting a weight tile to fp16
// in shared memory doubles its bytes and the MMA then reads it back, so shared
// memory rather than HBM set the pace of a kernel doing that.  Here each weight
// row (the operator's layout: one row per output channel, K contiguous) is
// converted by one thread straight into its TMEM lane with tcgen05.st, which
// the MMA reads as A (row m in lane m, element k in column k / 2).
//
// Structure (one CTA per SM, 608 threads).  Three rings run on one running
// k-block index per CTA: the int8 weight rows in shared memory (eight deep,
// freed as soon as they are converted, so the weight stream runs well ahead),
// the TMEM slots of converted weights (four) and the shared-memory tiles of
// token codes (five: the codes' latency, not the MMAs, set the pace with four).
// A k-block is made ready by one barrier, its code stage's, on which both the
// converters and the code loaders arrive, and released by one, on which the
// code loaders and (kQ8Slots k-blocks later) the converters wait, so each MMA
// thread does one wait, four MMAs and one commit per k-block.
//   warp 0       TMA: int8 weight rows, two blocks of 128 rows x 64 k per k-block
//                (Linear1: gate rows and the matching up rows; Linear2: 256
//                output channels)
//   warps 1, 18  MMA: warp 1 allocates TMEM (512 columns: two accumulators of
//                128 tokens, four weight slots of 2 x 32 columns); one lane of
//                each issues tcgen05.mma (M 128, N = the tile's token count
//                rounded up to 16, K 16, A from TMEM) into its own accumulator
//   warps 2..5   epilogue: thread = output channel, looping over the tile's tokens
//   warp 6       token codes: the tile of expert-ordered code rows (the token
//                quantiser writes each token's codes to its k rows) by TMA, K-major
//                with 128-byte swizzle, for Linear1 and Linear2 alike
//   warps 10..17 converters, two groups of four taking alternate k-blocks: thread
//                j turns row j of both weight blocks (64 int8 each) into 32
//                words of fp16 pairs in the k-block's TMEM slot
#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_tile.cuh"

namespace moe {
namespace {

constexpr int kQ8Tok = 128;                      // tokens per tile (largest MMA N)
constexpr int kQ8RawBytes = 2 * 128 * kBK;       // int8 weight rows of a k-block: 16 KB
constexpr int kQ8CodeBytes = kQ8Tok * kBK * 2;   // fp16 token codes of a k-block: 16 KB
constexpr int kQ8RawStages = 8;
constexpr int kQ8Slots = 4;                      // TMEM weight slots
// token-code stages: deeper than the slots, since the codes' latency (~1.3 us
// under the weight stream) sets the pace otherwise; a k-block's "ready"
// barrier is the code stage's
constexpr int kQ8CodeStages = 5;
constexpr int kQ8ConvGroups = 2;
constexpr int kQ8CodeRing = kQ8CodeStages * kQ8CodeBytes;  // first: 1024-aligned for the swizzle
constexpr int kQ8Ring = kQ8CodeRing + kQ8RawStages * kQ8RawBytes;
constexpr int kQ8Bars = 2 * kQ8RawStages + 2 * kQ8CodeStages + 2;
constexpr int kQ8BarBytes = 512;
constexpr int kQ8ScaleBytes = 4 * kQ8Tok * 4;    // per epilogue warp: the tile's token scales
constexpr int kQ8Smem = kQ8Ring + 1024 + kQ8BarBytes + kQ8ScaleBytes;
constexpr int kQ8Threads = 608;
constexpr int kQ8MmaWarp2 = 18;                  // the second MMA thread's warp
constexpr int kQ8Slot0 = 256;                    // TMEM: accumulators 0..255, slots 256 + 64 s
static_assert(kQ8Slot0 + 64 * kQ8Slots <= 512, "TMEM columns");
static_assert(8 * kQ8Bars + 8 <= kQ8BarBytes, "barrier area");
static_assert(kQ8Smem <= 232448, "shared memory");
static_assert(kQ8Slots % kQ8ConvGroups == 0, "a slot belongs to one converter group");
// A TMEM slot's previous user, k-block it - kQ8Slots, signals its end on its
// code stage's release barrier, so the converters wait there (no barrier of
// the slots' own).  That wait cannot alias: the next completion of the same
// barrier is the MMAs of k-block it - kQ8Slots + kQ8CodeStages > it - 1, which
// need this converter's slot first.  And the converter of k-block
// it + kQ8CodeStages, which waits for the MMAs of it + kQ8CodeStages - kQ8Slots
// >= it, never arrives on a ready barrier whose previous phase is still open.
static_assert(kQ8CodeStages >= kQ8Slots, "code ring at least as deep as the slots");

// 4 int8 (one 32-bit word) -> 4 fp16, exactly: with b = x + 128 in [0, 255],
// the fp16 bit pattern 0x6400 | b is 1024 + b, and subtracting 1152 leaves x.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x5342);
  const __half2 k = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), k);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), k);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// 32 lanes x 32 consecutive 32-bit TMEM columns: thread i writes lane (base + i).
__device__ __forceinline__ void tmem_st_32x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], fp16 inputs, fp32 accumulator.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Stage and phase parity of running k-block `it` in a ring of `n` stages.
__device__ __forceinline__ uint32_t ring_stage(unsigned it, int n) { return it % n; }
__device__ __forceinline__ uint32_t ring_phase(unsigned it, int n) { return (it / n) & 1u; }

template <bool SWIGLU>
__global__ void __launch_bounds__(kQ8Threads, 1)
    gemm_q8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bar_area = smem + kQ8Ring;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * kQ8Bars);
  float* scale_area = reinterpret_cast<float*>(bar_area + kQ8BarBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t codes0 = smem_u32(smem);
  const uint32_t raw0 = codes0 + kQ8CodeRing;
  const uint32_t rawfull0 = smem_u32(bar_area);                // weight rows landed
  const uint32_t rawempty0 = rawfull0 + 8 * kQ8RawStages;      // weight rows converted
  const uint32_t full0 = rawempty0 + 8 * kQ8RawStages;         // k-block ready: slot written, codes landed
  const uint32_t cempty0 = full0 + 8 * kQ8CodeStages;          // the k-block's MMAs are done
  const uint32_t tfull = cempty0 + 8 * kQ8CodeStages;
  const uint32_t tempty = tfull + 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQ8RawStages; ++s) {
      mbar_init(rawfull0 + 8 * s, 1);
      mbar_init(rawempty0 + 8 * s, 128);
    }
    for (int s = 0; s < kQ8CodeStages; ++s) {
      // converters, and the codes' TMA
      mbar_init(full0 + 8 * s, 128 + 1);
      mbar_init(cempty0 + 8 * s, 2);  // one commit per MMA thread
    }
    mbar_init(tfull, 2);
    mbar_init(tempty, 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = __ldg(p.tile_off + p.num_groups) * p.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ weight TMA
    if (lane == 0) {
      const uint64_t evict_first = l2_policy_evict_first();
      unsigned it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo t = decode_tile(p, tile);
        const int r0 = SWIGLU ? t.n * 128 : t.n * 256;
        const int r1 = SWIGLU ? p.up_off + t.n * 128 : t.n * 256 + 128;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t st = ring_stage(it, kQ8RawStages);
          if (!mbar_wait(rawempty0 + 8 * st, ring_phase(it, kQ8RawStages) ^ 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = rawfull0 + 8 * st;
          const uint32_t dst = raw0 + st * kQ8RawBytes;
          mbar_arrive_expect_tx(fb, kQ8RawBytes);
          if (p.l2_hint && t.stream) {
            tma_load_3d_hint(dst, &tmW, fb, kb * kBK, r0, t.group, evict_first);
            tma_load_3d_hint(dst + kQ8RawBytes / 2, &tmW, fb, kb * kBK, r1, t.group, evict_first);
          } else {
            tma_load_3d(dst, &tmW, fb, kb * kBK, r0, t.group);
            tma_load_3d(dst + kQ8RawBytes / 2, &tmW, fb, kb * kBK, r1, t.group);
          }
        }
      }
    }
  } else if (warp >= 6 && warp < 10) {
    // ------------------------------------------------------------ token codes
    // One lane of warp 6 loads the tile of expert-ordered code rows [128 x 64]
    // by TMA (rows past the group's end are the next group's or zero fill:
    // their products reach accumulator columns that are never stored); warps
    // 7..9 have no role (the converters' warp numbers fix their TMEM quarters).
    if (warp == 6 && lane == 0) {
      unsigned it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo t = decode_tile(p, tile);
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t st = ring_stage(it, kQ8CodeStages);
          if (!mbar_wait(cempty0 + 8 * st, ring_phase(it, kQ8CodeStages) ^ 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * st;
          mbar_arrive_expect_tx(fb, kQ8CodeBytes);
          tma_load_2d(codes0 + st * kQ8CodeBytes, &tmB, fb, kb * kBK, t.row0);
        }
      }
    }
  } else if (warp >= 10 && warp < 18) {
    // ------------------------------------------------------------ converters
    // TMEM lane quarter (warp % 4) -> weight rows 32 (warp % 4) .. + 31 of both
    // blocks; thread row j reads its 64 int8 of the block (4 x 16 bytes) and
    // writes 32 columns of fp16 pairs (k = 2c, 2c + 1 in column c).  Group g
    // takes the k-blocks whose running index is g modulo kQ8ConvGroups.
    const int q = warp & 3;
    const int grp = (warp - 10) >> 2;
    const int j = 32 * q + lane;
    const int sx = (j >> 1) & 3;
    unsigned it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        if (static_cast<int>(it % kQ8ConvGroups) != grp) continue;
        const uint32_t rs = ring_stage(it, kQ8RawStages);
        const uint32_t sl = ring_stage(it, kQ8Slots);
        bool w = true;
        if (lane == 0)
          w = mbar_wait(rawfull0 + 8 * rs, ring_phase(it, kQ8RawStages), p.status, abort_flag);
          if (w && it >= static_cast<unsigned>(kQ8Slots)) {
            // the slot's previous user, k-block it - kQ8Slots, is done
            const unsigned j = it - kQ8Slots;
            w = mbar_wait(cempty0 + 8 * ring_stage(j, kQ8CodeStages), ring_phase(j, kQ8CodeStages), p.status,
                          abort_flag);
          }
        if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* sw = smem + kQ8CodeRing + rs * kQ8RawBytes;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint4* row = reinterpret_cast<const uint4*>(sw + b * (kQ8RawBytes / 2) + j * kBK);
          uint32_t h[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = row[c ^ sx];  // the TMA's 64-byte swizzle
            i8x4_to_f16x4(v.x, h[8 * c + 0], h[8 * c + 1]);
            i8x4_to_f16x4(v.y, h[8 * c + 2], h[8 * c + 3]);
            i8x4_to_f16x4(v.z, h[8 * c + 4], h[8 * c + 5]);
            i8x4_to_f16x4(v.w, h[8 * c + 6], h[8 * c + 7]);
          }
          tmem_st_32x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kQ8Slot0 + 64 * sl + 32 * b, h);
        }
        // the shared-memory rows were consumed by the conversions above
        mbar_arrive(rawempty0 + 8 * rs);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        mbar_arrive(full0 + 8 * ring_stage(it, kQ8CodeStages));
      }
    }
  } else if (warp == 1 || warp == kQ8MmaWarp2) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads on different schedulers, one per accumulator (Linear1: gate
    // and up; Linear2: the two 128-channel blocks); each does one wait, four
    // MMAs and one commit per k-block (ring position as a wrapping counter,
    // descriptors as increments).  The pace of this loop, not the tensor core,
    // bounds the kernel at these shapes, hence the split.
    if (lane == 0) {
      const int b = warp == 1 ? 0 : 1;
      int sl = 0, cs = 0;   // TMEM slot and code stage of the k-block
      uint32_t ph = 0;      // phase of the code stage's ready barrier
      int local = 0;
      bool ok = true;
      const uint64_t bd0 = smem_desc_sw128(codes0, 16, 1024);
      const uint32_t slot0 = tmem_base + kQ8Slot0;
      const uint32_t dacc = tmem_base + kQ8Tok * b;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++local) {
        const TileInfo t = decode_tile(p, tile);
        const int rows = t.row_end - t.row0;
        const int n = rows <= 16 ? 16 : (rows >= kQ8Tok ? kQ8Tok : (rows + 15) & ~15);
        const uint32_t idesc = idesc_f32acc(128, n, kFmtF16, false, false);
        if (!mbar_wait(tempty, (local & 1) ^ 1, p.status, abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(full0 + 8 * cs, ph, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // B: the token codes, K-major rows of 128 B; a 16-wide k step is 32 B
          // (+2 in the descriptor's address field)
          const uint64_t bd = bd0 + static_cast<uint64_t>(cs * (kQ8CodeBytes >> 4));
          const uint32_t slot = slot0 + 64 * sl;
          mma_f16_tmem_a(dacc, slot + 32 * b, bd, idesc, kb != 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < kBK / 16; ++kk)
            mma_f16_tmem_a(dacc, slot + 32 * b + 8 * kk, bd + 2 * kk, idesc, 1u);
          mma_commit(cempty0 + 8 * cs);
          if (++sl == kQ8Slots) sl = 0;
          if (++cs == kQ8CodeStages) { cs = 0; ph ^= 1; }
        }
        if (!ok) break;
        mma_commit(tfull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Thread = output channel (TMEM lane): channel j of both accumulators,
    // the tile's tokens in chunks of 32 columns; each store instruction of a
    // warp writes 32 consecutive channels of one token row.
    const int q = warp & 3;
    const int j = 32 * q + lane;
    float* sc = scale_area + q * kQ8Tok;  // this warp's copy of the token scales
    float* out = static_cast<float*>(p.out);
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const TileInfo t = decode_tile(p, tile);
      const int rows = t.row_end - t.row0;
      const int ncol = rows <= 32 ? 32 : (rows >= kQ8Tok ? kQ8Tok : (rows + 31) & ~31);
      // the token (Linear1) or row (Linear2) scale of each of the tile's rows
#pragma unroll
      for (int i = 0; i < kQ8Tok / 32; ++i) {
        const int row = t.row0 + 32 * i + lane;
        float s = 0.0f;
        if (row < t.row_end) s = __ldg(p.scale_row + row);
        sc[32 * i + lane] = s;
      }
      __syncwarp();
      const float* scol = p.scale_col + static_cast<long long>(t.group) * p.scale_ld;
      const int c0 = SWIGLU ? t.n * 128 + j : t.n * 256 + j;        // block 0 channel
      const int c1 = SWIGLU ? p.up_off + t.n * 128 + j : c0 + 128;  // block 1 channel
      const bool in0 = c0 < p.n_out;
      const bool in1 = SWIGLU ? in0 : c1 < p.n_out;
      const float s0 = in0 ? __ldg(scol + c0) : 0.0f;
      const float s1 = in1 ? __ldg(scol + c1) : 0.0f;
      const bool got = mbar_wait(tfull, local & 1, p.status, abort_flag);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < ncol; c += 32) {
        float a[32], b[32];
        tmem_ld_32x32(tb + c, a);
        tmem_ld_32x32(tb + kQ8Tok + c, b);
        if (c + 32 == ncol) {
          tc_fence_before();
          mbar_arrive(tempty);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int row = t.row0 + c + i;
          if (row >= t.row_end) continue;
          const float sr = sc[c + i];
          if (SWIGLU) {
            // H = (C * s^W1) * s^X, then SwiGLU
            const float hg = (a[i] * s0) * sr;
            const float hu = (b[i] * s1) * sr;
            if (in0) out[static_cast<long long>(row) * p.ldo + c0] = __fdividef(hg, 1.0f + __expf(-hg)) * hu;
          } else if (p.out_bf16) {
            // rows rounded once to bf16 (RNE) for the combine
            uint16_t* o16 = static_cast<uint16_t*>(p.out) + static_cast<long long>(row) * p.ldo;
            if (in0) o16[c0] = __bfloat16_as_ushort(__float2bfloat16_rn((a[i] * s0) * sr));
            if (in1) o16[c1] = __bfloat16_as_ushort(__float2bfloat16_rn((b[i] * s1) * sr));
          } else {
            if (in0) out[static_cast<long long>(row) * p.ldo + c0] = (a[i] * s0) * sr;
            if (in1) out[static_cast<long long>(row) * p.ldo + c1] = (b[i] * s1) * sr;
          }
        }
      }
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <bool SWIGLU>
cudaError_t launch_q8(const CUtensorMap& w, const CUtensorMap& b, const GemmParams& p, int grid,
                      cudaStream_t s) {
  auto kern = gemm_q8_kernel<SWIGLU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kQ8Smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kQ8Threads, kQ8Smem, s>>>(w, b, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_q8(bool swiglu, const CUtensorMap& w, const CUtensorMap& b,
                           const GemmParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  return swiglu ? launch_q8<true>(w, b, p, grid, s) : launch_q8<false>(w, b, p, grid, s);
}

}  // namespace moe
