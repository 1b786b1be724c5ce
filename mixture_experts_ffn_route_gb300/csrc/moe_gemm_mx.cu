// Persistent grouped GEMM for the MX forms on the block-scaled tensor cores
// (tcgen05.mma kind::mxf8f6f4: FP8 operands, one E8M0 scale per 32 k for
// every row of A and of B, fp32 accumulator in TMEM).
//
//   Linear1: Z = DQ(Xq_e) DQ(W1[e])^T, U = Z_g * sigma(Z_g) * Z_u, and U
//            re-quantised per 32 columns: FP8 codes + E8M0 scales out
//   Linear2: O = DQ(Uq) DQ(W2[e])^T, bf16 (or fp32) out
// These are the stages GMM1 + SwiGLU + MX quantisation and GMM2 of the MXFP
// scenario on the "mega_moe" page (section 计算过程).  The weights keep the
// pages' K-contiguous layout ([E, 2I, H] and [E, H, I]) with their scales
// [E, N, K/32].
//
// Structure (one CTA per SM, 352 threads):
//   warp 0      TMA producer: A tile [128 rows x 128 k] and B tile
//               [256 n x 128 k], both K-major with 128-byte swizzle (Linear1:
//               128 gate rows of W1 and the matching 128 up rows; Linear2: 256
//               rows of W2).  Linear1's A rows are the token codes already laid
//               out in expert order by the quantisation kernel.
//   warps 1, 10 MMA: warp 1 allocates TMEM (one 256-column accumulator and the
//               scale slots of every stage); one lane of each takes one half of
//               the accumulator (B rows 0..127 or 128..255): it copies the
//               stage's A scale atom and its B scale atom into TMEM slots of its
//               own (tcgen05.cp 32x128b.warpx4, ordered before its own MMAs)
//               and issues four MMAs (M 128, N 128, K 32) whose scale byte is
//               the k step.  Splitting the issue over two threads on different
//               schedulers shortens the per-k-block issue path, which bounds the
//               kernel when a k-block carries few weight bytes (E2M1).
//   warps 2..5  epilogue (one accumulator row per thread).
//   warps 6..9  per k-block, the 4 scale bytes of each of the 128 A rows and
//               256 B rows into the stage's three 512-byte atoms (cp.async).
// The tile is as wide as for bf16 so that each k-block moves one A byte per
// two B bytes; two 256-column accumulators would leave no TMEM for the scales,
// so there is one, and the stages the producer loads ahead carry the MMA over
// the epilogue.
// A scale atom holds 128 rows x 4 groups: row r's 4 bytes are the 32-bit word
// at byte (r % 32) * 16 + (r / 32) * 4.  Copied with warpx4, TMEM lane l then
// holds rows l % 32 + 32 c in column c, which is where the MMA reads the scale
// of A row m (lane m, column m / 32) and of B row n (lane n % 32 of each lane
// quarter, column n / 32 of the B slot of the MMA thread that owns row n: rows
// 128..255 are rows 0..127 of the second B atom, in the second thread's slot);
// the byte inside the word is the MMA's scale id.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_tile.cuh"

namespace moe {
namespace {

constexpr int kMxBN = 256;
constexpr int kMxA = kBM * kMxBK;     // 16 KB
constexpr int kMxB = kMxBN * kMxBK;   // 32 KB
constexpr int kMxAtom = 512;          // 128 rows x 4 scale bytes
// scale words per row per k-block: 1 (a k-block of 128 codes), or 2 for the
// packed E2M1 x E2M1 form (kind::mxf4, a k-block of 256 codes in the same
// 128-byte rows); a stage holds that many A atoms and B atoms per 128 B rows
constexpr int kMxWordsMax = 2;
constexpr int kMxAtoms = kMxWordsMax * (1 + kMxBN / 128);
constexpr int kMxStageBytes = ((kMxA + kMxB + kMxAtoms * kMxAtom + 1023) / 1024) * 1024;
constexpr int kMxStages = 4;
constexpr int kMxRing = kMxStages * kMxStageBytes;
constexpr int kMxBarBytes = 256;
constexpr int kMxStgWords = 36;       // staging row pitch (32 data words + 4 pad)
constexpr int kMxStg = 4 * 32 * kMxStgWords * 4;
constexpr int kMxSmem = kMxRing + 1024 + kMxBarBytes + kMxStg;
constexpr int kMxThreads = 352;
constexpr int kMxMmaWarp2 = 10;       // the second MMA thread's warp
constexpr int kMxTmemCols = 512;
// stage s, MMA thread b, scale word w: A scales at kMxSfCol + 32 s + 16 b + 4 w,
// its B scales 8 on
constexpr int kMxSfCol = kMxBN;
constexpr int kMxSfStride = 32;
static_assert(kMxSfCol + kMxSfStride * kMxStages <= kMxTmemCols, "TMEM columns");
static_assert(8 * (2 * kMxStages + 2) + 8 <= kMxBarBytes, "barrier area");
static_assert(kMxSmem <= 232448, "shared memory");

// 4-byte global -> shared copy.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Copy a 32-row x 16-byte matrix from shared memory to TMEM columns
// [taddr, taddr + 4), replicated into all four lane quarters.
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

// Shared-memory descriptor of an unswizzled matrix (layout type 0): 8-row
// core matrices of 16-byte rows, `sbo` bytes apart.
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// D[tmem] (+)= (A * sA)(B * sB)^T with FP8 A, B and E8M0 scales in TMEM.
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= (A * sA)(B * sB)^T with packed E2M1 A, B (two codes per byte,
// even element in the low nibble), K 64, and two E8M0 scales per row (one per
// 32 codes) read from bytes sid and sid + 1 of the row's scale word.
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of the block-scaled kind: bits 4-5 B scale id,
// 7-9 A format, 10-12 B format (0 = E4M3, 1 = E5M2, 5 = E2M1), 15/16 A/B major
// (0 = K-major), 17-22 N >> 3, 23 scale type (1 = E8M0), 24-28 M >> 4,
// 29-30 A scale id.
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t afmt, uint32_t bfmt) {
  return (afmt << 7) | (bfmt << 10) | ((static_cast<uint32_t>(N) >> 3) << 17) | (1u << 23) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}
// kind::mxf4: E2M1 is format 1 for both operands (probe-confirmed: all-ones
// tiles and random codes against a CPU product)
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N) { return idesc_mx(M, N, 1, 1); }
__host__ __device__ constexpr uint32_t idesc_sf_ids(uint32_t a_id, uint32_t b_id) {
  return (a_id << 29) | (b_id << 4);
}

// Element formats, by their tensor-core codes: 0 = E4M3, 1 = E5M2 (one code
// per byte), 5 = E2M1 (two codes per byte in memory, even element in the low
// nibble; TMA's 16U4_ALIGN16B type spreads each 16 of them over 16 bytes of
// shared memory, the layout the MMA reads).  EMAX: the largest power-of-two
// exponent of the format (448 = 1.75 * 2^8, 57344 = 1.75 * 2^15, 6 = 1.5 * 2^2).
template <int FMT>
struct MxFmt {
  static constexpr int EMAX = FMT == 0 ? 8 : (FMT == 1 ? 15 : 2);
  static constexpr bool FP4 = FMT == 5;
  static constexpr int GROUP_BYTES = FP4 ? 16 : 32;  // bytes of one group of 32 codes
  static constexpr __nv_fp8_interpretation_t KIND = FMT == 1 ? __NV_E5M2 : __NV_E4M3;
};

// Shared exponent of a group with maximum magnitude `amax` (the OCP MX rule):
// floor(log2 amax) - emax, clamped below at -127; read off the fp32 exponent
// field (a zero or subnormal maximum gives -127).
template <int FMT>
__device__ __forceinline__ int mx_exponent(float amax) {
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - MxFmt<FMT>::EMAX;
  return e < -127 ? -127 : e;
}

// Four values (already divided by the group scale) -> four FP8 codes, round to
// nearest even with saturation, first value in the lowest byte.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, MxFmt<FMT>::KIND);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, MxFmt<FMT>::KIND);
  return (lo & 0xFFFFu) | (hi << 16);
}

// Eight values -> eight E2M1 codes in one word, round to nearest even with
// saturation, first value in the lowest nibble.
__device__ __forceinline__ uint32_t fp4x8(const float* v) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w |= static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(make_float2(v[2 * i], v[2 * i + 1]), __NV_E2M1,
                                                        cudaRoundNearest) & 0xFFu) << (8 * i);
  return w;
}

// Quantise 32 values of one group: GROUP_BYTES / 4 words of codes (8 for
// FP8, 4 for E2M1), returns the scale code.
template <int FMT>
__device__ __forceinline__ uint32_t mx_group(const float (&v)[32], uint32_t (&w)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int X = mx_exponent<FMT>(amax);
  // 2^-X, exact: X is in [-127, 125] so 127 - X is a normal exponent field
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - X) << 23);
  if (MxFmt<FMT>::FP4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float s[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j] = v[8 * i + j] * inv;
      w[i] = fp4x8(s);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = fp8x4<FMT>(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
  }
  return static_cast<uint32_t>(X + 127);
}

template <bool SWIGLU, int AF, int BF, bool PACKED>
__global__ void __launch_bounds__(kMxThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  static_assert(!PACKED || (AF == 5 && BF == 5), "the packed form is E2M1 x E2M1");
  constexpr int WORDS = PACKED ? 2 : 1;        // scale words per row per k-block
  constexpr int KBX = PACKED ? 128 : kMxBK;   // TMA x step per k-block: bytes, or codes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bar_area = smem + kMxRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * (2 * kMxStages + 2));
  uint32_t* stg_area = reinterpret_cast<uint32_t*>(bar_area + kMxBarBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t tiles0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bar_area);
  const uint32_t empty0 = full0 + 8 * kMxStages;
  const uint32_t tfull = empty0 + 8 * kMxStages;  // accumulator ready for the epilogue
  const uint32_t tempty = tfull + 8;              // accumulator drained

  if (threadIdx.x == 0) {
    // a stage is complete when the TMA bytes have landed (one arrival with the
    // byte count) and the row threads' scales have: one arrival per row warp
    // (chunked loads) or per row thread (4-byte copies)
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(full0 + 8 * s, 1 + (p.sf_vec ? 4 : 128));
      mbar_init(empty0 + 8 * s, 2);  // one commit per MMA thread
    }
    mbar_init(tfull, 2);
    mbar_init(tempty, 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kMxTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = __ldg(p.tile_off + p.num_groups) * p.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t evict_first = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
        const TileInfo t = decode_tile(p, tile);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, p.status, abort_flag)) break;
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t sa = tiles0 + stage * kMxStageBytes;
          const uint32_t sb = sa + kMxA;
          const int kx = kb * KBX;
          // an unpacked E2M1 tile arrives as half as many bytes as it fills;
          // a packed one fills its tile
          if (PACKED)
            mbar_arrive_expect_tx(fb, kMxA + kMxB);
          else
            mbar_arrive_expect_tx(fb, (MxFmt<AF>::FP4 ? kMxA / 2 : kMxA) + (MxFmt<BF>::FP4 ? kMxB / 2 : kMxB));
          tma_load_2d(sa, &tmA, fb, kx, t.row0);
          if (p.l2_hint && t.stream) {
            if (SWIGLU) {
              tma_load_3d_hint(sb, &tmB, fb, kx, t.n * 128, t.group, evict_first);
              tma_load_3d_hint(sb + 128 * kMxBK, &tmB, fb, kx, p.up_off + t.n * 128, t.group,
                               evict_first);
            } else {
              tma_load_3d_hint(sb, &tmB, fb, kx, t.n * kMxBN, t.group, evict_first);
            }
          } else if (SWIGLU) {
            tma_load_3d(sb, &tmB, fb, kx, t.n * 128, t.group);
            tma_load_3d(sb + 128 * kMxBK, &tmB, fb, kx, p.up_off + t.n * 128, t.group);
          } else {
            tma_load_3d(sb, &tmB, fb, kx, t.n * kMxBN, t.group);
          }
          if (++stage == kMxStages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp >= 6 && warp < 10) {
    // ------------------------------------------------------------ row threads
    // Thread (gw, lane) places the scale word(s) of A row r and of B rows r
    // and r + 128, r = 8 gw + lane / 4 + 32 (lane % 4), for each k-block: the
    // 32 lanes of a warp then write 32 consecutive words of an atom.  A rows
    // past the group's end and B rows past the output's end are not copied:
    // whatever their stale scales hold only reaches accumulator entries that
    // are never stored.
    const int gw = warp - 6;
    const int sr = 8 * gw + (lane >> 2) + 32 * (lane & 3);
    const uint32_t atom_off = static_cast<uint32_t>(128 * gw + 4 * lane);
    // this thread's scale rows in a tile: A row sr, B rows sr and sr + 128
    // (Linear1: 128 gate rows, then the matching up rows); nullptr past the
    // group's end or the output's end
    auto row_ptrs = [&](int tile, const uint8_t* (&src)[3]) {
      const TileInfo t = decode_tile(p, tile);
      const int row = t.row0 + sr;
      src[0] = row < t.row_end ? p.sfa + static_cast<long long>(row) * p.sf_ld : nullptr;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = SWIGLU ? t.n * 128 + sr : t.n * kMxBN + 128 * h + sr;
        const int nr = SWIGLU ? (h == 0 ? c : p.up_off + c) : c;
        src[1 + h] = c < p.n_out ? p.sfb + t.group * p.sfb_ld + static_cast<long long>(nr) * p.sf_ld
                                 : nullptr;
      }
    };
    int stage = 0;
    uint32_t phase = 0;
    if (p.sf_vec) {
      // Scale rows are whole 16-byte chunks (4 FP8 k-blocks, or 2 packed
      // ones): each is loaded once into registers, a chunk ahead of its use
      // and across tiles, and each k-block's words are stored into the atoms.
      // A quarter of the 4-byte gathers' requests, and their latency is off
      // the stage's path.
      constexpr int KPC = 4 / WORDS;  // k-blocks per chunk
      const int nchunks = p.num_kb / KPC;
      int ltile = blockIdx.x, lchunk = 0;  // load cursor
      const uint8_t* lsrc[3] = {nullptr, nullptr, nullptr};
      if (ltile < total) row_ptrs(ltile, lsrc);
      auto load_next = [&](uint4 (&v)[3]) {
#pragma unroll
        for (int i = 0; i < 3; ++i)
          v[i] = (ltile < total && lsrc[i] != nullptr)
                     ? __ldg(reinterpret_cast<const uint4*>(lsrc[i] + 16 * lchunk))
                     : make_uint4(0u, 0u, 0u, 0u);
        if (++lchunk == nchunks) {
          lchunk = 0;
          ltile += gridDim.x;
          if (ltile < total) row_ptrs(ltile, lsrc);
        }
      };
      auto word = [](const uint4& v, int i) -> uint32_t {
        return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
      };
      uint4 cur[3], nxt[3];
      load_next(cur);
      load_next(nxt);
      bool fresh = true, ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (__shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0)) break;
        const uint8_t* src[3];
        row_ptrs(tile, src);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          const int j = kb % KPC;
          if (j == 0) {
            if (!fresh) {
#pragma unroll
              for (int i = 0; i < 3; ++i) cur[i] = nxt[i];
              load_next(nxt);
            }
            fresh = false;
          }
          bool w = true;
          if (lane == 0) w = mbar_wait(empty0 + 8 * stage, phase ^ 1, p.status, abort_flag);
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
          uint8_t* atoms = smem + stage * kMxStageBytes + kMxA + kMxB;
#pragma unroll
          for (int w2 = 0; w2 < WORDS; ++w2) {
            const int wi = j * WORDS + w2;
            if (src[0] != nullptr)
              *reinterpret_cast<uint32_t*>(atoms + w2 * kMxAtom + atom_off) = word(cur[0], wi);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (src[1 + h] != nullptr)
                *reinterpret_cast<uint32_t*>(atoms + (WORDS * (1 + h) + w2) * kMxAtom + atom_off) =
                    word(cur[1 + h], wi);
          }
          // the tcgen05.cp that reads the atoms goes through the async proxy;
          // one arrival per warp once all its lanes have written and fenced
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full0 + 8 * stage);
          if (++stage == kMxStages) { stage = 0; phase ^= 1; }
        }
      }
    } else {
      // Scale rows that are not whole 16-byte chunks: 4-byte cp.async per row
      // and k-block, each thread arriving when its copies have landed.
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        if (__shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0)) break;
        const uint8_t* src[3];
        row_ptrs(tile, src);
        bool ok = true;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          bool w = true;
          if (lane == 0) w = mbar_wait(empty0 + 8 * stage, phase ^ 1, p.status, abort_flag);
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
          const uint32_t atoms = tiles0 + stage * kMxStageBytes + kMxA + kMxB;
          // word w of the k-block's scales: A atom w, B atoms WORDS (1 + h) + w
#pragma unroll
          for (int w2 = 0; w2 < WORDS; ++w2) {
            const int off = (kb * WORDS + w2) * 4;
            if (src[0] != nullptr) cp_async4(atoms + w2 * kMxAtom + atom_off, src[0] + off);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (src[1 + h] != nullptr)
                cp_async4(atoms + (WORDS * (1 + h) + w2) * kMxAtom + atom_off, src[1 + h] + off);
          }
          cp_async_arrive(full0 + 8 * stage);
          if (++stage == kMxStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1 || warp == kMxMmaWarp2) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      const int b = warp == 1 ? 0 : 1;  // accumulator half = B rows 128 b ..
      constexpr uint32_t idesc = PACKED ? idesc_mxf4(kBM, kMxBN / 2) : idesc_mx(kBM, kMxBN / 2, AF, BF);
      const uint32_t d = tmem_base + (kMxBN / 2) * b;
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++local) {
        if (!mbar_wait(tempty, (local & 1) ^ 1, p.status, abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, p.status, abort_flag)) break;
          // the row threads' copies went through the generic proxy
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = tiles0 + stage * kMxStageBytes;
          const uint32_t sb = sa + kMxA + b * (kMxBN / 2) * kMxBK;
          const uint32_t atoms = sa + kMxA + kMxB;
          const uint32_t tsa = tmem_base + kMxSfCol + kMxSfStride * stage + 16 * b;
          const uint32_t tsb = tsa + 8;
          // scale atoms -> TMEM; executes before the MMAs this thread issues after it
#pragma unroll
          for (int w = 0; w < WORDS; ++w) {
            tmem_cp_atom(tsa + 4 * w, smem_desc_plain(atoms + w * kMxAtom, 128, 128));
            tmem_cp_atom(tsb + 4 * w, smem_desc_plain(atoms + (WORDS * (1 + b) + w) * kMxAtom, 128, 128));
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // K-major rows of 128 B; a k step (32 FP8 codes, or 64 packed E2M1
            // codes) is 32 B along the row
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(sb + kk * 32, 16, 1024);
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            if (PACKED) {
              // two groups of 32 per MMA: scale bytes 2 (kk % 2) and + 1 of word kk / 2
              const uint32_t w = static_cast<uint32_t>(kk >> 1), sid = 2u * static_cast<uint32_t>(kk & 1);
              mma_mxf4(d, ad, bd, idesc | idesc_sf_ids(sid, sid), tsa + 4 * w, tsb + 4 * w, acc);
            } else {
              mma_mx(d, ad, bd, idesc | idesc_sf_ids(kk, kk), tsa, tsb, acc);
            }
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == kMxStages) { stage = 0; phase ^= 1; }
        }
        mma_commit(tfull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    uint32_t* stg = stg_area + q * 32 * kMxStgWords;
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const TileInfo t = decode_tile(p, tile);
      const bool got = mbar_wait(tfull, local & 1, p.status, abort_flag);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int wrow0 = t.row0 + q * 32;
      const int row = wrow0 + lane;
      if (wrow0 >= t.row_end) {
        // all 32 rows of this warp lie past the group's end: nothing to store
        tc_fence_before();
        mbar_arrive(tempty);
        continue;
      }
      if (SWIGLU) {
        // 128 SwiGLU columns = four scale groups, each held whole by this
        // thread: codes staged as 128 (FP8) or 64 (E2M1) bytes per row,
        // scales as one word
        constexpr int GB = MxFmt<AF>::GROUP_BYTES;
        uint8_t* out = static_cast<uint8_t*>(p.out);
        const int col = t.n * 128;
        uint32_t sc = 0;
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
          float g[32], u[32];
          tmem_ld_32x32(tb + 32 * h, g);
          tmem_ld_32x32(tb + 128 + 32 * h, u);
#pragma unroll
          // SiLU(g) * u; the fast divide (2 ulp) returns 0 once 1 + e^-g
          // exceeds 2^126, the limit of g / (1 + e^-g) there
          for (int i = 0; i < 32; ++i) g[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
          uint32_t w[8];
          sc |= mx_group<AF>(g, w) << (8 * h);
          uint4* srow4 = reinterpret_cast<uint4*>(stg + lane * kMxStgWords + (GB / 4) * h);
          srow4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          if (GB == 32) srow4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        // the accumulator has been read: the next tile's MMAs may start
        tc_fence_before();
        mbar_arrive(tempty);
        __syncwarp();
        // one store instruction: 4 rows x 128 bytes (FP8) or 8 rows x 64 bytes
        // (E2M1); p.ldo is the row pitch in bytes
        constexpr int LPR = GB / 4;  // lanes per row
        const int qd = lane % LPR;
        const long long cbytes = static_cast<long long>(col) * GB / 32;
        if (col < p.n_out) {
#pragma unroll
          for (int rr = 0; rr < 32; rr += 32 / LPR) {
            const int r = rr + lane / LPR;
            const uint4 v = reinterpret_cast<const uint4*>(stg + r * kMxStgWords)[qd];
            const int grow = wrow0 + r;
            if (grow < t.row_end)
              *reinterpret_cast<uint4*>(out + static_cast<long long>(grow) * p.ldo + cbytes + 16 * qd) = v;
          }
        }
        if (row < t.row_end) {
          // scale bytes of the groups inside the output (a last tile past I
          // keeps only its first two)
          uint8_t* sdst = p.out_sf + static_cast<long long>(row) * p.out_sf_ld + 4 * t.n;
          if (col + 128 <= p.n_out)
            *reinterpret_cast<uint32_t*>(sdst) = sc;
          else
            *reinterpret_cast<uint16_t*>(sdst) = static_cast<uint16_t>(sc);
        }
        __syncwarp();
      } else if (p.out_bf16) {
        // rows rounded once to bf16 (RNE) for the combine
        uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll 1
        for (int c = 0; c < kMxBN; c += 32) {
          float v[32];
          tmem_ld_32x32(tb + c, v);
          if (c + 32 == kMxBN) {
            tc_fence_before();
            mbar_arrive(tempty);
          }
          const int col = t.n * kMxBN + c;
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
          uint4* srow4 = reinterpret_cast<uint4*>(stg + lane * kMxStgWords);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            srow4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          __syncwarp();
          // 8 rows x 64 bytes per store instruction
          const int qd = lane & 3;
          if (col < p.n_out) {
#pragma unroll
            for (int rr = 0; rr < 32; rr += 8) {
              const int r = rr + (lane >> 2);
              const uint4 x = reinterpret_cast<const uint4*>(stg + r * kMxStgWords)[qd];
              const int grow = wrow0 + r;
              if (grow < t.row_end)
                *reinterpret_cast<uint4*>(out + static_cast<long long>(grow) * p.ldo + col + 8 * qd) = x;
            }
          }
          __syncwarp();
        }
      } else {
        float* out = static_cast<float*>(p.out);
#pragma unroll 1
        for (int c = 0; c < kMxBN; c += 32) {
          float v[32];
          tmem_ld_32x32(tb + c, v);
          if (c + 32 == kMxBN) {
            tc_fence_before();
            mbar_arrive(tempty);
          }
          const int col = t.n * kMxBN + c;
          float4* srow4 = reinterpret_cast<float4*>(stg + lane * kMxStgWords);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            srow4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          __syncwarp();
          // 4 rows x 128 bytes per store instruction
          const int qd = lane & 7;
          if (col < p.n_out) {
#pragma unroll
            for (int rr = 0; rr < 32; rr += 4) {
              const int r = rr + (lane >> 3);
              const float4 x = reinterpret_cast<const float4*>(stg + r * kMxStgWords)[qd];
              const int grow = wrow0 + r;
              if (grow < t.row_end)
                *reinterpret_cast<float4*>(out + static_cast<long long>(grow) * p.ldo + col + 4 * qd) = x;
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
    tmem_dealloc(tmem_base, kMxTmemCols);
  }
}

// Q_MX of bf16 rows: one warp per row, one lane per group of 32 at a time.
// With `inv` set, row t's codes and scales go to rows inv[t * k + j] (j < k,
// skipping dropped assignments, inv = -1) of the outputs: the rows in expert
// order that the MX Linear1 reads, each token quantised once.
template <int FMT>
__global__ void __launch_bounds__(256)
    mx_quant_rows_kernel(const uint16_t* __restrict__ x, int rows, int cols,
                         uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                         const int* __restrict__ inv, int k) {
  constexpr int GB = MxFmt<FMT>::GROUP_BYTES;
  const int lane = threadIdx.x & 31;
  const int groups = cols / 32;
  const long long row_bytes = static_cast<long long>(groups) * GB;
  const int wpb = blockDim.x >> 5;
  for (int row = blockIdx.x * wpb + (threadIdx.x >> 5); row < rows; row += gridDim.x * wpb) {
    const uint16_t* xr = x + static_cast<long long>(row) * cols;
    int dst[16];
    int ndst = 1;
    dst[0] = row;
    if (inv != nullptr) {
      ndst = 0;
      for (int j = 0; j < k; ++j) {
        const int r = __ldg(inv + static_cast<long long>(row) * k + j);
        if (r >= 0 && in_bounds(r, static_cast<long long>(rows) * k)) dst[ndst++] = r;
      }
    }
    for (int g = lane; g < groups; g += 32) {
      const uint4* src = reinterpret_cast<const uint4*>(xr + 32 * g);
      float v[32];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 b = __ldcs(src + j);
        const uint32_t u[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[8 * j + 2 * i] = bf16_lo(u[i]);
          v[8 * j + 2 * i + 1] = bf16_hi(u[i]);
        }
      }
      uint32_t w[8];
      const uint32_t sc = mx_group<FMT>(v, w);
      for (int d = 0; d < ndst; ++d) {
        uint4* out = reinterpret_cast<uint4*>(codes + static_cast<long long>(dst[d]) * row_bytes + GB * g);
        out[0] = make_uint4(w[0], w[1], w[2], w[3]);
        if (GB == 32) out[1] = make_uint4(w[4], w[5], w[6], w[7]);
        scales[static_cast<long long>(dst[d]) * groups + g] = static_cast<uint8_t>(sc);
      }
    }
  }
}

template <bool SWIGLU, int AF, int BF, bool PACKED = false>
cudaError_t launch_mx(const GemmMaps& m, const GemmParams& p, int grid, cudaStream_t s) {
  auto kern = gemm_mx_kernel<SWIGLU, AF, BF, PACKED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kMxThreads, kMxSmem, s>>>(m.a, m.b, p);
  return cudaGetLastError();
}

template <bool SWIGLU>
cudaError_t launch_mx_pair(int afmt, int bfmt, bool packed, const GemmMaps& m, const GemmParams& p,
                           int grid, cudaStream_t s) {
  if (packed) return afmt == 5 && bfmt == 5 ? launch_mx<SWIGLU, 5, 5, true>(m, p, grid, s) : cudaErrorInvalidValue;
  if (afmt == 0 && bfmt == 0) return launch_mx<SWIGLU, 0, 0>(m, p, grid, s);
  if (afmt == 1 && bfmt == 1) return launch_mx<SWIGLU, 1, 1>(m, p, grid, s);
  if (afmt == 0 && bfmt == 5) return launch_mx<SWIGLU, 0, 5>(m, p, grid, s);
  if (afmt == 1 && bfmt == 5) return launch_mx<SWIGLU, 1, 5>(m, p, grid, s);
  if (afmt == 5 && bfmt == 5) return launch_mx<SWIGLU, 5, 5>(m, p, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace

bool mx_pair_supported(int afmt, int bfmt) {
  return (afmt == bfmt && (afmt == 0 || afmt == 1 || afmt == 5)) || ((afmt == 0 || afmt == 1) && bfmt == 5);
}

cudaError_t launch_gemm_mx(bool swiglu, int afmt, int bfmt, bool packed, const GemmMaps& maps,
                           const GemmParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  return swiglu ? launch_mx_pair<true>(afmt, bfmt, packed, maps, p, grid, s)
                : launch_mx_pair<false>(afmt, bfmt, packed, maps, p, grid, s);
}

cudaError_t launch_mx_quant_rows(int fmt, const uint16_t* x, int rows, int cols, uint8_t* codes,
                                 uint8_t* scales, const int* inv, int k, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (inv != nullptr && (k < 1 || k > 16)) return cudaErrorInvalidValue;
  const int wpb = 8;
  long long blocks = (rows + wpb - 1) / wpb;
  if (blocks > 8LL * num_sms()) blocks = 8LL * num_sms();
  const int b = static_cast<int>(blocks);
  if (fmt == 0)
    mx_quant_rows_kernel<0><<<b, 32 * wpb, 0, s>>>(x, rows, cols, codes, scales, inv, k);
  else if (fmt == 1)
    mx_quant_rows_kernel<1><<<b, 32 * wpb, 0, s>>>(x, rows, cols, codes, scales, inv, k);
  else if (fmt == 5)
    mx_quant_rows_kernel<5><<<b, 32 * wpb, 0, s>>>(x, rows, cols, codes, scales, inv, k);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

MOE_DEFINE_BOUNDS_TAKE(gemm_mx)

}  // namespace moe
