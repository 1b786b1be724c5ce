// Fused router: gating GEMM on the tensor cores with the routing decision in
// its epilogue.
//
// "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例", section 路由与负载 / 路由张量:
// the gating linear l = X Wg ([n, h] -> [n, E]), the affinity a = score(l),
// the selection I_t = TopK(a + beta) and the mixing weights g = alpha a /
// sum_{I_t} a; section 路由与负载 / Hash 路由: the ids are the table row
// tid2eid[token], the gates unchanged.  The softmax gate of "Megatron
// 分布式训练全维度并行技术文档" (section 4.2) selects the top-k of the logits.
//
// One CTA owns a 128-row tile of X and all E <= 384 logit columns, over one
// slice of the contraction H.  S CTAs (a thread-block cluster, S in {1, 2, 4,
// 8}) split H so that the grid covers the SMs; they add their partial logits
// through distributed shared memory, in a fixed order, and each then decides
// 128 / S of the tile's rows.  No fp32 logits go to memory.
//
//   warp 0      TMA producer: X tile [128 rows x 64 k] K-major and Wg tile
//               [64 k x E] MN-major (Wg's own [H, E] layout), 128-byte swizzle.
//   warp 1      TMEM allocation; one lane issues tcgen05.mma (M 128, N <= 256,
//               K 16; a second MMA for columns 256..383) into one accumulator.
//   warps 2-5   during the main loop: write their share of Wg transposed
//               (one 64-row block of Wg per CTA at most), which the float64
//               re-decision reads; then copy the accumulator, one row per
//               thread, into shared memory over the drained operand ring
//               (16-byte chunks XOR-swizzled by row, conflict-free both ways).
//   all warps   after the cluster barrier: one warp per row sums the S partial
//               rows (ranks 0..S-1 in order), scores them, adds the selection
//               bias, takes k+1 warp arg-max rounds (larger score first, equal
//               scores to the lower id), writes ids and gates, and lists a
//               token whose first k+1 scores hold a pair closer than the
//               decision band, with its candidates, for the float64 re-decision
//               (moe_route.cu), exactly as the general path does.
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_route.cuh"

namespace moe {

namespace {

constexpr int kThreads = 320;
constexpr int kFusedMaxE = 384;                 // 6 boxes of 64 columns
constexpr int kRingMax = 6 * 128 * 64 * 4;      // 192 KB: the dump of 384 fp32 columns
constexpr int kBoxBytes = 64 * kBK * 2;         // one 64 x 64 bf16 box of Wg: 8 KB
constexpr int kABytes = kBM * kBK * 2;          // X tile: 16 KB

struct FusedParams {
  int T, H, E, k, fn, renorm, V, select;
  float alpha;
  int S, kbs, nkb, nbx, stages, stage_bytes, ring_bytes, tmem_cols, n_rt;
  const uint16_t* Wg;
  const float* bias;
  const int32_t* token_ids;
  const int32_t* tid2eid;
  int32_t* E_ids;
  float* G;
  float* logits_out;
  uint16_t* WgT;
  RouteScratch rs;
  int* status;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster passes both cluster barriers,
// whatever happened before (a timed-out wait included), so no CTA can wait
// for one that has left.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Shared-memory address of the same location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Wait for a barrier phase at teardown, whether or not the kernel is
// aborting (copies or MMAs still in flight must finish before the CTA leaves
// or frees TMEM); gives up after limit_ns.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return;
}

// Byte offset of 16-byte chunk c (4 columns) of accumulator row r in the
// dump: rows of cpr chunks, chunk index XOR (r mod 8).  A thread writing its
// row and a warp reading one row both touch 8 distinct bank quads per phase.
__device__ __forceinline__ uint32_t dump_off(int r, int c, int cpr) {
  return static_cast<uint32_t>((r * cpr + (c ^ (r & 7))) * 16);
}

// WgT[e][h] for the 64 rows h of k-block kb: thread i takes experts 2i, 2i+1
// (one 32-bit word of each Wg row), 16 rows at a time.
__device__ __forceinline__ void transpose_block(const FusedParams& p, int kb, int tid, int nthreads) {
  const int E = p.E, H = p.H;
  for (int pr = tid; pr < E / 2; pr += nthreads) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.Wg) + pr;  // column pair pr
#pragma unroll 1
    for (int i0 = 0; i0 < 64; i0 += 16) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = __ldg(src + static_cast<long long>(kb * 64 + i0 + i) * (E / 2));
      uint32_t lo[8], hi[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        lo[m] = (w[2 * m] & 0xFFFFu) | (w[2 * m + 1] << 16);
        hi[m] = (w[2 * m] >> 16) | (w[2 * m + 1] & 0xFFFF0000u);
      }
      uint4* d0 = reinterpret_cast<uint4*>(p.WgT + static_cast<long long>(2 * pr) * H + kb * 64 + i0);
      uint4* d1 = reinterpret_cast<uint4*>(p.WgT + static_cast<long long>(2 * pr + 1) * H + kb * 64 + i0);
      d0[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      d0[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
      d1[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      d1[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    }
  }
}

// The routing decision of token t from its fp32 logits, one warp: lane l
// holds the logits of chunks l, l + 32, l + 64 (columns 4c .. 4c + 3).
__device__ __forceinline__ void decide_row(const FusedParams& p, int t, const float (&lg)[12],
                                           int lane) {
  const int E = p.E, k = p.k, fn = p.fn;
  // column of register slot i
  auto col = [&](int i) { return 4 * (lane + 32 * (i >> 2)) + (i & 3); };
  float lmax = 0.0f, zsum = 1.0f;
  if (fn == 2) {
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < 12; ++i)
      if (col(i) < E) m = fmaxf(m, lg[i]);
    lmax = warp_max(m);
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < 12; ++i)
      if (col(i) < E) z += expf(lg[i] - lmax);
    zsum = warp_sum(z);
  }
  int my_sel = -1;    // lane j < k: the j-th id
  float my_l = 0.0f;  // and its logit
  bool tok_ok = true;
  if (p.token_ids != nullptr) {
    // ---------------------------------------------------------------- hash
    const int tok = __ldg(p.token_ids + t);
    tok_ok = tok >= 0 && tok < p.V;
    if (!tok_ok && lane == 0) set_flag(p.status, kFlagBadToken);
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      const int e = tok_ok ? __ldg(p.tid2eid + static_cast<long long>(tok) * k + j) : -1;
      float mine = 0.0f;
#pragma unroll
      for (int i = 0; i < 12; ++i)
        if (col(i) == e) mine = lg[i];
      const float le = __shfl_sync(0xffffffffu, mine, e >= 0 ? (e >> 2) & 31 : 0);
      if (lane == j) {
        my_sel = e;
        my_l = le;
      }
    }
  } else {
    // ---------------------------------------------------------------- top-k
    float sc[12];
#pragma unroll
    for (int i = 0; i < 12; ++i) {
      const int e = col(i);
      sc[i] = -FLT_MAX;
      if (e < E) {
        float v = score_f32(lg[i], fn);
        if (p.bias != nullptr) v += __ldg(p.bias + e);
        sc[i] = v;
      }
    }
    const int rounds = (k < E) ? k + 1 : k;
    bool close = false;
    float prev = 0.0f, kth = 0.0f;
#pragma unroll 1
    for (int r = 0; r < rounds; ++r) {
      float best = -FLT_MAX;
      int bid = 0x7fffffff;
      float bl = 0.0f;
#pragma unroll
      for (int i = 0; i < 12; ++i)
        if (col(i) < E && before(sc[i], col(i), best, bid)) {
          best = sc[i];
          bid = col(i);
          bl = lg[i];
        }
      warp_argmax_payload(best, bid, bl);
#pragma unroll
      for (int i = 0; i < 12; ++i)
        if (col(i) == bid) sc[i] = -FLT_MAX;  // taken
      if (r > 0) close |= (prev - best) < band_at(prev, fn);
      prev = best;
      if (r == k - 1) kth = best;
      if (r < k && lane == r) {
        my_sel = bid;
        my_l = bl;
      }
    }
    if (close) {
      // candidates: every expert within twice the band below the k-th score
      const float lim = kth - 2.0f * band_at(kth, fn);
      int count = 0;
      bool cand[12];
#pragma unroll
      for (int i = 0; i < 12; ++i) {
        const int e = col(i);
        bool c = false;
        if (e < E) {
          float v = score_f32(lg[i], fn);
          if (p.bias != nullptr) v += __ldg(p.bias + e);
          c = v >= lim;
        }
        cand[i] = c;
        count += __popc(__ballot_sync(0xffffffffu, c));
      }
      int base = 0;
      if (lane == 0) {
        base = atomicAdd(p.rs.counters + 1, count);
        const int fi = atomicAdd(p.rs.counters + 0, 1);
        p.rs.flagged[fi] = make_int4(t, base, count, 0);
        p.rs.fnorm[fi] = make_float2(lmax, zsum);
      }
      base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
      for (int i = 0; i < 12; ++i) {
        const unsigned bm = __ballot_sync(0xffffffffu, cand[i]);
        if (cand[i]) {
          const int at = base + __popc(bm & ((1u << lane) - 1u));
          p.rs.pairs[at] = make_int2(t, col(i));
          p.rs.plogit[at] = lg[i];
        }
        base += __popc(bm);
      }
    }
  }
  // gates (a close token's ids and gates are rewritten by the re-decision)
  float a = 0.0f;
  if (lane < k) {
    if (my_sel >= 0 && my_sel < E) {
      a = affinity_f32(my_l, fn, lmax, zsum);
    } else if (tok_ok) {
      set_flag(p.status, kFlagBadExpert);  // a table entry outside [0, E)
    }
  }
  float den = 0.0f;
  for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, a, j);
  if (lane < k) {
    float g = p.alpha * a;
    if (p.renorm) g = den > 0.0f ? p.alpha * a / den : 0.0f;
    p.E_ids[static_cast<long long>(t) * k + lane] = my_sel;
    p.G[static_cast<long long>(t) * k + lane] = g;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    route_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bar_area = smem + p.ring_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bar_area);
  const uint32_t empty0 = full0 + 8 * p.stages;
  const uint32_t tfull = empty0 + 8 * p.stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * (2 * p.stages + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int S = p.S;
  const int rank = S > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int rt = blockIdx.x / S;
  const int row0 = rt * kBM;
  const int kb0 = rank * p.kbs;
  const int kb1 = min(kb0 + p.kbs, p.nkb);
  const int ncols = p.nbx * 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int kb = kb0; kb < kb1 && !*abort_flag; ++kb) {
        if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, p.status, abort_flag)) break;
        const uint32_t fb = full0 + 8 * stage;
        const uint32_t sa = ring0 + stage * p.stage_bytes;
        mbar_arrive_expect_tx(fb, p.stage_bytes);
        tma_load_2d(sa, &tmX, fb, kb * kBK, row0);
        for (int j = 0; j < p.nbx; ++j)
          tma_load_3d(sa + kABytes + j * kBoxBytes, &tmW, fb, j * 64, kb * kBK, 0);
        ++issued;
        if (++stage == p.stages) { stage = 0; phase ^= 1; }
      }
      // let the copies still in flight land before the ring is reused or the
      // CTA leaves (they have all landed already unless a wait gave up)
      for (int i = 0; i < min(issued, p.stages); ++i) {
        if (--stage < 0) { stage = p.stages - 1; phase ^= 1; }
        drain_wait(full0 + 8 * stage, phase, 10000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const int n1 = ncols < 256 ? ncols : 256;
      const int n2 = ncols - n1;
      const uint32_t id1 = idesc_f32acc(kBM, n1, kFmtBF16, false, true);
      const uint32_t id2 = idesc_f32acc(kBM, n2 > 0 ? n2 : 64, kFmtBF16, false, true);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(full0 + 8 * stage, phase, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t sa = ring0 + stage * p.stage_bytes;
        const uint32_t sb = sa + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
          const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
          // B: MN-major 64-column boxes 8 KB apart (LBO), 8-row groups 1 KB apart
          mma_f16(tmem_base, ad, smem_desc_sw128(sb + kk * 16 * 128, kBoxBytes, 1024), id1, acc);
          if (n2 > 0)
            mma_f16(tmem_base + 256, ad, smem_desc_sw128(sb + 4 * kBoxBytes + kk * 16 * 128, kBoxBytes, 1024),
                    id2, acc);
        }
        mma_commit(empty0 + 8 * stage);
        if (++stage == p.stages) { stage = 0; phase ^= 1; }
      }
      mma_commit(tfull);  // also after a break: every MMA issued completes before teardown
      drain_wait(tfull, 0, 10000000ull);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ transpose, dump
    const int tid = threadIdx.x - 64;
    if (p.WgT != nullptr) {
      for (int j = rt; j < kb1 - kb0; j += p.n_rt) transpose_block(p, kb0 + j, tid, 128);
    }
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const bool got = mbar_wait(tfull, 0, p.status, abort_flag);
    if (__all_sync(0xffffffffu, got)) {
      tc_fence_after();
      const int r = 32 * q + lane;
      const int cpr = ncols / 4;
#pragma unroll 1
      for (int c0 = 0; c0 < ncols; c0 += 32) {
        float v[32];
        tmem_ld_32x32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + c0, v);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4*>(smem + dump_off(r, c0 / 4 + i, cpr)) =
              make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
  }

  tc_fence_before();
  if (S > 1) cluster_sync_all(); else __syncthreads();

  // ---------------------------------------------------------------- reduce
  // This CTA decides rows [rank R, rank R + R).  Their partial sums sit in
  // that band of every CTA's dump; the band of this CTA's own dump is read by
  // no other CTA, so the sums (ranks added in order) overwrite it there.  All
  // S loads of a chunk are issued before any is used (distributed shared
  // memory is far slower than local).
  const int R = kBM / S;
  const int cpr = ncols / 4;
  if (S > 1 && !*abort_flag) {
    uint32_t part[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) part[s] = s < S ? map_rank(ring0, s) : 0u;
    const int n_chunks = R * cpr;
#pragma unroll 2
    for (int i = threadIdx.x; i < n_chunks; i += kThreads) {
      const int r = rank * R + i / cpr;
      const uint32_t off = dump_off(r, i % cpr, cpr);
      float4 x[8];
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s < S) x[s] = ld_cluster_f4(part[s] + off);
      float4 acc = x[0];
#pragma unroll
      for (int s = 1; s < 8; ++s)
        if (s < S) {
          acc.x += x[s].x; acc.y += x[s].y; acc.z += x[s].z; acc.w += x[s].w;
        }
      *reinterpret_cast<float4*>(smem + off) = acc;
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- decide
  if (!*abort_flag) {
    for (int rr = warp; rr < R; rr += kThreads / 32) {
      const int r = rank * R + rr;
      const int t = row0 + r;
      if (t >= p.T) break;
      float lg[12];
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int c = lane + 32 * j;
        const float4 x = c < cpr ? *reinterpret_cast<const float4*>(smem + dump_off(r, c, cpr))
                                 : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        lg[4 * j] = x.x; lg[4 * j + 1] = x.y; lg[4 * j + 2] = x.z; lg[4 * j + 3] = x.w;
      }
      if (p.logits_out != nullptr) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int c = lane + 32 * j;
          if (4 * c < p.E)
            *reinterpret_cast<float4*>(p.logits_out + static_cast<long long>(t) * p.E + 4 * c) =
                make_float4(lg[4 * j], lg[4 * j + 1], lg[4 * j + 2], lg[4 * j + 3]);
        }
      }
      if (p.select) decide_row(p, t, lg, lane);
    }
  }

  if (S > 1) cluster_sync_all();  // partial rows stay readable until every CTA is done
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

struct FusedShape {
  int S, kbs, stages, stage_bytes, ring_bytes, tmem_cols, smem_bytes;
};

int pow2_at_least(int v) {
  int x = 32;
  while (x < v) x <<= 1;
  return x;
}

// Largest number of co-resident clusters of S CTAs of this kernel (cached per
// device and S).
int max_active_clusters(int S, int smem_bytes) {
  static std::mutex mu;
  static int cache[64][4][8] = {};  // [device][S][stage-size class] + 1
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int slot = S == 2 ? 0 : S == 4 ? 1 : S == 8 ? 2 : 3;
  const int cls = (smem_bytes >> 15) & 7;
  std::lock_guard<std::mutex> g(mu);
  if (cache[dev][slot][cls] != 0) return cache[dev][slot][cls] - 1;
  if (cudaFuncSetAttribute(route_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S * 64, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, route_fused_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev][slot][cls] = n + 1;
  return n;
}

FusedShape fused_shape(int T, int H, int E) {
  FusedShape f;
  const int nbx = (E + 63) / 64;
  const int nkb = H / kBK;
  const int n_rt = (T + kBM - 1) / kBM;
  f.stage_bytes = kABytes + nbx * kBoxBytes;
  f.stages = kRingMax / f.stage_bytes;
  if (f.stages > 8) f.stages = 8;
  const int dump = kBM * nbx * 64 * 4;
  f.ring_bytes = f.stages * f.stage_bytes > dump ? f.stages * f.stage_bytes : dump;
  f.tmem_cols = pow2_at_least(nbx * 64);
  f.smem_bytes = f.ring_bytes + 1024 + 256;
  f.S = 1;
  const int sms = num_sms();
  for (int cand : {8, 4, 2}) {
    if (n_rt * cand > sms || nkb < 8 * cand) continue;
    if (max_active_clusters(cand, f.smem_bytes) < n_rt) continue;
    f.S = cand;
    break;
  }
  f.kbs = (nkb + f.S - 1) / f.S;
  return f;
}

}  // namespace

bool route_fused_supported(int E, int H) {
  return E > 0 && E <= kFusedMaxE && E % 8 == 0 && H > 0 && H % kBK == 0;
}

cudaError_t launch_route_fused(const RouteFusedArgs& a, cudaStream_t s) {
  if (!route_fused_supported(a.E, a.H)) return cudaErrorNotSupported;
  if (a.T <= 0) return cudaSuccess;
  CUtensorMap mx, mw;
  if (!make_map_rows(&mx, a.X, a.T, a.H)) return cudaErrorInvalidValue;
  if (!make_map_weights(&mw, a.Wg, 1, a.H, a.E)) return cudaErrorInvalidValue;
  const FusedShape f = fused_shape(a.T, a.H, a.E);
  FusedParams p;
  p.T = a.T; p.H = a.H; p.E = a.E; p.k = a.k; p.fn = a.score_fn; p.renorm = a.renorm; p.V = a.V;
  p.select = a.select;
  p.alpha = a.alpha;
  p.S = f.S; p.kbs = f.kbs; p.nkb = a.H / kBK; p.nbx = (a.E + 63) / 64;
  p.stages = f.stages; p.stage_bytes = f.stage_bytes; p.ring_bytes = f.ring_bytes;
  p.tmem_cols = f.tmem_cols;
  p.n_rt = (a.T + kBM - 1) / kBM;
  p.Wg = a.Wg; p.bias = a.bias; p.token_ids = a.token_ids; p.tid2eid = a.tid2eid;
  p.E_ids = a.E_ids; p.G = a.G; p.logits_out = a.logits_out; p.WgT = a.WgT;
  p.rs = a.rs;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(route_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       f.smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_rt * f.S, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(f.smem_bytes);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = f.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = f.S > 1 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, route_fused_kernel, mx, mw, p);
  if (e != cudaSuccess) return e;
  if (a.select && a.token_ids == nullptr)
    return launch_route_recheck(a.X, a.WgT, a.bias, a.H, a.score_fn, a.k, a.alpha, a.renorm, a.E_ids,
                                a.G, a.rs, s);
  return cudaSuccess;
}

}  // namespace moe
