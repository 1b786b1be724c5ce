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
//   warps 6-15  fetch the selection bias (or the hash table rows) into
//               shared memory, then run the decision once on stand-in rows so
//               that its code is cached.
//   all warps   after the cluster barrier: sum the S partial rows of this
//               CTA's band (ranks 0..S-1 in order); then one warp per row (two
//               side by side) scores them, adds the selection bias, keeps each
//               lane's best three keys and takes k+1 warp arg-max rounds
//               (larger score first, equal scores to the lower id), writes ids
//               and gates, and lists a token whose first k+1 scores hold a
//               pair closer than the decision band, with its candidates, in
//               the CTA's segment of the list for the float64 re-decision
//               (moe_route.cu), which runs as this kernel's programmatic
//               dependent.
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_route.cuh"

namespace moe {

namespace {

constexpr int kThreads = 512;  // 16 warps: the decision has one warp per row
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

// Order-preserving 32-bit key of a float: larger float, larger key.
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// fp32 logit of column e of dump row `row`.
__device__ __forceinline__ float dump_logit(const uint8_t* smem, int row, int e, int cpr) {
  return *reinterpret_cast<const float*>(smem + dump_off(row, e >> 2, cpr) + 4 * (e & 3));
}

// Selection key of column e: the score plus the selection bias b (when the
// layer has one) as an order-preserving integer, its low 9 bits replaced by
// 511 - e.  Keys are then unique, a larger key is a larger score or, among
// scores equal to 2^-14 relative, the lower id, and the id comes back from
// the key.  0 (below every key) past the last expert.  Scores that close
// are far inside the decision band, so their order is settled by the float64
// re-decision: the closeness test takes the winners' full fp32 scores.
__device__ __forceinline__ uint32_t sel_key(float l, float b, bool has_bias, int e, int E, int fn) {
  if (e >= E) return 0u;
  const float v = score_f32(l, fn);
  return (fkey(has_bias ? v + b : v) & 0xFFFFFE00u) | static_cast<uint32_t>(511 - e);
}
__device__ __forceinline__ int key_id(uint32_t k) { return 511 - static_cast<int>(k & 511u); }

// A lane's best three keys, best first: a sorting network of integer
// min/max, no branches.
struct Top3 {
  uint32_t k0, k1, k2;
  __device__ __forceinline__ void clear() { k0 = k1 = k2 = 0u; }
  __device__ __forceinline__ void offer(uint32_t k) {
    const uint32_t x = min(k0, k);
    k0 = max(k0, k);
    const uint32_t y = min(k1, x);
    k1 = max(k1, x);
    k2 = max(k2, y);
  }
  __device__ __forceinline__ void pop() {
    k0 = k1;
    k1 = k2;
    k2 = 0u;
  }
};

// The routing decision of NR tokens from their fp32 logits (rows `row` of
// the reduced dump), one warp.  Lane l owns the columns of chunks l, l + 32,
// ... (columns 4c .. 4c + 3); it scores them once and keeps its best three
// keys.  Each arg-max round is then one single-instruction warp reduction
// over the lanes' best keys; the winning lane drops its key and, once its
// three are gone, rescans its columns for the keys below it.  The NR rows are decided side by side, so their dependency
// chains overlap.  bias_s: the selection bias in shared memory (or null);
// ids_s[r]: in hash mode row r's k table entries, prefetched into shared
// memory, then a 1 for a token id outside [0, V) (flagged there).  Rows with
// valid[r] false are stand-ins (computed, neither listed nor written).
template <int NCH, int NR>
__device__ __forceinline__ void decide_rows(const FusedParams& p, const uint8_t* smem, int cpr,
                                            const int (&row)[NR], const int (&t)[NR],
                                            const bool (&valid)[NR], const float* bias_s,
                                            const int* const (&ids_s)[NR], int* stage_n, int4* stage_f,
                                            float2* stage_n2, int band_t0, int* out_ids, float* out_g,
                                            int lane) {
  const int E = p.E, k = p.k, fn = p.fn;
  float lmax[NR], zsum[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    lmax[r] = 0.0f;
    zsum[r] = 1.0f;
  }
  if (fn == 2) {
    float m[NR], z[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) m[r] = -FLT_MAX;
#pragma unroll 1
    for (int j = 0; j < NCH; ++j) {
      const int c = lane + 32 * j;
      if (c >= cpr) break;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(smem + dump_off(row[r], c, cpr));
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (4 * c + q < E) m[r] = fmaxf(m[r], xs[q]);
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      lmax[r] = warp_max(m[r]);
      z[r] = 0.0f;
    }
#pragma unroll 1
    for (int j = 0; j < NCH; ++j) {
      const int c = lane + 32 * j;
      if (c >= cpr) break;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(smem + dump_off(row[r], c, cpr));
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (4 * c + q < E) z[r] += __expf(xs[q] - lmax[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) zsum[r] = warp_sum(z[r]);
  }
  int my_sel[NR];    // lane j < k: the j-th id
  float my_l[NR];    // and its logit
  bool tok_ok[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    my_sel[r] = -1;
    my_l[r] = 0.0f;
    tok_ok[r] = true;
  }
  if (p.token_ids != nullptr) {
    // ---------------------------------------------------------------- hash
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      tok_ok[r] = ids_s[r][kMaxK] == 0;
      if (lane < k) {
        const int e = ids_s[r][lane];
        my_sel[r] = e;
        if (e >= 0 && e < E) my_l[r] = dump_logit(smem, row[r], e, cpr);
      }
    }
  } else {
    // ---------------------------------------------------------------- top-k
    Top3 tl[NR];
    int left[NR];  // this lane's columns not yet taken
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      tl[r].clear();
      left[r] = 0;
    }
    const bool hb = bias_s != nullptr;
#pragma unroll 1
    for (int j = 0; j < NCH; ++j) {
      const int c = lane + 32 * j;
      if (c >= cpr) break;
      const float4 b4 = hb ? *reinterpret_cast<const float4*>(bias_s + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float bs[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(smem + dump_off(row[r], c, cpr));
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) tl[r].offer(sel_key(xs[q], bs[q], hb, 4 * c + q, E, fn));
        left[r] += max(0, min(4, E - 4 * c));
      }
    }
    const int rounds = (k < E) ? k + 1 : k;
    int wid[NR];  // lane j < rounds: the j-th winner
#pragma unroll
    for (int r = 0; r < NR; ++r) wid[r] = E;
#pragma unroll 1
    for (int rd = 0; rd < rounds; ++rd) {
      uint32_t m[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) m[r] = __reduce_max_sync(0xffffffffu, tl[r].k0);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (tl[r].k0 == m[r]) {  // the owner of the winning column
          tl[r].pop();
          --left[r];
          if (tl[r].k0 == 0u && left[r] > 0) {
            // refill: the lane's best three among its keys below m
#pragma unroll 1
            for (int j = 0; j < NCH; ++j) {
              const int c = lane + 32 * j;
              if (c >= cpr) break;
              const float4 x = *reinterpret_cast<const float4*>(smem + dump_off(row[r], c, cpr));
              const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int e = 4 * c + q;
                const uint32_t key = sel_key(xs[q], hb ? bias_s[e] : 0.0f, hb, e, E, fn);
                if (key < m[r]) tl[r].offer(key);
              }
            }
          }
        }
        if (lane == rd) wid[r] = key_id(m[r]);
      }
    }
    // the winners' full fp32 scores, one per lane: a pair of consecutive
    // winners closer than the band (or out of order: keys tie scores within
    // 2^-14) lists the token for the re-decision
    bool close[NR];
    float kth[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float ev = 0.0f;
      if (lane < rounds && wid[r] < E) {
        const float l = dump_logit(smem, row[r], wid[r], cpr);
        const float v = score_f32(l, fn);
        ev = hb ? v + bias_s[wid[r]] : v;
        if (lane < k) {
          my_sel[r] = wid[r];
          my_l[r] = l;
        }
      }
      const float pv = __shfl_up_sync(0xffffffffu, ev, 1);
      close[r] = __any_sync(0xffffffffu, lane >= 1 && lane < rounds && (pv - ev) < band_at(pv, fn));
      kth[r] = __shfl_sync(0xffffffffu, ev, k - 1);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      if (!close[r] || !valid[r]) continue;  // warp-uniform
      // candidates: every expert within twice the band below the k-th score;
      // the token's go to its own slots [t E, t E + count) of the pair
      // lists, and the token to the CTA's staging list, which the CTA
      // writes out as its segment of the re-decision list at the end
      const float lim = kth[r] - 2.0f * band_at(kth[r], fn);
      int base = t[r] * E;
      const int base0 = base;
#pragma unroll 1
      for (int j = 0; j < NCH; ++j) {
        const int c = lane + 32 * j;
        float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (c < cpr) x = *reinterpret_cast<const float4*>(smem + dump_off(row[r], c, cpr));
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = 4 * c + q;
          bool cand = false;
          if (c < cpr && e < E) {
            const float v = score_f32(xs[q], fn);
            cand = (bias_s != nullptr ? v + bias_s[e] : v) >= lim;
          }
          const unsigned bm = __ballot_sync(0xffffffffu, cand);
          if (cand) {
            const int at = base + __popc(bm & ((1u << lane) - 1u));
            if (in_bounds(at, static_cast<long long>(p.T) * E)) {
              p.rs.pairs[at] = make_int2(t[r], e);
              p.rs.plogit[at] = xs[q];
            }
          }
          base += __popc(bm);
        }
      }
      if (lane == 0) {
        const int fi = atomicAdd(stage_n, 1);
        stage_f[fi] = make_int4(t[r], base0, base - base0, 0);
        stage_n2[fi] = make_float2(lmax[r], zsum[r]);
      }
    }
  }
  // gates (a close token's ids and gates are rewritten by the re-decision)
  float a[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    a[r] = 0.0f;
    if (lane < k) {
      if (my_sel[r] >= 0 && my_sel[r] < E) {
        a[r] = affinity_f32(my_l[r], fn, lmax[r], zsum[r]);
      } else if (tok_ok[r] && valid[r]) {
        set_flag(p.status, kFlagBadExpert);  // a table entry outside [0, E)
      }
    }
  }
  float den[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) den[r] = warp_sum(a[r]);  // lanes >= k hold 0
#pragma unroll
  for (int r = 0; r < NR; ++r)
    if (lane < k && valid[r]) {
      float g = p.alpha * a[r];
      if (p.renorm) g = den[r] > 0.0f ? p.alpha * a[r] / den[r] : 0.0f;
      // into the band's staging rows, written out whole after the decisions
      const int rb = t[r] - band_t0;
      out_ids[rb * k + lane] = my_sel[r];
      out_g[rb * k + lane] = g;
    }
}

// Rows [rank R, rank R + R) of the tile, NR per warp at a time: their logits
// from this CTA's (reduced) dump, optionally written out, then decided.  A
// dry pass decides one group of stand-in rows (all invalid: nothing is
// written or listed) on whatever the shared memory holds, only so that the
// code is in the instruction caches when the real pass comes.
template <int NCH, int NR>
__device__ __forceinline__ void decide_band(const FusedParams& p, const uint8_t* smem, int rank,
                                            int R, int row0, int cpr, const float* bias_s,
                                            const int* ids_base, int* stage_n, int4* stage_f,
                                            float2* stage_n2, int* out_ids, float* out_g, int warp,
                                            int lane, bool dry) {
  constexpr int NW = kThreads / 32;
  for (int rr0 = warp; rr0 < R; rr0 += NR * NW) {
    int row[NR], t[NR];
    bool valid[NR];
    const int* ids[NR];
    int nvalid = 0;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      int rr = rr0 + r * NW;
      valid[r] = !dry && rr < R && row0 + rank * R + rr < p.T;
      nvalid += valid[r] ? 1 : 0;
      if (!valid[r]) rr = rr0;  // a stand-in row
      row[r] = rank * R + rr;
      t[r] = row0 + row[r];
      ids[r] = ids_base + rr * (kMaxK + 1);
    }
    if (nvalid == 0 && !dry) break;
    if (p.logits_out != nullptr) {
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll 1
        for (int c = lane; c < cpr; c += 32)
          if (valid[r] && 4 * c < p.E)
            *reinterpret_cast<float4*>(p.logits_out + static_cast<long long>(t[r]) * p.E + 4 * c) =
                *reinterpret_cast<const float4*>(smem + dump_off(row[r], c, cpr));
    }
    if (p.select)
      decide_rows<NCH, NR>(p, smem, cpr, row, t, valid, bias_s, ids, stage_n, stage_f, stage_n2,
                           row0 + rank * R, out_ids, out_g, lane);
    if (dry) break;
  }
}

// Sum of the S partial dumps over this CTA's band of rows [rank R, rank R + R)
// (R = 128 / S), written over the band in this CTA's own dump, which no other
// CTA reads.  Ranks are added in order.  Each thread issues the loads of U
// chunks (all S partials of each) before using any (distributed shared memory
// is slow to answer); U S <= 8 keeps them within 32 registers.
template <int S>
__device__ __forceinline__ void reduce_band(uint8_t* smem, uint32_t ring0, int rank, int cpr) {
  constexpr int R = kBM / S;
  constexpr int U = S >= 8 ? 1 : S == 4 ? 2 : 3;
  uint32_t part[S];
#pragma unroll
  for (int s = 0; s < S; ++s) part[s] = map_rank(ring0, s);
  const int n_chunks = R * cpr;
  for (int i0 = threadIdx.x; i0 < n_chunks; i0 += U * kThreads) {
    float4 x[U][S];
    uint32_t off[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kThreads;
      off[u] = i < n_chunks ? dump_off(rank * R + i / cpr, i % cpr, cpr) : 0u;
      if (i < n_chunks) {
#pragma unroll
        for (int s = 0; s < S; ++s) x[u][s] = ld_cluster_f4(part[s] + off[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i0 + u * kThreads < n_chunks) {
        float4 acc = x[u][0];
#pragma unroll
        for (int s = 1; s < S; ++s) {
          acc.x += x[u][s].x; acc.y += x[u][s].y; acc.z += x[u][s].z; acc.w += x[u][s].w;
        }
        *reinterpret_cast<float4*>(smem + off[u]) = acc;
      }
    }
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
  // side tables for the decision: the selection bias [E] and, in hash mode,
  // each decided row's table entries [R][kMaxK + 1] (the last: 1 for a token
  // id outside [0, V))
  float* bias_s = reinterpret_cast<float*>(bar_area + 256);
  int* ids_s = reinterpret_cast<int*>(bar_area + 256 + kFusedMaxE * 4);
  // the CTA's close tokens, appended to the global list at the end
  int4* stage_f = reinterpret_cast<int4*>(bar_area + 256 + kFusedMaxE * 4 + kBM * (kMaxK + 1) * 4);
  float2* stage_n2 = reinterpret_cast<float2*>(stage_f + kBM);
  int* stage_n = reinterpret_cast<int*>(tmem_slot + 2);
  // the band's ids and gates, written out with whole-sector stores at the end
  int* out_ids = reinterpret_cast<int*>(stage_n2 + kBM);
  float* out_g = reinterpret_cast<float*>(out_ids + kBM * kMaxK);

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
    *stage_n = 0;
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
  } else if (warp >= 6) {
    // ------------------------------------------------------------ side tables
    // idle until the decision: fetch what it reads from global memory
    const int tid = threadIdx.x - 6 * 32, nt = kThreads - 6 * 32;
    if (p.select && p.bias != nullptr)
      for (int e = tid; e < p.E; e += nt) bias_s[e] = __ldg(p.bias + e);
    if (p.select && p.token_ids != nullptr) {
      const int R = kBM / S;
      for (int rr = tid; rr < R; rr += nt) {
        const int t = row0 + rank * R + rr;
        int* row = ids_s + rr * (kMaxK + 1);
        if (t >= p.T) continue;
        const int tok = __ldg(p.token_ids + t);
        const bool ok = tok >= 0 && tok < p.V;
        if (!ok) set_flag(p.status, kFlagBadToken);
        for (int j = 0; j < p.k; ++j)
          row[j] = ok ? __ldg(p.tid2eid + static_cast<long long>(tok) * p.k + j) : -1;
        row[kMaxK] = ok ? 0 : 1;
      }
    }
  } else {
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

  // Warps 6-15 (idle until now) first run the decision once on stand-in
  // rows (the dry pass: it writes nothing), so that its instructions are
  // cached when every warp runs it for real, after the reduction.  Only
  // where the main loop is long enough to hide it (8 k-blocks or more).
  const int R = kBM / S;
  const int cpr = ncols / 4;
  const float* bs = p.bias != nullptr ? bias_s : nullptr;
#pragma unroll 1
  for (int pass = (warp >= 6 && p.select && kb1 - kb0 >= 8) ? 0 : 1; pass < 2; ++pass) {
    if (pass == 1) {
      tc_fence_before();
      if (S > 1) cluster_sync_all(); else __syncthreads();

      // ------------------------------------------------------------ reduce
      // This CTA decides rows [rank R, rank R + R).  Their partial sums sit
      // in that band of every CTA's dump; the band of this CTA's own dump is
      // read by no other CTA, so the sums (ranks added in order) overwrite
      // it there.  All S loads of a chunk are issued before any is used
      // (distributed shared memory is far slower than local).
      if (S > 1 && !*abort_flag) {
        if (S == 2) reduce_band<2>(smem, ring0, rank, cpr);
        else if (S == 4) reduce_band<4>(smem, ring0, rank, cpr);
        else reduce_band<8>(smem, ring0, rank, cpr);
      }
      __syncthreads();
    }

    // -------------------------------------------------------------- decide
    if (!*abort_flag) {
      const bool dry = pass == 0;
      if (cpr <= 32)
        decide_band<1, 2>(p, smem, rank, R, row0, cpr, bs, ids_s, stage_n, stage_f, stage_n2, out_ids, out_g,
                         warp, lane, dry);
      else if (cpr <= 64)
        decide_band<2, 2>(p, smem, rank, R, row0, cpr, bs, ids_s, stage_n, stage_f, stage_n2, out_ids, out_g,
                         warp, lane, dry);
      else
        decide_band<3, 2>(p, smem, rank, R, row0, cpr, bs, ids_s, stage_n, stage_f, stage_n2, out_ids, out_g,
                         warp, lane, dry);
    }
  }

  __syncthreads();
  if (p.select && !*abort_flag) {
    // the band's ids and gates, and (top-k) its close tokens: this CTA's
    // segment of the re-decision list, flagged[b R ..) with b = blockIdx.x
    // (the band starts at token b R), and its length
    const int t0 = row0 + rank * R;
    const int n_out = (min(p.T, t0 + R) - t0) * p.k;
    for (int i = threadIdx.x; i < n_out; i += kThreads) {
      p.E_ids[static_cast<long long>(t0) * p.k + i] = out_ids[i];
      p.G[static_cast<long long>(t0) * p.k + i] = out_g[i];
    }
    if (p.token_ids == nullptr) {
      const int nf = *stage_n;
      for (int i = threadIdx.x; i < nf; i += kThreads) {
        if (!in_bounds(t0 + i, p.T)) continue;
        p.rs.flagged[t0 + i] = stage_f[i];
        p.rs.fnorm[t0 + i] = stage_n2[i];
      }
      if (threadIdx.x == 0) p.rs.seg_n[blockIdx.x] = nf;
    }
  } else if (p.select && p.token_ids == nullptr && threadIdx.x == 0) {
    p.rs.seg_n[blockIdx.x] = 0;
  }
  // the re-decision may launch now (it waits for this grid's writes)
  asm volatile("griddepcontrol.launch_dependents;");
  // partial rows stay readable until every CTA of the cluster is done with
  // them: their loads have all returned by the time a CTA arrives here, so
  // the arrival needs no memory ordering
  if (S > 1) asm volatile("barrier.cluster.arrive.relaxed;\n\tbarrier.cluster.wait;" ::: "memory");
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
  f.smem_bytes = f.ring_bytes + 1024 + 256 + kFusedMaxE * 4 + kBM * (kMaxK + 1) * 4 +
                 kBM * (sizeof(int4) + sizeof(float2)) + 2 * kBM * kMaxK * 4;
  f.S = 1;
  const int sms = num_sms();
  // the largest S whose clusters are all co-resident in one wave and whose
  // ranks all get k-blocks; the decision's rows are split S ways as well, so
  // small layers take clusters too
  for (int cand : {8, 4, 2}) {
    const int per = (nkb + cand - 1) / cand;
    if (n_rt * cand > sms || cand > nkb || (cand - 1) * per >= nkb) continue;
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
    return launch_route_recheck(a.X, a.WgT, a.bias, a.T, a.H, a.E, a.score_fn, a.k, a.alpha, a.renorm,
                                a.E_ids, a.G, a.rs, a.rs.seg_n, p.n_rt * f.S, kBM / f.S, false, true, s);
  return cudaSuccess;
}

MOE_DEFINE_BOUNDS_TAKE(route_fused)

}  // namespace moe
