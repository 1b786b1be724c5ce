// Router selection over fp32 logits (the general path, for layers whose
// experts do not fit the fused router of moe_route_fused.cu), and the
// float64 re-decision of close tokens that both paths share.
//
// "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例", section 路由与负载 / 路由张量:
//   a = score(l);  I_t = TopK(a + beta);  g = alpha * a / sum_{I_t} a
// (beta selects only; the weights use the raw affinity).  The softmax gate of
// "Megatron 分布式训练全维度并行技术文档" (section 4.2) selects the top-k of
// softmax(l), which is the top-k of l itself.  Section 路由与负载 / Hash 路由:
// the ids are a table row of the token id, the gate formula is unchanged.
//
// Exact ids from inexact logits.  The fp32 tensor-core logit is within a few
// 1e-5 of the exact value, so the fp32 selection is final unless two
// neighbouring scores among the first k+1 lie within a decision band.  Such a
// token is re-decided in two steps:
//   select    fp32 top-(k+1) by k+1 warp arg-max rounds; a close token appends
//             every expert scoring within twice the band of its k-th score to
//             a list of (token, expert) pairs, with the pair's fp32 logit (and
//             the token's softmax normaliser);
//   redecide  one block per close token: the candidates within a band of
//             another get their logit sum_h X[t,h] Wg[h,e] recomputed to ~48
//             bits over a transposed copy of Wg (contiguous rows; each bf16
//             product is exact in fp32 and the sum is carried as float pairs),
//             each candidate's row split over the block's warps, and a float64
//             selection score; the others keep their fp32 score; the ranks of
//             the scores (larger first, equal scores to the lower id) give the
//             k ids in order, with gates from the listed fp32 logits.  The list
//             comes in segments (one per CTA of the fused router, one for the
//             general path, whose counters the last block zeroes for the next
//             call).
// The ids then equal those of an exact evaluation except at exact ties.
#include <float.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_route.cuh"

namespace moe {

constexpr int kWarps = 8;  // tokens (or pairs) per 256-thread block
// Softmax normaliser of one token's logits: max and sum of exp(l - max).
__device__ __forceinline__ void softmax_norm(const float* lrow, int E, int lane, float& lmax,
                                             float& zsum) {
  lmax = -FLT_MAX;
  for (int e = lane; e < E; e += 32) lmax = fmaxf(lmax, lrow[e]);
  lmax = warp_max(lmax);
  zsum = 0.0f;
  for (int e = lane; e < E; e += 32) zsum += expf(lrow[e] - lmax);
  zsum = warp_sum(zsum);
}

// The whole warp writes ids and gates of one token from the fp32 logits:
// lane j < k loads its own logit, the warp sums the affinities.
__device__ __forceinline__ void write_gates(const float* lrow, int E, int k, int fn, float alpha,
                                            int renorm, int my_sel, bool tok_ok, float lmax,
                                            float zsum, int lane, int32_t* ids, float* G,
                                            int* status) {
  float a = 0.0f;
  const bool mine = lane < k;
  if (mine) {
    if (my_sel >= 0 && my_sel < E) {
      const float l = lrow[my_sel];
      a = (fn == 2) ? expf(l - lmax) / zsum : score_f32(l, fn);
    } else if (tok_ok) {
      set_flag(status, kFlagBadExpert);  // a table entry outside [0, E)
    }
  }
  // sum over j < k in j order (lanes beyond k hold 0)
  float den = 0.0f;
  for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, a, j);
  if (mine) {
    float g = alpha * a;
    if (renorm) g = den > 0.0f ? alpha * a / den : 0.0f;
    ids[lane] = my_sel;
    G[lane] = g;
  }
}

// Lane j of the warp receives sel[j] (k <= 16 <= 32).
__device__ __forceinline__ int lane_sel(const int* sel, int k, int lane) {
  int v = -1;
#pragma unroll 1
  for (int j = 0; j < k; ++j) v = (lane == j) ? sel[j] : v;
  return v;
}

__global__ void __launch_bounds__(kWarps * 32)
    route_select_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                        const int32_t* __restrict__ token_ids, const int32_t* __restrict__ tid2eid,
                        int V, int T, int E, int k, int fn, float alpha, int renorm,
                        int32_t* __restrict__ E_ids, float* __restrict__ G, RouteScratch rs,
                        int* status) {
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + warp;
  if (t >= T) return;
  float* s = sh + warp * E;  // selection scores of this token
  const float* lrow = logits + static_cast<long long>(t) * E;

  float lmax = 0.0f, zsum = 1.0f;
  if (fn == 2) softmax_norm(lrow, E, lane, lmax, zsum);

  int sel[kMaxK];
  bool tok_ok = true;
  if (token_ids != nullptr) {
    // ---------------------------------------------------------------- hash
    const int tok = token_ids[t];
    tok_ok = tok >= 0 && tok < V;
    if (!tok_ok && lane == 0) set_flag(status, kFlagBadToken);
#pragma unroll 1
    for (int j = 0; j < k; ++j) sel[j] = tok_ok ? tid2eid[static_cast<long long>(tok) * k + j] : -1;
  } else {
    // ---------------------------------------------------------------- top-k
#pragma unroll 8
    for (int e = lane; e < E; e += 32) {
      float v = score_f32(__ldg(lrow + e), fn);
      if (bias != nullptr) v += __ldg(bias + e);
      s[e] = v;
    }
    __syncwarp();
    const int rounds = (k < E) ? k + 1 : k;
    float top[kMaxK + 1];
#pragma unroll 1
    for (int r = 0; r < rounds; ++r) {
      float best = -FLT_MAX;
      int bid = 0x7fffffff;
      for (int e = lane; e < E; e += 32) {
        const float v = s[e];
        if (before(v, e, best, bid)) { best = v; bid = e; }
      }
      warp_argmax(best, bid);
      top[r] = best;
      if (r < k) sel[r] = bid;
      if (lane == 0 && in_bounds(bid, E)) s[bid] = -FLT_MAX;  // taken
      __syncwarp();
    }
    bool close = false;
#pragma unroll 1
    for (int r = 0; r + 1 < rounds; ++r) close |= (top[r] - top[r + 1]) < band_at(top[r], fn);
    if (close) {
      // candidates: every expert within twice the band below the k-th score
      // (the k winners among them); restore the scores and list the pairs.
      for (int e = lane; e < E; e += 32) {
        float v = score_f32(lrow[e], fn);
        if (bias != nullptr) v += bias[e];
        s[e] = v;
      }
      __syncwarp();
      const float kth = top[k - 1];
      const float lim = kth - 2.0f * band_at(kth, fn);
      int count = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        count += __popc(__ballot_sync(0xffffffffu, e < E && s[e] >= lim));
      }
      int base = 0;
      if (lane == 0) {
        base = atomicAdd(rs.counters + 1, count);
        const int fi = atomicAdd(rs.counters + 0, 1);
        if (in_bounds(fi, T)) {
          rs.flagged[fi] = make_int4(t, base, count, 0);
          rs.fnorm[fi] = make_float2(lmax, zsum);
        }
      }
      base = __shfl_sync(0xffffffffu, base, 0);
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool cand = e < E && s[e] >= lim;
        const unsigned m = __ballot_sync(0xffffffffu, cand);
        if (cand) {
          const int at = base + __popc(m & ((1u << lane) - 1u));
          if (in_bounds(at, static_cast<long long>(T) * E)) {
            rs.pairs[at] = make_int2(t, e);
            rs.plogit[at] = lrow[e];
          }
        }
        base += __popc(m);
      }
    }
  }
  // fp32 decision (a close token's ids and gates are rewritten by reselect)
  write_gates(lrow, E, k, fn, alpha, renorm, lane_sel(sel, k, lane), tok_ok, lmax, zsum, lane,
              E_ids + static_cast<long long>(t) * k, G + static_cast<long long>(t) * k, status);
}

// Error-free sum of two floats (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// (H, L) += (h, l) for unevaluated float pairs: TwoSum of the high parts,
// the low parts added to the error, renormalised (Fast2Sum).
__device__ __forceinline__ void ff_add(float& H, float& L, float h, float l) {
  float s, e;
  two_sum(H, h, s, e);
  e += L + l;
  H = s + e;
  L = e - (H - s);
}

// Order-preserving 64-bit key of a double: larger double, larger key.
__device__ __forceinline__ unsigned long long order_key(double v) {
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(v));
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

constexpr int kRedecideWarps = 16;
constexpr int kRedecideList = 512;  // candidates a token's shared lists hold
constexpr int kRedecideBatch = 14;  // 16-byte loads of Wg^T in flight per lane

// Sum over the 16-byte vectors [v_begin, v_end) of the token row xs (shared
// memory) and Wg^T row e of the bf16 x bf16 products, one warp: each product
// is exact in fp32; the products are summed as unevaluated float pairs
// (hi, lo) with TwoSum on the fp32 pipes (GB300's fp64 rate is low), eight
// pairs per lane, folded as float pairs across the lanes in a fixed order.
// Returns the pair (H, L) in every lane.
__device__ __forceinline__ float2 pair_dot(const uint4* __restrict__ xs, const uint16_t* __restrict__ WgT,
                                           int H, int e, int v_begin, int v_end, int lane) {
  const uint4* wr = reinterpret_cast<const uint4*>(WgT + static_cast<long long>(e) * H);
  float hi[8], lo[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) hi[q] = lo[q] = 0.0f;
  for (int v0 = v_begin + lane; v0 < v_end; v0 += kRedecideBatch * 32) {
    uint4 b[kRedecideBatch];
#pragma unroll
    for (int u = 0; u < kRedecideBatch; ++u) {  // all loads of this round first
      const int v = v0 + u * 32;
      b[u] = v < v_end ? __ldg(wr + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kRedecideBatch; ++u) {
      const int v = v0 + u * 32;
      const uint4 a = v < v_end ? xs[v] : make_uint4(0, 0, 0, 0);
      const float p[8] = {bf16_lo(a.x) * bf16_lo(b[u].x), bf16_hi(a.x) * bf16_hi(b[u].x),
                          bf16_lo(a.y) * bf16_lo(b[u].y), bf16_hi(a.y) * bf16_hi(b[u].y),
                          bf16_lo(a.z) * bf16_lo(b[u].z), bf16_hi(a.z) * bf16_hi(b[u].z),
                          bf16_lo(a.w) * bf16_lo(b[u].w), bf16_hi(a.w) * bf16_hi(b[u].w)};
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float sum, err;
        two_sum(hi[q], p[q], sum, err);
        hi[q] = sum;
        lo[q] += err;
      }
    }
  }
  float H0 = hi[0], L0 = lo[0];
#pragma unroll
  for (int q = 1; q < 8; ++q) ff_add(H0, L0, hi[q], lo[q]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    ff_add(H0, L0, __shfl_xor_sync(0xffffffffu, H0, o), __shfl_xor_sync(0xffffffffu, L0, o));
  return make_float2(H0, L0);
}

// Re-decide the close tokens: one block per listed token.  The list is n_seg
// segments (launch_route_recheck); block b takes entries j = b, b +
// gridDim.x, ... of the order "entry j / n_seg of segment j mod n_seg".  The
// token's row of X and its candidates (ids, listed fp32 logits, fp32 scores)
// go to shared memory.  A candidate at least a band away from every other
// candidate has a certain place in the order, and its fp32 score is its key;
// the others are scored in float64 (each candidate's row split over the warps
// the group of candidates leaves, the float-pair partial sums added in a
// fixed order).  The k candidates of rank below k (larger key first, equal
// keys lower id first) are the selection, in rank order, with gates from
// their listed fp32 logits (and, for softmax, the token's listed
// normaliser).  A list longer than the shared arrays keeps its keys in
// memory and is taken in k arg-max rounds.  With zero_counters, the last
// block to finish zeroes the general path's list counters for the next call.
__global__ void __launch_bounds__(kRedecideWarps * 32)
    route_redecide_kernel(const uint16_t* __restrict__ X, const uint16_t* __restrict__ WgT,
                          const float* __restrict__ bias, int H, int k, int fn, float alpha, int renorm,
                          int32_t* __restrict__ E_ids, float* __restrict__ G, RouteScratch rs,
                          const int* seg_n, int n_seg, int seg_len, int zero_counters, int T, int E) {
  // launched as the fused router's programmatic dependent: its writes are
  // visible from here on (a no-op after an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint4 xs[];  // [H / 8], then the partial sums, the exact list, the segment counts
  float2* part = reinterpret_cast<float2*>(xs + H / 8);             // [kRedecideWarps]
  int* exact = reinterpret_cast<int*>(part + kRedecideWarps);       // [kRedecideList]
  int* cnt_s = exact + kRedecideList;                               // [n_seg]
  __shared__ float sc[kRedecideList];
  __shared__ float pl_s[kRedecideList];
  __shared__ int n_exact, n_total;
  __shared__ int wsum_s[kRedecideWarps];
  __shared__ unsigned long long key_s[kRedecideList];
  __shared__ int id_s[kRedecideList];
  __shared__ int sel_s[kMaxK];
  __shared__ float aff_s[kMaxK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int vecs = H / 8;
  // exclusive prefix of the segment counts (in place): entry j of the
  // list is entry j - pre[b] of segment b, the last b with pre[b] <= j
  {
    const int per = (n_seg + blockDim.x - 1) / blockDim.x;
    const int lo = min(n_seg, static_cast<int>(threadIdx.x) * per), hi = min(n_seg, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) {
      cnt_s[i] = reinterpret_cast<const volatile int*>(seg_n)[i];
      sum += cnt_s[i];
    }
    int incl = sum;  // inclusive scan over the threads: warps, then warp totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum_s[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kRedecideWarps ? wsum_s[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += v;
      }
      if (lane < kRedecideWarps) wsum_s[lane] = w;  // inclusive
    }
    __syncthreads();
    int run = incl - sum + (warp > 0 ? wsum_s[warp - 1] : 0);
    for (int i = lo; i < hi; ++i) {
      const int c = cnt_s[i];
      cnt_s[i] = run;
      run += c;
    }
    if (threadIdx.x == 0) n_total = wsum_s[kRedecideWarps - 1];
    __syncthreads();
  }
  for (int j = blockIdx.x; j < n_total; j += gridDim.x) {
    int seg = 0;
    for (int span = n_seg; span > 1;) {  // the last segment starting at or before j
      const int half = span >> 1;
      if (cnt_s[seg + half] <= j) seg += half;
      span -= half;
    }
    const int idx = j - cnt_s[seg];
    const int4 f = rs.flagged[static_cast<long long>(seg) * seg_len + idx];
    const int t = f.x, base = f.y, count = f.z;
    const long long n_pairs = static_cast<long long>(T) * E;
    if (!in_bounds(t, T) || !in_bounds(base, n_pairs) || !in_bounds(base + count - 1, n_pairs))
      continue;  // block-uniform
    const bool small = count <= kRedecideList;
    // the token row and the candidates, their loads issued together
    const uint4* xr = reinterpret_cast<const uint4*>(X + static_cast<long long>(t) * H);
    for (int v = threadIdx.x; v < vecs; v += blockDim.x) xs[v] = __ldg(xr + v);
    for (int i = threadIdx.x; small && i < count; i += blockDim.x) {
      int e = rs.pairs[base + i].y;
      if (!in_bounds(e, E)) e = 0;
      const float l = rs.plogit[base + i];
      float v = score_f32(l, fn);
      if (bias != nullptr) v += bias[e];
      id_s[i] = e;
      pl_s[i] = l;
      sc[i] = v;
    }
    __syncthreads();
    if (small) {
      // the fp32 selection score of each candidate, as the first decision
      // took it: only candidates within a band of another are recomputed
      for (int i = threadIdx.x; i < count; i += blockDim.x) {
        bool near = false;
        for (int q = 0; q < count && !near; ++q)
          near = q != i && fabsf(sc[i] - sc[q]) < band_at(fmaxf(sc[i], sc[q]), fn);
        exact[i] = near ? 1 : 0;
        if (!near) key_s[i] = order_key(static_cast<double>(sc[i]));
      }
      __syncthreads();
      if (warp == 0) {  // the recomputed candidates' list, in candidate order
        int m = 0;
        for (int c = 0; c < count; c += 32) {
          const bool near = c + lane < count && exact[c + lane] != 0;
          const unsigned b = __ballot_sync(0xffffffffu, near);
          __syncwarp();
          if (near) exact[m + __popc(b & ((1u << lane) - 1u))] = c + lane;
          m += __popc(b);
        }
        if (lane == 0) n_exact = m;
      }
      __syncthreads();
    }
    const int ne = small ? n_exact : count;
    auto exact_at = [&](int c) { return small ? exact[c] : c; };
    // exact candidates in groups of g = min(ne, warps); the warps of a group's
    // candidate split the row (ns parts), their float pairs added in order
    for (int c0 = 0; c0 < ne; c0 += kRedecideWarps) {
      const int g = min(ne - c0, kRedecideWarps);
      const int ns = kRedecideWarps / g;
      const int c = warp % g, part_i = warp / g;
      if (part_i < ns) {
        const int len = (vecs + ns - 1) / ns;
        const int vb = part_i * len, ve = min(vecs, vb + len);
        const int ci = exact_at(c0 + c);
        int ce = small ? id_s[ci] : rs.pairs[base + ci].y;
        if (!in_bounds(ce, E)) ce = 0;
        const float2 d = pair_dot(xs, WgT, H, ce, vb, ve, lane);
        if (lane == 0) part[warp] = d;
      }
      __syncthreads();
      if (warp == 0 && lane < g) {
        float2 acc = part[lane];
        for (int q = 1; q < ns; ++q) {
          const float2 d = part[q * g + lane];
          ff_add(acc.x, acc.y, d.x, d.y);
        }
        const int i = exact_at(c0 + lane);
        int e = small ? id_s[i] : rs.pairs[base + i].y;
        if (!in_bounds(e, E)) e = 0;
        double v = score_f64(static_cast<double>(acc.x) + static_cast<double>(acc.y), fn);
        if (bias != nullptr) v += static_cast<double>(bias[e]);
        if (small) key_s[i] = order_key(v);
        else rs.key[base + i] = order_key(v);
      }
      __syncthreads();
    }
    if (small) {
      // rank of each candidate among the others (larger key first, equal keys
      // lower id first): the k ranks below k are the selection, in order
      const float2 nrm = rs.fnorm[static_cast<long long>(seg) * seg_len + idx];
      for (int i = threadIdx.x; i < count; i += blockDim.x) {
        const unsigned long long v = key_s[i];
        const int e = id_s[i];
        int rank = 0;
        for (int q = 0; q < count; ++q) rank += before(key_s[q], id_s[q], v, e) ? 1 : 0;
        if (rank < k) {
          sel_s[rank] = e;
          aff_s[rank] = affinity_f32(pl_s[i], fn, nrm.x, nrm.y);
        }
      }
      __syncthreads();
      if (warp == 0) {
        float den = 0.0f;
        for (int jj = 0; jj < k; ++jj) den += aff_s[jj];  // in rank order
        if (lane < k) {
          const float a = aff_s[lane];
          float g = alpha * a;
          if (renorm) g = den > 0.0f ? alpha * a / den : 0.0f;
          E_ids[static_cast<long long>(t) * k + lane] = sel_s[lane];
          G[static_cast<long long>(t) * k + lane] = g;
        }
      }
      __syncthreads();
      continue;
    }
    if (warp == 0) {
      const float2 nrm = rs.fnorm[static_cast<long long>(seg) * seg_len + idx];
      // candidates held in registers, up to 4 per lane (count <= 128); more
      // candidates than that are read from memory each round
      constexpr int kHold = 4;
      unsigned long long cv[kHold];
      int ce[kHold];
      float cl[kHold];
#pragma unroll
      for (int h = 0; h < kHold; ++h) {
        const int i = lane + 32 * h;
        cv[h] = i < count ? rs.key[base + i] : 0ull;
        ce[h] = i < count ? rs.pairs[base + i].y : 0x7fffffff;
        cl[h] = i < count ? rs.plogit[base + i] : 0.0f;
      }
      int my_sel = -1;
      float my_l = 0.0f;
      unsigned long long last_v = ~0ull;
      int last_id = -1;
      // round r: the best candidate strictly after the previous winner in the
      // (larger score, lower id) order, so no candidate is taken twice
#pragma unroll 1
      for (int r = 0; r < k; ++r) {
        unsigned long long best = 0ull;
        int bid = 0x7fffffff;
        float bl = 0.0f;
#pragma unroll
        for (int h = 0; h < kHold; ++h)
          if (before(last_v, last_id, cv[h], ce[h]) && before(cv[h], ce[h], best, bid)) {
            best = cv[h];
            bid = ce[h];
            bl = cl[h];
          }
        for (int i = lane + 32 * kHold; i < count; i += 32) {
          const int e = rs.pairs[base + i].y;
          const unsigned long long v = rs.key[base + i];
          if (before(last_v, last_id, v, e) && before(v, e, best, bid)) {
            best = v;
            bid = e;
            bl = rs.plogit[base + i];
          }
        }
        warp_argmax_payload(best, bid, bl);
        if (lane == r) {
          my_sel = bid;
          my_l = bl;
        }
        last_v = best;
        last_id = bid;
      }
      const float a = lane < k ? affinity_f32(my_l, fn, nrm.x, nrm.y) : 0.0f;
      float den = 0.0f;
      for (int jj = 0; jj < k; ++jj) den += __shfl_sync(0xffffffffu, a, jj);
      if (lane < k) {
        float g = alpha * a;
        if (renorm) g = den > 0.0f ? alpha * a / den : 0.0f;
        E_ids[static_cast<long long>(t) * k + lane] = my_sel;
        G[static_cast<long long>(t) * k + lane] = g;
      }
    }
    __syncthreads();
  }
  // the last block to finish zeroes the counters (every block has read them)
  if (zero_counters && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(rs.counters + 2, 1) == static_cast<int>(gridDim.x) - 1) {
      rs.counters[0] = 0;
      rs.counters[1] = 0;
      rs.counters[2] = 0;
    }
  }
}

// WgT[e][h] = Wg[h][e], 32 x 32 tiles through shared memory.
__global__ void transpose_wg_kernel(const uint16_t* __restrict__ Wg, int H, int E,
                                    uint16_t* __restrict__ WgT) {
  __shared__ uint16_t tile[32][33];
  const int e0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int h = h0 + i, e = e0 + threadIdx.x;
    if (h < H && e < E) tile[i][threadIdx.x] = Wg[static_cast<long long>(h) * E + e];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int e = e0 + i, h = h0 + threadIdx.x;
    if (h < H && e < E) WgT[static_cast<long long>(e) * H + h] = tile[threadIdx.x][i];
  }
}

cudaError_t launch_transpose_wg(const uint16_t* Wg, int H, int E, uint16_t* WgT, cudaStream_t s) {
  dim3 grid((E + 31) / 32, (H + 31) / 32);
  transpose_wg_kernel<<<grid, dim3(32, 8), 0, s>>>(Wg, H, E, WgT);
  return cudaGetLastError();
}

cudaError_t launch_route_recheck(const uint16_t* X, const uint16_t* WgT, const float* bias, int T, int H,
                                 int E, int score_fn, int k, float alpha, int renorm, int32_t* E_ids,
                                 float* G, const RouteScratch& rs, const int* seg_n, int n_seg,
                                 int seg_len, bool zero_counters, bool pdl, cudaStream_t s) {
  const size_t sh = static_cast<size_t>(H) * 2 + kRedecideWarps * sizeof(float2) +
                    kRedecideList * sizeof(int) + static_cast<size_t>(n_seg) * sizeof(int);
  if (sh > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_redecide_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sh));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_sms(), 1, 1);
  cfg.blockDim = dim3(kRedecideWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = sh;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, route_redecide_kernel, X, WgT, bias, H, k, score_fn, alpha, renorm,
                            E_ids, G, rs, seg_n, n_seg, seg_len, zero_counters ? 1 : 0, T, E);
}

cudaError_t launch_route_select(const float* logits, const uint16_t* X, const uint16_t* WgT,
                                const float* bias, const int32_t* token_ids,
                                const int32_t* tid2eid, int V, int T, int H, int E, int k,
                                int score_fn, float alpha, int renorm, int32_t* E_ids, float* G,
                                const RouteScratch& rs, int* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int blocks = (T + kWarps - 1) / kWarps;
  const size_t sh = static_cast<size_t>(kWarps) * E * sizeof(float);
  if (sh > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sh));
    if (e != cudaSuccess) return e;
  }
  route_select_kernel<<<blocks, kWarps * 32, sh, s>>>(logits, bias, token_ids, tid2eid, V, T, E,
                                                      k, score_fn, alpha, renorm, E_ids, G, rs,
                                                      status);
  if (token_ids != nullptr) return cudaGetLastError();
  // one segment: the compact list and its counter, zeroed after use
  return launch_route_recheck(X, WgT, bias, T, H, E, score_fn, k, alpha, renorm, E_ids, G, rs, rs.counters,
                              1, T, true, false, s);
}

MOE_DEFINE_BOUNDS_TAKE(route)

}  // namespace moe
