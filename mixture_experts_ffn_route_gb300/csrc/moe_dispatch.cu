// Dispatch and combine: the on-device permute and un-permute around the
// expert GEMMs.
//
// "mega_moe" page, section 计算公式 / EP Dispatch: expert e receives the rows
// of the tokens that selected it, stacked in a fixed order, and row(i, k) is
// the unique row of token i in the block of its k-th expert.  "Megatron-LM 的
// MoE 并行：以 DeepSeek-V4 为例", section AlltoAll 的前向 / 计数与重排: count the
// assignments of each expert, then permute with duplication so each expert's
// rows are contiguous.  Here the fixed order inside a block is ascending flat
// assignment index f = t*k + j, which makes the result deterministic.
//
//   count   : per chunk of kChunk assignments, per-expert counts (smem atomics)
//   scan    : per-expert exclusive prefix over chunks, then over experts
//             (row offsets) and over 128-row tiles (tile offsets for the GEMMs)
//   place   : one block per chunk: each warp ranks its 128 ids among equal
//             ids (match_any), per-warp counts are prefix-summed per expert,
//             and each assignment gets row = row_off[e] + (rows of e in
//             earlier chunks, warps, and earlier in its warp); writes
//             perm[row] = f and inv[f] = row.  (Experts beyond 1024: one warp
//             per (expert, chunk) with ballot-prefix ranks.)
// The permuted token rows themselves are never written: Linear1 copies them
// from X by perm while it loads its A tiles.
//   combine : "mega_moe" page, section Token Combine: y_t = sum_j G[t, j] *
//             Yp[inv[t*k + j]] (+ the shared expert's row); Yp is fp32, the sum
//             is fp32 and y_t is rounded to bf16 once
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kChunk = 4096;
constexpr int kThreads = 1024;

int dispatch_chunks(int A) { return A <= 0 ? 0 : (A + kChunk - 1) / kChunk; }

__global__ void __launch_bounds__(kThreads)
    dispatch_count_kernel(const int32_t* __restrict__ E_ids, int A, int E, int* __restrict__ chunk_cnt,
                          int* __restrict__ inv, int* status) {
  extern __shared__ int hist[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int f0 = blockIdx.x * kChunk;
  const int f1 = min(A, f0 + kChunk);
  bool bad = false;
  for (int f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
    const int e = E_ids[f];
    if (e >= 0 && e < E) {
      atomicAdd(&hist[e], 1);
    } else {
      inv[f] = -1;
      bad = true;
    }
  }
  if (bad) set_flag(status, kFlagBadExpert);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) chunk_cnt[static_cast<long long>(blockIdx.x) * E + i] = hist[i];
}

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ int block_exclusive_scan(int v, int* out, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < static_cast<int>(blockDim.x >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
  const int total = warp_tot[(blockDim.x >> 5) - 1];
  *out = before;
  __syncthreads();
  return total;
}

// Single block.  After it: chunk_cnt[c][e] = rows of expert e in chunks < c;
// counts[e]; row_off[e] (exclusive, row_off[E] = valid assignments); tile_off.
// With a shared expert, group E is the T shared rows placed after all
// routed rows: counts[E] = T, row_off[E + 1] = row_off[E] + T.  With tile_doff
// set, tile_doff and tile_soff are the same running count of row tiles taken
// over the groups of at least dense_mt row tiles and over the rest.
__global__ void __launch_bounds__(kThreads)
    dispatch_scan_kernel(int* __restrict__ chunk_cnt, int nchunk, int E, int T, int has_shared,
                         int* __restrict__ counts, int* __restrict__ row_off, int* __restrict__ tile_off,
                         int* __restrict__ tile_doff, int* __restrict__ tile_soff, int dense_mt) {
  __shared__ int warp_tot[32];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int c = 0; c < nchunk; ++c) {
      const long long i = static_cast<long long>(c) * E + e;
      const int v = chunk_cnt[i];
      chunk_cnt[i] = run;
      run += v;
    }
    counts[e] = run;
  }
  __syncthreads();
  // exclusive scans over experts, kThreads experts per pass
  const bool split = tile_doff != nullptr;
  int row_carry = 0, tile_carry = 0, dense_carry = 0;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    const int n = (e < E) ? counts[e] : 0;
    const int mt = (n + kBM - 1) / kBM;
    int rb, tb, db = 0;
    const int rt = block_exclusive_scan(n, &rb, warp_tot);
    const int tt = block_exclusive_scan(mt, &tb, warp_tot);
    const int dt = split ? block_exclusive_scan(mt >= dense_mt ? mt : 0, &db, warp_tot) : 0;
    if (e < E) {
      row_off[e] = row_carry + rb;
      tile_off[e] = tile_carry + tb;
      if (split) {
        tile_doff[e] = dense_carry + db;
        tile_soff[e] = (tile_carry + tb) - (dense_carry + db);
      }
    }
    row_carry += rt;
    tile_carry += tt;
    dense_carry += dt;
  }
  if (threadIdx.x == 0) {
    row_off[E] = row_carry;
    tile_off[E] = tile_carry;
    int dense_end = dense_carry;
    if (has_shared) {
      const int mt = (T + kBM - 1) / kBM;
      counts[E] = T;
      row_off[E + 1] = row_carry + T;
      tile_off[E + 1] = tile_carry + mt;
      if (mt >= dense_mt) dense_end += mt;
    }
    if (split) {
      tile_doff[E] = dense_carry;
      tile_soff[E] = tile_carry - dense_carry;
      if (has_shared) {
        tile_doff[E + 1] = dense_end;
        tile_soff[E + 1] = tile_off[E + 1] - dense_end;
      }
    }
  }
}

// One block per (32 experts, chunk): the chunk's ids are staged in shared
// memory once; warp w ranks expert 32 * blockIdx.x + w with ballots, in
// ascending flat index order.
__global__ void __launch_bounds__(kThreads)
    dispatch_place_kernel(const int32_t* __restrict__ E_ids, int A, int E, int nchunk,
                          const int* __restrict__ chunk_base, const int* __restrict__ counts,
                          const int* __restrict__ row_off, int* __restrict__ perm, int* __restrict__ inv) {
  __shared__ int ids[kChunk];
  const int c = blockIdx.y;
  const int f0 = c * kChunk;
  const int n = min(A - f0, kChunk);
  for (int i = threadIdx.x; i < n; i += blockDim.x) ids[i] = E_ids[f0 + i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + warp;
  if (e >= E) return;
  const int b0 = chunk_base[static_cast<long long>(c) * E + e];
  const int b1 = (c + 1 < nchunk) ? chunk_base[static_cast<long long>(c + 1) * E + e] : counts[e];
  if (b1 == b0) return;  // no assignment of e in this chunk
  int pos = row_off[e] + b0;
  for (int i0 = 0; i0 < n && pos < row_off[e] + b1; i0 += 32) {
    const int i = i0 + lane;
    const bool mine = (i < n) && (ids[i] == e);
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    if (mine) {
      const int row = pos + __popc(m & ((1u << lane) - 1u));
      if (in_bounds(row, A)) {
        perm[row] = f0 + i;
        inv[f0 + i] = row;
      }
    }
    pos += __popc(m);
  }
}

constexpr int kPlaceMaxE = 1024;  // per-warp expert counts in shared memory: 32 * E ints

// One block per chunk of kChunk assignments; warp w takes ids [128 w, 128 w +
// 128) in four rounds of 32.  In a round, the lanes holding the same expert
// find each other (match_any): a lane's rank is the number of equal ids in
// lower lanes plus the warp's running count of that expert, which the lowest
// of them then advances.  The per-warp counts become an exclusive prefix over
// the warps, so rows follow ascending flat index inside each expert.
__global__ void __launch_bounds__(kThreads)
    dispatch_place_match_kernel(const int32_t* __restrict__ E_ids, int A, int E,
                                const int* __restrict__ chunk_base, const int* __restrict__ row_off,
                                int* __restrict__ perm, int* __restrict__ inv) {
  extern __shared__ int sm[];
  int* ids = sm;                // [kChunk]
  int* rank = sm + kChunk;      // [kChunk] rank among equal ids of the same warp
  int* cnt = sm + 2 * kChunk;   // [32][E]  per-warp counts, then their prefix over warps
  const int c = blockIdx.x;
  const int f0 = c * kChunk;
  const int n = min(A - f0, kChunk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) cnt[i] = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) ids[i] = E_ids[f0 + i];
  __syncthreads();
  int* wcnt = cnt + warp * E;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = 128 * warp + 32 * r + lane;
    int e = i < n ? ids[i] : -1;
    if (e >= E) e = -1;  // ids outside [0, E) are not placed (the count flagged them)
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int below = __popc(peers & ((1u << lane) - 1u));
    const int base = e >= 0 ? wcnt[e] : 0;
    __syncwarp();
    if (e >= 0 && below == 0) wcnt[e] = base + __popc(peers);
    __syncwarp();
    if (i < n) rank[i] = base + below;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  const int* cb = chunk_base + static_cast<long long>(c) * E;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = ids[i];
    if (e < 0 || e >= E) continue;
    const int row = __ldg(row_off + e) + __ldg(cb + e) + cnt[(i >> 7) * E + e] + rank[i];
    if (!in_bounds(row, A)) continue;
    perm[row] = f0 + i;
    inv[f0 + i] = row;
  }
}

cudaError_t launch_dispatch(const int32_t* E_ids, int T, int k, int E, int has_shared,
                            const DispatchBufs& b, int* status, cudaStream_t s) {
  const int A = T * k;
  if (A > 0) {
    const size_t sh = static_cast<size_t>(E) * sizeof(int);
    if (sh > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(dispatch_count_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(sh));
      if (e != cudaSuccess) return e;
    }
    dispatch_count_kernel<<<b.nchunk, kThreads, sh, s>>>(E_ids, A, E, b.chunk_cnt, b.inv, status);
  }
  dispatch_scan_kernel<<<1, kThreads, 0, s>>>(b.chunk_cnt, b.nchunk, E, T, has_shared, b.counts,
                                              b.row_off, b.tile_off, b.tile_doff, b.tile_soff,
                                              b.dense_mt);
  if (A > 0 && E <= kPlaceMaxE) {
    const int sh = (2 * kChunk + 32 * E) * static_cast<int>(sizeof(int));
    cudaError_t e = cudaFuncSetAttribute(dispatch_place_match_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, sh);
    if (e != cudaSuccess) return e;
    dispatch_place_match_kernel<<<b.nchunk, kThreads, sh, s>>>(E_ids, A, E, b.chunk_cnt, b.row_off,
                                                               b.perm, b.inv);
  } else if (A > 0) {
    dispatch_place_kernel<<<dim3((E + 31) / 32, b.nchunk), kThreads, 0, s>>>(E_ids, A, E, b.nchunk,
                                                                 b.chunk_cnt, b.counts, b.row_off,
                                                                 b.perm, b.inv);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------- combine
constexpr int kCombineThreads = 128;

// 8 consecutive elements of an expert output row (fp32 or bf16) as fp32.
__device__ __forceinline__ void load_row8(const float* row, int c, float (&x)[8]) {
  const float4* src = reinterpret_cast<const float4*>(row) + 2 * c;
  const float4 u = __ldcs(src), v = __ldcs(src + 1);  // read once
  x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w; x[4] = v.x; x[5] = v.y; x[6] = v.z; x[7] = v.w;
}
__device__ __forceinline__ void load_row8(const uint16_t* row, int c, float (&x)[8]) {
  const uint4 u = __ldcs(reinterpret_cast<const uint4*>(row) + c);
  x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

template <typename In>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const In* __restrict__ Yp, const int* __restrict__ inv,
                   const float* __restrict__ G, const int* __restrict__ row_off, int k, int H,
                   int E, int has_shared, uint16_t* __restrict__ Y) {
  __shared__ int rows[17];
  __shared__ float w[17];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    rows[threadIdx.x] = inv[static_cast<long long>(t) * k + threadIdx.x];
    w[threadIdx.x] = G[static_cast<long long>(t) * k + threadIdx.x];
  }
  if (threadIdx.x == 0 && has_shared) {
    rows[k] = row_off[E] + t;
    w[k] = 1.0f;
  }
  __syncthreads();
  const int n = k + (has_shared ? 1 : 0);
  const int vecs = H / 8;
  const long long n_rows = static_cast<long long>(gridDim.x) * (k + (has_shared ? 1 : 0));  // rows of Yp
  for (int c = threadIdx.x; c < vecs; c += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < n; ++j) {
      const int p = rows[j];
      if (p < 0 || !in_bounds(p, n_rows)) continue;
      float x[8];
      load_row8(Yp + static_cast<long long>(p) * H, c, x);
      const float g = w[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += g * x[i];
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(Y + static_cast<long long>(t) * H)[c] = o;
  }
}

// One warp per token: a token whose single assignment was dropped has no
// Linear2 row, so its output row is written here as zeros.
__global__ void __launch_bounds__(256)
    zero_dropped_kernel(const int* __restrict__ inv, int T, int H, uint16_t* __restrict__ Y) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T || __ldg(inv + t) >= 0) return;
  uint4* row = reinterpret_cast<uint4*>(Y + static_cast<long long>(t) * H);
  for (int c = lane; c < H / 8; c += 32) row[c] = make_uint4(0u, 0u, 0u, 0u);
}

cudaError_t launch_zero_dropped_rows(const int* inv, int T, int H, uint16_t* Y, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  zero_dropped_kernel<<<(T + 7) / 8, 256, 0, s>>>(inv, T, H, Y);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* Yp, const int* inv, const float* G, const int* row_off,
                           int T, int k, int H, int E, int has_shared, uint16_t* Y, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  combine_kernel<float><<<T, kCombineThreads, 0, s>>>(Yp, inv, G, row_off, k, H, E, has_shared, Y);
  return cudaGetLastError();
}

cudaError_t launch_combine_bf16(const uint16_t* Yp, const int* inv, const float* G,
                                const int* row_off, int T, int k, int H, int E, int has_shared,
                                uint16_t* Y, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  combine_kernel<uint16_t><<<T, kCombineThreads, 0, s>>>(Yp, inv, G, row_off, k, H, E, has_shared, Y);
  return cudaGetLastError();
}

MOE_DEFINE_BOUNDS_TAKE(dispatch)

}  // namespace moe
