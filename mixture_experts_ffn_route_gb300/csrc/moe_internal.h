// Internal interface between the C ABI (moe_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

#ifdef MOE_DEBUG_BOUNDS
// The bounds words of the debug build, one per translation unit that checks
// (MOE_DEFINE_BOUNDS_TAKE in moe_common.cuh).
int bounds_take_api();
int bounds_take_dispatch();
int bounds_take_gemm();
int bounds_take_gemm_mx();
int bounds_take_quant();
int bounds_take_backward();
int bounds_take_route();
int bounds_take_route_fused();
#endif

constexpr int kBM = 128;  // GEMM tile rows (tokens)
constexpr int kBK = 64;   // GEMM k-block (one 128-byte swizzle row of bf16)

enum GemmKind {
  kGemmRouter = 0,     // fp32 logits
  kGemmSwiGLU = 1,     // Linear1 + SwiGLU, bf16 out
  kGemmPlain = 2,      // Linear2, fp32 out
  kGemmCombineK1 = 4   // Linear2 with the top-1 combine: gate-scaled bf16 rows
                       // written to their tokens' rows of Y
};

// One grouped GEMM launch.  Groups are row ranges [row_off[g], row_off[g+1])
// of the A operand and of the output; tile_off[g] is the running count of
// 128-row tiles before group g.  Both arrays live on the device (written by
// the dispatch scan) so no host synchronisation is needed.  With
// row_off == nullptr there is one group of `dense_rows` rows.
struct GemmParams {
  const int* row_off;
  const int* tile_off;
  int num_groups;
  int dense_rows;
  int shared_group;  // group served by the second tensor maps, or -1
  int a2_shared;     // 1: that group's A rows come from map a2, starting at row 0
  int n_tiles;       // output column tiles per 128-row tile
  int num_kb;        // K / 64
  int n_out;         // valid output columns
  int up_off;        // SwiGLU: column of the first "up" column of W1 (= I)
  // Linear1 row gather: when gather_src is set, the A rows of a routed group
  // are the token rows gather_src[gather_perm[row] / gather_k] and those of the
  // shared group are gather_src[row - its first row]; they are copied by four
  // gather warps instead of TMA (map a is unused).
  const uint16_t* gather_src;  // X [gather_rows, K]
  const int* gather_perm;
  int gather_k;
  int gather_rows;
  // int8 forms: per-column weight scales of group g at scale_col + g *
  // scale_ld, and the per-row activation scales (Linear1: indexed by token,
  // Linear2: by assignment row)
  const float* scale_col;
  long long scale_ld;
  const float* scale_row;
  void* out;
  long long ldo;     // output row stride, elements
  int* status;
  // MX forms (FP8 codes, one E8M0 scale per 32 consecutive k): row r of A
  // has its scales at sfa + r * sf_ld; weight row n of group g at
  // sfb + g * sfb_ld + n * sf_ld.  The SwiGLU form writes
  // its output re-quantised: codes to out, scales to out_sf (out_sf_ld per row).
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sf_ld;
  long long sfb_ld;
  uint8_t* out_sf;
  int out_sf_ld;
  int sf_vec;        // 1: sf_ld, sfb_ld and both scale bases are 16-byte multiples
  // Linear1 (bf16): when set, the pre-activations (gate and up halves, bf16)
  // are also written to h_out [rows, 2 up_off], kept for the backward
  uint16_t* h_out;
  // Linear2 of the quantised forms: 1 = write the rows to out as bf16 (RNE)
  // instead of fp32
  int out_bf16;
  // kGemmCombineK1: the gates G [T] (k = 1); gather_perm maps a row to its token
  const float* gate;
  // Interleaved tile order (optional): tile_doff and tile_soff are tile_off
  // counted over the dense groups only (those of at least dense_mt row tiles,
  // whose weights are reused across row tiles) and over the others; the
  // dense groups' tiles are then spread evenly through the sparse groups'
  // weight stream (decode_tile).  Null: plain group order.
  const int* tile_doff;
  const int* tile_soff;
  // 1: the weight loads of sparse-group tiles (read once) carry an L2
  // evict_first policy, so that they pass through L2 without displacing the
  // token rows and the dense groups' weight blocks that are read again
  int l2_hint;
};

struct GemmMaps {
  CUtensorMap a, a2, b, b2;
};

// Tensor-map helpers (host).  Return false if the driver rejects the map.
bool make_map_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols);
bool make_map_weights(CUtensorMap* m, const void* base, int64_t groups, int64_t K, int64_t N);

// Per-row int8 quantisation ("mega_moe" A8W8): s = max|x| / 127 and codes
// round(x / s) (halves away from zero), written as fp16 values.  rows_dev,
// when set, gives the row count on the device (rows is then an upper bound).
// With inv (k <= 16), row t's codes and scale go to rows inv[t * k + j] of the
// outputs (the token rows in expert order), each token quantised once.
cudaError_t launch_quant_rows_bf16(const uint16_t* x, int rows, int cols, uint16_t* codes,
                                   float* scales, const int* inv, int k, cudaStream_t s);
cudaError_t launch_quant_rows_f32(const float* x, const int* rows_dev, int rows_max, int cols,
                                  uint16_t* codes, float* scales, cudaStream_t s);

// MX forms ("mega_moe" MXFP scenario).  Formats by tensor-core code:
// 0 = FLOAT8_E4M3FN, 1 = FLOAT8_E5M2, 5 = FLOAT4_E2M1 (two codes per byte).
// Rows quantised per group of 32 (cols a multiple of 32): codes [rows, cols]
// bytes (E2M1: [rows, cols / 2]), scales [rows, cols / 32]; with inv (the
// dispatch's inverse permutation, k <= 16) row t is written to rows
// inv[t k + j] instead of row t.
cudaError_t launch_mx_quant_rows(int fmt, const uint16_t* x, int rows, int cols, uint8_t* codes,
                                 uint8_t* scales, const int* inv, int k, cudaStream_t s);
// [rows, cols] codes, box of one 128-byte row segment x 128 rows, 128-byte
// swizzle; the weights [groups, N, K] as a 3-D map with box 128 bytes x
// box_rows n x 1.  Layouts: kMxFp8 one code per byte (box 128 codes);
// kMxFp4Spread packed E2M1 in memory, which the map type spreads to the
// shared-memory layout of kind::mxf8f6f4 (16 codes per 16 bytes, box 128
// codes); kMxFp4Packed packed E2M1 kept packed for kind::mxf4 (box 256 codes).
enum MxLayout { kMxFp8 = 0, kMxFp4Spread = 1, kMxFp4Packed = 2 };
bool make_map_mx_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int layout);
bool make_map_mx_weights(CUtensorMap* m, const void* base, int64_t groups, int64_t N, int64_t K,
                         int box_rows, int layout);
// Linear1 (SwiGLU, re-quantised to the activation format) or Linear2 (bf16 or
// fp32 out); A rows in expert order (map a), their scales at sfa.  K must be a
// multiple of 128 (of kMxBKPacked when packed).  afmt / bfmt: activation /
// weight formats; packed (E2M1 x E2M1 only): kind::mxf4 on packed tiles, maps
// of layout kMxFp4Packed, p.num_kb = K / kMxBKPacked.
bool mx_pair_supported(int afmt, int bfmt);
cudaError_t launch_gemm_mx(bool swiglu, int afmt, int bfmt, bool packed, const GemmMaps& maps,
                           const GemmParams& p, int grid, cudaStream_t s);
constexpr int kMxBK = 128;        // MX k-block: 128 FP8 codes (one 128-byte swizzle row) = 4 groups
constexpr int kMxBKPacked = 256;  // packed E2M1 k-block: 256 codes in the same row = 8 groups

// Backward GEMMs (bf16 operands, fp32 accumulation).  Groups split the rows
// (M) as in the forward (row_off / tile_off, shared group on map b2), or, for
// the weight gradients, the contraction (K): group g contracts rows
// [row_off[g], row_off[g + 1]) of both operands into its own [M, N] output.
enum BwdEpi { kBwdF32 = 0, kBwdSwiGLU = 1 };
struct BwdParams {
  const int* row_off;
  const int* tile_off;
  int num_groups;
  int dense_rows;    // split-M mode without groups: one group of this many rows
  int shared_group;  // split-M: group served by map b2; split-K: group written to out2
  int m_tiles;       // split-K: 128-row tiles of each group's output
  int n_tiles;       // 256-column tiles of the output
  int num_kb;        // split-M: K / 64 (rounded up)
  int M, N;          // output rows per group (split-K) and valid output columns
  void* out;         // fp32 [rows or M, ldo], or bf16 dH for the SwiGLU backward
  long long ldo;
  long long out_group_stride;  // split-K: elements between group outputs
  void* out2;                  // split-K: output of the shared group
  const uint16_t* h_in;        // SwiGLU backward: pre-activations [rows, 2I]
  int up_off;                  // column of the up half in h_in and out (= I)
  int* status;
};
// A_MN / B_MN: the operand's contiguous dimension is M / N (else K).
// Maps: A K-major [rows, K] box 64 x 128; A MN-major [K rows, M] box 64 x 64;
// B K-major [groups, N, K] box 64 x 256 x 1; B MN-major [K rows, N] box 64 x 64.
bool make_map_bf16_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols,
                      int box_rows);
bool make_map_bf16_kmajor_b(CUtensorMap* m, const void* base, int64_t groups, int64_t N, int64_t K);
cudaError_t launch_gemm_bwd(bool a_mn, bool b_mn, int epi, bool split_k, const CUtensorMap& a,
                            const CUtensorMap& b, const CUtensorMap& b2, const BwdParams& p,
                            int grid, cudaStream_t s);

// Elementwise steps of the backward (moe_backward.cu).  Permuted rows are the
// routed rows [0, row_off[E]) then, with a shared expert, its T rows.
cudaError_t launch_unpermute_bwd(const uint16_t* dY, const float* G, const int* perm,
                                 const int* row_off, const float* Yp, int rows_max, int k, int H,
                                 int E, int has_shared, uint16_t* dYp, float* dG, cudaStream_t s);
cudaError_t launch_gather_rows(const uint16_t* X, const int* perm, const int* row_off, int rows_max,
                               int k, int H, int E, int has_shared, uint16_t* Xp, cudaStream_t s);
cudaError_t launch_dx_reduce(const float* dXp, const int* inv, const int* row_off, const float* dXr,
                             int T, int k, int H, int E, int has_shared, uint16_t* dX, cudaStream_t s);
cudaError_t launch_router_bwd(const float* logits, const int32_t* E_ids, const float* dG, int T,
                              int E, int k, int score_fn, float alpha, int renorm, uint16_t* dl,
                              cudaStream_t s);

// A8W8 GEMMs with the int8 weights converted into TMEM as the MMA's A operand
// (moe_gemm_q8.cu).  w: int8 weight rows [groups, N, K] (K contiguous), box
// 64 k x 128 rows x 1, 64-byte swizzle (the 16-byte chunk c of row r lands at
// chunk c ^ ((r >> 1) & 3), so that a warp reading one row per thread hits
// every bank once); b: fp16 codes [rows, K] in expert order (one row per
// assignment) as make_map_rows.  p.scale_col / scale_ld: per-channel weight
// scales; p.scale_row: per-row activation scales; p.out [rows, ldo], fp32 (or
// bf16 for Linear2 with p.out_bf16).
bool make_map_i8_rows(CUtensorMap* m, const void* base, int64_t groups, int64_t N, int64_t K);
cudaError_t launch_gemm_q8(bool swiglu, const CUtensorMap& w, const CUtensorMap& b,
                           const GemmParams& p, int grid, cudaStream_t s);

// Launch the tcgen05 GEMM of the given kind on `grid` persistent CTAs.
cudaError_t launch_gemm(GemmKind kind, const GemmMaps& maps, const GemmParams& p, int grid,
                        cudaStream_t s);
int gemm_block_n(GemmKind kind);

// Router.  Scratch of the float64 re-decision of close tokens:
struct RouteScratch {
  int* counters;  // [0] close tokens, [1] candidate pairs, [2] re-decision blocks
                  // done; zero between calls (the re-decision's last block
                  // zeroes them).  General path only.
  int* seg_n;     // [T / 16]  fused router: close tokens of each CTA's band of
                  //           rows (its list: flagged[b R .. b R + seg_n[b]))
  int4* flagged;  // [T]      {token, first pair, pair count, 0}
  float2* fnorm;  // [T]      softmax normaliser of a close token {max logit, sum exp}
  int2* pairs;    // [T * E]  {token, expert}
  float* plogit;  // [T * E]  fp32 logit of each pair (for the gates)
  unsigned long long* key;  // [T * E]  order-preserving key of each pair's float64 score
};
cudaError_t launch_transpose_wg(const uint16_t* Wg, int H, int E, uint16_t* WgT, cudaStream_t s);
// Selection over fp32 logits [T, E] (top-k with the float64 re-decision of
// close tokens, or the hash lookup).
cudaError_t launch_route_select(const float* logits, const uint16_t* X, const uint16_t* WgT,
                                const float* bias, const int32_t* token_ids,
                                const int32_t* tid2eid, int V, int T, int H, int E, int k,
                                int score_fn, float alpha, int renorm, int32_t* E_ids, float* G,
                                const RouteScratch& rs, int* status, cudaStream_t s);
// The float64 re-decision of the tokens listed in rs (one kernel).
// Float64 re-decision of the listed close tokens.  The list is n_seg
// segments of at most seg_len entries: segment b holds seg_n[b] entries at
// flagged[b seg_len ..).  The general path passes one segment (its counters,
// which the last block zeroes); the fused router one per CTA, and launches
// the kernel as its programmatic dependent (pdl).
cudaError_t launch_route_recheck(const uint16_t* X, const uint16_t* WgT, const float* bias, int T, int H,
                                 int E, int score_fn, int k, float alpha, int renorm, int32_t* E_ids,
                                 float* G, const RouteScratch& rs, const int* seg_n, int n_seg,
                                 int seg_len, bool zero_counters, bool pdl, cudaStream_t s);
// Fused router (moe_route_fused.cu): the gating GEMM on the tensor cores with
// the scores, the selection bias, the top-k (or the hash lookup), the gates
// and the listing of close tokens in its epilogue; split over K across a
// cluster of CTAs whose partial logits are summed through distributed shared
// memory.  Writes Wg transposed into WgT (for the re-decision) when WgT is
// set, and the fp32 logits into logits_out when that is set; select = 0
// writes only those.  Returns cudaErrorNotSupported for shapes it does not
// take (E > 384 or H % 64 != 0), so the caller can use the general path.
struct RouteFusedArgs {
  const uint16_t* X;
  const uint16_t* Wg;
  const float* bias;
  const int32_t* token_ids;
  const int32_t* tid2eid;
  int V, T, H, E, k, score_fn, renorm;
  float alpha;
  int select;
  int32_t* E_ids;
  float* G;
  float* logits_out;
  uint16_t* WgT;
  RouteScratch rs;
  int* status;
};
bool route_fused_supported(int E, int H);
cudaError_t launch_route_fused(const RouteFusedArgs& a, cudaStream_t s);

// Dispatch: counts, offsets, permutation, inverse, tile offsets, gathered rows.
struct DispatchBufs {
  int* chunk_cnt;    // [nchunk * E]
  int* counts;       // [E + 1]
  int* row_off;      // [E + 2]
  int* tile_off;     // [E + 2]
  int* tile_doff;    // [E + 2] dense groups' tile offsets, or null
  int* tile_soff;    // [E + 2] sparse groups' tile offsets, or null
  int* perm;         // [T * k]
  int* inv;          // [T * k]
  int nchunk;
  int dense_mt;      // row tiles from which a group counts as dense
};
int dispatch_chunks(int A);
cudaError_t launch_dispatch(const int32_t* E_ids, int T, int k, int E, int has_shared,
                            const DispatchBufs& b, int* status, cudaStream_t s);
cudaError_t launch_combine(const float* Yp, const int* inv, const float* G,
                           const int* row_off, int T, int k, int H, int E, int has_shared,
                           uint16_t* Y, cudaStream_t s);
// Top-1 forward with the combine fused into Linear2: zero the rows of Y whose
// token's one id was dropped (inv < 0), as the combine would.
cudaError_t launch_zero_dropped_rows(const int* inv, int T, int H, uint16_t* Y, cudaStream_t s);
cudaError_t launch_combine_bf16(const uint16_t* Yp, const int* inv, const float* G,
                           const int* row_off, int T, int k, int H, int E, int has_shared,
                           uint16_t* Y, cudaStream_t s);

int num_sms();

}  // namespace moe
