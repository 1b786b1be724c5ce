// C ABI of the routed MoE FFN forward pass (declared in include/moe_ffn.h):
// argument validation, workspace layout and the launch sequence.
#include <string.h>

#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_ffn.h"
#include "moe_internal.h"

namespace moe {

int num_sms() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> g(mu);
  if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout (byte offsets, each 256-aligned).
struct WsLayout {
  size_t status, logits, wgt, flagged, fnorm, pairs, plogit, s64, segn, chunk_cnt, counts, row_off,
      tile_off, perm, inv, act, yp, total;
};

// The status header (256 bytes, zeroed by moe_workspace_init): the status
// word at byte 0; the router's re-decision list counters at byte 64; the
// debug build's bounds self-test array at byte 128.
constexpr size_t kRouteCountersAt = 64;

static WsLayout layout(const moe_params& p) {
  WsLayout L;
  const size_t T = static_cast<size_t>(p.T), E = static_cast<size_t>(p.E);
  const size_t A = T * static_cast<size_t>(p.k);
  const size_t Tsh = p.has_shared ? T : 0;
  const size_t nchunk = static_cast<size_t>(dispatch_chunks(static_cast<int>(A)));
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.status = take(256);
  L.logits = take(T * E * sizeof(float));  // general router path only
  L.wgt = take(static_cast<size_t>(p.H) * E * 2);
  L.flagged = take(T * 4 * sizeof(int));
  L.fnorm = take(T * 2 * sizeof(float));
  L.pairs = take(T * E * 2 * sizeof(int));
  L.plogit = take(T * E * sizeof(float));
  L.s64 = take(T * E * sizeof(double));
  L.segn = take((T / 16 + 8) * sizeof(int));  // fused router: one count per CTA
  L.chunk_cnt = take((nchunk > 0 ? nchunk : 1) * E * sizeof(int));
  L.counts = take((E + 2) * sizeof(int));
  L.row_off = take((E + 2) * sizeof(int));
  L.tile_off = take(3 * (E + 2) * sizeof(int));  // tile_off, tile_doff, tile_soff
  L.perm = take(A * sizeof(int));
  L.inv = take(A * sizeof(int));
  L.act = take((A + Tsh) * static_cast<size_t>(p.I) * 2);
  L.yp = take((A + Tsh) * static_cast<size_t>(p.H) * sizeof(float));
  L.total = o;
  return L;
}

// Workspace layout of the A8W8 forward.
struct WsLayoutQ {
  size_t status, chunk_cnt, counts, row_off, tile_off, perm, inv, xq, sx, act, aq, sa, yp, total;
};

static WsLayoutQ layout_a8w8(const moe_params& p) {
  WsLayoutQ L;
  const size_t T = static_cast<size_t>(p.T), E = static_cast<size_t>(p.E);
  const size_t A = T * static_cast<size_t>(p.k);
  const size_t H = static_cast<size_t>(p.H), I = static_cast<size_t>(p.I);
  const size_t nchunk = static_cast<size_t>(dispatch_chunks(static_cast<int>(A)));
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.status = take(256);
  L.chunk_cnt = take((nchunk > 0 ? nchunk : 1) * E * sizeof(int));
  L.counts = take((E + 2) * sizeof(int));
  L.row_off = take((E + 2) * sizeof(int));
  L.tile_off = take(3 * (E + 2) * sizeof(int));  // tile_off, tile_doff, tile_soff
  L.perm = take(A * sizeof(int));
  L.inv = take(A * sizeof(int));
  L.xq = take(A * H * 2);          // token codes in expert order (one row per assignment)
  L.sx = take(A * sizeof(float));
  L.act = take(A * I * sizeof(float));
  L.aq = take(A * I * 2);
  L.sa = take(A * sizeof(float));
  L.yp = take(A * H * sizeof(float));
  L.total = o;
  return L;
}

// Workspace layout of the MX forward.
struct WsLayoutMX {
  size_t status, chunk_cnt, counts, row_off, tile_off, perm, inv, xq, sx, uq, su, yp, total;
};

static WsLayoutMX layout_mx(const moe_params& p) {
  WsLayoutMX L;
  const size_t T = static_cast<size_t>(p.T), E = static_cast<size_t>(p.E);
  const size_t A = T * static_cast<size_t>(p.k);
  const size_t H = static_cast<size_t>(p.H), I = static_cast<size_t>(p.I);
  const size_t nchunk = static_cast<size_t>(dispatch_chunks(static_cast<int>(A)));
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.status = take(256);
  L.chunk_cnt = take((nchunk > 0 ? nchunk : 1) * E * sizeof(int));
  L.counts = take((E + 2) * sizeof(int));
  L.row_off = take((E + 2) * sizeof(int));
  L.tile_off = take(3 * (E + 2) * sizeof(int));  // tile_off, tile_doff, tile_soff
  L.perm = take(A * sizeof(int));
  L.inv = take(A * sizeof(int));
  L.xq = take(A * H);
  L.sx = take(A * H / 32);
  L.uq = take(A * I);
  L.su = take(A * I / 32);
  L.yp = take(A * H * sizeof(float));
  L.total = o;
  return L;
}

// Training workspace: the forward's layout, then what the backward keeps or
// builds.  Rows R = T k (+ T with a shared expert) in the forward's order.
struct WsLayoutTrain {
  WsLayout f;
  size_t h, dyp, dh, xp, dxr, dl, dg, koff, total;
};

static WsLayoutTrain layout_train(const moe_params& p) {
  WsLayoutTrain L;
  L.f = layout(p);
  const size_t T = static_cast<size_t>(p.T), E = static_cast<size_t>(p.E);
  const size_t R = T * static_cast<size_t>(p.k) + (p.has_shared ? T : 0);
  const size_t H = static_cast<size_t>(p.H), I = static_cast<size_t>(p.I);
  size_t o = L.f.total;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.h = take(R * 2 * I * 2);      // Linear1 pre-activations, bf16
  L.dyp = take(R * H * 2);        // un-permuted output gradient rows, bf16
  L.dh = take(R * 2 * I * 2);     // gradient of the pre-activations, bf16
  L.xp = take(R * H * 2);         // token rows in expert order, bf16
  L.dxr = take(T * H * 4);        // router part of dX, fp32
  L.dl = take(T * E * 2);         // logit gradient, bf16
  L.dg = take(T * static_cast<size_t>(p.k) * 4);
  L.koff = take(2 * sizeof(int));
  L.total = o;
  return L;
}

static bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

static moe_status check_params(const moe_params* p) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->H <= 0 || p->E <= 0 || p->I <= 0 || p->k <= 0) return MOE_ERR_INVALID_ARG;
  if (p->k > p->E || p->score_fn < 0 || p->score_fn > 2) return MOE_ERR_INVALID_ARG;
  if (p->has_shared != 0 && p->has_shared != 1) return MOE_ERR_INVALID_ARG;
  if (p->k > 16 || p->E > 4096) return MOE_ERR_UNSUPPORTED;
  if (p->H % 64 != 0 || p->I % 64 != 0) return MOE_ERR_UNSUPPORTED;
  // 32-bit row and element counts inside the kernels
  const long long A = static_cast<long long>(p->T) * p->k;
  if (A + p->T > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static moe_status check_ws(const moe_params* p, void* ws, size_t ws_bytes) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < layout(*p).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename T>
static T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

static moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static moe_status run_router_gemm(const moe_params* p, const uint16_t* X, const uint16_t* Wg,
                                  float* logits, int* status, cudaStream_t s) {
  GemmMaps maps;
  if (!make_map_rows(&maps.a, X, p->T, p->H)) return MOE_ERR_CUDA;
  if (!make_map_weights(&maps.b, Wg, 1, p->H, p->E)) return MOE_ERR_CUDA;
  maps.a2 = maps.a;
  maps.b2 = maps.b;
  GemmParams g;
  memset(&g, 0, sizeof(g));
  g.row_off = nullptr;
  g.tile_off = nullptr;
  g.num_groups = 1;
  g.dense_rows = p->T;
  g.shared_group = -1;
  g.a2_shared = 0;
  g.n_tiles = (p->E + gemm_block_n(kGemmRouter) - 1) / gemm_block_n(kGemmRouter);
  g.num_kb = p->H / kBK;
  g.n_out = p->E;
  g.up_off = 0;
  g.out = logits;
  g.ldo = p->E;
  g.status = status;
  const int tiles = ((p->T + kBM - 1) / kBM) * g.n_tiles;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return cuda_status(launch_gemm(kGemmRouter, maps, g, grid, s));
}

// L2 capacity of the current device in bytes (cached per device).
static size_t l2_bytes() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0) return 0;
    cache[dev] = v;
  }
  return static_cast<size_t>(cache[dev]);
}

// Waits on an mbarrier that nothing ever arrives on: the bounded wait must
// give up after limit_ns and record kFlagTimeout in the status word.
__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status, &abort_flag, limit_ns);
}

#ifdef MOE_DEBUG_BOUNDS
// Writes element `index` of a 32-int array through the debug build's bounds
// check (an index outside [0, 32) is recorded and skipped).
__global__ void selftest_bounds_kernel(int* arr, long long index) {
  if (in_bounds(index, 32)) arr[index] = 1;
}
#endif

MOE_DEFINE_BOUNDS_TAKE(api)

#ifdef MOE_DEBUG_BOUNDS
// Any translation unit's bounds word set since the last call (all cleared).
static bool take_bounds() {
  int v = 0;
  for (int w : {bounds_take_api(), bounds_take_dispatch(), bounds_take_gemm(), bounds_take_gemm_mx(),
                bounds_take_quant(), bounds_take_backward(), bounds_take_route(), bounds_take_route_fused()})
    v |= w;
  return v != 0;
}
#endif

}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_abi_version(void) { return 1; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id outside [0, E)";
    case MOE_ERR_BAD_TOKEN_ID: return "hash token id outside [0, V)";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_BOUNDS: return "index outside its array (debug build)";
  }
  return "unknown status";
}

size_t moe_workspace_size(const moe_params* p) {
  if (check_params(p) != MOE_OK) return 0;
  return layout(*p).total;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream)));
}

moe_status moe_sync_status(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || ws_bytes < 256) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int flags = 0;
  if (cudaMemcpyAsync(&flags, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
#ifdef MOE_DEBUG_BOUNDS
  const bool bounds = take_bounds();
#else
  const bool bounds = false;
#endif
  if (flags & kFlagTimeout) return MOE_ERR_TIMEOUT;
  if (bounds) return MOE_ERR_BOUNDS;
  if (flags & kFlagBadToken) return MOE_ERR_BAD_TOKEN_ID;
  if (flags & kFlagBadExpert) return MOE_ERR_BAD_EXPERT_ID;
  return MOE_OK;
}

moe_status moe_selftest_bounds(void* ws, size_t ws_bytes, int64_t index, void* stream) {
  if (ws == nullptr || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
#ifdef MOE_DEBUG_BOUNDS
  selftest_bounds_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(at<int>(ws, 128),
                                                                      static_cast<long long>(index));
  return cuda_status(cudaGetLastError());
#else
  (void)index;
  (void)stream;
  return MOE_ERR_UNSUPPORTED;
#endif
}

moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us,
                                      void* stream) {
  if (ws == nullptr || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  if (limit_us == 0 || limit_us > 1000000u) return MOE_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      at<int>(ws, 0), static_cast<unsigned long long>(limit_us) * 1000ull);
  return cuda_status(cudaGetLastError());
}

static RouteScratch route_scratch(void* ws, const WsLayout& L) {
  RouteScratch rs;
  rs.counters = at<int>(ws, kRouteCountersAt);
  rs.seg_n = at<int>(ws, L.segn);
  rs.flagged = at<int4>(ws, L.flagged);
  rs.fnorm = at<float2>(ws, L.fnorm);
  rs.pairs = at<int2>(ws, L.pairs);
  rs.plogit = at<float>(ws, L.plogit);
  rs.key = at<unsigned long long>(ws, L.s64);
  return rs;
}

moe_status moe_route_logits(const moe_params* p, const uint16_t* X, const uint16_t* Wg,
                            float* logits, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = check_params(p);
  if (st != MOE_OK) return st;
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  if (p->E % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (p->T == 0) return MOE_OK;
  if (!X || !Wg || !logits || !aligned16(X) || !aligned16(Wg) || !aligned16(logits))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!route_fused_supported(p->E, p->H))
    return run_router_gemm(p, X, Wg, logits, at<int>(ws, 0), s);
  // the fused router's own logits (the ones its decisions are taken on)
  const WsLayout L = layout(*p);
  RouteFusedArgs a;
  memset(&a, 0, sizeof(a));
  a.X = X;
  a.Wg = Wg;
  a.T = p->T; a.H = p->H; a.E = p->E; a.k = p->k; a.score_fn = p->score_fn; a.renorm = p->renorm;
  a.alpha = p->alpha;
  a.select = 0;
  a.logits_out = logits;
  a.rs = route_scratch(ws, L);
  a.status = at<int>(ws, L.status);
  return cuda_status(launch_route_fused(a, s));
}

moe_status moe_route(const moe_params* p, const uint16_t* X, const uint16_t* Wg,
                     const float* bias, const int32_t* token_ids, const int32_t* tid2eid,
                     int32_t V, int32_t* E_ids, float* G, void* ws, size_t ws_bytes,
                     void* stream) {
  moe_status st = check_params(p);
  if (st != MOE_OK) return st;
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  if (p->E % 8 != 0) return MOE_ERR_UNSUPPORTED;
  const bool hash = token_ids != nullptr;
  if (hash && (tid2eid == nullptr || V <= 0 || bias != nullptr)) return MOE_ERR_INVALID_ARG;
  if (!hash && tid2eid != nullptr) return MOE_ERR_INVALID_ARG;
  if (bias != nullptr && p->score_fn == MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
  if (p->T == 0) return MOE_OK;
  if (!X || !Wg || !E_ids || !G || !aligned16(X) || !aligned16(Wg)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(*p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = at<int>(ws, L.status);
  uint16_t* WgT = at<uint16_t>(ws, L.wgt);
  const RouteScratch rs = route_scratch(ws, L);
  if (route_fused_supported(p->E, p->H)) {
    // one launch: gating GEMM + scores + top-k (or hash lookup) + gates; for
    // top-k two more that re-decide the close tokens from float64 logits
    RouteFusedArgs a;
    a.X = X;
    a.Wg = Wg;
    a.bias = bias;
    a.token_ids = token_ids;
    a.tid2eid = tid2eid;
    a.V = V;
    a.T = p->T; a.H = p->H; a.E = p->E; a.k = p->k; a.score_fn = p->score_fn; a.renorm = p->renorm;
    a.alpha = p->alpha;
    a.select = 1;
    a.E_ids = E_ids;
    a.G = G;
    a.logits_out = nullptr;
    a.WgT = hash ? nullptr : WgT;
    a.rs = rs;
    a.status = status;
    return cuda_status(launch_route_fused(a, s));
  }
  // general path: fp32 logits to the workspace, then the selection
  float* logits = at<float>(ws, L.logits);
  if (!hash && launch_transpose_wg(Wg, p->H, p->E, WgT, s) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = run_router_gemm(p, X, Wg, logits, status, s)) != MOE_OK) return st;
  return cuda_status(launch_route_select(logits, X, WgT, bias, token_ids, tid2eid, V, p->T, p->H,
                                         p->E, p->k, p->score_fn, p->alpha, p->renorm, E_ids, G,
                                         rs, status, s));
}

// Interleaved tile order of the grouped forward GEMMs (decode_tile): the
// groups of at least kDenseMt row tiles, whose weight blocks are reused across
// row tiles, are spread evenly through the other groups' weight stream, and
// the stream's weight loads carry an L2 evict_first policy.  On a layer of
// T 4096, H 7168, 384 experts top-6 of I 2048 plus a shared expert, under a
// Zipf(1.1) load, this took Linear1 from 3.69 to 3.51 ms and Linear2 from 1.88
// to 1.76 ms; thresholds of 3 and 4 gained less, and the order without the
// policy lost (the stream then displaced the reused operands).
constexpr int kDenseMt = 2;
constexpr int kL2Hint = 1;

static void set_tile_split(DispatchBufs* b, int E) {
  b->tile_doff = b->tile_off + (E + 2);
  b->tile_soff = b->tile_off + 2 * (E + 2);
  b->dense_mt = kDenseMt;
}

static void set_schedule(GemmParams* g, const DispatchBufs& b) {
  g->tile_doff = b.dense_mt > 0 ? b.tile_doff : nullptr;
  g->tile_soff = b.dense_mt > 0 ? b.tile_soff : nullptr;
  g->l2_hint = kL2Hint;
}

static DispatchBufs dispatch_bufs(const moe_params* p, void* ws, const WsLayout& L) {
  DispatchBufs b;
  b.chunk_cnt = at<int>(ws, L.chunk_cnt);
  b.counts = at<int>(ws, L.counts);
  b.row_off = at<int>(ws, L.row_off);
  b.tile_off = at<int>(ws, L.tile_off);
  b.perm = at<int>(ws, L.perm);
  b.inv = at<int>(ws, L.inv);
  b.nchunk = dispatch_chunks(p->T * p->k);
  set_tile_split(&b, p->E);
  return b;
}

moe_status moe_dispatch(const moe_params* p, const int32_t* E_ids, int32_t* counts,
                        int32_t* offsets, int32_t* perm, void* ws, size_t ws_bytes,
                        void* stream) {
  moe_status st = check_params(p);
  if (st != MOE_OK) return st;
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  if (!counts || !offsets || (p->T > 0 && (!E_ids || !perm))) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(*p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const DispatchBufs b = dispatch_bufs(p, ws, L);
  cudaError_t e = launch_dispatch(E_ids, p->T, p->k, p->E, 0, b, at<int>(ws, L.status), s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const size_t A = static_cast<size_t>(p->T) * p->k;
  e = cudaMemcpyAsync(counts, b.counts, p->E * sizeof(int), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(offsets, b.row_off, (p->E + 1) * sizeof(int), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && A > 0)
    e = cudaMemcpyAsync(perm, b.perm, A * sizeof(int), cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

}  // extern "C"

// The bf16 forward; with h_out set, Linear1 also keeps its pre-activations.
static moe_status forward_impl(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                               const float* G, const uint16_t* W1, const uint16_t* W2,
                               const uint16_t* Ws1, const uint16_t* Ws2, uint16_t* Y, void* ws,
                               size_t ws_bytes, void* stream, void* const* stage_events,
                               uint16_t* h_out) {
  moe_status st = check_params(p);
  if (st != MOE_OK) return st;
  if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK) return st;
  if (p->T == 0) return MOE_OK;
  if (!X || !E_ids || !G || !W1 || !W2 || !Y) return MOE_ERR_INVALID_ARG;
  if (p->has_shared && (!Ws1 || !Ws2)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W1) || !aligned16(W2) || !aligned16(Y)) return MOE_ERR_INVALID_ARG;
  if (p->has_shared && (!aligned16(Ws1) || !aligned16(Ws2))) return MOE_ERR_INVALID_ARG;

  const WsLayout L = layout(*p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = at<int>(ws, L.status);
  const DispatchBufs b = dispatch_bufs(p, ws, L);
  const int T = p->T, H = p->H, E = p->E, k = p->k, I = p->I;
  const int A = T * k;
  const int Tsh = p->has_shared ? T : 0;
  uint16_t* Act = at<uint16_t>(ws, L.act);
  float* Yp = at<float>(ws, L.yp);

  auto mark = [&](int i) -> cudaError_t {
    if (stage_events == nullptr || stage_events[i] == nullptr) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s);
  };
  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = launch_dispatch(E_ids, T, k, E, p->has_shared, b, status, s);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  const int groups = E + (p->has_shared ? 1 : 0);
  const int mt_bound = (A + kBM - 1) / kBM + E + (Tsh + kBM - 1) / kBM;

  // Linear1 + SwiGLU:  Act = SwiGLU(X[rows of e] W1[e]), the rows gathered from
  // X by the permutation inside the GEMM; the shared group takes X as it is.
  // Where the experts average two row tiles or more and X is larger than L2
  // (the large-FFN layer), the token rows are first copied into expert order
  // (over Yp, which Linear2 writes only later) and Linear1 loads them by TMA:
  // whole boxes of consecutive rows instead of 128 scattered row segments.
  const bool rows_by_tma = A >= 2 * kBM * E && static_cast<size_t>(T) * H * 2 > l2_bytes();
  {
    GemmMaps maps;
    uint16_t* Xp = reinterpret_cast<uint16_t*>(Yp);
    bool ok = make_map_rows(&maps.a, rows_by_tma ? Xp : X, rows_by_tma ? A : T, H) &&
              make_map_weights(&maps.b, W1, E, H, 2 * I);
    if (ok) ok = rows_by_tma ? make_map_rows(&maps.a2, X, T, H) : (maps.a2 = maps.a, true);
    if (ok) ok = p->has_shared ? make_map_weights(&maps.b2, Ws1, 1, H, 2 * I) : (maps.b2 = maps.b, true);
    if (!ok) return MOE_ERR_CUDA;
    if (rows_by_tma && launch_gather_rows(X, b.perm, b.row_off, A, k, H, E, 0, Xp, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    GemmParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.tile_off = b.tile_off;
    g.num_groups = groups;
    g.shared_group = p->has_shared ? E : -1;
    g.a2_shared = rows_by_tma && p->has_shared ? 1 : 0;
    set_schedule(&g, b);
    g.gather_src = rows_by_tma ? nullptr : X;
    g.gather_perm = b.perm;
    g.gather_k = k;
    g.gather_rows = T;
    g.n_tiles = (I + 127) / 128;
    g.num_kb = H / kBK;
    g.n_out = I;
    g.up_off = I;
    g.out = Act;
    g.ldo = I;
    g.h_out = h_out;
    g.status = status;
    const long long tiles = static_cast<long long>(mt_bound) * g.n_tiles;
    const int grid = tiles < num_sms() ? static_cast<int>(tiles) : num_sms();
    if ((e = launch_gemm(kGemmSwiGLU, maps, g, grid, s)) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(2) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // Linear2:  Yp = Act W2[e] (shared group uses Ws2), fp32 rows: the layer
  // output is rounded to bf16 once, in the combine.  Top-1 without a shared
  // expert: the combine is one gate-scaled row per token, written by Linear2's
  // epilogue straight into Y (no Yp round trip); the training forward keeps
  // the rows, which the backward's gate gradient reads.
  const bool fuse_k1 = h_out == nullptr && k == 1 && !p->has_shared;
  {
    GemmMaps maps;
    bool ok = make_map_rows(&maps.a, Act, A + Tsh, I) && make_map_weights(&maps.b, W2, E, I, H);
    if (ok) ok = p->has_shared ? make_map_weights(&maps.b2, Ws2, 1, I, H) : (maps.b2 = maps.b, true);
    if (!ok) return MOE_ERR_CUDA;
    maps.a2 = maps.a;
    GemmParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.tile_off = b.tile_off;
    g.num_groups = groups;
    g.shared_group = p->has_shared ? E : -1;
    g.a2_shared = 0;
    set_schedule(&g, b);
    g.n_tiles = (H + 255) / 256;
    g.num_kb = I / kBK;
    g.n_out = H;
    g.up_off = 0;
    g.out = fuse_k1 ? static_cast<void*>(Y) : static_cast<void*>(Yp);
    g.ldo = H;
    g.status = status;
    if (fuse_k1) {
      g.gather_perm = b.perm;
      g.gather_k = 1;
      g.gather_rows = T;  // the extent of G and of Y's rows
      g.gate = G;
    }
    const long long tiles = static_cast<long long>(mt_bound) * g.n_tiles;
    const int grid = tiles < num_sms() ? static_cast<int>(tiles) : num_sms();
    const GemmKind kind = fuse_k1 ? kGemmCombineK1 : kGemmPlain;
    if ((e = launch_gemm(kind, maps, g, grid, s)) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (fuse_k1)
    e = launch_zero_dropped_rows(b.inv, T, H, Y, s);
  else
    e = launch_combine(Yp, b.inv, G, b.row_off, T, k, H, E, p->has_shared, Y, s);
  if (e == cudaSuccess) e = mark(4);
  return cuda_status(e);
}

extern "C" {

moe_status moe_forward_timed(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                             const float* G, const uint16_t* W1, const uint16_t* W2,
                             const uint16_t* Ws1, const uint16_t* Ws2, uint16_t* Y, void* ws,
                             size_t ws_bytes, void* stream, void* const* stage_events) {
  return forward_impl(p, X, E_ids, G, W1, W2, Ws1, Ws2, Y, ws, ws_bytes, stream, stage_events,
                      nullptr);
}

moe_status moe_forward(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                       const float* G, const uint16_t* W1, const uint16_t* W2,
                       const uint16_t* Ws1, const uint16_t* Ws2, uint16_t* Y, void* ws,
                       size_t ws_bytes, void* stream) {
  return moe_forward_timed(p, X, E_ids, G, W1, W2, Ws1, Ws2, Y, ws, ws_bytes, stream, nullptr);
}

size_t moe_workspace_size_a8w8(const moe_params* p) {
  if (check_params(p) != MOE_OK) return 0;
  return layout_a8w8(*p).total;
}

moe_status moe_forward_a8w8(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                            const float* G, const int8_t* W1q, const float* S1,
                            const int8_t* W2q, const float* S2, uint16_t* Y, void* ws,
                            size_t ws_bytes, void* stream, void* const* stage_events) {
  moe_status st = check_params(p);
  if (st != MOE_OK) return st;
  if (p->has_shared) return MOE_ERR_UNSUPPORTED;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 ||
      ws_bytes < layout_a8w8(*p).total)
    return MOE_ERR_WORKSPACE;
  if (p->T == 0) return MOE_OK;
  if (!X || !E_ids || !G || !W1q || !S1 || !W2q || !S2 || !Y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W1q) || !aligned16(W2q) || !aligned16(Y)) return MOE_ERR_INVALID_ARG;

  const WsLayoutQ L = layout_a8w8(*p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = at<int>(ws, L.status);
  DispatchBufs b;
  b.chunk_cnt = at<int>(ws, L.chunk_cnt);
  b.counts = at<int>(ws, L.counts);
  b.row_off = at<int>(ws, L.row_off);
  b.tile_off = at<int>(ws, L.tile_off);
  b.perm = at<int>(ws, L.perm);
  b.inv = at<int>(ws, L.inv);
  b.nchunk = dispatch_chunks(p->T * p->k);
  set_tile_split(&b, p->E);
  // The A8W8 kernel is bound by its MMA loop and its code conversion, not by
  // the weight stream: the interleaved order left its time unchanged and made
  // Linear1 read its expert-ordered code rows from DRAM again (14.0 against
  // 12.6 GB on the 384-expert layer), so it keeps the group order
  b.dense_mt = 0;
  const int T = p->T, H = p->H, E = p->E, k = p->k, I = p->I;
  const int A = T * k;
  uint16_t* Xq = at<uint16_t>(ws, L.xq);
  float* sX = at<float>(ws, L.sx);
  float* Act = at<float>(ws, L.act);
  uint16_t* Aq = at<uint16_t>(ws, L.aq);
  float* sA = at<float>(ws, L.sa);
  float* Yp = at<float>(ws, L.yp);
  auto mark = [&](int i) -> cudaError_t {
    if (stage_events == nullptr || stage_events[i] == nullptr) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s);
  };
  const int mt_bound = (A + kBM - 1) / kBM + E;

  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = launch_dispatch(E_ids, T, k, E, 0, b, status, s);
  if (e == cudaSuccess) e = launch_quant_rows_bf16(X, T, H, Xq, sX, b.inv, k, s);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  // Linear1: C = Q_e W1q[e]^T on the token codes in expert order (TMA),
  // dequantised, SwiGLU, fp32 out; the weights are the MMA's A operand in TMEM
  {
    CUtensorMap mw, mb;
    if (!make_map_rows(&mb, Xq, A, H) || !make_map_i8_rows(&mw, W1q, E, 2LL * I, H)) return MOE_ERR_CUDA;
    GemmParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.tile_off = b.tile_off;
    set_schedule(&g, b);
    g.num_groups = E;
    g.shared_group = -1;
    g.n_tiles = (I + 127) / 128;
    g.num_kb = H / kBK;
    g.n_out = I;
    g.up_off = I;
    g.out = Act;
    g.ldo = I;
    g.scale_col = S1;
    g.scale_ld = 2LL * I;
    g.scale_row = sX;
    g.status = status;
    const long long tiles = static_cast<long long>(mt_bound) * g.n_tiles;
    const int grid = tiles < num_sms() ? static_cast<int>(tiles) : num_sms();
    if (launch_gemm_q8(true, mw, mb, g, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(2) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // per-row re-quantisation of the SwiGLU output, then Linear2
  if (launch_quant_rows_f32(Act, b.row_off + E, A, I, Aq, sA, s) != cudaSuccess) return MOE_ERR_CUDA;
  {
    CUtensorMap mw, mb;
    if (!make_map_rows(&mb, Aq, A, I) || !make_map_i8_rows(&mw, W2q, E, H, I)) return MOE_ERR_CUDA;
    GemmParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.tile_off = b.tile_off;
    set_schedule(&g, b);
    g.num_groups = E;
    g.shared_group = -1;
    g.n_tiles = (H + 255) / 256;
    g.num_kb = I / kBK;
    g.n_out = H;
    g.out = Yp;  // bf16 rows
    g.out_bf16 = 1;
    g.ldo = H;
    g.scale_col = S2;
    g.scale_ld = H;
    g.scale_row = sA;
    g.status = status;
    const long long tiles = static_cast<long long>(mt_bound) * g.n_tiles;
    const int grid = tiles < num_sms() ? static_cast<int>(tiles) : num_sms();
    if (launch_gemm_q8(false, mw, mb, g, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;
  }
  e = launch_combine_bf16(reinterpret_cast<const uint16_t*>(Yp), b.inv, G, b.row_off, T, k, H, E, 0, Y, s);
  if (e == cudaSuccess) e = mark(4);
  return cuda_status(e);
}

size_t moe_workspace_size_train(const moe_params* p) {
  if (check_params(p) != MOE_OK) return 0;
  return layout_train(*p).total;
}

moe_status moe_forward_train(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                             const float* G, const uint16_t* W1, const uint16_t* W2,
                             const uint16_t* Ws1, const uint16_t* Ws2, uint16_t* Y, void* ws,
                             size_t ws_bytes, void* stream) {
  moe_status st = check_params(p);
  if (st != MOE_OK) return st;
  if (ws == nullptr || ws_bytes < layout_train(*p).total) return MOE_ERR_WORKSPACE;
  return forward_impl(p, X, E_ids, G, W1, W2, Ws1, Ws2, Y, ws, ws_bytes, stream, nullptr,
                      at<uint16_t>(ws, layout_train(*p).h));
}

moe_status moe_backward(const moe_params* p, const uint16_t* X, const uint16_t* Wg,
                        const int32_t* E_ids, const float* G, const uint16_t* W1,
                        const uint16_t* W2, const uint16_t* Ws1, const uint16_t* Ws2,
                        const uint16_t* dY, uint16_t* dX, float* dWg, float* dW1, float* dW2,
                        float* dWs1, float* dWs2, float* dG, void* ws, size_t ws_bytes,
                        void* stream, void* const* stage_events) {
  moe_status st = check_params(p);
  if (st != MOE_OK) return st;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 ||
      ws_bytes < layout_train(*p).total)
    return MOE_ERR_WORKSPACE;
  if (p->E % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (p->T == 0) return MOE_OK;
  if (!X || !Wg || !E_ids || !G || !W1 || !W2 || !dY || !dX || !dWg || !dW1 || !dW2)
    return MOE_ERR_INVALID_ARG;
  if (p->has_shared && (!Ws1 || !Ws2 || !dWs1 || !dWs2)) return MOE_ERR_INVALID_ARG;
  const void* al[] = {X, Wg, W1, W2, dY, dX, dWg, dW1, dW2};
  for (const void* q : al)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (p->has_shared && (!aligned16(Ws1) || !aligned16(Ws2) || !aligned16(dWs1) || !aligned16(dWs2)))
    return MOE_ERR_INVALID_ARG;

  const WsLayoutTrain L = layout_train(*p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = at<int>(ws, L.f.status);
  const DispatchBufs b = dispatch_bufs(p, ws, L.f);
  const int T = p->T, H = p->H, E = p->E, k = p->k, I = p->I;
  const int A = T * k;
  const int sh = p->has_shared ? 1 : 0;
  const int R = A + (sh ? T : 0);
  const int groups = E + sh;
  const int mt_bound = (A + kBM - 1) / kBM + E + (sh ? (T + kBM - 1) / kBM : 0);
  uint16_t* Act = at<uint16_t>(ws, L.f.act);
  float* Yp = at<float>(ws, L.f.yp);
  float* dXp = Yp;  // Yp is read by the un-permute backward before Linear1's dgrad writes here
  uint16_t* Hs = at<uint16_t>(ws, L.h);
  uint16_t* dYp = at<uint16_t>(ws, L.dyp);
  uint16_t* dH = at<uint16_t>(ws, L.dh);
  uint16_t* Xp = at<uint16_t>(ws, L.xp);
  float* dXr = at<float>(ws, L.dxr);
  uint16_t* dl = at<uint16_t>(ws, L.dl);
  float* dGw = dG != nullptr ? dG : at<float>(ws, L.dg);
  int* koff = at<int>(ws, L.koff);
  float* logits = at<float>(ws, L.f.logits);
  auto mark = [&](int i) -> cudaError_t {
    if (stage_events == nullptr || stage_events[i] == nullptr) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s);
  };
  auto grid_of = [&](long long tiles) { return tiles < num_sms() ? static_cast<int>(tiles) : num_sms(); };
  cudaError_t e = mark(0);
  // un-permute backward and the permuted token rows
  if (e == cudaSuccess) e = cudaMemsetAsync(dGw, 0, static_cast<size_t>(A) * sizeof(float), s);
  if (e == cudaSuccess)
    e = launch_unpermute_bwd(dY, G, b.perm, b.row_off, Yp, R, k, H, E, sh, dYp, dGw, s);
  if (e == cudaSuccess) e = launch_gather_rows(X, b.perm, b.row_off, R, k, H, E, sh, Xp, s);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  // dgrad of Linear2 with the SwiGLU backward: dH from dYp W2[e]^T and H
  {
    CUtensorMap ma, mb, mb2;
    bool ok = make_map_bf16_2d(&ma, dYp, R, H, 64, kBM) && make_map_bf16_kmajor_b(&mb, W2, E, I, H);
    if (ok) ok = sh ? make_map_bf16_kmajor_b(&mb2, Ws2, 1, I, H) : (mb2 = mb, true);
    if (!ok) return MOE_ERR_CUDA;
    BwdParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.tile_off = b.tile_off;
    g.num_groups = groups;
    g.shared_group = sh ? E : -1;
    g.n_tiles = (I + 255) / 256;
    g.num_kb = H / kBK;
    g.N = I;
    g.out = dH;
    g.ldo = 2LL * I;
    g.h_in = Hs;
    g.up_off = I;
    g.status = status;
    if (launch_gemm_bwd(false, false, kBwdSwiGLU, false, ma, mb, mb2, g,
                        grid_of(static_cast<long long>(mt_bound) * g.n_tiles), s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  // dgrad of Linear1: dXp = dH W1[e]^T, fp32
  {
    CUtensorMap ma, mb, mb2;
    bool ok = make_map_bf16_2d(&ma, dH, R, 2LL * I, 64, kBM) && make_map_bf16_kmajor_b(&mb, W1, E, H, 2LL * I);
    if (ok) ok = sh ? make_map_bf16_kmajor_b(&mb2, Ws1, 1, H, 2LL * I) : (mb2 = mb, true);
    if (!ok) return MOE_ERR_CUDA;
    BwdParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.tile_off = b.tile_off;
    g.num_groups = groups;
    g.shared_group = sh ? E : -1;
    g.n_tiles = (H + 255) / 256;
    g.num_kb = 2 * I / kBK;
    g.N = H;
    g.out = dXp;
    g.ldo = H;
    g.status = status;
    if (launch_gemm_bwd(false, false, kBwdF32, false, ma, mb, mb2, g,
                        grid_of(static_cast<long long>(mt_bound) * g.n_tiles), s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (mark(2) != cudaSuccess) return MOE_ERR_CUDA;
  // weight gradients: dW2[e] = Act_e^T dYp_e, dW1[e] = Xp_e^T dH_e (shared group -> dWs*)
  for (int w = 0; w < 2; ++w) {
    const int M = w == 0 ? I : H, N = w == 0 ? H : 2 * I;
    CUtensorMap ma, mb;
    const uint16_t* Aop = w == 0 ? Act : Xp;
    const uint16_t* Bop = w == 0 ? dYp : dH;
    if (!make_map_bf16_2d(&ma, Aop, R, M, 64, 64) || !make_map_bf16_2d(&mb, Bop, R, N, 64, 64))
      return MOE_ERR_CUDA;
    BwdParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.num_groups = groups;
    g.shared_group = sh ? E : -1;
    g.m_tiles = (M + kBM - 1) / kBM;
    g.n_tiles = (N + 255) / 256;
    g.M = M;
    g.N = N;
    g.out = w == 0 ? dW2 : dW1;
    g.out2 = w == 0 ? dWs2 : dWs1;
    g.out_group_stride = static_cast<long long>(M) * N;
    g.ldo = N;
    g.status = status;
    if (launch_gemm_bwd(true, true, kBwdF32, true, ma, mb, mb, g,
                        grid_of(static_cast<long long>(groups) * g.m_tiles * g.n_tiles), s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;
  // router backward: logits again, dL/dlogits, dWg = X^T dl, dXr = dl Wg^T
  if ((st = run_router_gemm(p, X, Wg, logits, status, s)) != MOE_OK) return st;
  if (launch_router_bwd(logits, E_ids, dGw, T, E, k, p->score_fn, p->alpha, p->renorm, dl, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  {
    const int kroff[2] = {0, T};
    if (cudaMemcpyAsync(koff, kroff, sizeof(kroff), cudaMemcpyHostToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    CUtensorMap ma, mb;
    if (!make_map_bf16_2d(&ma, X, T, H, 64, 64) || !make_map_bf16_2d(&mb, dl, T, E, 64, 64))
      return MOE_ERR_CUDA;
    BwdParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = koff;
    g.num_groups = 1;
    g.shared_group = -1;
    g.m_tiles = (H + kBM - 1) / kBM;
    g.n_tiles = (E + 255) / 256;
    g.M = H;
    g.N = E;
    g.out = dWg;
    g.ldo = E;
    g.status = status;
    if (launch_gemm_bwd(true, true, kBwdF32, true, ma, mb, mb, g, grid_of(g.m_tiles * g.n_tiles), s) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  }
  {
    CUtensorMap ma, mb;
    if (!make_map_bf16_2d(&ma, dl, T, E, 64, kBM) || !make_map_bf16_kmajor_b(&mb, Wg, 1, H, E))
      return MOE_ERR_CUDA;
    BwdParams g;
    memset(&g, 0, sizeof(g));
    g.dense_rows = T;
    g.num_groups = 1;
    g.shared_group = -1;
    g.n_tiles = (H + 255) / 256;
    g.num_kb = (E + kBK - 1) / kBK;
    g.N = H;
    g.out = dXr;
    g.ldo = H;
    g.status = status;
    if (launch_gemm_bwd(false, false, kBwdF32, false, ma, mb, mb, g,
                        grid_of(static_cast<long long>((T + kBM - 1) / kBM) * g.n_tiles), s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  e = launch_dx_reduce(dXp, b.inv, b.row_off, dXr, T, k, H, E, sh, dX, s);
  if (e == cudaSuccess) e = mark(4);
  return cuda_status(e);
}

moe_status moe_quantize_mx(int32_t fmt, const uint16_t* X, int32_t rows, int32_t cols,
                           uint8_t* Q, uint8_t* S, void* stream) {
  if (fmt != MOE_MX_E4M3 && fmt != MOE_MX_E5M2 && fmt != MOE_MX_E2M1) return MOE_ERR_INVALID_ARG;
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!X || !Q || !S || !aligned16(X) || !aligned16(Q)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_mx_quant_rows(fmt, X, rows, cols, Q, S, nullptr, 0,
                                          static_cast<cudaStream_t>(stream)));
}

size_t moe_workspace_size_mx(const moe_params* p) {
  if (check_params(p) != MOE_OK) return 0;
  return layout_mx(*p).total;
}

moe_status moe_forward_mx(const moe_params* p, int32_t fmt, int32_t wfmt, const uint16_t* X,
                          const int32_t* E_ids, const float* G, const uint8_t* W1,
                          const uint8_t* S1, const uint8_t* W2, const uint8_t* S2, uint16_t* Y,
                          void* ws, size_t ws_bytes, void* stream, void* const* stage_events) {
  moe_status st = check_params(p);
  if (st != MOE_OK) return st;
  auto known = [](int f) { return f == MOE_MX_E4M3 || f == MOE_MX_E5M2 || f == MOE_MX_E2M1; };
  if (!known(fmt) || !known(wfmt)) return MOE_ERR_INVALID_ARG;
  if (!mx_pair_supported(fmt, wfmt)) return MOE_ERR_UNSUPPORTED;
  const bool a4 = fmt == MOE_MX_E2M1, w4 = wfmt == MOE_MX_E2M1;
  if (p->has_shared) return MOE_ERR_UNSUPPORTED;
  if (p->H % kMxBK != 0 || p->I % kMxBK != 0) return MOE_ERR_UNSUPPORTED;
  // E2M1 x E2M1 runs kind::mxf4 on packed tiles when both K dims fill whole
  // 256-code k-blocks; otherwise kind::mxf8f6f4 on spread tiles
  const bool packed = a4 && w4 && p->H % kMxBKPacked == 0 && p->I % kMxBKPacked == 0;
  const int la = packed ? kMxFp4Packed : (a4 ? kMxFp4Spread : kMxFp8);
  const int lw = packed ? kMxFp4Packed : (w4 ? kMxFp4Spread : kMxFp8);
  const int kbk = packed ? kMxBKPacked : kMxBK;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 ||
      ws_bytes < layout_mx(*p).total)
    return MOE_ERR_WORKSPACE;
  if (p->T == 0) return MOE_OK;
  if (!X || !E_ids || !G || !W1 || !S1 || !W2 || !S2 || !Y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W1) || !aligned16(W2) || !aligned16(Y)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(S1) & 3u) != 0 || (reinterpret_cast<uintptr_t>(S2) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;

  const WsLayoutMX L = layout_mx(*p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = at<int>(ws, L.status);
  DispatchBufs b;
  b.chunk_cnt = at<int>(ws, L.chunk_cnt);
  b.counts = at<int>(ws, L.counts);
  b.row_off = at<int>(ws, L.row_off);
  b.tile_off = at<int>(ws, L.tile_off);
  b.perm = at<int>(ws, L.perm);
  b.inv = at<int>(ws, L.inv);
  b.nchunk = dispatch_chunks(p->T * p->k);
  set_tile_split(&b, p->E);
  // 8-bit codes against spread E2M1 weights: that kernel is bound by its MMA
  // loop rather than by the weight stream, so there is nothing to overlap, and
  // the interleaved order measured 2.4% slower on it; it keeps the group order
  if (!a4 && w4) b.dense_mt = 0;
  const int T = p->T, H = p->H, E = p->E, k = p->k, I = p->I;
  const int A = T * k;
  uint8_t* Xq = at<uint8_t>(ws, L.xq);
  uint8_t* SX = at<uint8_t>(ws, L.sx);
  uint8_t* Uq = at<uint8_t>(ws, L.uq);
  uint8_t* SU = at<uint8_t>(ws, L.su);
  float* Yp = at<float>(ws, L.yp);
  auto mark = [&](int i) -> cudaError_t {
    if (stage_events == nullptr || stage_events[i] == nullptr) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s);
  };
  const int mt_bound = (A + kBM - 1) / kBM + E;

  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = launch_dispatch(E_ids, T, k, E, 0, b, status, s);
  // each token row quantised once and written to its k rows in expert order
  if (e == cudaSuccess) e = launch_mx_quant_rows(fmt, X, T, H, Xq, SX, b.inv, k, s);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  // Linear1 + SwiGLU + Q_MX on the token codes in expert order
  {
    GemmMaps maps;
    if (!make_map_mx_rows(&maps.a, Xq, A, H, la) || !make_map_mx_weights(&maps.b, W1, E, 2LL * I, H, 128, lw))
      return MOE_ERR_CUDA;
    maps.a2 = maps.a;
    maps.b2 = maps.b;
    GemmParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.tile_off = b.tile_off;
    set_schedule(&g, b);
    g.num_groups = E;
    g.shared_group = -1;
    g.n_tiles = (I + 127) / 128;
    g.num_kb = H / kbk;
    g.n_out = I;
    g.up_off = I;
    g.out = Uq;
    g.ldo = a4 ? I / 2 : I;  // bytes per code row
    g.out_sf = SU;
    g.out_sf_ld = I / 32;
    g.sfa = SX;
    g.sfb = S1;
    g.sf_ld = H / 32;
    g.sfb_ld = 2LL * I * (H / 32);
    g.sf_vec = (g.sf_ld % 16 == 0 && g.sfb_ld % 16 == 0 && aligned16(g.sfa) && aligned16(g.sfb)) ? 1 : 0;
    g.status = status;
    const long long tiles = static_cast<long long>(mt_bound) * g.n_tiles;
    const int grid = tiles < num_sms() ? static_cast<int>(tiles) : num_sms();
    if (launch_gemm_mx(true, fmt, wfmt, packed, maps, g, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(2) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // Linear2 on the re-quantised SwiGLU rows, bf16 rows out
  {
    GemmMaps maps;
    if (!make_map_mx_rows(&maps.a, Uq, A, I, la) || !make_map_mx_weights(&maps.b, W2, E, H, I, 256, lw))
      return MOE_ERR_CUDA;
    maps.a2 = maps.a;
    maps.b2 = maps.b;
    GemmParams g;
    memset(&g, 0, sizeof(g));
    g.row_off = b.row_off;
    g.tile_off = b.tile_off;
    set_schedule(&g, b);
    g.num_groups = E;
    g.shared_group = -1;
    g.n_tiles = (H + 255) / 256;
    g.num_kb = I / kbk;
    g.n_out = H;
    g.out = Yp;
    g.out_bf16 = 1;
    g.ldo = H;
    g.sfa = SU;
    g.sfb = S2;
    g.sf_ld = I / 32;
    g.sfb_ld = static_cast<long long>(H) * (I / 32);
    g.sf_vec = (g.sf_ld % 16 == 0 && g.sfb_ld % 16 == 0 && aligned16(g.sfa) && aligned16(g.sfb)) ? 1 : 0;
    g.status = status;
    const long long tiles = static_cast<long long>(mt_bound) * g.n_tiles;
    const int grid = tiles < num_sms() ? static_cast<int>(tiles) : num_sms();
    if (launch_gemm_mx(false, fmt, wfmt, packed, maps, g, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;
  }
  e = launch_combine_bf16(reinterpret_cast<const uint16_t*>(Yp), b.inv, G, b.row_off, T, k, H, E, 0, Y, s);
  if (e == cudaSuccess) e = mark(4);
  return cuda_status(e);
}

}  // extern "C"
