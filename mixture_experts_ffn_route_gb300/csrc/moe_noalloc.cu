// moe_dispatch_noalloc: the dispatch (counts, offsets, permutation) for callers
// that cannot hand the library a workspace.
//
// Who needs it: code that may not allocate device memory at the point where it
// routes tokens -- for example a serving loop whose device memory is entirely
// owned by another allocator, or a latency-critical path where a cudaMalloc or
// cudaFree (which can synchronise the whole device) is not acceptable.  Such a
// caller still owns its inputs and outputs; only the scratch moves into the
// library, as one fixed array in device memory.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes (about
// 1.2 MB: per-chunk counts, tile offsets and the inverse permutation for up to
// 262144 assignments and 512 experts).  Every GPU that loads this library
// holds it until the process exits.  All calls share it and it keeps the last call's contents, so calls
// that overlap on the GPU (two streams, or two host threads) race; serialise
// them.  The kernels themselves are the ones moe_dispatch runs.
#include <mutex>

#include "moe_common.cuh"
#include "moe_ffn.h"
#include "moe_internal.h"

namespace moe {

constexpr int kNoAllocMaxAssignments = 262144;  // T * k
constexpr int kNoAllocMaxExperts = 512;
constexpr int kNoAllocMaxChunks = kNoAllocMaxAssignments / 4096;  // dispatch chunk = 4096
constexpr size_t kChunkCntBytes = sizeof(int) * kNoAllocMaxChunks * kNoAllocMaxExperts;
constexpr size_t kTileOffBytes = 4096;
constexpr size_t kInvBytes = sizeof(int) * kNoAllocMaxAssignments;
constexpr size_t kNoAllocScratchBytes = kChunkCntBytes + kTileOffBytes + kInvBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// The driver's cuCtxGetCurrent and cuCtxGetId, found through the runtime (no
// link-time dependency on the driver library).
static void context_fns(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
  static CtxGetCurrentFn f_cur = nullptr;
  static CtxGetIdFn f_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_cur = reinterpret_cast<CtxGetCurrentFn>(ptr);
    ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_id = reinterpret_cast<CtxGetIdFn>(ptr);
  });
  *cur = f_cur;
  *id = f_id;
}

// Unique id of the calling thread's current context, 0 if there is none (or
// the driver calls are unavailable).  Ids are never reused within a process,
// so a context created after a device reset gets a new one.
static unsigned long long current_context_id() {
  CtxGetCurrentFn cur;
  CtxGetIdFn id;
  context_fns(&cur, &id);
  CUcontext ctx = nullptr;
  unsigned long long v = 0;
  if (cur == nullptr || id == nullptr || cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  return id(ctx, &v) == CUDA_SUCCESS ? v : 0;
}

// Device address of the array in the current context (in host code the
// array's name is only a stand-in, not an address).  It is looked up with
// cudaGetSymbolAddress the first time a context calls, with its device
// current, and kept per context: a device reset ends the context, and the
// next call, from the new context, looks the address up again.
static void* noalloc_scratch_ptr(cudaError_t* err) {
  constexpr int kSlots = 64;
  static std::mutex mu;
  static unsigned long long ids[kSlots] = {0};
  static void* ptrs[kSlots] = {nullptr};
  static int next = 0;
  std::lock_guard<std::mutex> g(mu);
  unsigned long long ctx = current_context_id();
  if (ctx != 0)
    for (int i = 0; i < kSlots; ++i)
      if (ids[i] == ctx) return ptrs[i];
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the device's context current
  if (*err != cudaSuccess) return nullptr;
  ctx = current_context_id();
  if (ctx != 0) {
    ids[next] = ctx;
    ptrs[next] = p;
    next = (next + 1) % kSlots;
  }
  return p;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch_noalloc(const moe_params* p, const int32_t* E_ids,
                                           int32_t* counts, int32_t* offsets, int32_t* perm,
                                           void* stream) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->E <= 0 || p->k <= 0 || p->k > p->E) return MOE_ERR_INVALID_ARG;
  const long long A = static_cast<long long>(p->T) * p->k;
  if (A > kNoAllocMaxAssignments || p->E > kNoAllocMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || (A > 0 && (!E_ids || !perm))) return MOE_ERR_INVALID_ARG;

  cudaError_t err = cudaSuccess;
  unsigned char* base = static_cast<unsigned char*>(noalloc_scratch_ptr(&err));
  if (base == nullptr) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DispatchBufs b;
  b.chunk_cnt = reinterpret_cast<int*>(base);
  b.tile_off = reinterpret_cast<int*>(base + kChunkCntBytes);
  b.tile_doff = nullptr;  // no GEMM follows: the interleaved order is not needed
  b.tile_soff = nullptr;
  b.dense_mt = 0;
  b.inv = reinterpret_cast<int*>(base + kChunkCntBytes + kTileOffBytes);
  b.counts = counts;    // the scan writes counts[0, E) and offsets[0, E]
  b.row_off = offsets;  // straight into the caller's outputs
  b.perm = perm;
  b.nchunk = dispatch_chunks(static_cast<int>(A));
  // Nothing in the array has to start at zero: every word a call reads was
  // written earlier in the same call.  Ids outside [0, E) are dropped; there
  // is no status word here, so they show only as offsets[E] < T * k.
  err = launch_dispatch(E_ids, p->T, p->k, p->E, 0, b, nullptr, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
