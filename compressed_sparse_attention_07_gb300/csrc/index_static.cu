// csa2_index_topk_static: the indexer / top-k entry point for callers that
// cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a serving engine or plugin
// host that owns every device byte through its own fixed pool and hands the
// library no allocator, or a latency-critical decode loop where cudaMalloc /
// cudaFree would synchronise the device.  csa2_index_topk needs a workspace
// for the per-entry scores and HSI block maxima; this variant takes that
// scratch from one static device array compiled into the library instead.
//
// The array (kStaticScratchBytes) exists on every GPU that loads the
// library, for the life of the process.  All calls on a device share it and
// it keeps whatever the last call left there; the kernels write every score
// before reading it, so nothing has to be cleared between calls.  Two calls
// whose kernels overlap on the GPU (different streams without ordering, or
// different host threads) race on the array: order them on one stream.
#include <mutex>

#include <cuda.h>

#include "internal.h"

namespace csa2 {
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB
constexpr int kMaxContexts = 64;

static __device__ __align__(256) uint8_t g_index_scratch[kStaticScratchBytes];

// The array's device address depends on the context the module is loaded
// in (one per device for the primary context, another after a device reset
// or in a context the caller created), so resolved addresses are kept per
// context, keyed by the driver's context id (never reused in a process).
using CtxGetCurrent = CUresult (*)(CUcontext*);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long*);

std::mutex g_scratch_mu;
bool g_entry_looked_up = false;
CtxGetCurrent g_ctx_current = nullptr;
CtxGetId g_ctx_id = nullptr;
unsigned long long g_ctx_ids[kMaxContexts] = {};
void* g_ctx_addr[kMaxContexts] = {};
int g_n_ctx = 0;

// Device address of g_index_scratch in the current context.  In host code
// the array's name is only a host-side stand-in, so the address has to come
// from cudaGetSymbolAddress; it is asked once per context (the first call in
// a context also loads the module there, so make it before any capture).
cudaError_t scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_entry_looked_up) {
    g_entry_looked_up = true;
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
      g_ctx_current = reinterpret_cast<CtxGetCurrent>(f1);
      g_ctx_id = reinterpret_cast<CtxGetId>(f2);
    }
    (void)cudaGetLastError();
  }
  // make sure a context is current (the runtime creates the primary one)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned long long id = 0;
  bool keyed = false;
  if (g_ctx_current && g_ctx_id) {
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) == CUDA_SUCCESS && ctx && g_ctx_id(ctx, &id) == CUDA_SUCCESS) keyed = true;
  }
  if (keyed) {
    for (int i = 0; i < g_n_ctx; ++i)
      if (g_ctx_ids[i] == id) {
        *out = g_ctx_addr[i];
        return cudaSuccess;
      }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_index_scratch);
  if (e != cudaSuccess) return e;
  if (keyed && g_n_ctx < kMaxContexts) {
    g_ctx_ids[g_n_ctx] = id;
    g_ctx_addr[g_n_ctx] = p;
    ++g_n_ctx;
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace csa2

extern "C" {

size_t csa2_index_static_scratch_bytes(void) { return csa2::kStaticScratchBytes; }

int32_t csa2_index_topk_static(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q_idx,
                               const float* head_w, const int64_t* q_pos, const csa2_cache* idx_cache,
                               const int32_t* n_entries, int32_t max_entries, const int32_t* pool,
                               int32_t* topk_out, int32_t* pool_out, int32_t* status, void* stream) {
  using namespace csa2;
  // the same checks, in the same order, as csa2_index_topk with a workspace
  // of the array's size: a bad configuration or argument is reported as
  // such, and a query whose scratch exceeds the array as CSA2_ERR_CAPACITY,
  // all before anything is touched (the stand-in pointer only has the
  // array's alignment; it is never dereferenced)
  bool empty;
  const int32_t rc = check_index(cfg, B, Tq, q_idx, head_w, q_pos, idx_cache, n_entries, max_entries, pool, topk_out,
                                 pool_out, reinterpret_cast<const void*>(uintptr_t{256}), kStaticScratchBytes, status,
                                 &empty);
  if (rc != CSA2_OK || empty) return rc;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return CSA2_ERR_CUDA;
  const cudaError_t e = launch_index_topk(*cfg, B, Tq, q_idx, head_w, q_pos, *idx_cache, n_entries, max_entries, pool,
                                          topk_out, pool_out, scratch, kStaticScratchBytes, status,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

}  // extern "C"
