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

#include "internal.h"

namespace csa2 {
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_index_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_index_scratch on the current device, resolved once per
// device.  In host code the array's name is only a host-side stand-in, so the
// address has to come from cudaGetSymbolAddress.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_index_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
  if (!cfg) return CSA2_ERR_INVALID_ARG;
  if (B < 0 || Tq < 0 || max_entries < 0) return CSA2_ERR_INVALID_ARG;
  if (cfg->hsi_blocks < 0 || cfg->hsi_blocks > 4096) return CSA2_ERR_UNSUPPORTED;
  // one query's scores (and HSI block maxima) must fit in the static array;
  // larger requests are refused before anything is touched
  if (index_query_ws_bytes(*cfg, max_entries, pool != nullptr) > kStaticScratchBytes) return CSA2_ERR_CAPACITY;
  if (B == 0 || Tq == 0) return CSA2_OK;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return CSA2_ERR_CUDA;
  return csa2_index_topk(cfg, B, Tq, q_idx, head_w, q_pos, idx_cache, n_entries, max_entries, pool, topk_out,
                         pool_out, scratch, kStaticScratchBytes, status, stream);
}

}  // extern "C"
