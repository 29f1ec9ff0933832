// Internal launcher declarations shared by the CSA2 translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/csa2.h"
#include "csa2_device.cuh"

namespace csa2 {

// Launch with programmatic stream serialization: the grid may be scheduled
// while the previous kernel on the stream finishes; every kernel of the
// library waits for its predecessor (griddep_wait) before allocating tensor
// memory and before any global load whose value a kernel of the library may
// write -- before the wait a kernel issues L2 prefetch hints and reads only
// the attention's query and window rows, which only csa2_swa_encode writes,
// and that kernel lets its successor start only at its completion.
// cluster_x > 0 adds a cluster shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, int cluster_x,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster_x > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Format of the indexer cache under a layer configuration.
inline int idx_dtype(const csa2_cfg& cfg) {
  return (cfg.cache_dtype == CSA2_CACHE_FP4 && (cfg.formats & CSA2_FMT_IDX_68B)) ? CSA2_CACHE_FP4_S32 : cfg.cache_dtype;
}

inline CacheView view_of(const csa2_cache& c) {
  return CacheView{static_cast<uint8_t*>(c.data), static_cast<uint8_t*>(c.scales), c.block_table,
                   c.max_pages, c.num_pages};
}

cudaError_t launch_compress(const csa2_cfg& cfg, int B, int T, const uint16_t* x, const int64_t* pos0,
                            const float* merge_w, const uint16_t* w_idx, const csa2_cache& main_c,
                            const csa2_cache& idx_c, int32_t* n_entries, int32_t* status,
                            cudaStream_t stream);

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Tensor-core indexer scores for queries [q0, q0 + nq): every visible entry
// (pool == NULL) or the entries of each query's HSI pool.
cudaError_t launch_score_tc(const csa2_cfg& cfg, int q0, int nq, int Tq, const uint16_t* q_idx, const float* head_w,
                            const int64_t* q_pos, const csa2_cache& idx_c, const int32_t* n_entries,
                            int64_t max_entries, const int32_t* pool, float* scores, int64_t stride, float* bmax,
                            uint32_t* krange, int kr_stride, int* n_slots, int32_t* status, int num_sms,
                            cudaStream_t stream);

// Scoring CTAs per query (key-range slots written) of launch_score_tc for
// the same arguments.
int score_slots_used(const csa2_cfg& cfg, int q0, int nq, int Tq, int64_t max_entries, bool gather, int num_sms);

// Key-range slots per query in the indexer workspace: one per scoring CTA
// (at least four 128-entry tiles each).
inline int score_range_slots(int64_t tiles) { return (int)((tiles + 3) / 4); }

// Per-query workspace bytes of the indexer (scores + HSI block maxima).
size_t index_query_ws_bytes(const csa2_cfg& cfg, int max_entries, bool reindex);

// Host-side checks of csa2_index_topk's arguments, in the order that entry
// point applies them; *empty is set when there is nothing to launch.
int32_t check_index(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q_idx, const float* head_w,
                    const int64_t* q_pos, const csa2_cache* idx_cache, const int32_t* n_entries,
                    int32_t max_entries, const int32_t* pool, const int32_t* topk_out, const int32_t* pool_out,
                    const void* workspace, size_t workspace_bytes, const int32_t* status, bool* empty);

cudaError_t launch_index_topk(const csa2_cfg& cfg, int B, int Tq, const uint16_t* q_idx,
                              const float* head_w, const int64_t* q_pos, const csa2_cache& idx_c,
                              const int32_t* n_entries, int max_entries, const int32_t* pool,
                              int32_t* topk_out, int32_t* pool_out, void* ws, size_t ws_bytes,
                              int32_t* status, cudaStream_t stream);

// The two halves of launch_index_topk for a workspace that holds every
// query: the scores (and HSI block maxima when hsi_out) of all B * Tq
// queries, then the selection from them.
cudaError_t launch_index_score(const csa2_cfg& cfg, int B, int Tq, const uint16_t* q_idx, const float* head_w,
                               const int64_t* q_pos, const csa2_cache& idx_c, const int32_t* n_entries,
                               int max_entries, const int32_t* pool, bool hsi_out, void* ws, size_t ws_bytes,
                               int32_t* status, cudaStream_t stream);
cudaError_t launch_index_select(const csa2_cfg& cfg, int B, int Tq, const int64_t* q_pos, const int32_t* n_entries,
                                int max_entries, const int32_t* pool, int32_t* topk_out, int32_t* pool_out, void* ws,
                                size_t ws_bytes, cudaStream_t stream);

cudaError_t launch_attend(const csa2_cfg& cfg, int B, int Tq, const uint16_t* q, const csa2_cache& main_c,
                          const int32_t* n_entries, const int32_t* topk, const void* swa, int S,
                          const int32_t* swa_len, const int64_t* swa_pos0, const int64_t* q_pos,
                          float scale, float* out, float* lse, int32_t* status, bool ids_early, cudaStream_t stream);

// Whether the attention kernel fits top-k + window rows (TMEM and shared memory).
bool attend_tc_supported(int topk, int window);

// Whether csa2_attend takes the row-tile kernel (the one that reads MXFP8 window rows).
bool attend_rows_path(int topk, int window);

cudaError_t launch_swa_encode(int B, int T, const uint16_t* x, const int64_t* row0, void* rows, int S,
                              int32_t* status, cudaStream_t stream);

cudaError_t launch_gather_dequant(const csa2_cache& c, int cache_dtype, int B, int n, const int32_t* ids,
                                  float* out, int32_t* status, cudaStream_t stream);

}  // namespace csa2
