// C ABI of the CSA2 library: argument validation on the host, then the
// launches of the compressor, indexer / top-k and attention kernels, and the
// Full / Reindex / Reuse layer dispatcher.  No allocation, no synchronisation.
#include <cstring>

#include "internal.h"

using namespace csa2;

namespace {

bool cfg_supported(const csa2_cfg* c, int32_t* err) {
  if (!c) { *err = CSA2_ERR_INVALID_ARG; return false; }
  if ((c->formats & ~(CSA2_FMT_IDX_68B | CSA2_FMT_SWA_FP8 | CSA2_FMT_IDX_QFP4)) != 0 || !(c->rope_theta > 0.0) ||
      (c->cache_dtype != CSA2_CACHE_FP4 && c->cache_dtype != CSA2_CACHE_BF16) ||
      ((c->formats & CSA2_FMT_IDX_68B) && c->cache_dtype != CSA2_CACHE_FP4)) {
    *err = CSA2_ERR_INVALID_ARG;
    return false;
  }
  if (c->dim != kDim || c->rope_dims != kRope || c->n_heads != kHeads || c->idx_heads != kIdxHeads ||
      c->idx_dim != kIdxDim || c->hsi_block != kHsiBlock || c->topk < 1 || c->topk > 1024 || c->window < 0 ||
      c->window > 512 || !attend_tc_supported(c->topk, c->window) || (c->ratio != 1 && c->ratio != 2) || c->hsi_blocks < 0 || c->hsi_blocks > 4096) {
    *err = CSA2_ERR_UNSUPPORTED;
    return false;
  }
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Alignment the kernels' loads and stores need of a pointer (null passes:
// presence is checked separately).
bool al(const void* p, size_t a) { return !p || aligned(p, a); }

bool cache_ok(const csa2_cache* c, int channels, int dtype) {
  if (!c || !c->data || !c->block_table || c->max_pages <= 0 || c->num_pages <= 0 || c->reserved != 0) return false;
  if (!al(c->block_table, 4)) return false;
  if (c->channels != channels) return false;
  if (dtype != CSA2_CACHE_BF16 && !c->scales) return false;
  // 16-byte alignment of the page bases (128-bit loads)
  if ((reinterpret_cast<uintptr_t>(c->data) & 15) || (c->scales && (reinterpret_cast<uintptr_t>(c->scales) & 15)))
    return false;
  return true;
}

int32_t cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

}  // namespace

int csa2::num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

extern "C" {

size_t csa2_page_bytes(int32_t channels, int32_t cache_dtype, int32_t which) {
  if (channels <= 0 || channels % 16) return 0;
  if (cache_dtype == CSA2_CACHE_FP4) return which == 0 ? (size_t)kPage * channels / 2 : (size_t)kPage * channels / 16;
  if (cache_dtype == CSA2_CACHE_FP4_S32)
    return channels % 32 ? 0 : which == 0 ? (size_t)kPage * channels / 2 : (size_t)kPage * channels / 32;
  if (cache_dtype == CSA2_CACHE_BF16) return which == 0 ? (size_t)kPage * channels * 2 : 0;
  return 0;
}

const char* csa2_status_string(int32_t code) {
  switch (code) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported configuration";
    case CSA2_ERR_CUDA: return "CUDA launch failure";
    case CSA2_ERR_CAPACITY: return "workspace or cache capacity too small";
    case CSA2_ERR_BAD_PAGE: return "block table entry outside the page pool";
    case CSA2_ERR_BAD_INDEX: return "entry id outside the sequence";
    case CSA2_ERR_TIMEOUT: return "device wait timed out";
    case CSA2_ERR_RANGE: return "input beyond the f16 operand range";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace {

// Host-side argument checks of each entry point (nothing is enqueued).
// CSA2_OK means the call would launch; a call with nothing to do reports
// CSA2_OK through *empty.
int32_t check_compress(const csa2_cfg* cfg, int32_t B, int32_t T, const uint16_t* x, const int64_t* pos0,
                       const float* merge_w, const uint16_t* w_idx, const csa2_cache* main_cache,
                       const csa2_cache* idx_cache, const int32_t* n_entries, const int32_t* status, bool* empty) {
  int32_t err;
  *empty = false;
  if (!cfg_supported(cfg, &err)) return err;
  if (B < 0 || T < 0 || T % cfg->ratio) return CSA2_ERR_INVALID_ARG;
  if (B == 0 || T == 0) {
    *empty = true;
    return CSA2_OK;
  }
  if (!x || !pos0 || !merge_w || !w_idx || !n_entries) return CSA2_ERR_INVALID_ARG;
  if (!al(x, 4) || !al(pos0, 8) || !al(merge_w, 4) || !al(w_idx, 8) || !al(n_entries, 4) || !al(status, 4))
    return CSA2_ERR_INVALID_ARG;
  if (!cache_ok(main_cache, kDim, cfg->cache_dtype) || !cache_ok(idx_cache, kIdxDim, idx_dtype(*cfg)))
    return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

}  // namespace

int32_t csa2::check_index(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q_idx, const float* head_w,
                          const int64_t* q_pos, const csa2_cache* idx_cache, const int32_t* n_entries,
                          int32_t max_entries, const int32_t* pool, const int32_t* topk_out, const int32_t* pool_out,
                          const void* workspace, size_t workspace_bytes, const int32_t* status, bool* empty) {
  int32_t err;
  *empty = false;
  if (!cfg_supported(cfg, &err)) return err;
  if (B < 0 || Tq < 0 || max_entries < 0) return CSA2_ERR_INVALID_ARG;
  if (B == 0 || Tq == 0) {
    *empty = true;
    return CSA2_OK;
  }
  if (!q_idx || !q_pos || !n_entries || !topk_out || !workspace) return CSA2_ERR_INVALID_ARG;
  if (!al(q_idx, 16) || !al(head_w, 4) || !al(q_pos, 8) || !al(n_entries, 4) || !al(pool, 4) || !al(topk_out, 4) ||
      !al(pool_out, 4) || !al(status, 4))
    return CSA2_ERR_INVALID_ARG;
  if (!cache_ok(idx_cache, kIdxDim, idx_dtype(*cfg))) return CSA2_ERR_INVALID_ARG;
  if ((int64_t)max_entries > (int64_t)idx_cache->max_pages * kPage) return CSA2_ERR_CAPACITY;
  if (pool && pool_out) return CSA2_ERR_INVALID_ARG;
  if ((pool || pool_out) && cfg->hsi_blocks <= 0) return CSA2_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return CSA2_ERR_INVALID_ARG;
  if (workspace_bytes < index_query_ws_bytes(*cfg, max_entries, pool != nullptr)) return CSA2_ERR_CAPACITY;
  return CSA2_OK;
}

namespace {

int32_t check_attend(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q, const csa2_cache* main_cache,
                     const int32_t* n_entries, const int32_t* topk, const void* swa, int32_t S,
                     const int32_t* swa_len, const int64_t* swa_pos0, const int64_t* q_pos, float scale,
                     const float* out, const float* lse, const int32_t* status, bool* empty) {
  int32_t err;
  *empty = false;
  if (!cfg_supported(cfg, &err)) return err;
  if (B < 0 || Tq < 0 || S < 0) return CSA2_ERR_INVALID_ARG;
  if (B == 0 || Tq == 0) {
    *empty = true;
    return CSA2_OK;
  }
  if (!q || !n_entries || !topk || !q_pos || !out) return CSA2_ERR_INVALID_ARG;
  if (!al(q, 16) || !al(n_entries, 4) || !al(topk, 4) || !al(swa_len, 4) || !al(swa_pos0, 8) || !al(q_pos, 8) ||
      !al(out, 16) || !al(lse, 4) || !al(status, 4))
    return CSA2_ERR_INVALID_ARG;
  if (cfg->window > 0 && (!swa || !swa_len || !swa_pos0 || S == 0 || !aligned(swa, 16))) return CSA2_ERR_INVALID_ARG;
  if (!cache_ok(main_cache, kDim, cfg->cache_dtype)) return CSA2_ERR_INVALID_ARG;
  if (!(scale == scale)) return CSA2_ERR_INVALID_ARG;
  if ((cfg->formats & CSA2_FMT_SWA_FP8) && !attend_rows_path(cfg->topk, cfg->window)) return CSA2_ERR_UNSUPPORTED;
  return CSA2_OK;
}

}  // namespace

extern "C" {

int32_t csa2_compress(const csa2_cfg* cfg, int32_t B, int32_t T, const uint16_t* x, const int64_t* pos0,
                      const float* merge_w, const uint16_t* w_idx, const csa2_cache* main_cache,
                      const csa2_cache* idx_cache, int32_t* n_entries, int32_t* status, void* stream) {
  bool empty;
  const int32_t rc = check_compress(cfg, B, T, x, pos0, merge_w, w_idx, main_cache, idx_cache, n_entries, status, &empty);
  if (rc != CSA2_OK || empty) return rc;
  return cuda_status(launch_compress(*cfg, B, T, x, pos0, merge_w, w_idx, *main_cache, *idx_cache, n_entries, status,
                                     static_cast<cudaStream_t>(stream)));
}

size_t csa2_index_workspace_bytes(const csa2_cfg* cfg, int32_t B, int32_t Tq, int32_t max_entries, int32_t reindex) {
  int32_t err;
  if (!cfg_supported(cfg, &err) || B < 0 || Tq < 0 || max_entries < 0) return 0;
  return (size_t)B * Tq * index_query_ws_bytes(*cfg, max_entries, reindex != 0);
}

int32_t csa2_index_topk(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q_idx, const float* head_w,
                        const int64_t* q_pos, const csa2_cache* idx_cache, const int32_t* n_entries,
                        int32_t max_entries, const int32_t* pool, int32_t* topk_out, int32_t* pool_out,
                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  bool empty;
  const int32_t rc = check_index(cfg, B, Tq, q_idx, head_w, q_pos, idx_cache, n_entries, max_entries, pool, topk_out,
                                 pool_out, workspace, workspace_bytes, status, &empty);
  if (rc != CSA2_OK || empty) return rc;
  return cuda_status(launch_index_topk(*cfg, B, Tq, q_idx, head_w, q_pos, *idx_cache, n_entries, max_entries, pool,
                                       topk_out, pool_out, workspace, workspace_bytes, status,
                                       static_cast<cudaStream_t>(stream)));
}

// The indexer in two calls: checks of csa2_index_topk, plus a workspace
// that holds every query (one scoring and one selection launch).
static int32_t check_split(const csa2_cfg* cfg, int32_t B, int32_t Tq, int32_t max_entries, const int32_t* pool,
                           size_t workspace_bytes) {
  const size_t per_q = index_query_ws_bytes(*cfg, max_entries, pool != nullptr);
  if ((int64_t)B * Tq > 65535) return CSA2_ERR_UNSUPPORTED;
  if (workspace_bytes / per_q < (size_t)B * Tq) return CSA2_ERR_CAPACITY;
  return CSA2_OK;
}

int32_t csa2_index_score(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q_idx, const float* head_w,
                         const int64_t* q_pos, const csa2_cache* idx_cache, const int32_t* n_entries,
                         int32_t max_entries, const int32_t* pool, int32_t hsi, void* workspace,
                         size_t workspace_bytes, int32_t* status, void* stream) {
  bool empty;
  if (hsi && pool) return CSA2_ERR_INVALID_ARG;
  // a stand-in for the outputs (never written here) so that the shared
  // checks apply; an HSI request is checked as a pool output
  const int32_t* fake_out = reinterpret_cast<const int32_t*>(uintptr_t{256});
  int32_t rc = check_index(cfg, B, Tq, q_idx, head_w, q_pos, idx_cache, n_entries, max_entries, pool, fake_out,
                           hsi ? fake_out : nullptr, workspace, workspace_bytes, status, &empty);
  if (rc != CSA2_OK || empty) return rc;
  rc = check_split(cfg, B, Tq, max_entries, pool, workspace_bytes);
  if (rc != CSA2_OK) return rc;
  return cuda_status(launch_index_score(*cfg, B, Tq, q_idx, head_w, q_pos, *idx_cache, n_entries, max_entries, pool,
                                        hsi != 0, workspace, workspace_bytes, status,
                                        static_cast<cudaStream_t>(stream)));
}

int32_t csa2_index_select(const csa2_cfg* cfg, int32_t B, int32_t Tq, const int64_t* q_pos,
                          const csa2_cache* idx_cache, const int32_t* n_entries, int32_t max_entries,
                          const int32_t* pool, int32_t* topk_out, int32_t* pool_out, void* workspace,
                          size_t workspace_bytes, int32_t* status, void* stream) {
  bool empty;
  const uint16_t* fake_q = reinterpret_cast<const uint16_t*>(uintptr_t{256});
  int32_t rc = check_index(cfg, B, Tq, fake_q, nullptr, q_pos, idx_cache, n_entries, max_entries, pool, topk_out,
                           pool_out, workspace, workspace_bytes, status, &empty);
  if (rc != CSA2_OK || empty) return rc;
  rc = check_split(cfg, B, Tq, max_entries, pool, workspace_bytes);
  if (rc != CSA2_OK) return rc;
  return cuda_status(launch_index_select(*cfg, B, Tq, q_pos, n_entries, max_entries, pool, topk_out, pool_out,
                                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

int32_t csa2_attend(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q, const csa2_cache* main_cache,
                    const int32_t* n_entries, const int32_t* topk, const void* swa, int32_t S,
                    const int32_t* swa_len, const int64_t* swa_pos0, const int64_t* q_pos, float scale, float* out,
                    float* lse, int32_t* status, void* stream) {
  bool empty;
  const int32_t rc = check_attend(cfg, B, Tq, q, main_cache, n_entries, topk, swa, S, swa_len, swa_pos0, q_pos, scale,
                                  out, lse, status, &empty);
  if (rc != CSA2_OK || empty) return rc;
  return cuda_status(launch_attend(*cfg, B, Tq, q, *main_cache, n_entries, topk, swa, S, swa_len, swa_pos0, q_pos,
                                   scale, out, lse, status, false, static_cast<cudaStream_t>(stream)));
}

int32_t csa2_gather_dequant(const csa2_cache* cache, int32_t cache_dtype, int32_t B, int32_t n, const int32_t* ids,
                            float* out, int32_t* status, void* stream) {
  if (!cache || (cache->channels != kDim && cache->channels != kIdxDim)) return CSA2_ERR_INVALID_ARG;
  if (cache_dtype != CSA2_CACHE_FP4 && cache_dtype != CSA2_CACHE_BF16 && cache_dtype != CSA2_CACHE_FP4_S32)
    return CSA2_ERR_INVALID_ARG;
  if (cache_dtype == CSA2_CACHE_FP4_S32 && cache->channels != kIdxDim) return CSA2_ERR_INVALID_ARG;
  if (!cache_ok(cache, cache->channels, cache_dtype)) return CSA2_ERR_INVALID_ARG;
  if (B < 0 || n < 0) return CSA2_ERR_INVALID_ARG;
  if (B == 0 || n == 0) return CSA2_OK;
  if (!ids || !out || !al(ids, 4) || !al(out, 4) || !al(status, 4)) return CSA2_ERR_INVALID_ARG;
  return cuda_status(launch_gather_dequant(*cache, cache_dtype, B, n, ids, out, status, static_cast<cudaStream_t>(stream)));
}

int32_t csa2_swa_encode(int32_t B, int32_t T, const uint16_t* x, const int64_t* row0, void* rows, int32_t S,
                        int32_t* status, void* stream) {
  if (B < 0 || T < 0 || S < 0) return CSA2_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return CSA2_OK;
  if (!x || !row0 || !rows || !al(x, 16) || !al(rows, 16) || !al(row0, 8) || !al(status, 4) || T > S)
    return CSA2_ERR_INVALID_ARG;
  return cuda_status(launch_swa_encode(B, T, x, row0, rows, S, status, static_cast<cudaStream_t>(stream)));
}

int32_t csa2_layer(const csa2_cfg* cfg, int32_t mode, csa2_group_state* st, const csa2_layer_io* io, void* stream) {
  int32_t err;
  if (!cfg_supported(cfg, &err)) return err;
  if (!st || !io) return CSA2_ERR_INVALID_ARG;
  if (mode != CSA2_MODE_FULL && mode != CSA2_MODE_REINDEX && mode != CSA2_MODE_REUSE) return CSA2_ERR_INVALID_ARG;
  if (!st->topk) return CSA2_ERR_INVALID_ARG;
  if (mode == CSA2_MODE_REINDEX && (!st->pool || cfg->hsi_blocks <= 0)) return CSA2_ERR_INVALID_ARG;
  // every stage's arguments are checked before the first launch, so an
  // argument error leaves the caches, the published top-k and the pool as
  // they were
  const bool comp = mode == CSA2_MODE_FULL && io->x;
  const bool index = mode != CSA2_MODE_REUSE;
  const int32_t* pool_in = mode == CSA2_MODE_REINDEX ? st->pool : nullptr;
  int32_t* pool_out = (mode == CSA2_MODE_FULL && cfg->hsi_blocks > 0) ? st->pool : nullptr;
  bool e_comp = true, e_index = true, e_att;
  int32_t rc;
  if (comp) {
    rc = check_compress(cfg, io->B, io->T, io->x, io->pos0, io->merge_w, io->w_idx, &st->main_cache, &st->idx_cache,
                        st->n_entries, st->status, &e_comp);
    if (rc) return rc;
  }
  if (index) {
    rc = check_index(cfg, io->B, io->Tq, io->q_idx, io->head_w, io->q_pos, &st->idx_cache, st->n_entries,
                     st->max_entries, pool_in, st->topk, pool_out, st->workspace, st->workspace_bytes, st->status,
                     &e_index);
    if (rc) return rc;
  }
  rc = check_attend(cfg, io->B, io->Tq, io->q, &st->main_cache, st->n_entries, st->topk, io->swa, io->S, io->swa_len,
                    io->swa_pos0, io->q_pos, io->scale, io->out, io->lse, st->status, &e_att);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!e_comp) {
    rc = cuda_status(launch_compress(*cfg, io->B, io->T, io->x, io->pos0, io->merge_w, io->w_idx, st->main_cache,
                                     st->idx_cache, st->n_entries, st->status, s));
    if (rc) return rc;
  }
  if (!e_index) {
    rc = cuda_status(launch_index_topk(*cfg, io->B, io->Tq, io->q_idx, io->head_w, io->q_pos, st->idx_cache,
                                       st->n_entries, st->max_entries, pool_in, st->topk, pool_out, st->workspace,
                                       st->workspace_bytes, st->status, s));
    if (rc) return rc;
  }
  if (e_att) return CSA2_OK;
  // a Reuse layer's attention gathers its rows before it waits for the
  // kernel enqueued just before it (that kernel writes no top-k or cache)
  return cuda_status(launch_attend(*cfg, io->B, io->Tq, io->q, st->main_cache, st->n_entries, st->topk, io->swa,
                                   io->S, io->swa_len, io->swa_pos0, io->q_pos, io->scale, io->out, io->lse,
                                   st->status, mode == CSA2_MODE_REUSE, s));
}

}  // extern "C"
