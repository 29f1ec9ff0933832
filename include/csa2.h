/*
 * csa2.h -- C ABI of the GB300 CSA2 compressed-sparse-attention library.
 *
 * CSA2 is the attention of DeepSeek-V4.1-Flash as described in
 * "DeepSeek-V4.1 Flash ..." (hn.213312.xyz) sec. 2.3 and in "What black
 * technologies does DeepSeek V4.1 Flash adopt" (36kr), section "CSA2": a
 * compressor writes one 512-channel latent entry per r tokens into a main-KV
 * cache shared across layers, an indexer projected from that cache scores
 * the entries and keeps the top 512, and 64 query heads attend over the
 * selected entries together with the layer's own sliding window of 128 rows,
 * with one latent vector serving as both key and value.
 *
 * Conventions for every entry point:
 *  - All pointers are DEVICE pointers unless stated, owned by the caller; the
 *    library allocates nothing and never synchronises.  Calls are enqueued on
 *    `stream` (a cudaStream_t passed as void*, NULL = legacy default stream).
 *  - Every kernel is launched as a programmatic dependent launch: it may
 *    start while the kernel enqueued just before it on the stream finishes.
 *    Each kernel of this library waits for that kernel's completion (and
 *    the visibility of its writes) before reading any argument, with two
 *    exceptions: the selection reads q_pos and n_entries before that wait
 *    (its predecessor is the scoring kernel of the same indexer call, which
 *    writes neither; csa2_index_select follows csa2_index_score with the
 *    same q_pos and n_entries), and the decode attention reads q, the
 *    window rows and their positions before it (named at csa2_attend and
 *    csa2_layer).
 *    Because every kernel of this library waits before it lets its own
 *    successor start, placing any call of this library between the kernel
 *    that writes those inputs and the attention satisfies the rule.
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major.
 *  - The return value reports argument errors found on the host before any
 *    launch (CSA2_ERR_INVALID_ARG / CSA2_ERR_UNSUPPORTED / CSA2_ERR_CAPACITY)
 *    and launch failures (CSA2_ERR_CUDA).  Errors found on the device (a page
 *    id or entry id out of range) are written to `*status`, a device int32
 *    that the caller zeroes; the first error wins and the faulty access is
 *    skipped.  No call aborts the process or raises across the ABI.
 *  - Every pointer has at least its element's natural alignment (2 bytes for
 *    bf16, 4 for int32 / float, 8 for int64); 16 bytes are required of the
 *    cache pages, the indexer queries `q_idx`, the attention queries `q`,
 *    the attention output `out`, window rows and the csa2_swa_encode input;
 *    8 of the indexer projection `w_idx`; 4 of the compressor input `x`;
 *    256 of index workspaces.  A pointer short of this is an argument
 *    error (CSA2_ERR_INVALID_ARG), found before any launch.
 *  - Sizes fixed by the model and accepted only at these values: dim 512,
 *    rope_dims 64, n_heads 64, idx_heads 32, idx_dim 128, hsi_block 8.
 *    topk (1..1024), window (0..512), ratio (1 or 2), hsi_blocks (0..4096)
 *    and rope_theta are free.
 *  - f16 operands: the tensor cores multiply in f16 with fp32 accumulation.
 *    FP4 and MXFP8 values and FP4-encoded queries are exact in f16; bf16
 *    inputs made into f16 -- the attention queries `q`, bf16 window rows,
 *    the rows of a bf16 main cache, and the indexer queries `q_idx` over an
 *    FP4 cache -- keep their value for |x| in [2^-14, 65504] (below that an
 *    absolute error of at most 2^-25).  Such an input beyond 65504 in
 *    magnitude, or not finite, sets CSA2_ERR_RANGE in *status (the query's
 *    results are then unspecified); the call still completes.
 *
 * Paged cache layout (a build choice; the pages never mention paging).  A
 * page holds 64 consecutive entries of one sequence; entry j of sequence b
 * lives in page block_table[b * max_pages + j / 64], slot j % 64.
 *  FP4 (E2M1 elements, one E4M3 scale per 16 channels, no global scale;
 *  hn.213312.xyz sec. 2.4.4): element 2i in the low nibble of byte i.
 *   main (512 ch):   data page 64 x 256 B, slot s at s*256 (row-major);
 *                    scales page 64 x 32 B, slot s at s*32.
 *   indexer (128 ch): data page 64 x 64 B stored by 16-byte chunks:
 *                    chunk c (0..3) of slot s at (c*64 + s)*16;
 *                    scales page 64 x 8 B, slot s at s*8.
 *  BF16: main page 64 x 1024 B row-major; indexer page 64 x 256 B by 16-byte
 *   chunks, chunk c (0..15) of slot s at (c*64 + s)*16; no scales.
 *  FP4_S32 (indexer only; the 68-byte entry of hn.213312.xyz sec. 3.1: 64 B
 *   of codes + one E4M3 scale per 32 channels): data page as FP4 indexer;
 *   scales page 64 x 4 B, slot s at s*4.
 *
 * Window rows (the layer's sliding-window KV, passed to csa2_attend): bf16
 * [B][S][512], or with CSA2_FMT_SWA_FP8 rows of 528 bytes in the OCP MXFP8
 * layout (hn.213312.xyz sec. 2.4.4: the SWA KV stays in FP8): bytes 0..511
 * E4M3 elements (channel c at byte c), bytes 512..527 one E8M0 scale
 * 2^(e - 127) per 32 channels; value = E4M3(element) x scale.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad size or stride */
  CSA2_ERR_UNSUPPORTED = 2, /* a model size other than the ones listed above */
  CSA2_ERR_CUDA = 3,        /* a launch failed (cudaGetLastError) */
  CSA2_ERR_CAPACITY = 4,    /* workspace or cache too small for the request */
  /* device-side status codes (written to *status) */
  CSA2_ERR_BAD_PAGE = 16,   /* block_table entry outside [0, num_pages) */
  CSA2_ERR_BAD_INDEX = 17,  /* top-k / pool id outside the sequence's entries */
  CSA2_ERR_TIMEOUT = 18,    /* a bounded device-side wait gave up */
  CSA2_ERR_RANGE = 19       /* an input that becomes an f16 tensor-core operand is not finite
                               or beyond the f16 range (|x| > 65504); the affected query's
                               results are unspecified (see "f16 operands" below) */
};

enum { CSA2_CACHE_FP4 = 0, CSA2_CACHE_BF16 = 1, CSA2_CACHE_FP4_S32 = 2 };
/* csa2_cfg.formats flags (0 = FP4 indexer entries with one scale per 16
 * channels, bf16 window rows) */
enum {
  CSA2_FMT_IDX_68B = 1,  /* FP4 caches: the indexer cache is CSA2_CACHE_FP4_S32 */
  CSA2_FMT_SWA_FP8 = 2,  /* window rows are 528-byte MXFP8 rows */
  CSA2_FMT_IDX_QFP4 = 4  /* indexer queries scored in FP4: each head's q_idx is encoded like a
                            cache entry (E2M1, E4M3 per 16 channels) and read back (the FP4
                            indexer Q/K of hn.213312.xyz sec. 2.4.4) */
};
enum { CSA2_MODE_FULL = 0, CSA2_MODE_REINDEX = 1, CSA2_MODE_REUSE = 2 };

#define CSA2_PAGE_ENTRIES 64

/* Layer configuration; the model config list of hn.213312.xyz sec. 1.2 gives
 * head_dim 512, rope_head_dim 64, 64 heads, index 32 x 128, index_topk 512,
 * window 128, compress ratio 2 (encoder) / 1 (decoder), candidate blocks
 * 2048 x 8, theta 10000 / 160000. */
typedef struct csa2_cfg {
  int32_t dim;         /* latent channels (512) */
  int32_t rope_dims;   /* leading channels carrying RoPE (64) */
  int32_t n_heads;     /* main query heads (64) */
  int32_t idx_heads;   /* indexer heads (32) */
  int32_t idx_dim;     /* indexer channels (128) */
  int32_t topk;        /* entries kept per query (512) */
  int32_t window;      /* sliding-window rows per query (128) */
  int32_t ratio;       /* tokens merged per entry r (2 encoder, 1 decoder) */
  int32_t hsi_blocks;  /* HSI candidate blocks per query (2048); 0 = no HSI */
  int32_t hsi_block;   /* entries per HSI block (8) */
  int32_t cache_dtype; /* CSA2_CACHE_FP4 or CSA2_CACHE_BF16 (main cache) */
  int32_t formats;     /* CSA2_FMT_* flags; 0 for the default formats */
  double rope_theta;   /* RoPE base (10000 encoder, 160000 decoder) */
} csa2_cfg;

/* One paged cache (main KV or indexer K); see the layout above. */
typedef struct csa2_cache {
  void* data;                 /* FP4 codes or BF16 values, num_pages pages */
  void* scales;               /* FP4 E4M3 scales, num_pages pages; NULL for BF16 */
  const int32_t* block_table; /* [batch][max_pages] page ids */
  int32_t max_pages;          /* block_table row stride; capacity = 64 * max_pages */
  int32_t num_pages;          /* pages allocated behind data / scales */
  int32_t channels;           /* 512 (main) or 128 (indexer) */
  int32_t reserved;           /* must be 0 */
} csa2_cache;

/* Bytes of one page of a cache: which = 0 data, 1 scales (0 for BF16);
 * cache_dtype CSA2_CACHE_FP4, CSA2_CACHE_BF16 or CSA2_CACHE_FP4_S32. */
CSA2_API size_t csa2_page_bytes(int32_t channels, int32_t cache_dtype, int32_t which);

/* Human-readable name of a status code (static string). */
CSA2_API const char* csa2_status_string(int32_t code);

/* a1 -- compressor (hn.213312.xyz sec. 1.1 "sequence axis", sec. 2.3.1; 36kr
 * "CSA2"; FP4 encoding sec. 2.4.4).  For each sequence b, the T token latents
 * x[b] at positions pos0[b] .. pos0[b]+T-1 (pos0[b] a multiple of r, T a
 * multiple of r) form T/r entries j = pos0[b]/r + m:
 *   entry = sum_{i<r} merge_w[i] (.) x[b][r*m + i]      (per channel, fp32)
 *   RoPE on interleaved pairs of the first 64 channels at position r*j + r-1,
 *   frequency theta^(-2i/64), angle formed in fp64;
 *   encode (FP4: scale = RNE_E4M3(amax/6), code = RNE_E2M1(x/scale), ties to
 *   even, saturating; BF16: round to nearest even) into the main cache;
 *   indexer K = decoded stored entry . w_idx (fp32 accumulate), encoded the
 *   same way into the indexer cache.
 * x [B][T][512] bf16; pos0 [B] int64; merge_w [r][512] fp32;
 * w_idx [512][128] bf16; n_entries [B] int32 is set to pos0[b]/r + T/r. */
CSA2_API int32_t csa2_compress(const csa2_cfg* cfg, int32_t B, int32_t T, const uint16_t* x,
                      const int64_t* pos0, const float* merge_w, const uint16_t* w_idx,
                      const csa2_cache* main_cache, const csa2_cache* idx_cache,
                      int32_t* n_entries, int32_t* status, void* stream);

/* Workspace bytes csa2_index_topk needs to run all B*Tq queries in one pass
 * over sequences of at most max_entries entries; a smaller workspace makes it
 * run the queries in chunks (at least one query's worth is required). */
CSA2_API size_t csa2_index_workspace_bytes(const csa2_cfg* cfg, int32_t B, int32_t Tq, int32_t max_entries,
                                  int32_t reindex);

/* a3..a6 -- lightweight indexer, top-k, HSI pool, Reindex (hn.213312.xyz
 * sec. 2.3.1, 2.3.2, 2.3.4; 36kr "CSA2").  For query (b, t) at position
 * q_pos[b][t], entry j is visible iff r*j + r - 1 <= q_pos and
 * j < n_entries[b].  Score s_j = sum_h w_h ReLU(q_idx_h . K_j) (w_h = head_w
 * or 1).  Without `pool`: every visible entry is a candidate (Full); with
 * `pool` [B][Tq][hsi_blocks] (ascending block ids, -1 padded) only the
 * visible entries of those blocks are (Reindex).  topk_out [B][Tq][topk]
 * receives the k best candidates by (score desc, id asc), ascending, -1
 * padded.  pool_out (Full only, needs hsi_blocks > 0): block score = max over
 * the block's visible entries; the block of the latest visible entry is
 * always kept; the best hsi_blocks blocks by (score desc, id asc), ascending,
 * -1 padded.  max_entries bounds n_entries (grid sizing).  q_idx
 * [B][Tq][32][128] bf16; head_w [B][Tq][32] fp32 or NULL. */
CSA2_API int32_t csa2_index_topk(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q_idx,
                        const float* head_w, const int64_t* q_pos, const csa2_cache* idx_cache,
                        const int32_t* n_entries, int32_t max_entries, const int32_t* pool,
                        int32_t* topk_out, int32_t* pool_out, void* workspace,
                        size_t workspace_bytes, int32_t* status, void* stream);

/* a3..a6 and a4/a5 as two calls, for a caller that wants the scoring and
 * the selection on their own (to time or overlap them): csa2_index_score
 * writes the scores of all B*Tq queries (and, with hsi != 0 on a Full call,
 * the HSI block maxima) into `workspace`; csa2_index_select then selects
 * topk_out (and pool_out) from that workspace.  Together they compute what
 * csa2_index_topk computes with the same arguments.  Arguments and checks
 * are csa2_index_topk's, plus: the workspace must hold every query
 * (csa2_index_workspace_bytes(cfg, B, Tq, max_entries, pool != NULL)
 * bytes, else CSA2_ERR_CAPACITY); B*Tq <= 65535 (else CSA2_ERR_UNSUPPORTED);
 * hsi != 0 only without `pool` (CSA2_ERR_INVALID_ARG).  The select call
 * must follow the score call on the same stream with the same cfg, B, Tq,
 * q_pos, n_entries, max_entries and pool, the same workspace untouched in
 * between, and pool_out != NULL only if hsi was set; otherwise its output
 * is unspecified (every access stays inside the workspace). */
CSA2_API int32_t csa2_index_score(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q_idx,
                                  const float* head_w, const int64_t* q_pos, const csa2_cache* idx_cache,
                                  const int32_t* n_entries, int32_t max_entries, const int32_t* pool, int32_t hsi,
                                  void* workspace, size_t workspace_bytes, int32_t* status, void* stream);
CSA2_API int32_t csa2_index_select(const csa2_cfg* cfg, int32_t B, int32_t Tq, const int64_t* q_pos,
                                   const csa2_cache* idx_cache, const int32_t* n_entries, int32_t max_entries,
                                   const int32_t* pool, int32_t* topk_out, int32_t* pool_out, void* workspace,
                                   size_t workspace_bytes, int32_t* status, void* stream);

/* a7 -- sparse attention (hn.213312.xyz sec. 2.2.2 "global KV and local KV
 * concatenated and scored with Q", sec. 3.3.1 "key = value"; 36kr "CSA2").
 * For query (b, t) and head h: rows E = {main entries topk[b][t][i] >= 0} and
 * the window rows of swa[b] at positions max(0, q_pos-W+1) .. q_pos that lie
 * in [swa_pos0[b], swa_pos0[b] + swa_len[b]); logits l_e = scale * q_h . c_e,
 * p = softmax over E jointly, out_h = sum_e p_e c_e (all 512 channels).
 * q [B][Tq][64][512] bf16; topk [B][Tq][topk]; swa [B][S][512] bf16, or
 * [B][S] MXFP8 rows of 528 B with CSA2_FMT_SWA_FP8 (16-byte aligned; only
 * for topk + window <= 768, else CSA2_ERR_UNSUPPORTED);
 * out [B][Tq][64][512] fp32; lse [B][Tq][64] fp32 natural log, or NULL.
 * Read before the wait on the previous kernel (so that the loads overlap a
 * preceding selection): q, swa, swa_len, swa_pos0 and q_pos.  They must not
 * be written by the kernel enqueued immediately before this call on the
 * stream; of this library's calls only csa2_swa_encode writes any of them,
 * so enqueue another call (the indexer of a decode step) between the two.
 * topk, n_entries and the main cache are read after that kernel has
 * completed. */
CSA2_API int32_t csa2_attend(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q,
                    const csa2_cache* main_cache, const int32_t* n_entries, const int32_t* topk,
                    const void* swa, int32_t S, const int32_t* swa_len, const int64_t* swa_pos0,
                    const int64_t* q_pos, float scale, float* out, float* lse, int32_t* status,
                    void* stream);

/* FP8 window rows (hn.213312.xyz sec. 2.4.4: the SWA KV stays FP8), OCP
 * MXFP8: for each sequence b the T bf16 rows x[b] [T][512] are encoded into
 * rows[b][row0[b] + i] of a [B][S] array of 528-byte rows (layout above).
 * Per 32-channel block: scale 2^(floor(log2 amax) - 8) (E8M0, clamped to
 * 2^-127 .. 2^127; an all-zero block takes 2^-127); element = the E4M3 value
 * nearest to x / scale, ties to even, saturating at 448, +0 for values that
 * round to zero.  row0 [B] int64 (device); a sequence whose rows would fall
 * outside [0, S) is skipped and CSA2_ERR_BAD_INDEX written to *status.
 * A csa2_attend that reads these rows must not be the next call enqueued
 * on the stream (it reads window rows before waiting for its predecessor). */
CSA2_API int32_t csa2_swa_encode(int32_t B, int32_t T, const uint16_t* x, const int64_t* row0, void* rows,
                                 int32_t S, int32_t* status, void* stream);

/* csa2_index_topk without a caller-provided workspace, for callers that
 * cannot allocate device memory (a serving engine or plugin host that owns
 * all device memory in its own pool and offers no allocator, or a decode loop
 * that must not pay for cudaMalloc's device synchronisation).  The write-ups
 * have no counterpart to this call: it only changes where the scratch lives.
 * Same arguments, rules and results as csa2_index_topk; the scores and HSI
 * block maxima go to one static device array of
 * csa2_index_static_scratch_bytes() bytes (8 MiB) built into the library,
 * present on every GPU that loads it until the process exits.  One query's
 * scratch (about 4 B per entry, 4.5 B with HSI) must fit, else
 * CSA2_ERR_CAPACITY before any launch; larger batches run in chunks.
 * Allocates nothing.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress), so make that first call before any stream
 * capture.  Calls share the array and keep the previous call's contents
 * (nothing needs clearing); calls that overlap on the GPU race, so order them
 * on one stream. */
CSA2_API int32_t csa2_index_topk_static(const csa2_cfg* cfg, int32_t B, int32_t Tq, const uint16_t* q_idx,
                                        const float* head_w, const int64_t* q_pos, const csa2_cache* idx_cache,
                                        const int32_t* n_entries, int32_t max_entries, const int32_t* pool,
                                        int32_t* topk_out, int32_t* pool_out, int32_t* status, void* stream);

/* Size in bytes of the static scratch array behind csa2_index_topk_static. */
CSA2_API size_t csa2_index_static_scratch_bytes(void);

/* Decode entries of a cache to fp32: out[b][i][c] = value of entry
 * ids[b][i] of sequence b (ids < 0 give zeros).  ids [B][n]; out
 * [B][n][channels].  Exact for both cache formats. */
CSA2_API int32_t csa2_gather_dequant(const csa2_cache* cache, int32_t cache_dtype, int32_t B, int32_t n,
                            const int32_t* ids, float* out, int32_t* status, void* stream);

/* State shared by the layers of one cross-layer group (hn.213312.xyz
 * sec. 2.3.2, 3.2): the main-KV and indexer-K caches written by the Full
 * layer, the latest published top-k and the HSI pool. */
typedef struct csa2_group_state {
  csa2_cache main_cache;
  csa2_cache idx_cache;
  int32_t* n_entries;   /* [B] */
  int32_t max_entries;  /* capacity bound per sequence */
  int32_t reserved;
  int32_t* topk;        /* [B][Tq][topk] latest published top-k */
  int32_t* pool;        /* [B][Tq][hsi_blocks] HSI pool, or NULL */
  void* workspace;
  size_t workspace_bytes;
  int32_t* status;
} csa2_group_state;

/* Per-layer inputs and outputs of one CSA2 layer. */
typedef struct csa2_layer_io {
  int32_t B, Tq;
  const int64_t* q_pos;      /* [B][Tq] */
  /* compressor inputs, Full mode only; x == NULL skips compression */
  int32_t T;
  const uint16_t* x;
  const int64_t* pos0;
  const float* merge_w;
  const uint16_t* w_idx;
  /* indexer query, Full and Reindex */
  const uint16_t* q_idx;
  const float* head_w;
  /* attention, every mode */
  const uint16_t* q;
  const void* swa;           /* bf16 rows, or MXFP8 rows with CSA2_FMT_SWA_FP8 */
  int32_t S;
  const int32_t* swa_len;
  const int64_t* swa_pos0;
  float scale;
  float* out;
  float* lse;
} csa2_layer_io;

/* a8 -- one layer under its cross-layer mode (hn.213312.xyz sec. 2.3.2 and
 * the access table of sec. 3.2; 36kr "CSA2"):
 *  FULL    compress (if io->x), index the whole visible cache, publish top-k
 *          (and the HSI pool when cfg->hsi_blocks > 0), attend;
 *  REINDEX index only the pool's entries with this layer's q_idx, publish
 *          top-k, attend (no cache writes);
 *  REUSE   attend with the latest published top-k (no indexer, no writes).
 * The attention reads io's query and window arrays before it waits for the
 * kernel enqueued just before it (see csa2_attend); in REUSE mode it also
 * gathers its rows before that wait, reading the published top-k,
 * state->n_entries and the main cache.  In REUSE mode that kernel is the one
 * enqueued before this call, which therefore must write none of these (a
 * preceding csa2_layer call of the group writes none of them with its last
 * kernel). */
CSA2_API int32_t csa2_layer(const csa2_cfg* cfg, int32_t mode, csa2_group_state* state,
                   const csa2_layer_io* io, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
