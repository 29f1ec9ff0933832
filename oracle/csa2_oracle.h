/*
 * CSA2 CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 restatement of what the DeepSeek-V4.1-Flash write-ups
 * define for CSA2 compressed sparse attention (compressor, FP4 main-KV /
 * indexer-K encoding, lightweight indexer + top-k, hierarchical sparse
 * indexer, sparse attention over top-k plus the sliding window, and the
 * Full / Reindex / Reuse cross-layer modes).  It shares no code, header,
 * table or constant with the CUDA library, and the CUDA library never calls
 * it.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it.
 *
 * Sources (page title, then section):
 *  - "DeepSeek-V4.1 Flash ... (hn.213312.xyz)" sec. 1.1-1.2 (three compression
 *    axes, model config list), sec. 2.3.1 (CSA2 vs CSA: indexer K projected
 *    from main KV, no overlap, no absolute position embedding), sec. 2.3.2
 *    (Full / Reindex / Reuse), sec. 2.3.4 (HSI: block max, top-2048 blocks of
 *    8, forced latest block), sec. 2.4.4 (FP4 main KV: E2M1 with one E4M3
 *    scale per 16 channels, no global scale, quantised after RoPE; the SWA
 *    KV kept in FP8, read here as OCP MXFP8: E4M3 elements, one E8M0 scale
 *    per 32 channels),
 *    sec. 3.1 (288 B / 68 B per entry, 890 B/token table; 68 B read as 64 B
 *    of codes + one E4M3 scale per 32 channels), sec. 3.2 (mode
 *    access table), sec. 3.3.1 (key = value, convex-combination readout).
 *  - "What black technologies does DeepSeek V4.1 Flash adopt" (36kr),
 *    sections "CSA2" and "FP4 and Bounded Replay".
 *
 * Readings where the pages are silent (the same list is kept in the design
 * notes of the repository): indexer score s_j = sum_h w_h * ReLU(q_h . K_j);
 * FP4 scale = RNE_E4M3(amax / 6), code = RNE_E2M1(x / scale) saturating at 6,
 * ties to even, a value that rounds to zero gets code +0; merge then RoPE at
 * position r*j + r - 1 on interleaved pairs of the first rope_dims channels,
 * freq_i = theta^(-2i/rope_dims), no YaRN; indexer K = dequant(stored main
 * entry) . W_idx; entry j visible to a query at t iff r*j + r - 1 <= t and
 * j < n_entries; top-k ordered by (score desc, index asc), output ascending,
 * padded with -1; HSI forced block takes one of the block slots; one joint
 * softmax over the top-k entries and the window rows t-W+1..t.
 *
 * Canonical (unpaged) layouts used by every oracle function:
 *  - bf16 tensors are uint16 bit patterns, row-major;
 *  - FP4 entries of C channels: codes [N][C/2] bytes (element 2i in the low
 *    nibble of byte i), scales [N][C/16] E4M3 bytes ([N][C/32] for the
 *    68-byte indexer entry);
 *  - BF16 cache entries: [N][C] uint16;
 *  - MXFP8 window rows: [N][C + C/32] bytes (elements, then block scales).
 *
 * parity pins: every function here is pinned by tests/test_oracle_*.py
 * (codebook anchors, brute-force searches, closed forms and invariants).
 */
#ifndef CSA2_ORACLE_H
#define CSA2_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

#define ORC_CACHE_FP4 0
#define ORC_CACHE_BF16 1
/* FP4 main KV with the 68-byte indexer entry (sec. 3.1): the indexer cache
 * carries one E4M3 scale per 32 channels (64 B codes + 4 B scales). */
#define ORC_CACHE_FP4_G32 2
/* Window-row formats: bf16, or MXFP8 (sec. 2.4.4: the SWA KV stays FP8) */
#define ORC_SWA_BF16 0
#define ORC_SWA_MXFP8 1

/* ---- scalar codecs (OCP MX formats named by the pages, sec. 2.4.4) ---- */
double orc_bf16_value(uint16_t bits);
uint16_t orc_bf16_round(double x); /* round to nearest even, no NaN inputs */
double orc_e2m1_value(int code);   /* code in 0..15 */
double orc_e4m3_value(int byte);   /* byte in 0..255; NaN for S.1111.111 */
int orc_e4m3_nearest_code(double y);  /* y >= 0; nearest finite code, ties even, saturating */
int orc_e2m1_nearest_code(double x, double scale); /* code of x/scale, ties even, sat. */

/* FP4 encode / decode of one entry of C channels (C multiple of 16). */
void orc_fp4_encode(const double* x, int C, uint8_t* codes, uint8_t* scales);
void orc_fp4_decode(const uint8_t* codes, const uint8_t* scales, int C, double* out);
/* The same with one scale per `group` channels (16 or 32; C multiple of group). */
void orc_fp4_encode_g(const double* x, int C, int group, uint8_t* codes, uint8_t* scales);
void orc_fp4_decode_g(const uint8_t* codes, const uint8_t* scales, int C, int group, double* out);

/* OCP MX E8M0 scale value 2^(byte - 127) (NaN for 0xFF). */
double orc_e8m0_value(int byte);
/* MXFP8 window row of C channels (C multiple of 32): C E4M3 element bytes,
 * then C/32 E8M0 scale bytes; scale 2^(floor(log2 amax) - 8) per block. */
void orc_mxfp8_encode(const double* x, int C, uint8_t* row);
void orc_mxfp8_decode(const uint8_t* row, int C, double* out);

/* ---- a1: compressor ----
 * x      [B][T][D] bf16 token latents at positions pos0[b] + i (pos0 % r == 0, T % r == 0)
 * w      [r][D] fp32 per-channel merge weights
 * w_idx  [D][Ci] bf16 indexer-K projection
 * Writes entries j = pos0/r + m, m < T/r, into the canonical caches, whose
 * per-sequence capacity is n_cap entries:
 *   FP4:  main_codes [B][n_cap][D/2], main_scales [B][n_cap][D/16],
 *         idx_codes [B][n_cap][Ci/2], idx_scales [B][n_cap][Ci/16]
 *   BF16: main_bf16 [B][n_cap][D], idx_bf16 [B][n_cap][Ci]
 * Optional diagnostics (may be NULL), shaped [B][T/r][D] / [B][T/r][Ci]:
 *   pre_main / pre_idx: the values just before encoding;
 *   mag_main / mag_idx: sum of |terms| that formed each value (rounding
 *   error scale of any fp32 evaluation of the same value).
 * Returns 0, or -1 on bad arguments. */
int orc_compress(int B, int T, int D, int Ci, int rope_dims, int r, double theta, int cache_dtype,
                 const uint16_t* x, const int64_t* pos0, const float* w, const uint16_t* w_idx,
                 int n_cap,
                 uint8_t* main_codes, uint8_t* main_scales, uint16_t* main_bf16,
                 uint8_t* idx_codes, uint8_t* idx_scales, uint16_t* idx_bf16,
                 double* pre_main, double* mag_main, double* pre_idx, double* mag_idx);
/* (cache_dtype ORC_CACHE_FP4_G32: the main cache as FP4, the indexer cache
 * with idx_scales [B][n_cap][Ci/32].) */

/* ---- a3/a4/a5/a6: indexer scores, top-k, HSI pool, Reindex over a pool ----
 * q_idx  [B][Tq][H][Ci] bf16; head_w [B][Tq][H] fp32 or NULL (all ones)
 * q_pos  [B][Tq] query positions; n_entries [B]
 * idx cache canonical (see above), capacity n_cap per sequence
 * pool   [B][Tq][n_blocks] block ids (-1 padded) or NULL: when given, only the
 *        entries of those blocks (block size bs) are candidates (Reindex)
 * topk_out [B][Tq][k]: ascending entry ids, -1 padded
 * pool_out [B][Tq][n_blocks] or NULL: HSI block ids, ascending, -1 padded
 *          (requires pool == NULL and n_blocks > 0)
 * scores_out [B][Tq][n_cap] or NULL: s_j for candidates, -inf elsewhere */
int orc_index_topk(int B, int Tq, int H, int Ci, int r, int cache_dtype, int n_cap,
                   const uint8_t* idx_codes, const uint8_t* idx_scales, const uint16_t* idx_bf16,
                   const int32_t* n_entries, const uint16_t* q_idx, const float* head_w,
                   const int64_t* q_pos, int k, int n_blocks, int bs, const int32_t* pool,
                   int32_t* topk_out, int32_t* pool_out, double* scores_out);
/* The same with q_fp4 != 0: every head's indexer query is first encoded to
 * FP4 like a cache entry (E2M1, one E4M3 scale per 16 channels) and read
 * back, so the scores are FP4 x FP4 dot products (the FP4 indexer Q/K that
 * sec. 2.4.4 says V4 already trained with). */
int orc_index_topk_q(int B, int Tq, int H, int Ci, int r, int cache_dtype, int n_cap,
                     const uint8_t* idx_codes, const uint8_t* idx_scales, const uint16_t* idx_bf16,
                     const int32_t* n_entries, const uint16_t* q_idx, int q_fp4, const float* head_w,
                     const int64_t* q_pos, int k, int n_blocks, int bs, const int32_t* pool,
                     int32_t* topk_out, int32_t* pool_out, double* scores_out);

/* ---- a7: sparse attention over top-k entries and the sliding window ----
 * q      [B][Tq][Hm][D] bf16 (already rotated)
 * main cache canonical, capacity n_cap; topk [B][Tq][k] (-1 = empty slot)
 * swa    [B][S] rows at positions swa_pos0[b] + i, i < swa_len[b] <= S:
 *        swa_fmt ORC_SWA_BF16: [D] bf16; ORC_SWA_MXFP8: D + D/32 bytes
 * window W: a query at t reads the rows at positions max(0, t-W+1)..t present
 * out    [B][Tq][Hm][D]; lse [B][Tq][Hm] (natural log) or NULL */
int orc_attend(int B, int Tq, int Hm, int D, int cache_dtype, int n_cap,
               const uint8_t* main_codes, const uint8_t* main_scales, const uint16_t* main_bf16,
               const int32_t* n_entries, const uint16_t* q, const int32_t* topk, int k,
               const void* swa, int swa_fmt, int S, const int32_t* swa_len, const int64_t* swa_pos0,
               const int64_t* q_pos, int W, double scale, double* out, double* lse);

/* Dense attention over every visible entry and the window (no selection):
 * the k >= N limit, coded separately for the oracle's own pin -- its own
 * dot products and the softmax in pairwise form, weight_e =
 * 1 / sum_f exp(scale q.(c_f - c_e)), sharing nothing with orc_attend. */
int orc_attend_dense(int B, int Tq, int Hm, int D, int r, int cache_dtype, int n_cap,
                     const uint8_t* main_codes, const uint8_t* main_scales,
                     const uint16_t* main_bf16, const int32_t* n_entries, const uint16_t* q,
                     const void* swa, int swa_fmt, int S, const int32_t* swa_len, const int64_t* swa_pos0,
                     const int64_t* q_pos, int W, double scale, double* out);

/* Threads the oracle's parallel loops may use (OpenMP); returns the count. */
int orc_threads(void);

#ifdef __cplusplus
}
#endif
#endif
