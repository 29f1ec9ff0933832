/*
 * CSA2 CPU oracle (fp64) -- TEST INFRASTRUCTURE ONLY; see csa2_oracle.h for
 * the sources, the readings adopted where the pages are silent, and the
 * canonical layouts.  Plain loops, no blocking or fusion beyond the
 * definitions; parallel only across independent (sequence, query) units.
 */
#include "csa2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Scalar codecs                                                             */
/* ------------------------------------------------------------------------ */

double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16, ties to even, by comparing against the
 * exact midpoint of the two neighbouring bf16 values (both computable exactly
 * in double).  Saturation is not needed for the value ranges used here; an
 * overflowing input rounds to infinity as IEEE rounding would. */
uint16_t orc_bf16_round(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  float f = (float)x; /* nearest float: a bf16 neighbour pair brackets it */
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lo = u & 0xFFFF0000u;       /* truncation toward zero */
  uint32_t hi = lo + 0x00010000u;      /* next bf16 away from zero */
  double vlo = orc_bf16_value((uint16_t)(lo >> 16));
  double vhi = orc_bf16_value((uint16_t)(hi >> 16));
  double ax = fabs(x), alo = fabs(vlo), ahi = fabs(vhi);
  double mid = alo + (ahi - alo) / 2.0; /* exact: both have 8-bit significands */
  if (ax < mid) return (uint16_t)(lo >> 16);
  if (ax > mid) return (uint16_t)(hi >> 16);
  return ((lo >> 16) & 1u) ? (uint16_t)(hi >> 16) : (uint16_t)(lo >> 16);
}

/* OCP MX E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit, no inf/NaN. */
double orc_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* OCP E4M3 (the "FN" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * S.1111.111 is NaN, no infinities, largest finite magnitude 448. */
double orc_e4m3_value(int byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Nearest non-negative finite E4M3 code to y (y >= 0), ties to the even
 * code, saturating at 448.  Walks the 127 non-negative finite codes in
 * increasing order and stops at the first midpoint above y. */
int orc_e4m3_nearest_code(double y) {
  for (int c = 0; c < 126; ++c) {
    double mid = (orc_e4m3_value(c) + orc_e4m3_value(c + 1)) / 2.0; /* exact */
    if (y < mid) return c;
    if (y == mid) return (c & 1) ? c + 1 : c;
  }
  return 126; /* 448 */
}

/* E2M1 code of x / scale with round-to-nearest-even and saturation at 6.
 * The decision is taken by comparing |x| with scale * midpoint, a product
 * that is exact in double, so x / scale is never formed. */
int orc_e2m1_nearest_code(double x, double scale) {
  if (!(scale > 0.0)) return 0;
  double ax = fabs(x);
  int mag = 7; /* 6.0 */
  for (int c = 0; c < 7; ++c) {
    double mid = scale * ((orc_e2m1_value(c) + orc_e2m1_value(c + 1)) / 2.0);
    if (ax < mid) { mag = c; break; }
    if (ax == mid) { mag = (c & 1) ? c + 1 : c; break; }
  }
  if (mag == 0) return 0; /* a value that rounds to zero gets +0 */
  return (x < 0.0) ? (mag | 8) : mag;
}

/* One E4M3 scale per `group` consecutive channels (16: the main-KV format
 * of sec. 2.4.4; 32: the 68-byte indexer entry of sec. 3.1): scale =
 * RNE_E4M3(amax / 6), i.e. the E4M3 value nearest to amax / 6, decided by
 * comparing amax with 6 * midpoint (exact).  A zero scale gives all-zero
 * codes. */
void orc_fp4_encode_g(const double* x, int C, int group, uint8_t* codes, uint8_t* scales) {
  for (int g = 0; g < C / group; ++g) {
    double amax = 0.0;
    for (int i = 0; i < group; ++i) {
      double a = fabs(x[group * g + i]);
      if (a > amax) amax = a;
    }
    int sc = 126;
    for (int c = 0; c < 126; ++c) {
      double mid6 = 3.0 * (orc_e4m3_value(c) + orc_e4m3_value(c + 1)); /* 6 * midpoint, exact */
      if (amax < mid6) { sc = c; break; }
      if (amax == mid6) { sc = (c & 1) ? c + 1 : c; break; }
    }
    scales[g] = (uint8_t)sc;
    double s = orc_e4m3_value(sc);
    for (int i = 0; i < group; i += 2) {
      int c0 = orc_e2m1_nearest_code(x[group * g + i], s);
      int c1 = orc_e2m1_nearest_code(x[group * g + i + 1], s);
      codes[(group * g + i) / 2] = (uint8_t)(c0 | (c1 << 4));
    }
  }
}

void orc_fp4_decode_g(const uint8_t* codes, const uint8_t* scales, int C, int group, double* out) {
  for (int i = 0; i < C; ++i) {
    int byte = codes[i / 2];
    int code = (i & 1) ? (byte >> 4) : (byte & 15);
    out[i] = orc_e2m1_value(code) * orc_e4m3_value(scales[i / group]);
  }
}

void orc_fp4_encode(const double* x, int C, uint8_t* codes, uint8_t* scales) {
  orc_fp4_encode_g(x, C, 16, codes, scales);
}

void orc_fp4_decode(const uint8_t* codes, const uint8_t* scales, int C, double* out) {
  orc_fp4_decode_g(codes, scales, C, 16, out);
}

/* OCP MX E8M0 scale: 2^(byte - 127); 0xFF is NaN. */
double orc_e8m0_value(int byte) {
  if (byte == 255) return NAN;
  return ldexp(1.0, byte - 127);
}

/* MXFP8 row of C channels (E4M3 elements, one E8M0 scale per 32 channels,
 * OCP MX): row = C element bytes (channel c at byte c) then C/32 scale
 * bytes.  Per block: X = 2^(floor(log2 amax) - 8), 8 being the exponent of
 * E4M3's largest binade, so that amax / X lies in [256, 512); the scale byte
 * is clamped to 0..254; an all-zero block takes byte 0.  Element = the E4M3
 * code nearest to |x| / X (exact: X is a power of two), ties to the even
 * code, saturating at 448, sign bit set for negative values that do not
 * round to zero. */
void orc_mxfp8_encode(const double* x, int C, uint8_t* row) {
  for (int g = 0; g < C / 32; ++g) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      double a = fabs(x[32 * g + i]);
      if (a > amax) amax = a;
    }
    int sb = 0;
    if (amax > 0.0) {
      int ex;
      frexp(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
      sb = (ex - 1) - 8 + 127;
      if (sb < 0) sb = 0;
      if (sb > 254) sb = 254;
    }
    row[C + g] = (uint8_t)sb;
    double X = orc_e8m0_value(sb);
    for (int i = 0; i < 32; ++i) {
      double v = x[32 * g + i];
      int mag = orc_e4m3_nearest_code(fabs(v) / X);
      row[32 * g + i] = (uint8_t)((v < 0.0 && mag != 0) ? (mag | 0x80) : mag);
    }
  }
}

void orc_mxfp8_decode(const uint8_t* row, int C, double* out) {
  for (int i = 0; i < C; ++i) out[i] = orc_e4m3_value(row[i]) * orc_e8m0_value(row[C + i / 32]);
}

/* ------------------------------------------------------------------------ */
/* a1: compressor                                                            */
/* ------------------------------------------------------------------------ */

int orc_compress(int B, int T, int D, int Ci, int rope_dims, int r, double theta, int cache_dtype,
                 const uint16_t* x, const int64_t* pos0, const float* w, const uint16_t* w_idx,
                 int n_cap,
                 uint8_t* main_codes, uint8_t* main_scales, uint16_t* main_bf16,
                 uint8_t* idx_codes, uint8_t* idx_scales, uint16_t* idx_bf16,
                 double* pre_main, double* mag_main, double* pre_idx, double* mag_idx) {
  if (B < 0 || T < 0 || r < 1 || T % r || D % 16 || Ci % 16 || (cache_dtype == ORC_CACHE_FP4_G32 && Ci % 32) ||
      rope_dims % 2 || rope_dims > D)
    return -1;
  int M = T / r;
  for (int b = 0; b < B; ++b)
    if (pos0[b] < 0 || pos0[b] % r || pos0[b] / r + M > n_cap) return -1;

#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < B; ++b) {
    for (int m = 0; m < M; ++m) {
      double* v = (double*)malloc(sizeof(double) * D);
      double* mag = (double*)malloc(sizeof(double) * D);
      double* e = (double*)malloc(sizeof(double) * D);
      double* kv = (double*)malloc(sizeof(double) * Ci);
      double* kmag = (double*)malloc(sizeof(double) * Ci);
      int64_t j = pos0[b] / r + m;
      /* merge: entry = sum_i w_i (.) x_{r*j+i}, per channel */
      for (int c = 0; c < D; ++c) {
        double acc = 0.0, am = 0.0;
        for (int i = 0; i < r; ++i) {
          double t = (double)w[(size_t)i * D + c] *
                     orc_bf16_value(x[((size_t)b * T + (size_t)m * r + i) * D + c]);
          acc += t;
          am += fabs(t);
        }
        v[c] = acc;
        mag[c] = am;
      }
      /* RoPE at the entry's position p = r*j + r - 1, pairs (2i, 2i+1) */
      double p = (double)(r * j + r - 1);
      for (int i = 0; i < rope_dims / 2; ++i) {
        double f = pow(theta, -2.0 * i / rope_dims);
        double a = p * f;
        double cs = cos(a), sn = sin(a);
        double x0 = v[2 * i], x1 = v[2 * i + 1];
        v[2 * i] = x0 * cs - x1 * sn;
        v[2 * i + 1] = x0 * sn + x1 * cs;
        double pm = mag[2 * i] + mag[2 * i + 1];
        mag[2 * i] = pm;
        mag[2 * i + 1] = pm;
      }
      size_t slot = (size_t)b * n_cap + (size_t)j;
      size_t row = (size_t)b * M + m;
      if (pre_main) memcpy(pre_main + row * D, v, sizeof(double) * D);
      if (mag_main) memcpy(mag_main + row * D, mag, sizeof(double) * D);
      /* store, then read back the stored entry (indexer K is projected from it) */
      if (cache_dtype != ORC_CACHE_BF16) {
        orc_fp4_encode(v, D, main_codes + slot * (D / 2), main_scales + slot * (D / 16));
        orc_fp4_decode(main_codes + slot * (D / 2), main_scales + slot * (D / 16), D, e);
      } else {
        for (int c = 0; c < D; ++c) {
          main_bf16[slot * D + c] = orc_bf16_round(v[c]);
          e[c] = orc_bf16_value(main_bf16[slot * D + c]);
        }
      }
      /* indexer K_j = dequant(entry_j) . W_idx */
      for (int k = 0; k < Ci; ++k) {
        double acc = 0.0, am = 0.0;
        for (int c = 0; c < D; ++c) {
          double t = e[c] * orc_bf16_value(w_idx[(size_t)c * Ci + k]);
          acc += t;
          am += fabs(t);
        }
        kv[k] = acc;
        kmag[k] = am;
      }
      if (pre_idx) memcpy(pre_idx + row * Ci, kv, sizeof(double) * Ci);
      if (mag_idx) memcpy(mag_idx + row * Ci, kmag, sizeof(double) * Ci);
      if (cache_dtype == ORC_CACHE_FP4) {
        orc_fp4_encode(kv, Ci, idx_codes + slot * (Ci / 2), idx_scales + slot * (Ci / 16));
      } else if (cache_dtype == ORC_CACHE_FP4_G32) {
        orc_fp4_encode_g(kv, Ci, 32, idx_codes + slot * (Ci / 2), idx_scales + slot * (Ci / 32));
      } else {
        for (int k = 0; k < Ci; ++k) idx_bf16[slot * Ci + k] = orc_bf16_round(kv[k]);
      }
      free(v); free(mag); free(e); free(kv); free(kmag);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* a3-a6: indexer, top-k, HSI, Reindex                                       */
/* ------------------------------------------------------------------------ */

typedef struct {
  double score;
  int64_t id;
} orc_ranked;

/* (score desc, id asc): the reading adopted for the pages' unstated tie rule */
static int orc_rank_cmp(const void* pa, const void* pb) {
  const orc_ranked* a = (const orc_ranked*)pa;
  const orc_ranked* b = (const orc_ranked*)pb;
  if (a->score > b->score) return -1;
  if (a->score < b->score) return 1;
  return (a->id < b->id) ? -1 : (a->id > b->id);
}

static int orc_int_cmp(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/* Keep the first k of a ranked list, emit their ids ascending, pad with -1. */
static void orc_emit_topk(orc_ranked* cand, int n, int k, int32_t* out) {
  qsort(cand, (size_t)n, sizeof(orc_ranked), orc_rank_cmp);
  int m = n < k ? n : k;
  for (int i = 0; i < m; ++i) out[i] = (int32_t)cand[i].id;
  qsort(out, (size_t)m, sizeof(int32_t), orc_int_cmp);
  for (int i = m; i < k; ++i) out[i] = -1;
}

static void orc_load_entry(int cache_dtype, int C, size_t slot, const uint8_t* codes,
                           const uint8_t* scales, const uint16_t* bf, double* out) {
  if (cache_dtype == ORC_CACHE_FP4) {
    orc_fp4_decode(codes + slot * (C / 2), scales + slot * (C / 16), C, out);
  } else if (cache_dtype == ORC_CACHE_FP4_G32) {
    orc_fp4_decode_g(codes + slot * (C / 2), scales + slot * (C / 32), C, 32, out);
  } else {
    for (int c = 0; c < C; ++c) out[c] = orc_bf16_value(bf[slot * C + c]);
  }
}

/* number of entries visible to a query at position t: r*j + r - 1 <= t, j < n */
static int64_t orc_visible(int64_t t, int r, int64_t n) {
  if (t < r - 1) return 0;
  int64_t v = (t - (r - 1)) / r + 1;
  return v < n ? v : n;
}

int orc_index_topk(int B, int Tq, int H, int Ci, int r, int cache_dtype, int n_cap,
                   const uint8_t* idx_codes, const uint8_t* idx_scales, const uint16_t* idx_bf16,
                   const int32_t* n_entries, const uint16_t* q_idx, const float* head_w,
                   const int64_t* q_pos, int k, int n_blocks, int bs, const int32_t* pool,
                   int32_t* topk_out, int32_t* pool_out, double* scores_out) {
  return orc_index_topk_q(B, Tq, H, Ci, r, cache_dtype, n_cap, idx_codes, idx_scales, idx_bf16, n_entries, q_idx,
                          0, head_w, q_pos, k, n_blocks, bs, pool, topk_out, pool_out, scores_out);
}

int orc_index_topk_q(int B, int Tq, int H, int Ci, int r, int cache_dtype, int n_cap,
                     const uint8_t* idx_codes, const uint8_t* idx_scales, const uint16_t* idx_bf16,
                     const int32_t* n_entries, const uint16_t* q_idx, int q_fp4, const float* head_w,
                     const int64_t* q_pos, int k, int n_blocks, int bs, const int32_t* pool,
                     int32_t* topk_out, int32_t* pool_out, double* scores_out) {
  if (B < 0 || Tq < 0 || k < 1 || Ci % 16 || r < 1) return -1;
  if ((pool || pool_out) && (n_blocks < 1 || bs < 1)) return -1;
  if (pool && pool_out) return -1;

#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    for (int t = 0; t < Tq; ++t) {
      size_t qi = (size_t)b * Tq + t;
      int64_t nv = orc_visible(q_pos[qi], r, n_entries[b]);
      double* q = (double*)malloc(sizeof(double) * H * Ci);
      double* kv = (double*)malloc(sizeof(double) * Ci);
      for (int i = 0; i < H * Ci; ++i) q[i] = orc_bf16_value(q_idx[qi * H * Ci + i]);
      if (q_fp4) {
        /* FP4 indexer queries: each head's query encoded like a cache entry
         * (E2M1, one E4M3 scale per 16 channels) and read back */
        uint8_t* qc = (uint8_t*)malloc((size_t)Ci / 2);
        uint8_t* qs = (uint8_t*)malloc((size_t)Ci / 16);
        for (int h = 0; h < H; ++h) {
          orc_fp4_encode(q + (size_t)h * Ci, Ci, qc, qs);
          orc_fp4_decode(qc, qs, Ci, q + (size_t)h * Ci);
        }
        free(qc);
        free(qs);
      }
      /* candidate set: all visible entries, or the visible entries of the pool */
      char* cand = (char*)calloc((size_t)(nv > 0 ? nv : 1), 1);
      if (pool) {
        for (int pb = 0; pb < n_blocks; ++pb) {
          int32_t blk = pool[qi * n_blocks + pb];
          if (blk < 0) continue;
          for (int64_t j = (int64_t)blk * bs; j < (int64_t)(blk + 1) * bs && j < nv; ++j) cand[j] = 1;
        }
      } else {
        for (int64_t j = 0; j < nv; ++j) cand[j] = 1;
      }
      double* s = (double*)malloc(sizeof(double) * (size_t)(nv > 0 ? nv : 1));
      orc_ranked* rk = (orc_ranked*)malloc(sizeof(orc_ranked) * (size_t)(nv > 0 ? nv : 1));
      int nc = 0;
      for (int64_t j = 0; j < nv; ++j) {
        s[j] = -INFINITY;
        if (!cand[j]) continue;
        orc_load_entry(cache_dtype, Ci, (size_t)b * n_cap + (size_t)j, idx_codes, idx_scales,
                       idx_bf16, kv);
        double acc = 0.0;
        for (int h = 0; h < H; ++h) {
          double d = 0.0;
          for (int c = 0; c < Ci; ++c) d += q[h * Ci + c] * kv[c];
          double wh = head_w ? (double)head_w[qi * H + h] : 1.0;
          acc += wh * (d > 0.0 ? d : 0.0);
        }
        s[j] = acc;
        rk[nc].score = acc;
        rk[nc].id = j;
        ++nc;
      }
      if (scores_out) {
        for (int64_t j = 0; j < n_cap; ++j) scores_out[qi * n_cap + j] = (j < nv) ? s[j] : -INFINITY;
      }
      orc_emit_topk(rk, nc, k, topk_out + qi * k);

      if (pool_out) {
        /* HSI: block score = max over the block's visible entries; the block
         * holding the latest visible entry is always kept and takes a slot. */
        int64_t nb = (nv + bs - 1) / bs;
        int32_t* po = pool_out + qi * n_blocks;
        if (nb == 0) {
          for (int i = 0; i < n_blocks; ++i) po[i] = -1;
        } else {
          int64_t forced = (nv - 1) / bs;
          orc_ranked* br = (orc_ranked*)malloc(sizeof(orc_ranked) * (size_t)nb);
          int nr = 0;
          for (int64_t blk = 0; blk < nb; ++blk) {
            if (blk == forced) continue;
            double m = -INFINITY;
            for (int64_t j = blk * bs; j < (blk + 1) * bs && j < nv; ++j) m = s[j] > m ? s[j] : m;
            br[nr].score = m;
            br[nr].id = blk;
            ++nr;
          }
          po[0] = (int32_t)forced;
          orc_emit_topk(br, nr, n_blocks - 1, po + 1);
          /* po[1..] is ascending with -1 padding; merge the forced id in */
          int cnt = 1;
          for (int i = 1; i < n_blocks; ++i) cnt += po[i] >= 0;
          qsort(po, (size_t)cnt, sizeof(int32_t), orc_int_cmp);
          free(br);
        }
      }
      free(q); free(kv); free(cand); free(s); free(rk);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* a7: sparse attention                                                      */
/* ------------------------------------------------------------------------ */

/* One query token, all heads: softmax over the given rows jointly, output the
 * probability-weighted sum of the same rows (key = value). */
static void orc_attend_rows(int Hm, int D, const double* q, double* const* rows, int n,
                            double scale, double* out, double* lse) {
  double* l = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int h = 0; h < Hm; ++h) {
    const double* qh = q + (size_t)h * D;
    double mx = -INFINITY;
    for (int e = 0; e < n; ++e) {
      double d = 0.0;
      for (int c = 0; c < D; ++c) d += qh[c] * rows[e][c];
      l[e] = d * scale;
      if (l[e] > mx) mx = l[e];
    }
    double z = 0.0;
    for (int e = 0; e < n; ++e) z += exp(l[e] - mx);
    double* o = out + (size_t)h * D;
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    for (int e = 0; e < n; ++e) {
      double p = exp(l[e] - mx) / z;
      for (int c = 0; c < D; ++c) o[c] += p * rows[e][c];
    }
    if (lse) lse[h] = (n > 0) ? mx + log(z) : -INFINITY;
  }
  free(l);
}

/* Bytes of one window row: bf16 (2 per channel) or MXFP8 (1 per channel plus
 * one scale byte per 32). */
static size_t orc_swa_row_bytes(int fmt, int D) { return fmt == ORC_SWA_MXFP8 ? (size_t)D + D / 32 : 2 * (size_t)D; }

static int orc_window_rows(int64_t t, int W, const uint8_t* swa_b, int fmt, int D, int64_t p0,
                           int32_t len, double** rows, int n) {
  const size_t rb = orc_swa_row_bytes(fmt, D);
  for (int64_t pos = t - W + 1; pos <= t; ++pos) {
    if (pos < 0 || pos < p0 || pos >= p0 + len) continue;
    double* rw = (double*)malloc(sizeof(double) * D);
    const uint8_t* src = swa_b + (size_t)(pos - p0) * rb;
    if (fmt == ORC_SWA_MXFP8) {
      orc_mxfp8_decode(src, D, rw);
    } else {
      for (int c = 0; c < D; ++c) {
        uint16_t bits;
        memcpy(&bits, src + 2 * c, 2);
        rw[c] = orc_bf16_value(bits);
      }
    }
    rows[n++] = rw;
  }
  return n;
}

int orc_attend(int B, int Tq, int Hm, int D, int cache_dtype, int n_cap,
               const uint8_t* main_codes, const uint8_t* main_scales, const uint16_t* main_bf16,
               const int32_t* n_entries, const uint16_t* q, const int32_t* topk, int k,
               const void* swa, int swa_fmt, int S, const int32_t* swa_len, const int64_t* swa_pos0,
               const int64_t* q_pos, int W, double scale, double* out, double* lse) {
  if (B < 0 || Tq < 0 || k < 0 || D % 16 || (swa_fmt == ORC_SWA_MXFP8 && D % 32) || W < 0 || (swa_fmt != ORC_SWA_BF16 && swa_fmt != ORC_SWA_MXFP8))
    return -1;
  const size_t rb = orc_swa_row_bytes(swa_fmt, D);
  int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(| : bad)
  for (int b = 0; b < B; ++b) {
    for (int t = 0; t < Tq; ++t) {
      size_t qi = (size_t)b * Tq + t;
      double* qq = (double*)malloc(sizeof(double) * Hm * D);
      for (int i = 0; i < Hm * D; ++i) qq[i] = orc_bf16_value(q[qi * Hm * D + i]);
      double** rows = (double**)malloc(sizeof(double*) * (size_t)(k + W + 1));
      int n = 0;
      for (int i = 0; i < k; ++i) {
        int32_t j = topk[qi * k + i];
        if (j < 0) continue;
        if (j >= n_entries[b] || j >= n_cap) { bad = 1; continue; }
        rows[n] = (double*)malloc(sizeof(double) * D);
        orc_load_entry(cache_dtype, D, (size_t)b * n_cap + j, main_codes, main_scales, main_bf16,
                       rows[n]);
        ++n;
      }
      int32_t len = swa_len[b] < S ? swa_len[b] : S;
      n = orc_window_rows(q_pos[qi], W, (const uint8_t*)swa + (size_t)b * S * rb, swa_fmt, D, swa_pos0[b], len,
                          rows, n);
      orc_attend_rows(Hm, D, qq, rows, n, scale, out + qi * Hm * D, lse ? lse + qi * Hm : NULL);
      for (int i = 0; i < n; ++i) free(rows[i]);
      free(rows);
      free(qq);
    }
  }
  return bad ? -2 : 0;
}

/* Dense attention, written out without the selection path's softmax: for
 * each head the weight of row e is 1 / sum_f exp(scale q.(c_f - c_e)) (the
 * softmax of the logits in its pairwise form, which needs no running maximum
 * and never overflows), and the output is sum_e weight_e c_e.  Quadratic in
 * the rows, so only for the small inputs of the dense-limit pin. */
static void orc_dense_head(int D, const double* qh, double* const* rows, int n, double scale, double* o) {
  double* dot = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int e = 0; e < n; ++e) {
    double acc = 0.0;
    for (int c = 0; c < D; ++c) acc += rows[e][c] * qh[c];
    dot[e] = acc;
  }
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  for (int e = 0; e < n; ++e) {
    double den = 0.0;
    for (int f = 0; f < n; ++f) den += exp(scale * (dot[f] - dot[e]));
    const double wgt = 1.0 / den;
    for (int c = 0; c < D; ++c) o[c] += wgt * rows[e][c];
  }
  free(dot);
}

int orc_attend_dense(int B, int Tq, int Hm, int D, int r, int cache_dtype, int n_cap,
                     const uint8_t* main_codes, const uint8_t* main_scales,
                     const uint16_t* main_bf16, const int32_t* n_entries, const uint16_t* q,
                     const void* swa, int swa_fmt, int S, const int32_t* swa_len, const int64_t* swa_pos0,
                     const int64_t* q_pos, int W, double scale, double* out) {
  if (B < 0 || Tq < 0 || D % 16 || (swa_fmt == ORC_SWA_MXFP8 && D % 32) || W < 0 || r < 1 || (swa_fmt != ORC_SWA_BF16 && swa_fmt != ORC_SWA_MXFP8))
    return -1;
  const size_t rb = orc_swa_row_bytes(swa_fmt, D);
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < B; ++b) {
    for (int t = 0; t < Tq; ++t) {
      size_t qi = (size_t)b * Tq + t;
      double* qq = (double*)malloc(sizeof(double) * Hm * D);
      for (int i = 0; i < Hm * D; ++i) qq[i] = orc_bf16_value(q[qi * Hm * D + i]);
      int64_t nv = orc_visible(q_pos[qi], r, n_entries[b]);
      double** rows = (double**)malloc(sizeof(double*) * (size_t)(nv + W + 1));
      int n = 0;
      for (int64_t j = 0; j < nv; ++j) {
        rows[n] = (double*)malloc(sizeof(double) * D);
        orc_load_entry(cache_dtype, D, (size_t)b * n_cap + j, main_codes, main_scales, main_bf16,
                       rows[n]);
        ++n;
      }
      int32_t len = swa_len[b] < S ? swa_len[b] : S;
      n = orc_window_rows(q_pos[qi], W, (const uint8_t*)swa + (size_t)b * S * rb, swa_fmt, D, swa_pos0[b], len,
                          rows, n);
      for (int h = 0; h < Hm; ++h) orc_dense_head(D, qq + (size_t)h * D, rows, n, scale, out + (qi * Hm + h) * D);
      for (int i = 0; i < n; ++i) free(rows[i]);
      free(rows);
      free(qq);
    }
  }
  return 0;
}
