/*
 * csa_oracle.c — plain fp64 CPU oracle of the CSA indexer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only tests/, the smoke check and the CPU-baseline leg of the
 * benchmark do. It shares no code, header, table or constant with the CUDA
 * library; the two only see the same seeded input bytes.
 *
 * Every function restates one step of the method as the pages define it:
 *
 *   FlashMemory-DeepSeek-V4, "compressed_k format": a record is HEAD_DIM e4m3
 *     bytes followed by a 4-byte fp32 scale; k = e4m3(bytes) * scale.
 *   FlashMemory-DeepSeek-V4, "Retriever architecture":
 *     score = sigmoid( sum_heads( relu(k . q_h) * fused_w_h ) ), in [0, 1].
 *   FlashMemory-DeepSeek-V4, "Two-level recall algorithm", Level 2: keep the
 *     top-512 per query, over the full history or confined to the resident set
 *     (non-resident logits set to -inf, i.e. left out).
 *   BatchGen #153 commit log: relu is applied before the head-weighted sum;
 *     lengths count compressed records.
 *
 * Readings where the pages are silent:
 *   - e4m3 is the OCP "fn" variant (bias 7, no infinities, S.1111.111 = NaN).
 *   - The trailing scale is little-endian IEEE binary32.
 *   - All arithmetic is fp64 (the pages' `.float()` dequant rounds k to fp32,
 *     a relative change below 6e-8, far inside the tolerance).
 *   - Ties in the logit are broken by the lower logical position.
 *   - Fewer than k visible records: the tail is idx -1, score 0 (sigmoid(-inf)).
 *   - Invalid geometry (page id out of range, resident page past the length,
 *     request id out of range) drops the affected records and sets a flag bit.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC.
 * -ffp-contract=off keeps the result identical on x86 and Arm.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_D 128
#define OR_PAGE 64
#define OR_REC_BYTES (OR_D + 4)

/* Flag bits reported by the oracle (the oracle's own numbering). */
#define OR_FLAG_PAGE_OOB 1
#define OR_FLAG_RESIDENT_OOB 2
#define OR_FLAG_RANGE 4
#define OR_FLAG_BAD_REQUEST 16
#define OR_FLAG_LEN_OOB 32

/* Host-side description of one indexer problem (the oracle's own type). */
typedef struct oracle_problem {
  const uint16_t* q;          /* [num_q, H, D] bf16 bit patterns */
  const float* w;             /* [num_q, H] */
  int32_t num_q, H, D;
  const uint8_t* kv;          /* page p at kv + p * page_stride */
  int64_t num_pages, page_stride;
  const int32_t* page_table;  /* [num_req, pt_stride] */
  int32_t num_req, pt_stride;
  const int32_t* q_req;       /* NULL = identity */
  const int32_t* q_len;
  const int32_t* resident;    /* NULL = full history */
  const int32_t* n_resident;
  int32_t res_stride;
  int32_t format;             /* records: 0 = e4m3 + fp32 scale (132 B), 1 = MXFP4 (68 B) */
} oracle_problem;

/* FP4 (MXFP4) variant, defined in its section at the end of this file. */
#define OR_FP4_BLOCK 32
#define OR_FP4_REC_BYTES (OR_D / 2 + OR_D / OR_FP4_BLOCK)
void oracle_mxfp4_round(const float* x, int64_t n, double* out);
void oracle_fp4_decode(const uint8_t* rec, double* k);

/* OCP FP8 E4M3 ("fn") byte -> value. E = 0: subnormal m/8 * 2^-6; otherwise
 * (1 + m/8) * 2^(E-7); E = 15 and m = 7 is NaN. */
double oracle_e4m3(uint8_t b) {
  int sign = b >> 7;
  int E = (b >> 3) & 15;
  int m = b & 7;
  double v;
  if (E == 15 && m == 7) return NAN;
  if (E == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, E - 7);
  return sign ? -v : v;
}

/* bf16 bit pattern -> value: the upper half of an IEEE binary32. */
double oracle_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Trailing scale: bytes 128..131 of the record, little-endian binary32. */
double oracle_scale(const uint8_t* rec) {
  uint32_t u = (uint32_t)rec[OR_D] | ((uint32_t)rec[OR_D + 1] << 8) |
               ((uint32_t)rec[OR_D + 2] << 16) | ((uint32_t)rec[OR_D + 3] << 24);
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Request of query row b, or -1 when out of range. */
static int32_t row_request(const oracle_problem* P, int32_t b, int32_t* flags) {
  int32_t req = P->q_req ? P->q_req[b] : b;
  if (req < 0 || req >= P->num_req) {
    *flags |= OR_FLAG_BAD_REQUEST;
    return -1;
  }
  return req;
}

/* Visible length of row b in records: q_len clamped to [0, 64 * pt_stride]. */
static int64_t row_length(const oracle_problem* P, int32_t b, int32_t* flags) {
  int64_t L = P->q_len[b];
  if (L < 0) {
    *flags |= OR_FLAG_LEN_OOB;
    L = 0;
  }
  if (L > (int64_t)OR_PAGE * P->pt_stride) {
    *flags |= OR_FLAG_LEN_OOB;
    L = (int64_t)OR_PAGE * P->pt_stride;
  }
  return L;
}

/*
 * Lists the visible records of row b: their logical positions and the score
 * column each one occupies (full mode: column = position; resident mode:
 * column = j*64 + r for the j-th listed page). Returns the count; `pos` and
 * `col` may be NULL to count only.
 */
int64_t oracle_visible(const oracle_problem* P, int32_t b, int64_t* pos, int64_t* col,
                       int32_t* flags_out) {
  int32_t flags = 0;
  int64_t n = 0;
  int32_t req = row_request(P, b, &flags);
  if (req >= 0) {
    int64_t L = row_length(P, b, &flags);
    int64_t npages = (L + OR_PAGE - 1) / OR_PAGE;
    if (!P->resident) {
      for (int64_t p = 0; p < npages; ++p) {
        int32_t phys = P->page_table[(int64_t)req * P->pt_stride + p];
        if (phys < 0 || phys >= P->num_pages) {
          flags |= OR_FLAG_PAGE_OOB;
          continue;
        }
        for (int64_t r = 0; r < OR_PAGE && p * OR_PAGE + r < L; ++r) {
          if (pos) pos[n] = p * OR_PAGE + r;
          if (col) col[n] = p * OR_PAGE + r;
          ++n;
        }
      }
    } else {
      int64_t nres = P->n_resident[req];
      if (nres < 0) {
        flags |= OR_FLAG_LEN_OOB;
        nres = 0;
      }
      if (nres > P->res_stride) {
        flags |= OR_FLAG_LEN_OOB;
        nres = P->res_stride;
      }
      for (int64_t j = 0; j < nres; ++j) {
        int64_t p = P->resident[(int64_t)req * P->res_stride + j];
        if (p < 0 || p >= npages) {
          flags |= OR_FLAG_RESIDENT_OOB;
          continue;
        }
        int32_t phys = P->page_table[(int64_t)req * P->pt_stride + p];
        if (phys < 0 || phys >= P->num_pages) {
          flags |= OR_FLAG_PAGE_OOB;
          continue;
        }
        for (int64_t r = 0; r < OR_PAGE && p * OR_PAGE + r < L; ++r) {
          if (pos) pos[n] = p * OR_PAGE + r;
          if (col) col[n] = j * OR_PAGE + r;
          ++n;
        }
      }
    }
  }
  if (flags_out) *flags_out |= flags;
  return n;
}

/* q of row b decoded to fp64 and stored d-major: qT[d*H + h] = q[b][h][d]; with
 * MXFP4 records the query is block-rounded the same way, head by head. */
static void decode_query(const oracle_problem* P, int32_t b, double* qT) {
  const int H = P->H;
  const uint16_t* qb = P->q + (int64_t)b * H * OR_D;
  for (int h = 0; h < H; ++h)
    for (int d = 0; d < OR_D; ++d) qT[d * H + h] = oracle_bf16(qb[h * OR_D + d]);
  if (P->format == 1) {
    for (int h = 0; h < H; ++h) {
      float qf[OR_D];
      double qr[OR_D];
      for (int d = 0; d < OR_D; ++d) qf[d] = (float)qT[d * H + h];
      oracle_mxfp4_round(qf, OR_D, qr);
      for (int d = 0; d < OR_D; ++d) qT[d * H + h] = qr[d];
    }
  }
}

/*
 * logit of row b at a visible logical position, given the row's decoded query:
 * sum over heads of relu(k . q_h) * w_h, with k the dequantised record.
 * Each head's dot product is accumulated over d = 0..D-1 in order; the loop
 * runs d outermost so that all heads advance together, which leaves each
 * head's summation order unchanged.
 */
static double logit_at(const oracle_problem* P, int32_t b, const double* qT, int64_t position) {
  const int H = P->H;
  int32_t req = P->q_req ? P->q_req[b] : b;
  int64_t p = position / OR_PAGE, r = position % OR_PAGE;
  int32_t phys = P->page_table[(int64_t)req * P->pt_stride + p];
  const uint8_t* rec = P->kv + (int64_t)phys * P->page_stride + r * (P->format == 1 ? OR_FP4_REC_BYTES : OR_REC_BYTES);
  double dot[256];
  for (int h = 0; h < H; ++h) dot[h] = 0.0;
  if (P->format == 1) {
    double k[OR_D];
    oracle_fp4_decode(rec, k); /* dequantise: e2m1 codes times their block scales */
    for (int d = 0; d < OR_D; ++d) {
      const double* qd = qT + d * H;
      for (int h = 0; h < H; ++h) dot[h] += k[d] * qd[h];
    }
  } else {
    const double s = oracle_scale(rec);
    for (int d = 0; d < OR_D; ++d) {
      const double kd = oracle_e4m3(rec[d]) * s; /* dequantise: e4m3 value times scale */
      const double* qd = qT + d * H;
      for (int h = 0; h < H; ++h) dot[h] += kd * qd[h];
    }
  }
  double logit = 0.0;
  for (int h = 0; h < H; ++h) {
    const double relu = dot[h] > 0.0 ? dot[h] : 0.0; /* relu before the weighted sum */
    logit += relu * (double)P->w[(int64_t)b * H + h];
  }
  return logit;
}

/* logit of row b at one visible logical position (decodes q itself). */
double oracle_logit(const oracle_problem* P, int32_t b, int64_t position) {
  double* qT = (double*)malloc(sizeof(double) * OR_D * P->H);
  decode_query(P, b, qT);
  double v = logit_at(P, b, qT, position);
  free(qT);
  return v;
}

double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * Logits of every visible record, in score-matrix layout: out[b*stride + col].
 * Invisible columns are left untouched; valid[b*stride + col] is set to 1 for
 * written columns (valid may be NULL). Returns the OR of the flag bits.
 */
int32_t oracle_logits(const oracle_problem* P, double* out, uint8_t* valid, int64_t stride) {
  int32_t flags = 0;
  for (int32_t b = 0; b < P->num_q; ++b) {
    int64_t n = oracle_visible(P, b, NULL, NULL, &flags);
    if (n == 0) continue;
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * n);
    int64_t* col = (int64_t*)malloc(sizeof(int64_t) * n);
    oracle_visible(P, b, pos, col, NULL);
    double* qT = (double*)malloc(sizeof(double) * OR_D * P->H);
    decode_query(P, b, qT);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
      out[(int64_t)b * stride + col[i]] = logit_at(P, b, qT, pos[i]);
      if (valid) valid[(int64_t)b * stride + col[i]] = 1;
    }
    free(qT);
    free(pos);
    free(col);
  }
  return flags;
}

typedef struct {
  double logit;
  int64_t pos;
} ranked;

/* Order: logit descending, then position ascending. */
static int by_logit_then_position(const void* a, const void* b) {
  const ranked* x = (const ranked*)a;
  const ranked* y = (const ranked*)b;
  if (x->logit > y->logit) return -1;
  if (x->logit < y->logit) return 1;
  return (x->pos > y->pos) - (x->pos < y->pos);
}

/*
 * Top-k of every row: idx[b*k + i] (logical position, -1 padding), score
 * (sigmoid of the logit, 0 for padding) and logit (-inf for padding).
 * Any of score / logit may be NULL. Returns the OR of the flag bits.
 */
int32_t oracle_topk(const oracle_problem* P, int32_t k, int32_t* idx, double* score,
                    double* logit) {
  int32_t flags = 0;
  for (int32_t b = 0; b < P->num_q; ++b) {
    int64_t n = oracle_visible(P, b, NULL, NULL, &flags);
    ranked* all = (ranked*)malloc(sizeof(ranked) * (n > 0 ? n : 1));
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (n > 0 ? n : 1));
    oracle_visible(P, b, pos, NULL, NULL);
    double* qT = (double*)malloc(sizeof(double) * OR_D * P->H);
    decode_query(P, b, qT);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
      all[i].logit = logit_at(P, b, qT, pos[i]);
      all[i].pos = pos[i];
    }
    free(qT);
    qsort(all, (size_t)n, sizeof(ranked), by_logit_then_position);
    for (int32_t i = 0; i < k; ++i) {
      int64_t o = (int64_t)b * k + i;
      if (i < n) {
        idx[o] = (int32_t)all[i].pos;
        if (score) score[o] = oracle_sigmoid(all[i].logit);
        if (logit) logit[o] = all[i].logit;
      } else {
        idx[o] = -1;
        if (score) score[o] = 0.0;
        if (logit) logit[o] = -INFINITY;
      }
    }
    free(all);
    free(pos);
  }
  return flags;
}

/*
 * Same as oracle_topk for rows [b0, b1) only and for at most `max_records`
 * visible records per row (the first ones in column order). Used to time the
 * oracle on a bounded sample of a large workload.
 */
int64_t oracle_topk_sample(const oracle_problem* P, int32_t b0, int32_t b1, int64_t max_records,
                           int32_t k, int32_t* idx, double* score) {
  int64_t scored = 0;
  for (int32_t b = b0; b < b1; ++b) {
    int32_t flags = 0;
    int64_t n = oracle_visible(P, b, NULL, NULL, &flags);
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (n > 0 ? n : 1));
    oracle_visible(P, b, pos, NULL, NULL);
    if (n > max_records) n = max_records;
    ranked* all = (ranked*)malloc(sizeof(ranked) * (n > 0 ? n : 1));
    double* qT = (double*)malloc(sizeof(double) * OR_D * P->H);
    decode_query(P, b, qT);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
      all[i].logit = logit_at(P, b, qT, pos[i]);
      all[i].pos = pos[i];
    }
    free(qT);
    qsort(all, (size_t)n, sizeof(ranked), by_logit_then_position);
    for (int32_t i = 0; i < k; ++i) {
      int64_t o = (int64_t)(b - b0) * k + i;
      idx[o] = i < n ? (int32_t)all[i].pos : -1;
      if (score) score[o] = i < n ? oracle_sigmoid(all[i].logit) : 0.0;
    }
    scored += n;
    free(all);
    free(pos);
  }
  return scored;
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
int32_t oracle_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ writer
 *
 * The compressed-K writer, the step before the path: it quantises new key rows
 * into the record format and stores them in the paged cache.
 * FlashMemory-DeepSeek-V4, "compressed_k format" fixes the record (HEAD_DIM e4m3
 * bytes, then the fp32 scale; k = e4m3 * scale); the BatchGen #153 commit log
 * names a store kernel that writes the indexer pool in that [128B fp8 | 4B fp32
 * scale] layout. The scale and the rounding are the plainest reading of that
 * format and of the workloads' "fp32 scale = amax/448" (448 = largest e4m3):
 *   amax  = max_d |x_d|                      (exact)
 *   scale = amax / 448                       (binary32 division, nearest even)
 *   c_d   = e4m3(x_d / scale)                (x_d / scale in binary32, then the
 *                                            nearest e4m3 value, ties to the even
 *                                            mantissa; magnitudes past 448 saturate)
 *   a row whose scale is 0 (amax == 0, or amax so small that amax / 448
 *   underflows) is stored as zero codes and scale 0.
 * The code is decided in binary32, the precision of the pages' torch cast.
 */

/* binary32 -> OCP E4M3 "fn" byte: the nearest of the 127 non-negative finite
 * e4m3 values (searched one by one), ties to the even mantissa, with the sign of
 * the input. Values beyond 448, infinities included, get 448 (saturation). NaN
 * gives the NaN code 0x7F. */
uint8_t oracle_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);  /* the largest value is the nearest (infinities too) */
  int best = 0;
  double best_d = a;  /* distance to code 0 (value 0) */
  for (int c = 1; c < 127; ++c) {
    const double d = fabs(a - oracle_e4m3((uint8_t)c));
    if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

void oracle_e4m3_encode_many(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

/* One record from one row of OR_D binary32 values; returns OR_FLAG_RANGE (and
 * writes nothing) if a value is not finite. */
int32_t oracle_quantise_row(const float* x, uint8_t* rec) {
  float amax = 0.0f;
  for (int d = 0; d < OR_D; ++d) {
    if (!isfinite(x[d])) return OR_FLAG_RANGE;
    const float a = fabsf(x[d]);
    if (a > amax) amax = a;
  }
  const float scale = amax / 448.0f;
  for (int d = 0; d < OR_D; ++d) {
    if (scale == 0.0f) {
      rec[d] = 0;
    } else {
      const float y = x[d] / scale;
      rec[d] = oracle_e4m3_encode(y);
    }
  }
  uint32_t bits;
  memcpy(&bits, &scale, 4);
  for (int j = 0; j < 4; ++j) rec[OR_D + j] = (uint8_t)(bits >> (8 * j));  /* little-endian */
  return 0;
}

/*
 * Writes n rows into the cache in place. keys [n, OR_D] binary32 (bf16 rows are
 * widened exactly by the caller); row i goes to request req[i] (req NULL: request
 * i) at logical position pos[i]: physical page page_table[req][pos / 64], record
 * pos % 64. A row with a request outside [0, num_req), a position outside
 * [0, 64 * pt_stride), a physical page outside [0, num_pages) or a non-finite
 * value is skipped and flagged. Returns the OR of the flags.
 */
int32_t oracle_write_keys(const float* keys, int64_t n, const int32_t* req, const int32_t* pos, uint8_t* kv,
                          int64_t num_pages, int64_t page_stride, const int32_t* page_table, int32_t num_req,
                          int32_t pt_stride) {
  int32_t flags = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t r = req ? req[i] : i;
    if (r < 0 || r >= num_req) {
      flags |= OR_FLAG_BAD_REQUEST;
      continue;
    }
    const int64_t p = pos[i];
    if (p < 0 || p >= (int64_t)OR_PAGE * pt_stride) {
      flags |= OR_FLAG_LEN_OOB;
      continue;
    }
    const int64_t phys = page_table[r * pt_stride + p / OR_PAGE];
    if (phys < 0 || phys >= num_pages) {
      flags |= OR_FLAG_PAGE_OOB;
      continue;
    }
    uint8_t rec[OR_REC_BYTES];
    const int32_t f = oracle_quantise_row(keys + i * OR_D, rec);
    if (f) {
      flags |= f;
      continue;
    }
    memcpy(kv + phys * page_stride + (p % OR_PAGE) * OR_REC_BYTES, rec, OR_REC_BYTES);
  }
  return flags;
}

/* ------------------------------------------------------------------ Level-1 recall
 *
 * FlashMemory-DeepSeek-V4, "Two-level recall algorithm", Level 1, and "Joint
 * checkpoint + ensemble": the Memory Indexer scores the full history of each
 * query row at the target layers (each with its own 128-head query, weights
 * and compressed keys), the per-layer sigmoid scores are ensembled per chunk
 * (max, the default "union", or mean), and the resident set is the chunks whose
 * ensemble score reaches the threshold plus the recency tail and the attention
 * sink ("threshold + recent + sink"). The pages print neither the threshold nor
 * the tail and sink sizes: they are parameters here.
 *
 * keep [num_q, keep_stride]: 1 / 0 for positions below the row's visible
 * length; scores: the ensemble scores there (fp64). pages [num_q, pages_stride]:
 * the logical pages holding a resident chunk, ascending; n_pages their count.
 * The layers share num_q, num_req and pt_stride (not checked here); the rows
 * (q_len, q_req) are layer 0's in every layer. Reading for invalid geometry
 * (the pages do not speak of it): a chunk whose page is out of range in a
 * layer has no score from that layer and counts 0 there; the flag is raised.
 */
int32_t oracle_recall(const oracle_problem* layers, int32_t n_layers, int32_t ensemble_mean, double threshold,
                      int64_t sink, int64_t recent, uint8_t* keep, int64_t keep_stride, double* scores,
                      int32_t* pages, int32_t pages_stride, int32_t* n_pages) {
  const int32_t num_q = layers[0].num_q;
  const int64_t cells = (int64_t)num_q * keep_stride;
  double* logit = (double*)malloc(sizeof(double) * (cells > 0 ? cells : 1));
  uint8_t* valid = (uint8_t*)malloc(cells > 0 ? cells : 1);
  double* acc = (double*)calloc(cells > 0 ? cells : 1, sizeof(double));
  int64_t* len = (int64_t*)calloc(num_q > 0 ? num_q : 1, sizeof(int64_t));
  int32_t flags = 0;
  for (int32_t b = 0; b < num_q; ++b)
    len[b] = row_request(&layers[0], b, &flags) < 0 ? 0 : row_length(&layers[0], b, &flags);
  for (int32_t l = 0; l < n_layers; ++l) {
    oracle_problem P = layers[l];
    P.q_len = layers[0].q_len;
    P.q_req = layers[0].q_req;
    memset(valid, 0, cells > 0 ? cells : 1);
    flags |= oracle_logits(&P, logit, valid, keep_stride);
    for (int32_t b = 0; b < num_q; ++b) {
      for (int64_t n = 0; n < len[b]; ++n) {
        const int64_t o = (int64_t)b * keep_stride + n;
        const double sc = valid[o] ? oracle_sigmoid(logit[o]) : 0.0;
        double* a = &acc[o];
        if (l == 0)
          *a = sc;
        else
          *a = ensemble_mean ? *a + sc : (sc > *a ? sc : *a);
      }
    }
  }
  for (int32_t b = 0; b < num_q; ++b) {
    const int64_t L = len[b];
    int32_t listed = 0;
    int64_t last_page = -1;
    for (int64_t n = 0; n < L; ++n) {
      const int64_t o = (int64_t)b * keep_stride + n;
      const double e = ensemble_mean ? acc[o] / n_layers : acc[o];
      const int k = e >= threshold || n < sink || n >= L - recent;
      keep[o] = (uint8_t)k;
      if (scores) scores[o] = e;
      if (k && n / OR_PAGE != last_page) {
        last_page = n / OR_PAGE;
        pages[(int64_t)b * pages_stride + listed++] = (int32_t)last_page;
      }
    }
    n_pages[b] = listed;
  }
  free(logit);
  free(valid);
  free(acc);
  free(len);
  return flags;
}

/* ------------------------------------------------------------------ FP4 (MXFP4) variant
 *
 * BatchGen #153 commit log (the indexer quantisation notes) and the V4.1 runtime
 * page: the published model FP4-rounds the index query and key alike (e2m1,
 * "MXFP4", cvt.e2m1x2) before the index score. The pages name the element type
 * and MXFP4 but print neither the block size nor a record layout. Readings
 * follow the OCP MX format for MXFP4:
 *   - blocks of 32 consecutive elements along head_dim share one UE8M0 scale
 *     X = 2^(floor(log2(amax)) - 2), 2 being the largest e2m1 exponent; the
 *     exponent is clamped to [-127, 127]; a block of zeros takes X = 2^-127;
 *   - an element is stored as the nearest e2m1 value of x / X, ties to the even
 *     mantissa, magnitudes past 6 saturating to 6;
 *   - a key record is 64 bytes of codes (element 2j in the low nibble of byte j)
 *     followed by the 4 UE8M0 bytes of its blocks, 68 bytes; 64 records a page.
 * The logit is the indexer's, on the dequantised values:
 *   logit = sum_h relu(k . q_h) * w_h, with k and q_h both MXFP4-rounded.
 */
/* e2m1 code (4 bits): sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0;
 * exponent 0 is subnormal (value = mantissa * 0.5). No infinities or NaNs. */
double oracle_e2m1(uint8_t code) {
  const int sign = (code >> 3) & 1, E = (code >> 1) & 3, m = code & 1;
  const double v = E == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, E - 1);
  return sign ? -v : v;
}

/* UE8M0 scale byte: 2^(e - 127); 255 is NaN. */
double oracle_ue8m0(uint8_t e) { return e == 255 ? NAN : ldexp(1.0, (int)e - 127); }

/* Nearest e2m1 code of v (already divided by its block scale): every one of the
 * 8 magnitudes is tried; the closer wins, a tie goes to the even mantissa;
 * magnitudes at or past 6 saturate. */
uint8_t oracle_e2m1_encode(double v) {
  const uint8_t sign = (v < 0 || (v == 0 && signbit(v))) ? 8 : 0;
  const double a = fabs(v);
  if (a >= 6.0) return sign | 7;
  uint8_t best = 0;
  double best_d = INFINITY;
  for (uint8_t c = 0; c < 8; ++c) {
    const double d = fabs(oracle_e2m1(c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_d = d;
    }
  }
  return sign | best;
}

/* One block of 32 values: its UE8M0 scale byte and 32 codes (one per byte). */
void oracle_mxfp4_block(const float* x, uint8_t* codes, uint8_t* scale) {
  double amax = 0.0;
  for (int i = 0; i < OR_FP4_BLOCK; ++i) amax = fmax(amax, fabs((double)x[i]));
  int e = -127;
  if (amax > 0.0) {
    int E2;
    (void)frexp(amax, &E2); /* amax = f * 2^E2, f in [0.5, 1): floor(log2 amax) = E2 - 1 */
    e = (E2 - 1) - 2;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
  }
  *scale = (uint8_t)(e + 127);
  const double X = ldexp(1.0, e);
  for (int i = 0; i < OR_FP4_BLOCK; ++i) codes[i] = oracle_e2m1_encode((double)x[i] / X);
}

/* n values (n a multiple of 32) quantised and dequantised block by block. */
void oracle_mxfp4_round(const float* x, int64_t n, double* out) {
  uint8_t codes[OR_FP4_BLOCK], sc;
  for (int64_t b = 0; b + OR_FP4_BLOCK <= n; b += OR_FP4_BLOCK) {
    oracle_mxfp4_block(x + b, codes, &sc);
    for (int i = 0; i < OR_FP4_BLOCK; ++i) out[b + i] = oracle_e2m1(codes[i]) * oracle_ue8m0(sc);
  }
}

/* A key row of 128 values as a 68-byte FP4 record. */
void oracle_fp4_record(const float* x, uint8_t* rec) {
  uint8_t codes[OR_D];
  for (int blk = 0; blk < OR_D / OR_FP4_BLOCK; ++blk)
    oracle_mxfp4_block(x + blk * OR_FP4_BLOCK, codes + blk * OR_FP4_BLOCK, rec + OR_D / 2 + blk);
  for (int j = 0; j < OR_D / 2; ++j) rec[j] = (uint8_t)((codes[2 * j] & 15) | ((codes[2 * j + 1] & 15) << 4));
}

/* The 128 key values a 68-byte FP4 record holds. */
void oracle_fp4_decode(const uint8_t* rec, double* k) {
  for (int d = 0; d < OR_D; ++d) {
    const uint8_t code = (uint8_t)((rec[d / 2] >> (4 * (d & 1))) & 15);
    k[d] = oracle_e2m1(code) * oracle_ue8m0(rec[OR_D / 2 + d / OR_FP4_BLOCK]);
  }
}

/* Logit of one FP4 key record against an H-head bf16 query (bit patterns,
 * [H][128]) and fp32 head weights: both sides MXFP4-rounded, then the indexer's
 * relu'd, head-weighted sum in fp64. */
double oracle_fp4_logit(const uint8_t* rec, const uint16_t* q, const float* w, int32_t H) {
  double k[OR_D];
  oracle_fp4_decode(rec, k);
  double logit = 0.0;
  for (int32_t h = 0; h < H; ++h) {
    float qf[OR_D];
    double qr[OR_D];
    for (int d = 0; d < OR_D; ++d) qf[d] = (float)oracle_bf16(q[(int64_t)h * OR_D + d]);
    oracle_mxfp4_round(qf, OR_D, qr);
    double dot = 0.0;
    for (int d = 0; d < OR_D; ++d) dot += k[d] * qr[d];
    const double relu = dot > 0.0 ? dot : 0.0;
    logit += relu * (double)w[h];
  }
  return logit;
}

/* Key rows written into a paged MXFP4 cache: the 68-byte record of row i goes to
 * page_table[req][pos / 64], row pos % 64. The same checks as oracle_write_keys,
 * in the same order (request, position, page, a non-finite value): a failing row
 * is skipped and its flag bit set. */
int32_t oracle_fp4_write_keys(const float* keys, int64_t n, const int32_t* req, const int32_t* pos, uint8_t* kv,
                              int64_t num_pages, int64_t page_stride, const int32_t* page_table, int32_t num_req,
                              int32_t pt_stride) {
  int32_t flags = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t r = req ? req[i] : i;
    if (r < 0 || r >= num_req) {
      flags |= OR_FLAG_BAD_REQUEST;
      continue;
    }
    const int64_t p = pos[i];
    if (p < 0 || p >= (int64_t)OR_PAGE * pt_stride) {
      flags |= OR_FLAG_LEN_OOB;
      continue;
    }
    const int64_t phys = page_table[r * pt_stride + p / OR_PAGE];
    if (phys < 0 || phys >= num_pages) {
      flags |= OR_FLAG_PAGE_OOB;
      continue;
    }
    int finite = 1;
    for (int d = 0; d < OR_D; ++d) finite &= isfinite(keys[i * OR_D + d]) ? 1 : 0;
    if (!finite) {
      flags |= OR_FLAG_RANGE;
      continue;
    }
    oracle_fp4_record(keys + i * OR_D, kv + phys * page_stride + (p % OR_PAGE) * OR_FP4_REC_BYTES);
  }
  return flags;
}
