/*
 * Plain fp64 CPU oracle for MXFP4 MLA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test suite, the smoke check and the bench's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (single-token decode, absorbed MLA, one shared KV head):
 *   K[t][d] = e2m1(code[t][d]) * 2^(scale[t][d/32] - 127),  d < 576
 *   V[t][d] = K[t][d],                                         d < 512
 *   s_t     = sm_scale * sum_d q[h][d] * K[t][d]
 *   out[h]  = sum_t softmax(s)_t * V[t]          (empty sequence -> zeros)
 * Sources (kernelindex "amd-mixed-mla" submissions):
 *   - 608791, HIP common source: the e2m1 table kFp4Lut, e8m0_to_float
 *     (0x00 -> 2^-127, 0xFF -> NaN), unpack_mxfp4 (low nibble = even element),
 *     block of 32 elements per scale;
 *   - 717900, "_nibble_to_f32": sign / 2-bit exponent / 1-bit mantissa decode;
 *     layout comment "byte j -> fp4[2j] in bits[3:0], fp4[2j+1] in bits[7:4]";
 *   - 676098, "_naive_fallback": scores = q.k * sm_scale, softmax over the
 *     sequence's tokens, weighted sum of V = first 512 dims of the same row;
 *   - 608791, "mla_reduce_v1_like_kernel" and 676098 "_mla_reduce_kernel":
 *     split partials (normalised acc, lse) merged with weights exp(lse - max),
 *     empty splits skipped, all-empty -> zeros.
 * Everything is fp64; inputs q are bf16 bit patterns widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MXO_HEADS 16
#define MXO_QK 576
#define MXO_V 512
#define MXO_PACKED 288
#define MXO_NSCALE 18

/* e2m1 code -> value, as the table printed on page 608791 (codes 8..15 are the
 * negatives of 0..7, code 8 is -0). */
static const double kE2m1Table[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0};

double mxo_e2m1_table(int code) { return kE2m1Table[code & 15]; }

/* e2m1 code -> value from its fields (page 717900, _nibble_to_f32):
 * sign = bit 3, exponent = bits 2..1, mantissa = bit 0;
 * exponent 0 -> mantissa * 0.5, else (1 + mantissa/2) * 2^(exponent-1). */
double mxo_e2m1_fields(int code) {
  int sign = (code >> 3) & 1, ex = (code >> 1) & 3, man = code & 1;
  double mag = (ex == 0) ? man * 0.5 : (1.0 + man * 0.5) * ldexp(1.0, ex - 1);
  return sign ? -mag : mag;
}

/* E8M0 byte -> 2^(b-127); 0xFF encodes NaN (page 608791, e8m0_to_float). */
double mxo_e8m0(int b) {
  if ((b & 255) == 255) return NAN;
  return ldexp(1.0, (b & 255) - 127);
}

double mxo_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), directly from the exact
 * value: quantum = 2^(floor(log2|x|) - 7) for normals, 2^-133 below 2^-126. */
uint16_t mxo_double_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  double ax = fabs(x), r;
  if (ax == 0.0) {
    r = x;
  } else {
    int e;
    frexp(ax, &e); /* ax = m * 2^e, m in [0.5,1): floor(log2 ax) = e - 1 */
    int qexp = (e - 1 >= -126) ? (e - 1 - 7) : -133;
    r = ldexp(nearbyint(ldexp(x, -qexp)), qexp); /* default rounding: to even */
  }
  float f = (float)r; /* exact: r is a bf16 value (or overflows to inf) */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* Dequantise one token: 288 packed bytes + 18 scale bytes -> 576 doubles. */
void mxo_dequant_token(const uint8_t* packed, const uint8_t* scale, double* k) {
  for (int d = 0; d < MXO_QK; ++d) {
    uint8_t byte = packed[d / 2];
    int code = (d % 2 == 0) ? (byte & 15) : (byte >> 4);
    k[d] = mxo_e2m1_table(code) * mxo_e8m0(scale[d / 32]);
  }
}

int mxo_attend_heads(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                     int64_t row0, int64_t row1, double sm_scale, int h0, int h1, double* out);

/* Attention of all 16 heads of one query row over KV rows [row0, row1).
 * q: 16*576 bf16 bits; out: 16*512 doubles.  Returns 0, or -1 on allocation
 * failure. */
int mxo_attend(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
               int64_t row0, int64_t row1, double sm_scale, double* out) {
  return mxo_attend_heads(q, kv_packed, kv_scale, row0, row1, sm_scale, 0, MXO_HEADS, out);
}

/* Heads [h0, h1) of the above (out rows of the other heads are left untouched). */
int mxo_attend_heads(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                     int64_t row0, int64_t row1, double sm_scale, int h0, int h1, double* out) {
  int64_t n = row1 - row0;
  memset(out + (size_t)h0 * MXO_V, 0, sizeof(double) * (size_t)(h1 - h0) * MXO_V);
  if (n <= 0) return 0;
  double* k = (double*)malloc(sizeof(double) * (size_t)n * MXO_QK);
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  if (!k || !s) {
    free(k);
    free(s);
    return -1;
  }
  for (int64_t t = 0; t < n; ++t)
    mxo_dequant_token(kv_packed + (row0 + t) * MXO_PACKED, kv_scale + (row0 + t) * MXO_NSCALE,
                      k + t * MXO_QK);
  for (int h = h0; h < h1; ++h) {
    double qd[MXO_QK];
    for (int d = 0; d < MXO_QK; ++d) qd[d] = mxo_bf16_to_double(q[h * MXO_QK + d]);
    double m = -INFINITY;
    int any_nan = 0;
    for (int64_t t = 0; t < n; ++t) {
      double dot = 0.0;
      for (int d = 0; d < MXO_QK; ++d) dot += qd[d] * k[t * MXO_QK + d];
      s[t] = sm_scale * dot;
      if (isnan(s[t])) any_nan = 1;
      else if (s[t] > m) m = s[t];
    }
    double* o = out + h * MXO_V;
    if (any_nan) {
      for (int d = 0; d < MXO_V; ++d) o[d] = NAN;
      continue;
    }
    double l = 0.0;
    for (int64_t t = 0; t < n; ++t) {
      double w = exp(s[t] - m);
      l += w;
      for (int d = 0; d < MXO_V; ++d) o[d] += w * k[t * MXO_QK + d];
    }
    for (int d = 0; d < MXO_V; ++d) o[d] /= l;
  }
  free(k);
  free(s);
  return 0;
}

/* Whole decode call: q [batch,16,576] bf16 bits, kv_indptr [batch+1],
 * out [batch,16,512] doubles. */
int mxo_decode(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
               const int32_t* kv_indptr, int batch, double sm_scale, double* out) {
  for (int b = 0; b < batch; ++b) {
    int rc = mxo_attend(q + (size_t)b * MXO_HEADS * MXO_QK, kv_packed, kv_scale, kv_indptr[b],
                        kv_indptr[b + 1], sm_scale, out + (size_t)b * MXO_HEADS * MXO_V);
    if (rc) return rc;
  }
  return 0;
}

/* The same decode with the (sequence, head) pairs spread over `nthreads` OpenMP
 * threads (each pair runs the single-threaded code above for one head, so every
 * output element is computed by exactly the same operations in the same order).
 * Built without OpenMP it runs on one thread.  Returns 0, or -1 on allocation
 * failure. */

int mxo_decode_mt(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                  const int32_t* kv_indptr, int batch, double sm_scale, double* out, int nthreads) {
  int rc = 0;
  if (nthreads < 1) nthreads = 1;
  /* a whole sequence per task when there are enough sequences (the dequantised rows
   * are then shared by its 16 heads), else one task per (sequence, head) */
  const int per_head = batch < 2 * nthreads;
  const int64_t tasks = per_head ? (int64_t)batch * MXO_HEADS : batch;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : rc)
#endif
  for (int64_t i = 0; i < tasks; ++i) {
    const int b = per_head ? (int)(i / MXO_HEADS) : (int)i;
    const int h0 = per_head ? (int)(i % MXO_HEADS) : 0, h1 = per_head ? h0 + 1 : MXO_HEADS;
    rc |= mxo_attend_heads(q + (size_t)b * MXO_HEADS * MXO_QK, kv_packed, kv_scale, kv_indptr[b],
                           kv_indptr[b + 1], sm_scale, h0, h1, out + (size_t)b * MXO_HEADS * MXO_V);
  }
  return rc;
}

/* Threads an OpenMP region would use by default (1 without OpenMP), and the host's
 * online processors. */
int mxo_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
int mxo_online_cpus(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }

/* ---- query rows, paged KV, fp8 KV --------------------------------------------
 * Several query rows per sequence (676098, "_naive_fallback": q rows [qo_indptr[b],
 * qo_indptr[b+1]) of sequence b each attend, with no mask, to all of b's KV rows).
 * q [total_q,16,576], out [total_q,16,512]. */
int mxo_decode_rows(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                    const int32_t* qo_indptr, const int32_t* kv_indptr, int batch, double sm_scale,
                    double* out) {
  for (int b = 0; b < batch; ++b) {
    for (int r = qo_indptr[b]; r < qo_indptr[b + 1]; ++r) {
      int rc = mxo_attend(q + (size_t)r * MXO_HEADS * MXO_QK, kv_packed, kv_scale, kv_indptr[b],
                          kv_indptr[b + 1], sm_scale, out + (size_t)r * MXO_HEADS * MXO_V);
      if (rc) return rc;
    }
  }
  return 0;
}

/* Paged KV (676098, "_aiter_mla_decode": kv_indptr counts pages of kv_indices, kv_last_page_len
 * the rows used in each sequence's last page): sequence b's KV rows are, in order, rows
 * page * page_size + o of its pages kv_indices[kv_indptr[b] .. kv_indptr[b+1]), o < page_size
 * for every page but the last and o < kv_last_page_len[b] for the last.  The attention is
 * then the one above over those rows, gathered into a contiguous copy. */
int mxo_decode_paged(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                     const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                     const int32_t* kv_last_page_len, int page_size, int batch, double sm_scale,
                     double* out) {
  for (int b = 0; b < batch; ++b) {
    const int npages = kv_indptr[b + 1] - kv_indptr[b];
    const int64_t n = npages > 0 ? (int64_t)(npages - 1) * page_size + kv_last_page_len[b] : 0;
    uint8_t* gp = (uint8_t*)malloc((size_t)(n > 0 ? n : 1) * MXO_PACKED);
    uint8_t* gs = (uint8_t*)malloc((size_t)(n > 0 ? n : 1) * MXO_NSCALE);
    if (!gp || !gs) {
      free(gp);
      free(gs);
      return -1;
    }
    for (int64_t t = 0; t < n; ++t) {
      const int64_t row = (int64_t)kv_indices[kv_indptr[b] + t / page_size] * page_size + t % page_size;
      memcpy(gp + t * MXO_PACKED, kv_packed + row * MXO_PACKED, MXO_PACKED);
      memcpy(gs + t * MXO_NSCALE, kv_scale + row * MXO_NSCALE, MXO_NSCALE);
    }
    const int r0 = qo_indptr ? qo_indptr[b] : b, r1 = qo_indptr ? qo_indptr[b + 1] : b + 1;
    int rc = 0;
    for (int r = r0; r < r1 && rc == 0; ++r)
      rc = mxo_attend(q + (size_t)r * MXO_HEADS * MXO_QK, gp, gs, 0, n, sm_scale,
                      out + (size_t)r * MXO_HEADS * MXO_V);
    free(gp);
    free(gs);
    if (rc) return rc;
  }
  return 0;
}

/* fp8 e4m3 ("fn": no infinities) byte -> value, from the format's fields: sign bit 7,
 * exponent bits 6..3 with bias 7, mantissa bits 2..0; exponent 0 is subnormal
 * (mantissa / 8 * 2^-6); exponent 15 with mantissa 7 is NaN (so 448 is the largest). */
double mxo_e4m3(int byte) {
  const int b = byte & 255, sign = b >> 7, ex = (b >> 3) & 15, man = b & 7;
  double mag;
  if (ex == 15 && man == 7) return NAN;
  if (ex == 0) mag = ldexp((double)man, -9);
  else mag = ldexp(1.0 + man / 8.0, ex - 7);
  return sign ? -mag : mag;
}

/* fp8 KV with one per-tensor scale (676098 "_aiter_mla_decode", 717900 "_decode"):
 * K[t][d] = e4m3(kv[t][d]) * kv_scale, V = K[:, :512]; the query is used as given (bf16).
 * kv [rows,576] bytes. */
int mxo_decode_fp8(const uint16_t* q, const uint8_t* kv, double kv_scale, const int32_t* kv_indptr,
                   int batch, double sm_scale, double* out) {
  for (int b = 0; b < batch; ++b) {
    const int64_t r0 = kv_indptr[b], n = kv_indptr[b + 1] - r0;
    double* o = out + (size_t)b * MXO_HEADS * MXO_V;
    memset(o, 0, sizeof(double) * MXO_HEADS * MXO_V);
    if (n <= 0) continue;
    double* k = (double*)malloc(sizeof(double) * (size_t)n * MXO_QK);
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    if (!k || !s) {
      free(k);
      free(s);
      return -1;
    }
    for (int64_t t = 0; t < n; ++t)
      for (int d = 0; d < MXO_QK; ++d) k[t * MXO_QK + d] = mxo_e4m3(kv[(r0 + t) * MXO_QK + d]) * kv_scale;
    for (int h = 0; h < MXO_HEADS; ++h) {
      double qd[MXO_QK];
      for (int d = 0; d < MXO_QK; ++d) qd[d] = mxo_bf16_to_double(q[((size_t)b * MXO_HEADS + h) * MXO_QK + d]);
      double m = -INFINITY;
      int any_nan = 0;
      for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int d = 0; d < MXO_QK; ++d) dot += qd[d] * k[t * MXO_QK + d];
        s[t] = sm_scale * dot;
        if (isnan(s[t])) any_nan = 1;
        else if (s[t] > m) m = s[t];
      }
      double* oh = o + h * MXO_V;
      if (any_nan) {
        for (int d = 0; d < MXO_V; ++d) oh[d] = NAN;
        continue;
      }
      double l = 0.0;
      for (int64_t t = 0; t < n; ++t) {
        const double w = exp(s[t] - m);
        l += w;
        for (int d = 0; d < MXO_V; ++d) oh[d] += w * k[t * MXO_QK + d];
      }
      for (int d = 0; d < MXO_V; ++d) oh[d] /= l;
    }
    free(k);
    free(s);
  }
  return 0;
}

/* Split mode: each sequence's rows are cut into `nsplit` contiguous chunks of
 * ceil(n/nsplit) rows (the last ones may be short or empty).  Per chunk and
 * head: normalised acc = sum w V / l and lse = m + ln l, with m the chunk max.
 * Merge: M = max lse over non-empty chunks, out = sum e^(lse-M) acc / sum e^(lse-M).
 * Used to pin that the merge is invariant to the split count. */
int mxo_decode_split(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                     const int32_t* kv_indptr, int batch, double sm_scale, int nsplit,
                     double* out) {
  if (nsplit < 1) return -2;
  double* acc = (double*)malloc(sizeof(double) * (size_t)nsplit * MXO_HEADS * MXO_V);
  double* lse = (double*)malloc(sizeof(double) * (size_t)nsplit * MXO_HEADS);
  int* nonempty = (int*)malloc(sizeof(int) * (size_t)nsplit);
  if (!acc || !lse || !nonempty) {
    free(acc);
    free(lse);
    free(nonempty);
    return -1;
  }
  int rc = 0;
  for (int b = 0; b < batch && rc == 0; ++b) {
    int64_t r0 = kv_indptr[b], r1 = kv_indptr[b + 1], n = r1 - r0;
    int64_t chunk = (n + nsplit - 1) / nsplit;
    const uint16_t* qb = q + (size_t)b * MXO_HEADS * MXO_QK;
    for (int c = 0; c < nsplit && rc == 0; ++c) {
      int64_t c0 = r0 + c * chunk, c1 = c0 + chunk;
      if (c0 > r1) c0 = r1;
      if (c1 > r1) c1 = r1;
      nonempty[c] = c1 > c0;
      if (!nonempty[c]) continue;
      /* normalised partial = attention over the chunk alone */
      rc = mxo_attend(qb, kv_packed, kv_scale, c0, c1, sm_scale, acc + (size_t)c * MXO_HEADS * MXO_V);
      /* its log-sum-exp, from the chunk's scores */
      double* k = (double*)malloc(sizeof(double) * MXO_QK);
      if (!k) { rc = -1; break; }
      for (int h = 0; h < MXO_HEADS; ++h) {
        double qd[MXO_QK];
        for (int d = 0; d < MXO_QK; ++d) qd[d] = mxo_bf16_to_double(qb[h * MXO_QK + d]);
        double m = -INFINITY, l = 0.0;
        for (int64_t t = c0; t < c1; ++t) {
          mxo_dequant_token(kv_packed + t * MXO_PACKED, kv_scale + t * MXO_NSCALE, k);
          double dot = 0.0;
          for (int d = 0; d < MXO_QK; ++d) dot += qd[d] * k[d];
          double st = sm_scale * dot;
          if (st > m) { l = l * exp(m - st) + 1.0; m = st; }
          else l += exp(st - m);
        }
        lse[c * MXO_HEADS + h] = m + log(l);
      }
      free(k);
    }
    for (int h = 0; h < MXO_HEADS; ++h) {
      double* o = out + ((size_t)b * MXO_HEADS + h) * MXO_V;
      double M = -INFINITY;
      for (int c = 0; c < nsplit; ++c)
        if (nonempty[c] && lse[c * MXO_HEADS + h] > M) M = lse[c * MXO_HEADS + h];
      for (int d = 0; d < MXO_V; ++d) o[d] = 0.0;
      if (M == -INFINITY) continue; /* every chunk empty */
      double L = 0.0;
      for (int c = 0; c < nsplit; ++c) {
        if (!nonempty[c]) continue;
        double w = exp(lse[c * MXO_HEADS + h] - M);
        L += w;
        const double* a = acc + ((size_t)c * MXO_HEADS + h) * MXO_V;
        for (int d = 0; d < MXO_V; ++d) o[d] += w * a[d];
      }
      for (int d = 0; d < MXO_V; ++d) o[d] /= L;
    }
  }
  free(acc);
  free(lse);
  free(nonempty);
  return rc;
}
