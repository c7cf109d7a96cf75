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

/* Attention of all 16 heads of one query row over KV rows [row0, row1).
 * q: 16*576 bf16 bits; out: 16*512 doubles.  Returns 0, or -1 on allocation
 * failure. */
int mxo_attend(const uint16_t* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
               int64_t row0, int64_t row1, double sm_scale, double* out) {
  int64_t n = row1 - row0;
  memset(out, 0, sizeof(double) * MXO_HEADS * MXO_V);
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
  for (int h = 0; h < MXO_HEADS; ++h) {
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
