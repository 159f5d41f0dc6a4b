/*
 * fa_oracle.c -- plain FP64 reference for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it computes is the textbook definition, written out with no tiling,
 * no fusion and no reordering:
 *
 *   s_ij = scale * <q_i, k_j>                 (FlashAttention_01 page, 3.1 and
 *                                              the "Flash Attention" history
 *                                              page, 1.1: softmax(QK^T/sqrt d)V)
 *   visible(i, j) <=> k_start[b] <= j < k_end[b]  and  (!causal or j <= i + Sk - Sq)
 *                     and  key_mask[b][j] != 0 when a key mask is given
 *                     (per-key boolean mask, FlashAttention_01 page,
 *                     "interface and implementation constraints": masks and
 *                     ragged layouts are part of the kernel contract)
 *   m   = max over visible j of s_ij          (mask applied before the max,
 *   l   = sum_vis exp(s_ij - m)                FlashAttention_01 page, "online
 *   u   = sum_vis exp(s_ij - m) v_j            softmax derivation": m, l, u)
 *   O_i = u / l,  LSE_i = m + ln l
 *   no visible key: O_i = 0, LSE_i = -inf, m = -inf, l = 0 (no -inf - -inf
 *   is ever evaluated; the page asks for an explicit rule).
 *
 * Backward (FlashAttention_01 page, "backward recomputation" and the
 * "attention backward chain rule" section), with dO given:
 *   p_ij  = exp(s_ij - m_i) / l_i on visible entries, 0 elsewhere
 *   D_i   = sum_c dO_ic O_ic
 *   dP_ij = <dO_i, v_j>
 *   dS_ij = p_ij (dP_ij - D_i)
 *   dV_j  = sum_i p_ij dO_i
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j  = scale sum_i dS_ij q_i
 * With grouped K/V heads (GQA, "Flash Attention" practitioner page, 2.3)
 * query head h reads KV head h / (Hq/Hkv), and dK/dV of a KV head sum over
 * the query heads that read it.
 *
 * Dropout on the attention weights (FlashAttention_01 page, "why the
 * backward can recompute" and "interface and implementation constraints":
 * the random mask is part of the forward/backward contract and must be
 * reproduced element by element).  Weight (i, j) is dropped with
 * probability q = floor(p_drop * 2^16) / 2^16 (the draws are 16-bit) and the
 * kept ones are scaled by r = 1 / (1 - q), so each weight keeps its
 * expectation (inverted dropout):
 *   O_i   = u_i / l_i,  u_i = sum_vis exp(s_ij - m) keep_ij r v_j
 *   (m, l and LSE are those of the undropped weights)
 *   dP_ij = keep_ij r <dO_i, v_j>,  dV_j = sum_i p_ij keep_ij r dO_i
 * keep_ij comes from Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC 2011) with counter
 * (j / 8, i, b * Hq + h, offset) and key (seed low word, seed high word):
 * keep_ij <=> the 16-bit half (j mod 2) (0: low, 1: high) of word
 * ((j mod 8) / 2) is >= floor(p * 2^16).
 *
 * Inputs are either fp64 arrays or bf16 bit patterns (uint16); a bf16 value
 * is widened to fp64 exactly.  Layout is [B, H, S, d], d innermost.
 * OpenMP only distributes independent rows (or independent key rows for
 * dK/dV); every sum is evaluated in plain index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* exact bf16 -> fp64: a bf16 value is the top 16 bits of an IEEE binary32 */
static double bf16_bits_to_double(uint16_t h) {
  uint32_t w = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

typedef struct {
  const void* p;
  int bf16;
} src_t;

/* ---- Philox4x32-10, restated from the SC 2011 paper ----------------------
 * state: four 32-bit counter words and a two-word key.  One round maps
 * (c0, c1, c2, c3) to (hi(B*c2) ^ c1 ^ k0, lo(B*c2), hi(A*c0) ^ c3 ^ k1,
 * lo(A*c0)) with the paper's multipliers A, B; the key is advanced by the
 * paper's Weyl constants before every round but the first. */
static void philox4x32_10(const uint32_t ctr[4], uint32_t k0, uint32_t k1, uint32_t out[4]) {
  const uint64_t A = 0xD2511F53u, B = 0xCD9E8D57u;
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = A * (uint64_t)c0;
    const uint64_t p1 = B * (uint64_t)c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n1 = (uint32_t)p1;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    const uint32_t n3 = (uint32_t)p0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

void oracle_philox4x32_10(const uint32_t* ctr, uint32_t k0, uint32_t k1, uint32_t* out) {
  philox4x32_10(ctr, k0, k1, out);
}

typedef struct {
  int on;
  uint32_t thr;          /* floor(p * 2^16): keep iff the 16-bit draw is >= thr */
  double keep_scale;     /* 2^16 / (2^16 - thr): 1 / the keep probability */
  uint32_t seed_lo, seed_hi, offset;
} drop_t;

static drop_t make_drop(double p, unsigned long long seed, unsigned int offset) {
  drop_t d;
  d.on = p > 0.0;
  d.thr = d.on ? (uint32_t)floor(p * 65536.0) : 0u;
  d.keep_scale = d.on ? 65536.0 / (65536.0 - (double)d.thr) : 1.0;
  d.seed_lo = (uint32_t)(seed & 0xffffffffull);
  d.seed_hi = (uint32_t)(seed >> 32);
  d.offset = offset;
  return d;
}

/* keep_ij / P(keep) for query row i of query head bh (= b * Hq + h), key j */
static double drop_factor(const drop_t* d, long bh, long i, long j) {
  if (!d || !d->on) return 1.0;
  const uint32_t ctr[4] = {(uint32_t)(j / 8), (uint32_t)i, (uint32_t)bh, d->offset};
  uint32_t w[4];
  philox4x32_10(ctr, d->seed_lo, d->seed_hi, w);
  const uint32_t word = w[(j % 8) / 2];
  const uint32_t draw = (j % 2) ? (word >> 16) : (word & 0xffffu);
  return (draw >= d->thr) ? d->keep_scale : 0.0;
}

/* 1 when weight (i, j) of query head bh is kept, 0 when dropped */
int oracle_dropout_keep(double p, unsigned long long seed, unsigned int offset, long bh, long i,
                        long j) {
  const drop_t d = make_drop(p, seed, offset);
  return drop_factor(&d, bh, i, j) != 0.0;
}

static double ld(src_t s, long idx) {
  if (s.bf16) return bf16_bits_to_double(((const uint16_t*)s.p)[idx]);
  return ((const double*)s.p)[idx];
}

static void load_row(src_t s, long base, long d, double* out) {
  for (long c = 0; c < d; ++c) out[c] = ld(s, base + c);
}

/* km: this batch row's key mask (NULL: every key passes) */
static int is_visible(long i, long j, long Sq, long Sk, int causal, long ks, long ke,
                      const unsigned char* km) {
  if (j < ks || j >= ke) return 0;
  if (causal && j > i + Sk - Sq) return 0;
  if (km && !km[j]) return 0;
  return 1;
}

static const unsigned char* mask_row(const unsigned char* key_mask, long b, long Sk) {
  return key_mask ? key_mask + b * Sk : NULL;
}

static void key_range(const int* k_start, const int* k_end, long b, long Sk, long* ks, long* ke) {
  *ks = k_start ? (long)k_start[b] : 0;
  *ke = k_end ? (long)k_end[b] : Sk;
}

/*
 * One query row against n keys.  qrow[d]; key row j starts at index
 * kbase + j*d in k (and vbase + j*d in v).  Writes m, l, u[d], o[d], lse.
 * s is caller scratch of length >= n.
 */
static void row_attention(const double* qrow, src_t k, long kbase, src_t v, long vbase,
                          long n, long d, double scale, long i, long Sq, int causal,
                          long ks, long ke, const unsigned char* km, const drop_t* dr,
                          long bh, double* s, double* m_out, double* l_out,
                          double* u, double* o, double* lse_out) {
  double m = -INFINITY;
  long nvis = 0;
  for (long j = 0; j < n; ++j) {
    if (!is_visible(i, j, Sq, n, causal, ks, ke, km)) continue;
    double acc = 0.0;
    for (long c = 0; c < d; ++c) acc += qrow[c] * ld(k, kbase + j * d + c);
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
    ++nvis;
  }
  for (long c = 0; c < d; ++c) u[c] = 0.0;
  if (nvis == 0) {
    *m_out = -INFINITY;
    *l_out = 0.0;
    for (long c = 0; c < d; ++c) o[c] = 0.0;
    *lse_out = -INFINITY;
    return;
  }
  double l = 0.0;
  for (long j = 0; j < n; ++j) {
    if (!is_visible(i, j, Sq, n, causal, ks, ke, km)) continue;
    double e = exp(s[j] - m);
    l += e;
    const double ed = e * drop_factor(dr, bh, i, j);
    for (long c = 0; c < d; ++c) u[c] += ed * ld(v, vbase + j * d + c);
  }
  *m_out = m;
  *l_out = l;
  for (long c = 0; c < d; ++c) o[c] = u[c] / l;
  *lse_out = m + log(l);
}

/*
 * Single-row state (m, l, u, O, LSE) for one query against n keys, all
 * inputs fp64, no mask beyond the optional causal rule for row i of Sq.
 */
int oracle_row_state(const double* q, const double* k, const double* v, long n, long d,
                     double scale, double* m, double* l, double* u, double* o, double* lse) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  if (!s) return 1;
  src_t ks = {k, 0}, vs = {v, 0};
  row_attention(q, ks, 0, vs, 0, n, d, scale, 0, 1, 0, 0, n, NULL, NULL, 0, s, m, l, u, o, lse);
  free(s);
  return 0;
}

/*
 * Forward over [B, Hq, Sq, d] queries.  rows == NULL computes every row and
 * writes o[B*Hq*Sq*d], lse[B*Hq*Sq]; otherwise rows holds nrows flat row ids
 * ((b*Hq + h)*Sq + i) and o/lse are packed in that order.  m_out/l_out are
 * optional and follow the same packing.  key_mask is NULL or [B, Sk] bytes
 * (nonzero = the key may be seen).
 */
int oracle_fwd(const void* q, const void* k, const void* v, int in_bf16, long B, long Hq,
               long Hkv, long Sq, long Sk, long d, int causal, double scale,
               const int* k_start, const int* k_end, const unsigned char* key_mask,
               double p_drop, unsigned long long seed, unsigned int offset,
               long nrows, const long* rows,
               double* o, double* lse, double* m_out, double* l_out) {
  if (Hkv <= 0 || Hq % Hkv != 0) return 1;
  const drop_t dr = make_drop(p_drop, seed, offset);
  const long group = Hq / Hkv;
  const long total = rows ? nrows : B * Hq * Sq;
  src_t qs = {q, in_bf16}, kk = {k, in_bf16}, vv = {v, in_bf16};
  int err = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
    double* u = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !qrow || !u) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (long r = 0; r < total; ++r) {
        const long flat = rows ? rows[r] : r;
        const long i = flat % Sq;
        const long h = (flat / Sq) % Hq;
        const long b = flat / (Sq * Hq);
        const long hk = h / group;
        long ks, ke;
        key_range(k_start, k_end, b, Sk, &ks, &ke);
        load_row(qs, flat * d, d, qrow);
        const long kvbase = (b * Hkv + hk) * Sk * d;
        double m, l;
        row_attention(qrow, kk, kvbase, vv, kvbase, Sk, d, scale, i, Sq, causal, ks, ke,
                      mask_row(key_mask, b, Sk), &dr, b * Hq + h, s, &m, &l, u, o + r * d,
                      lse + r);
        if (m_out) m_out[r] = m;
        if (l_out) l_out[r] = l;
      }
    }
    free(s);
    free(qrow);
    free(u);
  }
  return err;
}

/*
 * Dense probabilities and score gradients for small problems:
 * p[B,Hq,Sq,Sk] and ds[B,Hq,Sq,Sk] (ds may be NULL, dout then unused).
 */
int oracle_probs(const void* q, const void* k, const void* v, const void* dout, int in_bf16,
                 long B, long Hq, long Hkv, long Sq, long Sk, long d, int causal,
                 double scale, const int* k_start, const int* k_end,
                 const unsigned char* key_mask, double p_drop, unsigned long long seed,
                 unsigned int offset, double* p, double* ds) {
  if (Hkv <= 0 || Hq % Hkv != 0) return 1;
  const drop_t dr = make_drop(p_drop, seed, offset);
  const long group = Hq / Hkv;
  src_t qs = {q, in_bf16}, kk = {k, in_bf16}, vv = {v, in_bf16}, dos = {dout, in_bf16};
  double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
  double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
  double* u = (double*)malloc(sizeof(double) * (size_t)d);
  double* orow = (double*)malloc(sizeof(double) * (size_t)d);
  if (!s || !qrow || !u || !orow) return 1;
  for (long b = 0; b < B; ++b)
    for (long h = 0; h < Hq; ++h)
      for (long i = 0; i < Sq; ++i) {
        const long flat = (b * Hq + h) * Sq + i;
        const long kvbase = (b * Hkv + h / group) * Sk * d;
        long ks, ke;
        key_range(k_start, k_end, b, Sk, &ks, &ke);
        load_row(qs, flat * d, d, qrow);
        double m, l, lse;
        const unsigned char* km = mask_row(key_mask, b, Sk);
        row_attention(qrow, kk, kvbase, vv, kvbase, Sk, d, scale, i, Sq, causal, ks, ke, km, &dr,
                      b * Hq + h, s, &m, &l, u, orow, &lse);
        double D = 0.0;
        if (ds)
          for (long c = 0; c < d; ++c) D += ld(dos, flat * d + c) * orow[c];
        for (long j = 0; j < Sk; ++j) {
          const long idx = flat * Sk + j;
          double pij = 0.0;
          if (l > 0.0 && is_visible(i, j, Sq, Sk, causal, ks, ke, km)) pij = exp(s[j] - m) / l;
          p[idx] = pij;
          if (ds) {
            double dp = 0.0;
            for (long c = 0; c < d; ++c) dp += ld(dos, flat * d + c) * ld(vv, kvbase + j * d + c);
            ds[idx] = pij * (dp * drop_factor(&dr, b * Hq + h, i, j) - D);
          }
        }
      }
  free(s);
  free(qrow);
  free(u);
  free(orow);
  return 0;
}

/*
 * dQ_i of one query row (flat row id), from its own statistics: m_i, l_i and
 * O_i from the definition, D_i = <dO_i, O_i>, then dQ_i = scale sum over
 * visible j of p_ij (dP_ij - D_i) k_j.  Writes dqr[d]; returns m_i, l_i, D_i.
 * s, qrow, dorow, u, orow are caller scratch.
 */
static void dq_row(src_t qs, src_t kk, src_t vv, src_t dos, long flat, long B, long Hq,
                   long Hkv, long Sq, long Sk, long d, int causal, double scale,
                   const int* k_start, const int* k_end, const unsigned char* key_mask,
                   const drop_t* dr, double* s, double* qrow, double* dorow, double* u,
                   double* orow, double* dqr, double* m_out, double* l_out, double* D_out) {
  const long group = Hq / Hkv;
  const long i = flat % Sq;
  const long h = (flat / Sq) % Hq;
  const long b = flat / (Sq * Hq);
  (void)B;
  const long kvbase = (b * Hkv + h / group) * Sk * d;
  long ks, ke;
  key_range(k_start, k_end, b, Sk, &ks, &ke);
  load_row(qs, flat * d, d, qrow);
  load_row(dos, flat * d, d, dorow);
  double lse, m, l;
  const unsigned char* km = mask_row(key_mask, b, Sk);
  row_attention(qrow, kk, kvbase, vv, kvbase, Sk, d, scale, i, Sq, causal, ks, ke, km, dr,
                b * Hq + h, s, &m, &l, u, orow, &lse);
  double D = 0.0;
  for (long c = 0; c < d; ++c) D += dorow[c] * orow[c];
  for (long c = 0; c < d; ++c) dqr[c] = 0.0;
  *m_out = m;
  *l_out = l;
  *D_out = D;
  if (l <= 0.0) return;
  for (long j = 0; j < Sk; ++j) {
    if (!is_visible(i, j, Sq, Sk, causal, ks, ke, km)) continue;
    const double pij = exp(s[j] - m) / l;
    double dp = 0.0;
    for (long c = 0; c < d; ++c) dp += dorow[c] * ld(vv, kvbase + j * d + c);
    const double dsij = pij * (dp * drop_factor(dr, b * Hq + h, i, j) - D);
    for (long c = 0; c < d; ++c) dqr[c] += scale * dsij * ld(kk, kvbase + j * d + c);
  }
}

/*
 * Full backward: dq[B,Hq,Sq,d], dk/dv[B,Hkv,Sk,d], all fp64.
 * Per-row statistics m_i, l_i and D_i are formed first from the definition;
 * every p_ij and dS_ij is then evaluated from them where it is needed.
 */
int oracle_bwd(const void* q, const void* k, const void* v, const void* dout, int in_bf16,
               long B, long Hq, long Hkv, long Sq, long Sk, long d, int causal, double scale,
               const int* k_start, const int* k_end, const unsigned char* key_mask,
               double p_drop, unsigned long long seed, unsigned int offset, double* dq,
               double* dk, double* dv) {
  if (Hkv <= 0 || Hq % Hkv != 0) return 1;
  const drop_t dr = make_drop(p_drop, seed, offset);
  const long group = Hq / Hkv;
  const long nrow = B * Hq * Sq;
  src_t qs = {q, in_bf16}, kk = {k, in_bf16}, vv = {v, in_bf16}, dos = {dout, in_bf16};
  double* M = (double*)malloc(sizeof(double) * (size_t)(nrow > 0 ? nrow : 1));
  double* L = (double*)malloc(sizeof(double) * (size_t)(nrow > 0 ? nrow : 1));
  double* Dv = (double*)malloc(sizeof(double) * (size_t)(nrow > 0 ? nrow : 1));
  if (!M || !L || !Dv) return 1;
  int err = 0;

  /* pass 1: row statistics m_i, l_i, D_i = <dO_i, O_i>, and dQ_i */
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
    double* dorow = (double*)malloc(sizeof(double) * (size_t)d);
    double* u = (double*)malloc(sizeof(double) * (size_t)d);
    double* orow = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !qrow || !dorow || !u || !orow) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (long flat = 0; flat < nrow; ++flat)
        dq_row(qs, kk, vv, dos, flat, B, Hq, Hkv, Sq, Sk, d, causal, scale, k_start, k_end,
               key_mask, &dr, s, qrow, dorow, u, orow, dq + flat * d, &M[flat], &L[flat],
               &Dv[flat]);
    }
    free(s);
    free(qrow);
    free(dorow);
    free(u);
    free(orow);
  }
  if (err) goto done;

  /* pass 2: dK_j and dV_j, summing over every query row of every query head
     in the group that reads KV head hk */
#pragma omp parallel
  {
    double* krow = (double*)malloc(sizeof(double) * (size_t)d);
    double* vrow = (double*)malloc(sizeof(double) * (size_t)d);
    if (!krow || !vrow) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (long flatk = 0; flatk < B * Hkv * Sk; ++flatk) {
        const long j = flatk % Sk;
        const long hk = (flatk / Sk) % Hkv;
        const long b = flatk / (Sk * Hkv);
        long ks, ke;
        key_range(k_start, k_end, b, Sk, &ks, &ke);
        const unsigned char* km = mask_row(key_mask, b, Sk);
        load_row(kk, flatk * d, d, krow);
        load_row(vv, flatk * d, d, vrow);
        double* dkr = dk + flatk * d;
        double* dvr = dv + flatk * d;
        for (long c = 0; c < d; ++c) dkr[c] = dvr[c] = 0.0;
        for (long g = 0; g < group; ++g) {
          const long h = hk * group + g;
          for (long i = 0; i < Sq; ++i) {
            if (!is_visible(i, j, Sq, Sk, causal, ks, ke, km)) continue;
            const long flat = (b * Hq + h) * Sq + i;
            if (L[flat] <= 0.0) continue;
            double sij = 0.0, dp = 0.0;
            for (long c = 0; c < d; ++c) sij += ld(qs, flat * d + c) * krow[c];
            sij *= scale;
            for (long c = 0; c < d; ++c) dp += ld(dos, flat * d + c) * vrow[c];
            const double pij = exp(sij - M[flat]) / L[flat];
            const double f = drop_factor(&dr, b * Hq + h, i, j);
            const double dsij = pij * (dp * f - Dv[flat]);
            for (long c = 0; c < d; ++c) {
              dvr[c] += pij * f * ld(dos, flat * d + c);
              dkr[c] += scale * dsij * ld(qs, flat * d + c);
            }
          }
        }
      }
    }
    free(krow);
    free(vrow);
  }
done:
  free(M);
  free(L);
  free(Dv);
  return err;
}

/*
 * dQ of selected query rows only (rows: nrows flat row ids (b*Hq + h)*Sq + i;
 * dq: [nrows, d]), each from its own statistics -- O(Sk * d) per row, so it
 * serves problems too large for the full backward.
 */
int oracle_bwd_dq_rows(const void* q, const void* k, const void* v, const void* dout,
                       int in_bf16, long B, long Hq, long Hkv, long Sq, long Sk, long d,
                       int causal, double scale, const int* k_start, const int* k_end,
                       const unsigned char* key_mask, double p_drop, unsigned long long seed,
                       unsigned int offset, long nrows, const long* rows, double* dq) {
  if (Hkv <= 0 || Hq % Hkv != 0) return 1;
  const drop_t dr = make_drop(p_drop, seed, offset);
  src_t qs = {q, in_bf16}, kk = {k, in_bf16}, vv = {v, in_bf16}, dos = {dout, in_bf16};
  int err = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
    double* dorow = (double*)malloc(sizeof(double) * (size_t)d);
    double* u = (double*)malloc(sizeof(double) * (size_t)d);
    double* orow = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !qrow || !dorow || !u || !orow) {
#pragma omp atomic write
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (long r = 0; r < nrows; ++r) {
        double m, l, D;
        dq_row(qs, kk, vv, dos, rows[r], B, Hq, Hkv, Sq, Sk, d, causal, scale, k_start, k_end,
               key_mask, &dr, s, qrow, dorow, u, orow, dq + r * d, &m, &l, &D);
      }
    }
    free(s);
    free(qrow);
    free(dorow);
    free(u);
    free(orow);
  }
  return err;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
