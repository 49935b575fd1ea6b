/*
 * specdec_oracle.c — plain, slow, fp64 CPU reference of the speculative
 * decoding verify/accept step and of the MTP shift/insert step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg may use it.  It shares no code, header, table
 * or constant with the CUDA path; it is written from the method's definition
 * (sources below) in scalar loops, so that a reader can check it by eye.
 *
 * Sources, cited by page title and section:
 *  [AS]  "Accelerating Sonar through speculation" (Perplexity Research,
 *        2025-06-10):
 *        §Speculative decoding — candidate prefixes are scored by probability,
 *            the longest acceptable prefix is kept, and the target gives one
 *            extra token, so at most n+1 tokens leave one step;
 *        §Speculative decoding, stage "Acceptance" — the target produces
 *            logits for each draft token and the accepted length follows;
 *        §Speculative decoding, stage "Target generation" — at the mismatch
 *            position or at the end of the draft the target row is sampled;
 *        §Target-draft — acceptance compares the full draft and target
 *            probability distributions; the draft takes the top token when it
 *            is greedy;
 *        §MTP — the input-token buffer is shifted left by one relative to the
 *            target's output hidden states;
 *        §Single-token MTP scheduling — after the shift, a GPU kernel inserts
 *            the next target token at its position, with no CPU sync; the
 *            slots after it are redundant work.
 *  [FI]  "Fast Inference from Transformers via Speculative Decoding" (listed
 *        in [AS] §References): accept draft x with probability
 *        min(1, p(x)/q(x)); on rejection sample from norm(max(0, p - q));
 *        when every draft is accepted sample one more token from p.
 *  [PH]  Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *        1, 2, 3" (SC'11): the Philox4x32-10 counter-based generator.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  R1  acceptance threshold = a uniform draw u_j; accept iff u_j < p/q.
 *  R2  one temperature T_b per request for target and draft; logits are
 *      multiplied by s = 1/T; T == 0 selects the greedy branch.
 *  R3  random numbers: Philox4x32-10, key = (seed low 32, seed high 32),
 *      counter = (v >> 2, o + j, b, purpose), word v & 3; purpose 0 is the
 *      acceptance draw (v = 0), purpose 1 the race draw for vocab entry v;
 *      o is the request's position offset (0 unless the caller gives one),
 *      so that draws can follow a request's absolute position rather than
 *      the row index within its draft window.
 *      U(w) = ((w >> 9) + 1/2) * 2^-23, in (0, 1), exact in fp32 and fp64.
 *  R4  sampling from weights r_v is the exponential race
 *      argmax_v r_v / E_v with E_v = -ln U_v, over entries with r_v > 0;
 *      the lowest index wins an exact tie.
 *  R5  greedy argmax: the lowest index holding the maximum wins.
 *  R6  a residual that is zero everywhere (p == q) falls back to the race on p.
 *  R7  invalid device data: a draft token outside [0, V) rejects its row;
 *      draft_len is clamped to [0, n_max]; T < 0, NaN, or 0 < T < 1e-6 is
 *      treated as greedy, and so is T > 0 without draft logits for a request
 *      that has drafts (L > 0).  Each sets a bit of the returned error word.
 *      A request with L == 0 needs no draft logits: its token is the race on
 *      the target row's p.
 *  R8  MTP: within segment [s, s+n] of the flattened token buffer,
 *      out[s+i] = in[s+i+1] for i < n, out[s+n] = in[s+n], then
 *      out[s+a] = next token.  Hidden states stay in place (copied bitwise
 *      when a distinct output buffer is given).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes used by this oracle's own interface */
#define ORACLE_F32 0
#define ORACLE_BF16 1

/* error-word bits (R7) */
#define ORACLE_ERR_TOKEN 1u
#define ORACLE_ERR_DRAFT_LEN 2u
#define ORACLE_ERR_TEMPERATURE 4u

/* ------------------------------------------------------------------ Philox */

/* [PH] Philox4x32 with 10 rounds.  One round multiplies counter words 0 and 2
 * by the two round multipliers, and the new counter is
 * (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)).
 * Between rounds the key is bumped by the Weyl constants. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
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

/* R3: one 32-bit word -> uniform in (0, 1). */
double oracle_uniform(uint32_t w) {
  return ((double)(w >> 9) + 0.5) * (1.0 / 8388608.0); /* 2^-23 */
}

/* R3: the word for (seed; request b, row j, vocab entry v, purpose). */
uint32_t oracle_draw(uint64_t seed, uint32_t b, uint32_t j, uint32_t v,
                     uint32_t purpose) {
  uint32_t ctr[4] = {v >> 2, j, b, purpose};
  uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return out[v & 3u];
}

/* ------------------------------------------------------------------ helpers */

static double logit_at(const void* base, int dtype, size_t idx) {
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f; /* bf16 -> fp32 -> fp64 is exact */
}

/* log-sum-exp of s * x over one row: max(s x) + ln sum exp(s x - max). */
static double row_lse(const void* base, int dtype, size_t row_off, int V,
                      double s) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double z = s * logit_at(base, dtype, row_off + (size_t)v);
    if (z > m) m = z;
  }
  double acc = 0.0;
  for (int v = 0; v < V; ++v) {
    double z = s * logit_at(base, dtype, row_off + (size_t)v);
    acc += exp(z - m);
  }
  return m + log(acc);
}

/* R5: first index holding the maximum value. */
static int row_argmax(const void* base, int dtype, size_t row_off, int V) {
  int best = 0;
  double bv = logit_at(base, dtype, row_off);
  for (int v = 1; v < V; ++v) {
    double x = logit_at(base, dtype, row_off + (size_t)v);
    if (x > bv) {
      bv = x;
      best = v;
    }
  }
  return best;
}

/* R4: exponential race over weights r[0..V-1] (entries with r <= 0 skipped).
 * Returns the winner (or -1 if no entry is positive); *gap receives the
 * relative gap (k1 - k2) / k1 between the two largest keys (1 if only one
 * entry competes). */
int oracle_race(const double* r, int V, uint64_t seed, uint32_t b, uint32_t j,
                double* gap) {
  int best = -1;
  double k1 = 0.0, k2 = 0.0;
  for (int v = 0; v < V; ++v) {
    if (!(r[v] > 0.0)) continue;
    double u = oracle_uniform(oracle_draw(seed, b, j, (uint32_t)v, 1u));
    double e = -log(u);
    double key = r[v] / e;
    if (best < 0 || key > k1) {
      k2 = (best < 0) ? 0.0 : k1;
      k1 = key;
      best = v;
    } else if (key > k2) {
      k2 = key;
    }
  }
  if (gap) *gap = (best < 0) ? NAN : (k1 > 0.0 ? (k1 - k2) / k1 : 0.0);
  return best;
}

/* --------------------------------------------------------------- verify */

/*
 * Verify/accept for requests listed in the batch.
 *
 * target [B, n_max+1, V], draft [B, n_max, V] (may be NULL when every request
 * is greedy or has no drafts), row-major, dtype ORACLE_F32 or ORACLE_BF16 (raw bf16 bits).
 * draft_tokens [B, n_max]; draft_len [B]; temperature [B].
 * req_ids: optional [B]; the request coordinate b that enters the random
 *   counter for local request i (NULL: b = i).  It lets a caller verify a
 *   sample of a larger batch and still draw that batch's numbers.
 * pos_off: optional [B]; the position offset o of R3 for local request i
 *   (NULL: o = 0).  Row j draws with counter word o + j (mod 2^32).
 * Outputs: accepted_len [B]; out_tokens [B, n_max+1] (a+1 tokens, rest -1);
 *   optional row_lse [B, n_max+1, 2] (LSE of s*target row j, LSE of s*draft
 *   row j; NaN where not defined); optional accept_margin [B, n_max]
 *   (|u_j - min(1, p/q)| / u_j for rows whose test ran, NaN elsewhere);
 *   optional race_gap [B] (relative top-2 key gap of the race that produced
 *   the last emitted token; NaN for greedy requests).
 * Returns the OR of the error bits of R7.
 */
uint32_t oracle_spec_verify(const void* target, const void* draft, int dtype,
                            int B, int n_max, int V,
                            const int32_t* draft_tokens,
                            const int32_t* draft_len, const float* temperature,
                            uint64_t seed, const int32_t* req_ids,
                            const int32_t* pos_off,
                            int32_t* accepted_len, int32_t* out_tokens,
                            double* row_lse_out, double* accept_margin,
                            double* race_gap) {
  uint32_t err = 0;
  const size_t rows_t = (size_t)n_max + 1;
  double* r = (double*)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
  if (!r) return 0xFFFFFFFFu;

  for (int i = 0; i < B; ++i) {
    const uint32_t b = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
    const uint32_t o = pos_off ? (uint32_t)pos_off[i] : 0u;
    const int32_t* x = draft_tokens + (size_t)i * (size_t)n_max;
    int32_t* out = out_tokens + (size_t)i * rows_t;

    /* R7: clamp the draft length. */
    int L = draft_len[i];
    if (L < 0 || L > n_max) {
      err |= ORACLE_ERR_DRAFT_LEN;
      L = L < 0 ? 0 : n_max;
    }
    /* R2 / R7: temperature. */
    double T = (double)temperature[i];
    int greedy = 0;
    if (T == 0.0) {
      greedy = 1;
    } else if (!(T > 0.0) || T < 1e-6) { /* negative, NaN or too small */
      err |= ORACLE_ERR_TEMPERATURE;
      greedy = 1;
    }
    /* A request with drafts needs the draft distribution; one without
     * (L == 0) samples its only token from the target row alone. */
    if (!greedy && draft == NULL && L > 0) {
      err |= ORACLE_ERR_TEMPERATURE;
      greedy = 1;
    }

    if (row_lse_out)
      for (size_t k = 0; k < rows_t * 2; ++k)
        row_lse_out[(size_t)i * rows_t * 2 + k] = NAN;
    if (accept_margin)
      for (int k = 0; k < n_max; ++k)
        accept_margin[(size_t)i * (size_t)n_max + (size_t)k] = NAN;
    if (race_gap) race_gap[i] = NAN;

    int a = L, y = -1;
    if (greedy) {
      /* [AS] §Target-draft, T = 0: accept while the draft token equals the
       * target argmax; the first mismatch (or the row after the last draft)
       * emits the target argmax. */
      for (int j = 0; j <= L; ++j) {
        size_t off_t = ((size_t)i * rows_t + (size_t)j) * (size_t)V;
        int g = row_argmax(target, dtype, off_t, V);
        if (j == L) {
          a = L;
          y = g;
          break;
        }
        if (x[j] < 0 || x[j] >= V) err |= ORACLE_ERR_TOKEN;
        if (x[j] != g) {
          a = j;
          y = g;
          break;
        }
      }
    } else {
      const double s = 1.0 / T;
      /* [AS] stage "Acceptance" + [FI]: test the drafts in order. */
      a = L;
      for (int j = 0; j < L; ++j) {
        size_t off_t = ((size_t)i * rows_t + (size_t)j) * (size_t)V;
        size_t off_d = ((size_t)i * (size_t)n_max + (size_t)j) * (size_t)V;
        double lse_t = row_lse(target, dtype, off_t, V, s);
        double lse_d = row_lse(draft, dtype, off_d, V, s);
        if (row_lse_out) {
          row_lse_out[((size_t)i * rows_t + (size_t)j) * 2 + 0] = lse_t;
          row_lse_out[((size_t)i * rows_t + (size_t)j) * 2 + 1] = lse_d;
        }
        int tok = x[j];
        int rejected;
        if (tok < 0 || tok >= V) {
          err |= ORACLE_ERR_TOKEN;
          rejected = 1;
        } else {
          double lp = s * logit_at(target, dtype, off_t + (size_t)tok) - lse_t;
          double lq = s * logit_at(draft, dtype, off_d + (size_t)tok) - lse_d;
          double ratio = exp(lp - lq); /* p(x)/q(x) */
          double u = oracle_uniform(oracle_draw(seed, b, o + (uint32_t)j, 0u, 0u));
          if (accept_margin) {
            double thr = ratio < 1.0 ? ratio : 1.0;
            accept_margin[(size_t)i * (size_t)n_max + (size_t)j] =
                fabs(u - thr) / u;
          }
          rejected = !(u < ratio);
        }
        if (rejected) {
          /* [AS] stage "Target generation" + [FI]: sample the replacement
           * from norm(max(0, p - q)) on this row. */
          for (int v = 0; v < V; ++v) {
            double p = exp(s * logit_at(target, dtype, off_t + (size_t)v) - lse_t);
            double q = exp(s * logit_at(draft, dtype, off_d + (size_t)v) - lse_d);
            double d = p - q;
            r[v] = d > 0.0 ? d : 0.0;
          }
          double gap = NAN;
          y = oracle_race(r, V, seed, b, o + (uint32_t)j, &gap);
          if (y < 0) { /* R6: residual vanished; race on p instead */
            for (int v = 0; v < V; ++v)
              r[v] = exp(s * logit_at(target, dtype, off_t + (size_t)v) - lse_t);
            y = oracle_race(r, V, seed, b, o + (uint32_t)j, &gap);
          }
          if (race_gap) race_gap[i] = gap;
          a = j;
          break;
        }
      }
      if (a == L) {
        /* Every draft accepted: the bonus token from the target's row L. */
        size_t off_t = ((size_t)i * rows_t + (size_t)L) * (size_t)V;
        double lse_t = row_lse(target, dtype, off_t, V, s);
        if (row_lse_out)
          row_lse_out[((size_t)i * rows_t + (size_t)L) * 2 + 0] = lse_t;
        for (int v = 0; v < V; ++v)
          r[v] = exp(s * logit_at(target, dtype, off_t + (size_t)v) - lse_t);
        double gap = NAN;
        y = oracle_race(r, V, seed, b, o + (uint32_t)L, &gap);
        if (race_gap) race_gap[i] = gap;
      }
    }

    /* [AS] §Speculative decoding: at most n+1 tokens leave the step. */
    accepted_len[i] = a;
    for (size_t k = 0; k < rows_t; ++k) out[k] = -1;
    for (int k = 0; k < a; ++k) out[k] = x[k];
    out[a] = y;
  }
  free(r);
  return err;
}

/* Per-row statistics for every valid row, for comparison with a kernel that
 * scores all rows of a request (not only those up to the first rejection).
 * row_lse [B, n_max+1, 2] as in oracle_spec_verify; NaN for rows beyond
 * draft_len, for draft rows of the last row, and for greedy requests. */
void oracle_row_lse_all(const void* target, const void* draft, int dtype,
                        int B, int n_max, int V, const int32_t* draft_len,
                        const float* temperature, double* row_lse_out) {
  const size_t rows_t = (size_t)n_max + 1;
  for (int i = 0; i < B; ++i) {
    int L = draft_len[i];
    if (L < 0) L = 0;
    if (L > n_max) L = n_max;
    double T = (double)temperature[i];
    int greedy = !(T > 0.0) || T < 1e-6 || (draft == NULL && L > 0);
    for (size_t k = 0; k < rows_t * 2; ++k)
      row_lse_out[(size_t)i * rows_t * 2 + k] = NAN;
    if (greedy) continue;
    const double s = 1.0 / T;
    for (int j = 0; j <= L; ++j) {
      size_t off_t = ((size_t)i * rows_t + (size_t)j) * (size_t)V;
      row_lse_out[((size_t)i * rows_t + (size_t)j) * 2 + 0] =
          row_lse(target, dtype, off_t, V, s);
      if (j < L) {
        size_t off_d = ((size_t)i * (size_t)n_max + (size_t)j) * (size_t)V;
        row_lse_out[((size_t)i * rows_t + (size_t)j) * 2 + 1] =
            row_lse(draft, dtype, off_d, V, s);
      }
    }
  }
}

/* ------------------------------------------------------- MTP shift/insert */

/*
 * [AS] §MTP and §Single-token MTP scheduling, reading R8.
 * tokens_in / tokens_out [R] (may be the same buffer); segment b starts at
 * seg_start[b] (NULL: b * (R / B)) and holds draft_len[b] + 1 slots.  The
 * replacement token of request b is next_token[b] when next_token_stride is
 * 0, else next_token[b * next_token_stride + accepted_len[b]].
 * hidden_in / hidden_out [R, H] of elem_bytes each: copied bitwise when both
 * are given and distinct.  Slots outside every segment are not written.
 * Returns 0, or 1 for a segment or index outside the buffers.
 */
int oracle_mtp_shift_insert(const int32_t* tokens_in, int32_t* tokens_out,
                            const void* hidden_in, void* hidden_out, int R,
                            int H, int elem_bytes, const int32_t* seg_start,
                            const int32_t* draft_len,
                            const int32_t* accepted_len,
                            const int32_t* next_token, int next_token_stride,
                            int B) {
  int32_t* tmp = (int32_t*)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
  if (!tmp) return 1;
  memcpy(tmp, tokens_in, sizeof(int32_t) * (size_t)R); /* in-place safe */
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    int s = seg_start ? seg_start[b] : b * (R / B);
    int n = draft_len[b];
    int a = accepted_len[b];
    if (s < 0 || n < 0 || s + n >= R || a < 0 || a > n) {
      bad = 1;
      continue;
    }
    for (int i = 0; i < n; ++i) tokens_out[s + i] = tmp[s + i + 1];
    tokens_out[s + n] = tmp[s + n];
    int tok = next_token_stride == 0 ? next_token[b]
                                     : next_token[(size_t)b * (size_t)next_token_stride + (size_t)a];
    tokens_out[s + a] = tok;
  }
  free(tmp);
  if (hidden_in && hidden_out && hidden_in != hidden_out)
    memcpy(hidden_out, hidden_in, (size_t)R * (size_t)H * (size_t)elem_bytes);
  return bad;
}
