/*
 * hdp_oracle.c -- plain, slow, fp64 CPU oracle for document-masked causal
 * attention over a packed micro-batch cut into capacity-C chunks.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Source: "ByteScale: Communication-Efficient Scaling of LLM Training with a
 * 2048K Context Length on 16384 GPUs" (AI training network primer research
 * digest).
 *   - capacity C and the ceil(s/C) ranks of a sequence: section 1 and
 *     section 3.1 (Figure 2);
 *   - short sequences packed onto one rank by best fit: section 3.1,
 *     Figure 2(b);
 *   - a query attends only to its own sequence; one C x C block per ring step,
 *     partial results combined across steps: section 3.2;
 *   - attention time grows as O(s^2): section 1, section 2.
 *
 * Everything is written as the plain definition: explicit loops in fp64,
 * exact two-pass softmax per (query, head), no tiling, no online rescaling.
 * Readings where the pages are silent (best-fit-decreasing tie-breaks, shard
 * numbering, natural-log LSE, consecutive GQA grouping) are stated next to
 * the code that takes them.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ENOMEM 2

/* bf16 bit pattern -> double, exactly (a bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Threads the oracle's parallel loops use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ plan */

/* Number of chunks of a sequence of length s at capacity C, counted by
 * walking the sequence C tokens at a time (section 3.1: a sequence longer than
 * C spans ceil(s/C) ranks). */
static int32_t count_chunks(int32_t s, int32_t C) {
  int32_t n = 0;
  for (int64_t t = 0; t < s; t += C) n++;
  return n;
}

/* Totals needed to size the plan tables. */
int oracle_plan_sizes(const int32_t* lengths, int32_t n, int32_t C, int32_t* num_chunks, int64_t* num_blocks,
                      int64_t* total_tokens) {
  if (n < 0 || C < 1) return ORC_EINVAL;
  int64_t nc = 0, nb = 0, tt = 0;
  for (int32_t i = 0; i < n; i++) {
    if (lengths[i] < 1) return ORC_EINVAL;
    int32_t c = count_chunks(lengths[i], C);
    nc += c;
    /* blocks (qc, kc) with 0 <= kc <= qc < c, counted one by one */
    for (int32_t qc = 0; qc < c; qc++)
      for (int32_t kc = 0; kc <= qc; kc++) nb++;
    tt += lengths[i];
  }
  *num_chunks = (int32_t)nc;
  *num_blocks = nb;
  *total_tokens = tt;
  return ORC_OK;
}

/* Piece of a sequence shorter than C, to be packed by best fit. */
typedef struct {
  int32_t len, doc, chunk;
} piece_t;

/* Best-fit-decreasing order: length descending, then document ascending. */
static int piece_cmp(const void* a, const void* b) {
  const piece_t* x = (const piece_t*)a;
  const piece_t* y = (const piece_t*)b;
  if (x->len != y->len) return x->len > y->len ? -1 : 1;
  return x->doc < y->doc ? -1 : (x->doc > y->doc ? 1 : 0);
}

/*
 * The sharding plan.
 *   cu_seqlens[n+1]    exclusive prefix sum of lengths (token offsets)
 *   chunk_offsets[n+1] exclusive prefix sum of chunks per sequence
 *   block_offsets[n+1] exclusive prefix sum of causal (qc, kc) blocks per sequence
 *   chunk_table[Nc][4] {doc, index within doc, first global token, length}
 *   block_table[Nb][2] {global q chunk, global kv chunk}, ordered by doc, then
 *                      q chunk, then kv chunk ascending
 *   chunk_pairs[Nc]    causal (query, key) pairs whose query lies in the chunk
 *   shard_of_chunk[Nc] rank ("shard") holding the chunk
 *
 * Shards (section 3.1, Figure 2(b): full C-token slices get a rank each,
 * shorter sequences are packed onto one rank by best fit).  Reading: every
 * chunk of exactly C tokens gets its own shard, numbered in chunk order; then
 * each piece shorter than C (a short sequence or the tail of a long one),
 * taken in best-fit-decreasing order (length desc, doc asc), goes to the
 * open piece shard with the least remaining capacity that still fits, the
 * lowest shard id on ties, or else opens a new shard.
 */
int oracle_plan(const int32_t* lengths, int32_t n, int32_t C, int32_t* cu_seqlens, int32_t* chunk_offsets,
                int64_t* block_offsets, int32_t* chunk_table, int32_t* block_table, int64_t* chunk_pairs,
                int32_t* shard_of_chunk, int32_t* num_shards) {
  if (n < 0 || C < 1) return ORC_EINVAL;
  int64_t tok = 0, ch = 0, blk = 0;
  for (int32_t i = 0; i < n; i++) {
    if (lengths[i] < 1) return ORC_EINVAL;
    cu_seqlens[i] = (int32_t)tok;
    chunk_offsets[i] = (int32_t)ch;
    block_offsets[i] = blk;
    const int32_t s = lengths[i];
    const int64_t first_chunk = ch;
    int32_t idx = 0;
    for (int64_t a = 0; a < s; a += C, idx++) {
      int64_t b = a + C < s ? a + C : s;
      chunk_table[ch * 4 + 0] = i;
      chunk_table[ch * 4 + 1] = idx;
      chunk_table[ch * 4 + 2] = (int32_t)(tok + a);
      chunk_table[ch * 4 + 3] = (int32_t)(b - a);
      /* doc-local query p sees keys 0..p: p+1 pairs */
      int64_t pairs = 0;
      for (int64_t p = a; p < b; p++) pairs += p + 1;
      chunk_pairs[ch] = pairs;
      ch++;
    }
    for (int32_t qc = 0; qc < idx; qc++)
      for (int32_t kc = 0; kc <= qc; kc++) {
        block_table[blk * 2 + 0] = (int32_t)(first_chunk + qc);
        block_table[blk * 2 + 1] = (int32_t)(first_chunk + kc);
        blk++;
      }
    tok += s;
  }
  cu_seqlens[n] = (int32_t)tok;
  chunk_offsets[n] = (int32_t)ch;
  block_offsets[n] = blk;

  /* shards: full chunks first, in chunk order (skipped when the caller passes
   * shard_of_chunk = NULL) */
  if (!shard_of_chunk) {
    *num_shards = 0;
    return ORC_OK;
  }
  int32_t ns = 0;
  int64_t npieces = 0;
  for (int64_t c = 0; c < ch; c++) {
    if (chunk_table[c * 4 + 3] == C)
      shard_of_chunk[c] = ns++;
    else
      npieces++;
  }
  if (npieces > 0) {
    piece_t* pcs = (piece_t*)malloc(sizeof(piece_t) * (size_t)npieces);
    int64_t* remaining = (int64_t*)malloc(sizeof(int64_t) * (size_t)npieces);
    int32_t* shard_id = (int32_t*)malloc(sizeof(int32_t) * (size_t)npieces);
    if (!pcs || !remaining || !shard_id) {
      free(pcs);
      free(remaining);
      free(shard_id);
      return ORC_ENOMEM;
    }
    int64_t k = 0;
    for (int64_t c = 0; c < ch; c++)
      if (chunk_table[c * 4 + 3] != C) {
        pcs[k].len = chunk_table[c * 4 + 3];
        pcs[k].doc = chunk_table[c * 4 + 0];
        pcs[k].chunk = (int32_t)c;
        k++;
      }
    qsort(pcs, (size_t)npieces, sizeof(piece_t), piece_cmp);
    int64_t nopen = 0; /* open piece shards, in order of opening (ascending id) */
    for (int64_t p = 0; p < npieces; p++) {
      int64_t best = -1;
      for (int64_t s = 0; s < nopen; s++)
        if (remaining[s] >= pcs[p].len && (best < 0 || remaining[s] < remaining[best])) best = s;
      if (best < 0) {
        best = nopen++;
        remaining[best] = C;
        shard_id[best] = ns++;
      }
      remaining[best] -= pcs[p].len;
      shard_of_chunk[pcs[p].chunk] = shard_id[best];
    }
    free(pcs);
    free(remaining);
    free(shard_id);
  }
  *num_shards = ns;
  return ORC_OK;
}

/* ------------------------------------------------------------------ FLOPs */

/* Useful causal attention FLOPs: for every (query, key) pair with the key at
 * or before the query in the same sequence, d multiply-adds for q.k and d for
 * p.v (2 FLOPs each), per query head: 4*d*Hq per pair.  Pairs are counted
 * one by one. */
int64_t oracle_flops_total(const int32_t* lengths, int32_t n, int32_t d, int32_t hq) {
  int64_t pairs = 0;
  for (int32_t i = 0; i < n; i++)
    for (int64_t p = 0; p < lengths[i]; p++) pairs += p + 1;
  return pairs * 4 * (int64_t)d * hq;
}

/* Per-shard FLOPs: each chunk's pairs, times 4*d*Hq, summed into its shard. */
int oracle_flops_per_shard(const int64_t* chunk_pairs, const int32_t* shard_of_chunk, int32_t num_chunks,
                           int32_t num_shards, int32_t d, int32_t hq, int64_t* out) {
  for (int32_t s = 0; s < num_shards; s++) out[s] = 0;
  for (int32_t c = 0; c < num_chunks; c++) {
    int32_t s = shard_of_chunk[c];
    if (s < 0 || s >= num_shards) return ORC_EINVAL;
    out[s] += chunk_pairs[c] * 4 * (int64_t)d * hq;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ attention */

/* Document containing global token t (cu_seqlens ascending). */
static int32_t doc_of_token(const int32_t* cu, int32_t n, int64_t t) {
  int32_t lo = 0, hi = n - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) / 2;
    if (cu[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

/*
 * Attention of one query row against the keys of its own document whose
 * doc-local position j satisfies key_lo <= j < key_hi and j <= p (causal).
 * With key_lo = 0 and key_hi = s this is the full row; a narrower range is a
 * partial block of the ring step in section 3.2.  An empty range gives
 * lse = -inf and o = 0.
 *   scores  S_j = scale * sum_c q[c] k_j[c]
 *   lse     = m + ln sum_j exp(S_j - m),  m = max_j S_j
 *   o       = sum_j exp(S_j - lse) v_j
 * Layouts: q [T][hq][d], k and v [T][hkv][d] (bf16 bits); query head h reads
 * kv head h / (hq / hkv) (consecutive grouping).
 */
static void attend_row(const uint16_t* q, const uint16_t* k, const uint16_t* v, int32_t hq, int32_t hkv,
                       int32_t d, double scale, int64_t doc_start, int64_t p, int32_t h, int64_t key_lo,
                       int64_t key_hi, double* o, double* lse, double* scores) {
  const int32_t g = h / (hq / hkv);
  const uint16_t* qrow = q + ((doc_start + p) * hq + h) * (int64_t)d;
  int64_t hi = key_hi < p + 1 ? key_hi : p + 1;
  for (int32_t c = 0; c < d; c++) o[c] = 0.0;
  if (key_lo >= hi) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t j = key_lo; j < hi; j++) {
    const uint16_t* krow = k + ((doc_start + j) * hkv + g) * (int64_t)d;
    double s = 0.0;
    for (int32_t c = 0; c < d; c++) s += bf16_to_double(qrow[c]) * bf16_to_double(krow[c]);
    s *= scale;
    scores[j - key_lo] = s;
    if (s > m) m = s;
  }
  double sum = 0.0;
  for (int64_t j = key_lo; j < hi; j++) sum += exp(scores[j - key_lo] - m);
  const double L = m + log(sum);
  for (int64_t j = key_lo; j < hi; j++) {
    const double w = exp(scores[j - key_lo] - L);
    const uint16_t* vrow = v + ((doc_start + j) * hkv + g) * (int64_t)d;
    for (int32_t c = 0; c < d; c++) o[c] += w * bf16_to_double(vrow[c]);
  }
  *lse = L;
}

static int check_heads(int32_t hq, int32_t hkv, int32_t d) {
  if (hq < 1 || hkv < 1 || d < 1 || hq % hkv != 0) return ORC_EINVAL;
  return ORC_OK;
}

/*
 * Full document-masked causal attention over the packed batch.
 *   o   [T][hq][d]  fp64 (not rounded)
 *   lse [hq][T]     fp64, natural log
 */
int oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* cu_seqlens,
                     int32_t n, int32_t hq, int32_t hkv, int32_t d, double scale, double* o, double* lse) {
  if (check_heads(hq, hkv, d) != ORC_OK || n < 1) return ORC_EINVAL;
  const int64_t T = cu_seqlens[n];
  int32_t maxlen = 0;
  for (int32_t i = 0; i < n; i++)
    if (cu_seqlens[i + 1] - cu_seqlens[i] > maxlen) maxlen = cu_seqlens[i + 1] - cu_seqlens[i];
  int err = ORC_OK;
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    if (!scores) {
#pragma omp atomic write
      err = ORC_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t w = 0; w < T * hq; w++) {
        const int64_t t = w / hq;
        const int32_t h = (int32_t)(w % hq);
        const int32_t i = doc_of_token(cu_seqlens, n, t);
        const int64_t start = cu_seqlens[i];
        const int64_t s = cu_seqlens[i + 1] - start;
        attend_row(q, k, v, hq, hkv, d, scale, start, t - start, h, 0, s, o + (t * hq + h) * (int64_t)d,
                   lse + (int64_t)h * T + t, scores);
      }
      free(scores);
    }
  }
  return err;
}

/*
 * Sampled rows: for sample i, query token tokens[i] with head heads[i],
 * restricted to doc-local keys [key_lo[i], key_hi[i]) (pass NULL for the
 * whole document).  o_out [ns][d], lse_out [ns].
 */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* cu_seqlens,
                          int32_t n, int32_t hq, int32_t hkv, int32_t d, double scale, const int64_t* tokens,
                          const int32_t* heads, const int64_t* key_lo, const int64_t* key_hi, int64_t ns,
                          double* o_out, double* lse_out) {
  if (check_heads(hq, hkv, d) != ORC_OK || n < 1) return ORC_EINVAL;
  const int64_t T = cu_seqlens[n];
  for (int64_t i = 0; i < ns; i++)
    if (tokens[i] < 0 || tokens[i] >= T || heads[i] < 0 || heads[i] >= hq) return ORC_EINVAL;
  int32_t maxlen = 0;
  for (int32_t i = 0; i < n; i++)
    if (cu_seqlens[i + 1] - cu_seqlens[i] > maxlen) maxlen = cu_seqlens[i + 1] - cu_seqlens[i];
  int err = ORC_OK;
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    if (!scores) {
#pragma omp atomic write
      err = ORC_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < ns; i++) {
        const int64_t t = tokens[i];
        const int32_t di = doc_of_token(cu_seqlens, n, t);
        const int64_t start = cu_seqlens[di];
        const int64_t s = cu_seqlens[di + 1] - start;
        const int64_t lo = key_lo ? key_lo[i] : 0;
        const int64_t hi = key_hi ? key_hi[i] : s;
        attend_row(q, k, v, hq, hkv, d, scale, start, t - start, heads[i], lo < 0 ? 0 : lo, hi > s ? s : hi,
                   o_out + i * (int64_t)d, lse_out + i, scores);
      }
      free(scores);
    }
  }
  return err;
}

/* ------------------------------------------------------------------ merge */

/*
 * Exact log-sum-exp combination of m partial results of the same rows
 * (section 3.2: partial blocks from each ring step are combined):
 *   M   = max_k lse_k
 *   lse = M + ln sum_k exp(lse_k - M)
 *   o   = sum_k exp(lse_k - lse) o_k
 * A partial with lse_k = -inf contributes nothing; if all are -inf the row's
 * lse is -inf and o is 0.
 * o_parts [m][rows][d], lse_parts [m][rows]; o_out [rows][d], lse_out [rows].
 */
int oracle_merge(int32_t m, int64_t rows, int32_t d, const double* o_parts, const double* lse_parts, double* o_out,
                 double* lse_out) {
  if (m < 1 || rows < 0 || d < 1) return ORC_EINVAL;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; r++) {
    double M = -INFINITY;
    for (int32_t k = 0; k < m; k++)
      if (lse_parts[k * rows + r] > M) M = lse_parts[k * rows + r];
    double* o = o_out + r * (int64_t)d;
    for (int32_t c = 0; c < d; c++) o[c] = 0.0;
    if (M == -INFINITY) {
      lse_out[r] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int32_t k = 0; k < m; k++) sum += exp(lse_parts[k * rows + r] - M);
    const double L = M + log(sum);
    for (int32_t k = 0; k < m; k++) {
      const double w = exp(lse_parts[k * rows + r] - L);
      if (w == 0.0) continue;
      const double* ok = o_parts + (k * rows + r) * (int64_t)d;
      for (int32_t c = 0; c < d; c++) o[c] += w * ok[c];
    }
    lse_out[r] = L;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ backward */

/*
 * The training step the pages time runs a forward and a backward pass over
 * the same packed micro-batch (review and digest, section 5: forward plus
 * backward bars).  The backward of document-masked causal attention is the
 * gradient of L = sum_{t,h,c} O[t][h][c] dO[t][h][c] with respect to q, k, v,
 * written out from its definition.  For query row a of query head h (kv head
 * g = h / (hq/hkv)) and the keys b <= a of a's own document:
 *   S_ab  = scale q_a . k_b
 *   P_ab  = exp(S_ab - lse_a),  lse_a = ln sum_b exp(S_ab)     (two passes)
 *   dP_ab = dO_a . v_b
 *   Dl_a  = sum_b P_ab dP_ab
 *   dS_ab = P_ab (dP_ab - Dl_a)
 *   dq_a  = scale sum_b dS_ab k_b
 *   dk_b += scale dS_ab q_a        (summed over the query heads of g)
 *   dv_b += P_ab dO_a              (summed over the query heads of g)
 * Inputs and outputs are fp64 so that finite differences of the forward
 * below can pin it; callers with bf16 data convert exactly.
 */

/* Forward on fp64 inputs (same definition as oracle_attention). */
int oracle_attention_f64(const double* q, const double* k, const double* v, const int32_t* cu_seqlens, int32_t n,
                         int32_t hq, int32_t hkv, int32_t d, double scale, double* o, double* lse) {
  if (check_heads(hq, hkv, d) != ORC_OK || n < 1) return ORC_EINVAL;
  const int64_t T = cu_seqlens[n];
  const int32_t grp = hq / hkv;
  for (int64_t t = 0; t < T; t++) {
    const int32_t i = doc_of_token(cu_seqlens, n, t);
    const int64_t start = cu_seqlens[i];
    for (int32_t h = 0; h < hq; h++) {
      const int32_t g = h / grp;
      const double* qa = q + (t * hq + h) * (int64_t)d;
      double m = -INFINITY;
      for (int64_t b = start; b <= t; b++) {
        double s = 0.0;
        for (int32_t c = 0; c < d; c++) s += qa[c] * k[(b * hkv + g) * (int64_t)d + c];
        s *= scale;
        if (s > m) m = s;
      }
      double sum = 0.0;
      for (int64_t b = start; b <= t; b++) {
        double s = 0.0;
        for (int32_t c = 0; c < d; c++) s += qa[c] * k[(b * hkv + g) * (int64_t)d + c];
        sum += exp(s * scale - m);
      }
      const double L = m + log(sum);
      double* oa = o + (t * hq + h) * (int64_t)d;
      for (int32_t c = 0; c < d; c++) oa[c] = 0.0;
      for (int64_t b = start; b <= t; b++) {
        double s = 0.0;
        for (int32_t c = 0; c < d; c++) s += qa[c] * k[(b * hkv + g) * (int64_t)d + c];
        const double p = exp(s * scale - L);
        for (int32_t c = 0; c < d; c++) oa[c] += p * v[(b * hkv + g) * (int64_t)d + c];
      }
      lse[(int64_t)h * T + t] = L;
    }
  }
  return ORC_OK;
}

/* One query row of the backward: fills P (probabilities) and dS for keys
 * b = start..a, accumulates dq_a.  p and ds have room for a - start + 1. */
static void bwd_row(const double* q, const double* k, const double* v, const double* dout, int32_t hq, int32_t hkv,
                    int32_t d, double scale, int64_t start, int64_t a, int32_t h, double* p, double* ds,
                    double* dq_a) {
  const int32_t g = h / (hq / hkv);
  const double* qa = q + (a * hq + h) * (int64_t)d;
  const double* doa = dout + (a * hq + h) * (int64_t)d;
  const int64_t nk = a - start + 1;
  double m = -INFINITY;
  for (int64_t j = 0; j < nk; j++) {
    const double* kb = k + ((start + j) * hkv + g) * (int64_t)d;
    double s = 0.0;
    for (int32_t c = 0; c < d; c++) s += qa[c] * kb[c];
    p[j] = s * scale;
    if (p[j] > m) m = p[j];
  }
  double sum = 0.0;
  for (int64_t j = 0; j < nk; j++) sum += exp(p[j] - m);
  const double L = m + log(sum);
  double dl = 0.0;
  for (int64_t j = 0; j < nk; j++) {
    p[j] = exp(p[j] - L);
    const double* vb = v + ((start + j) * hkv + g) * (int64_t)d;
    double dp = 0.0;
    for (int32_t c = 0; c < d; c++) dp += doa[c] * vb[c];
    ds[j] = dp;
    dl += p[j] * dp;
  }
  for (int32_t c = 0; c < d; c++) dq_a[c] = 0.0;
  for (int64_t j = 0; j < nk; j++) {
    ds[j] = p[j] * (ds[j] - dl);
    const double* kb = k + ((start + j) * hkv + g) * (int64_t)d;
    for (int32_t c = 0; c < d; c++) dq_a[c] += scale * ds[j] * kb[c];
  }
}

/* Full backward.  dq [T][hq][d], dk and dv [T][hkv][d], all fp64. */
int oracle_attention_bwd(const double* q, const double* k, const double* v, const double* dout,
                         const int32_t* cu_seqlens, int32_t n, int32_t hq, int32_t hkv, int32_t d, double scale,
                         double* dq, double* dk, double* dv) {
  if (check_heads(hq, hkv, d) != ORC_OK || n < 1) return ORC_EINVAL;
  const int64_t T = cu_seqlens[n];
  const int32_t grp = hq / hkv;
  memset(dk, 0, sizeof(double) * (size_t)(T * hkv * d));
  memset(dv, 0, sizeof(double) * (size_t)(T * hkv * d));
  int32_t maxlen = 0;
  for (int32_t i = 0; i < n; i++)
    if (cu_seqlens[i + 1] - cu_seqlens[i] > maxlen) maxlen = cu_seqlens[i + 1] - cu_seqlens[i];
  int err = ORC_OK;
  /* one (document, kv head) per iteration: its dk/dv rows and the dq rows of
   * its query heads are written by that iteration alone */
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    double* ds = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    if (!p || !ds) {
#pragma omp atomic write
      err = ORC_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t w = 0; w < (int64_t)n * hkv; w++) {
        const int32_t i = (int32_t)(w / hkv), g = (int32_t)(w % hkv);
        const int64_t start = cu_seqlens[i], end = cu_seqlens[i + 1];
        for (int32_t h = g * grp; h < (g + 1) * grp; h++) {
          for (int64_t a = start; a < end; a++) {
            bwd_row(q, k, v, dout, hq, hkv, d, scale, start, a, h, p, ds, dq + (a * hq + h) * (int64_t)d);
            const double* qa = q + (a * hq + h) * (int64_t)d;
            const double* doa = dout + (a * hq + h) * (int64_t)d;
            for (int64_t j = 0; j <= a - start; j++) {
              double* dkb = dk + ((start + j) * hkv + g) * (int64_t)d;
              double* dvb = dv + ((start + j) * hkv + g) * (int64_t)d;
              for (int32_t c = 0; c < d; c++) {
                dkb[c] += scale * ds[j] * qa[c];
                dvb[c] += p[j] * doa[c];
              }
            }
          }
        }
      }
    }
    free(p);
    free(ds);
  }
  return err;
}

/* dk and dv of selected keys of one document for one kv head g: the same sums
 * as oracle_attention_bwd (over the group's query heads h and the document's
 * queries a >= key), arranged by query row so that each row's softmax and dS
 * are computed once for all the selected keys.  keys[i] are doc-local
 * positions.  The rows are split over the threads; each thread sums into its
 * own buffer and the buffers are added in thread order at the end. */
int oracle_attention_bwd_dkv_doc(const double* q, const double* k, const double* v, const double* dout,
                                 const int32_t* cu_seqlens, int32_t n, int32_t hq, int32_t hkv, int32_t d,
                                 double scale, int32_t doc, int32_t g, const int64_t* keys, int64_t nk,
                                 double* dk_out, double* dv_out) {
  if (check_heads(hq, hkv, d) != ORC_OK || n < 1 || doc < 0 || doc >= n || g < 0 || g >= hkv || nk < 1)
    return ORC_EINVAL;
  const int64_t start = cu_seqlens[doc], end = cu_seqlens[doc + 1], len = end - start;
  int64_t kmin = len;
  for (int64_t i = 0; i < nk; i++) {
    if (keys[i] < 0 || keys[i] >= len) return ORC_EINVAL;
    if (keys[i] < kmin) kmin = keys[i];
  }
  const int32_t grp = hq / hkv;
  const int nthreads = omp_get_max_threads();
  const size_t per = (size_t)nk * (size_t)d * 2;
  double* acc = (double*)calloc(per * (size_t)nthreads, sizeof(double));
  if (!acc) return ORC_ENOMEM;
  int err = ORC_OK;
  const int64_t rows = (int64_t)grp * (len - kmin);
#pragma omp parallel num_threads(nthreads)
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)len);
    double* ds = (double*)malloc(sizeof(double) * (size_t)len);
    double* dq_a = (double*)malloc(sizeof(double) * (size_t)d);
    double* mine = acc + per * (size_t)omp_get_thread_num();
    if (!p || !ds || !dq_a) {
#pragma omp atomic write
      err = ORC_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 8)
      for (int64_t r = 0; r < rows; r++) {
        const int32_t h = g * grp + (int32_t)(r / (len - kmin));
        const int64_t a = start + kmin + r % (len - kmin);
        bwd_row(q, k, v, dout, hq, hkv, d, scale, start, a, h, p, ds, dq_a);
        const double* qa = q + (a * hq + h) * (int64_t)d;
        const double* doa = dout + (a * hq + h) * (int64_t)d;
        for (int64_t i = 0; i < nk; i++) {
          const int64_t j = keys[i];
          if (start + j > a) continue;  /* key after the query: masked */
          double* dkb = mine + (size_t)i * d * 2;
          double* dvb = dkb + d;
          for (int32_t c = 0; c < d; c++) {
            dkb[c] += scale * ds[j] * qa[c];
            dvb[c] += p[j] * doa[c];
          }
        }
      }
    }
    free(p);
    free(ds);
    free(dq_a);
  }
  for (int64_t i = 0; i < nk; i++)
    for (int32_t c = 0; c < d; c++) {
      double sk = 0.0, sv = 0.0;
      for (int t = 0; t < nthreads; t++) {
        sk += acc[per * (size_t)t + (size_t)i * d * 2 + c];
        sv += acc[per * (size_t)t + (size_t)i * d * 2 + d + c];
      }
      dk_out[i * d + c] = sk;
      dv_out[i * d + c] = sv;
    }
  free(acc);
  return err;
}

/* Sampled dq rows: dq_out[i] = dq of token tokens[i], query head heads[i]. */
int oracle_attention_bwd_dq_rows(const double* q, const double* k, const double* v, const double* dout,
                                 const int32_t* cu_seqlens, int32_t n, int32_t hq, int32_t hkv, int32_t d,
                                 double scale, const int64_t* tokens, const int32_t* heads, int64_t ns,
                                 double* dq_out) {
  if (check_heads(hq, hkv, d) != ORC_OK || n < 1) return ORC_EINVAL;
  const int64_t T = cu_seqlens[n];
  int32_t maxlen = 0;
  for (int32_t i = 0; i < n; i++)
    if (cu_seqlens[i + 1] - cu_seqlens[i] > maxlen) maxlen = cu_seqlens[i + 1] - cu_seqlens[i];
  for (int64_t i = 0; i < ns; i++)
    if (tokens[i] < 0 || tokens[i] >= T || heads[i] < 0 || heads[i] >= hq) return ORC_EINVAL;
  int err = ORC_OK;
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    double* ds = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    if (!p || !ds) {
#pragma omp atomic write
      err = ORC_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < ns; i++) {
        const int32_t doc = doc_of_token(cu_seqlens, n, tokens[i]);
        bwd_row(q, k, v, dout, hq, hkv, d, scale, cu_seqlens[doc], tokens[i], heads[i], p, ds,
                dq_out + i * (int64_t)d);
      }
    }
    free(p);
    free(ds);
  }
  return err;
}

/* Sampled dk / dv rows: key token tokens[i] of kv head kv_heads[i]; sums over
 * the query heads of that group and the queries a >= the key in its document.
 * dk_out, dv_out [ns][d].  Cost per sample: (group x later queries) rows of
 * O(s d) each, so keys near the end of long documents are cheap. */
int oracle_attention_bwd_dkv_rows(const double* q, const double* k, const double* v, const double* dout,
                                  const int32_t* cu_seqlens, int32_t n, int32_t hq, int32_t hkv, int32_t d,
                                  double scale, const int64_t* tokens, const int32_t* kv_heads, int64_t ns,
                                  double* dk_out, double* dv_out) {
  if (check_heads(hq, hkv, d) != ORC_OK || n < 1) return ORC_EINVAL;
  const int64_t T = cu_seqlens[n];
  const int32_t grp = hq / hkv;
  int32_t maxlen = 0;
  for (int32_t i = 0; i < n; i++)
    if (cu_seqlens[i + 1] - cu_seqlens[i] > maxlen) maxlen = cu_seqlens[i + 1] - cu_seqlens[i];
  for (int64_t i = 0; i < ns; i++)
    if (tokens[i] < 0 || tokens[i] >= T || kv_heads[i] < 0 || kv_heads[i] >= hkv) return ORC_EINVAL;
  int err = ORC_OK;
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    double* ds = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    double* dq_a = (double*)malloc(sizeof(double) * (size_t)d);
    if (!p || !ds || !dq_a) {
#pragma omp atomic write
      err = ORC_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < ns; i++) {
        const int64_t b = tokens[i];
        const int32_t g = kv_heads[i];
        const int32_t doc = doc_of_token(cu_seqlens, n, b);
        const int64_t start = cu_seqlens[doc], end = cu_seqlens[doc + 1];
        double* dkb = dk_out + i * (int64_t)d;
        double* dvb = dv_out + i * (int64_t)d;
        for (int32_t c = 0; c < d; c++) dkb[c] = dvb[c] = 0.0;
        for (int32_t h = g * grp; h < (g + 1) * grp; h++) {
          for (int64_t a = b; a < end; a++) {
            bwd_row(q, k, v, dout, hq, hkv, d, scale, start, a, h, p, ds, dq_a);
            const double* qa = q + (a * hq + h) * (int64_t)d;
            const double* doa = dout + (a * hq + h) * (int64_t)d;
            for (int32_t c = 0; c < d; c++) {
              dkb[c] += scale * ds[b - start] * qa[c];
              dvb[c] += p[b - start] * doa[c];
            }
          }
        }
      }
    }
    free(p);
    free(ds);
    free(dq_a);
  }
  return err;
}
