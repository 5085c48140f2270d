/*
 * CPU oracle for the routed-expert MoE layer: TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct C.  Only the tests, the package's smoke
 * check and bench.py's cpu_baseline / reference leg may call it; the CUDA
 * library never links or calls it, and the two share no code, header,
 * table or constant.
 *
 * Sources (Hebrus "Agent Field Notes"):
 *  - AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus: evidence before
 *    execution", section "Phase 1: separate math from acceleration":
 *    float32 router softmax and normalized top-10 selection; zero-centred
 *    RMS normalisation.
 *  - AFN-019 "Hide SSD misses before the router knows they exist", section
 *    "Why overlap alone cannot defeat the byte roofline": expert geometry
 *    (gate + up + down), deduplication of repeated routes across a verifier
 *    block, grouping token rows by expert.
 *  - AFN-019, section "Hypothesis H4: ExpertMajor should stream as a
 *    wavefront, not a barrier": gate and up are used together, down after
 *    the SwiGLU intermediate exists; the weighted sum follows a
 *    deterministic route-rank order.
 *  - AFN-019, section "Hypothesis H7: DFlash block size must follow I/O
 *    cost": 48 * U_B * record bytes per block, break-even U_B < 10 tau(B).
 *  - AFN-019, section "Two storage workloads, not one": an expert miss moves
 *    a whole record; replacement by score(record) = P(use before eviction)
 *    x expected exposed latency avoided / resident bytes, measured against
 *    least-recently-used replacement as the baseline.
 *  - AFN-021 "Replay decode as prefill: a training flywheel for predictive
 *    MoE I/O", section "What feature should the sidecar see?": feature ->
 *    shared low-rank trunk -> plus target-layer embedding -> shared
 *    expert-head embeddings -> one score per expert -> ranked candidates.
 *  - AFN-021 "Replay decode as prefill: a training flywheel for predictive
 *    MoE I/O", section "The key equivalence -- and where it breaks": expert
 *    IDs and their rank order must match exactly; weights within a declared
 *    tolerance.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - selection key is the fp32 logit (sum accumulated in fp64, plus bias,
 *    rounded once to fp32); ties break towards the lower expert ID;
 *  - "normalized top-k" = softmax restricted to the k selected logits
 *    (identical to full softmax divided by the top-k mass);
 *  - SwiGLU h = silu(g) * u with silu(z) = z / (1 + exp(-z));
 *  - gate/up rows are [I,H] (out x in), down is [H,I];
 *  - rows of one expert are grouped in ascending flat route order t*k + j;
 *  - int4 g64: w = scale * q, q signed in [-8,7], 64 consecutive inputs per
 *    scale, even input index in the low nibble.
 *
 * Everything that is floating point is evaluated in fp64 and stored as fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_bits_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int oracle_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* ---- router logits: L[t,e] = fp32( sum_h x[t,h] * Wr[e,h] + b[e] ) ------ */
void oracle_router_logits(const uint16_t *x, const uint16_t *wr, const float *bias,
                          int T, int H, int E, float *logits) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h)
        s += bf16_bits_to_f64(x[(size_t)t * H + h]) * bf16_bits_to_f64(wr[(size_t)e * H + h]);
      if (bias) s += (double)bias[e];
      logits[(size_t)t * E + e] = (float)s;
    }
  }
}

/* Same, for an fp32 input row (the RMS-normalised residual of the stack). */
void oracle_router_logits_f32(const float *x, const uint16_t *wr, const float *bias,
                              int T, int H, int E, float *logits) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h)
        s += (double)x[(size_t)t * H + h] * bf16_bits_to_f64(wr[(size_t)e * H + h]);
      if (bias) s += (double)bias[e];
      logits[(size_t)t * E + e] = (float)s;
    }
  }
}

/* ---- top-k over fp32 logits ---------------------------------------------
 * Full sort of every row by (logit descending, expert ID ascending); the
 * first k IDs in that order are the route, in rank order.  Weights are the
 * softmax over those k logits:  w_j = exp(L_j - L_0) / sum_j' exp(L_j' - L_0).
 * gap[t] = L(k-th) - L((k+1)-th), +inf when k == E.                        */
typedef struct {
  float v;
  int e;
} scored;

static int cmp_scored(const void *pa, const void *pb) {
  const scored *a = (const scored *)pa, *b = (const scored *)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->e < b->e) ? -1 : (a->e > b->e);
}

void oracle_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w, float *gap) {
#pragma omp parallel
  {
    scored *row = (scored *)malloc(sizeof(scored) * (size_t)E);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      for (int e = 0; e < E; ++e) {
        row[e].v = logits[(size_t)t * E + e];
        row[e].e = e;
      }
      qsort(row, (size_t)E, sizeof(scored), cmp_scored);
      double denom = 0.0;
      for (int j = 0; j < k; ++j) denom += exp((double)row[j].v - (double)row[0].v);
      for (int j = 0; j < k; ++j) {
        ids[(size_t)t * k + j] = row[j].e;
        w[(size_t)t * k + j] = (float)(exp((double)row[j].v - (double)row[0].v) / denom);
      }
      if (gap) gap[t] = (k < E) ? (float)((double)row[k - 1].v - (double)row[k].v) : INFINITY;
    }
    free(row);
  }
}

/* ---- grouping token rows by expert: stable counting sort ----------------
 * counts[e] = #{r : ids[r] == e};  offsets = exclusive scan (offsets[E] = R);
 * slots of expert e hold its routes r = t*k + j in ascending r;
 * perm[slot] = r and inv[r] = slot.  Returns -1 on an ID outside [0,E).    */
int oracle_permute(const int32_t *ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                   int32_t *perm, int32_t *inv) {
  const int R = T * k;
  if (E <= 0) return -1;
  for (int r = 0; r < R; ++r)
    if (ids[r] < 0 || ids[r] >= E) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int r = 0; r < R; ++r) counts[ids[r]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  for (int r = 0; r < R; ++r) {
    int e = ids[r];
    int s = offsets[e] + fill[e]++;
    perm[s] = r;
    inv[r] = s;
  }
  free(fill);
  return 0;
}

/* ---- one expert: y = Wd * (silu(Wg x) .* (Wu x)), all in fp64 ----------- */
static void expert_forward(const double *xin, int H, int I, const float *wg, const float *wu,
                           const float *wd, double *hbuf, double *y) {
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int h = 0; h < H; ++h) {
      g += (double)wg[(size_t)i * H + h] * xin[h];
      u += (double)wu[(size_t)i * H + h] * xin[h];
    }
    hbuf[i] = g / (1.0 + exp(-g)) * u;
  }
  for (int o = 0; o < H; ++o) {
    double s = 0.0;
    for (int i = 0; i < I; ++i) s += (double)wd[(size_t)o * I + i] * hbuf[i];
    y[o] = s;
  }
}

/* int4 g64 -> fp32: w[row][c] = scale[row][c/64] * q[row][c]. */
void oracle_dequant_int4(const uint8_t *q, const uint16_t *s, int rows, int K, float *w) {
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < K; ++c) {
      uint8_t byte = q[(size_t)r * (K / 2) + c / 2];
      int nib = (c & 1) ? (byte >> 4) : (byte & 0xF);
      int qv = (nib >= 8) ? nib - 16 : nib;
      w[(size_t)r * K + c] = (float)(bf16_bits_to_f64(s[(size_t)r * (K / 64) + c / 64]) * (double)qv);
    }
}

static void expert_weights_bf16(const uint16_t *wgu, const uint16_t *wd, int e, int H, int I,
                                float *g, float *u, float *d) {
  const uint16_t *base = wgu + (size_t)e * 2 * I * H;
  for (size_t n = 0; n < (size_t)I * H; ++n) {
    g[n] = (float)bf16_bits_to_f64(base[n]);
    u[n] = (float)bf16_bits_to_f64(base[(size_t)I * H + n]);
  }
  const uint16_t *db = wd + (size_t)e * H * I;
  for (size_t n = 0; n < (size_t)H * I; ++n) d[n] = (float)bf16_bits_to_f64(db[n]);
}

static void expert_weights_int4(const uint8_t *wgu_q, const uint16_t *sgu, const uint8_t *wd_q,
                                const uint16_t *sd, int e, int H, int I, float *g, float *u,
                                float *d) {
  oracle_dequant_int4(wgu_q + (size_t)e * 2 * I * (H / 2), sgu + (size_t)e * 2 * I * (H / 64), I, H, g);
  oracle_dequant_int4(wgu_q + (size_t)e * 2 * I * (H / 2) + (size_t)I * (H / 2),
                      sgu + (size_t)e * 2 * I * (H / 64) + (size_t)I * (H / 64), I, H, u);
  oracle_dequant_int4(wd_q + (size_t)e * H * (I / 2), sd + (size_t)e * H * (I / 64), H, I, d);
}

/* ---- expert outputs + weighted combine for n tokens ---------------------
 * xin [n,H] fp32 is the expert input (bf16 x widened, or RMSNorm output).
 * out[t] = sum_{j=0..k-1} w[t,j] * y_{ids[t,j]}(x_t), summed in rank order j.
 * Exactly one of (wgu, wd) or (wgu_q, sgu, wd_q, sd) is given.             */
void oracle_experts_combine(const float *xin, int n, int H, int I, int k, const int32_t *ids,
                            const float *w, const uint16_t *wgu, const uint16_t *wd,
                            const uint8_t *wgu_q, const uint16_t *sgu, const uint8_t *wd_q,
                            const uint16_t *sd, float *out) {
#pragma omp parallel
  {
    float *g = (float *)malloc(sizeof(float) * (size_t)I * H);
    float *u = (float *)malloc(sizeof(float) * (size_t)I * H);
    float *d = (float *)malloc(sizeof(float) * (size_t)H * I);
    double *xd = (double *)malloc(sizeof(double) * (size_t)H);
    double *hb = (double *)malloc(sizeof(double) * (size_t)I);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
    for (int t = 0; t < n; ++t) {
      for (int h = 0; h < H; ++h) {
        xd[h] = (double)xin[(size_t)t * H + h];
        acc[h] = 0.0;
      }
      for (int j = 0; j < k; ++j) {
        int e = ids[(size_t)t * k + j];
        if (wgu)
          expert_weights_bf16(wgu, wd, e, H, I, g, u, d);
        else
          expert_weights_int4(wgu_q, sgu, wd_q, sd, e, H, I, g, u, d);
        expert_forward(xd, H, I, g, u, d, hb, y);
        double wj = (double)w[(size_t)t * k + j];
        for (int h = 0; h < H; ++h) acc[h] += wj * y[h];
      }
      for (int h = 0; h < H; ++h) out[(size_t)t * H + h] = (float)acc[h];
    }
    free(g); free(u); free(d); free(xd); free(hb); free(y); free(acc);
  }
}

/* One expert applied to fp32 rows (no routing): y[n,H].  Exposed so that
 * single-expert special cases can be checked against plain matmuls.        */
void oracle_expert_rows(const float *xin, int n, int H, int I, const uint16_t *wgu,
                        const uint16_t *wd, int e, float *y) {
  float *g = (float *)malloc(sizeof(float) * (size_t)I * H);
  float *u = (float *)malloc(sizeof(float) * (size_t)I * H);
  float *d = (float *)malloc(sizeof(float) * (size_t)H * I);
  double *xd = (double *)malloc(sizeof(double) * (size_t)H);
  double *hb = (double *)malloc(sizeof(double) * (size_t)I);
  double *yd = (double *)malloc(sizeof(double) * (size_t)H);
  expert_weights_bf16(wgu, wd, e, H, I, g, u, d);
  for (int t = 0; t < n; ++t) {
    for (int h = 0; h < H; ++h) xd[h] = (double)xin[(size_t)t * H + h];
    expert_forward(xd, H, I, g, u, d, hb, yd);
    for (int h = 0; h < H; ++h) y[(size_t)t * H + h] = (float)yd[h];
  }
  free(g); free(u); free(d); free(xd); free(hb); free(yd);
}

/* ---- combine alone: out[t] = sum_j w[t,j] * y[inv[t*k+j]] in rank order j.
 * y [R,H] holds one expert output per slot.                                */
void oracle_combine(const float *y, const int32_t *inv, const float *w, int T, int k, int H,
                    const float *residual, float *out) {
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += (double)w[(size_t)t * k + j] * (double)y[(size_t)inv[(size_t)t * k + j] * H + h];
      if (residual) acc += (double)residual[(size_t)t * H + h];
      out[(size_t)t * H + h] = (float)acc;
    }
}

/* ---- recall of a predicted route ------------------------------------------
 * hits[t] = |{pred[t,:]} intersect {ref[t,:]}| (AFN-019, section
 * "Hypothesis H2": a predictor is scored against the exact top-k).          */
void oracle_recall(const int32_t *pred, const int32_t *ref, int T, int k, int32_t *hits) {
  for (int t = 0; t < T; ++t) {
    int h = 0;
    for (int j = 0; j < k; ++j)
      for (int i = 0; i < k; ++i)
        if (ref[(size_t)t * k + j] == pred[(size_t)t * k + i]) {
          ++h;
          break;
        }
    hits[t] = h;
  }
}

/* fp32 -> bf16 bit patterns, round to nearest, ties to even (NaN kept
 * quiet).  Reading for the residual stack: the MoE layer's input x is bf16
 * in every workload of the layer (the Qwen4Exp geometry's tokens are bf16),
 * and in the stack that input is RMSNorm(x_l); so the normalised residual is
 * rounded to bf16 once before routing and the experts, while the residual
 * stream itself stays fp32.                                                 */
void oracle_round_bf16(const float *x, size_t n, uint16_t *out) {
  for (size_t i = 0; i < n; ++i) {
    uint32_t u;
    memcpy(&u, &x[i], 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) {
      out[i] = (uint16_t)((u >> 16) | 0x40u);
      continue;
    }
    uint32_t lsb = (u >> 16) & 1u;
    out[i] = (uint16_t)((u + 0x7fffu + lsb) >> 16);
  }
}

/* ---- zero-centred RMSNorm: n = x / sqrt(mean(x^2) + eps) * (1 + gamma) --- */
void oracle_rmsnorm(const float *x, const float *gamma, int T, int H, double eps, float *out) {
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int h = 0; h < H; ++h) ss += (double)x[(size_t)t * H + h] * (double)x[(size_t)t * H + h];
    double r = 1.0 / sqrt(ss / H + eps);
    for (int h = 0; h < H; ++h)
      out[(size_t)t * H + h] =
          (float)((double)x[(size_t)t * H + h] * r * (1.0 + (gamma ? (double)gamma[h] : 0.0)));
  }
}

/* ---- block deduplication --------------------------------------------------
 * ids [L, Ttot, k].  Block b covers tokens [b*B, min((b+1)*B, Ttot)).
 * mask[l,b] = set of experts routed by any token of the block in layer l,
 * U[l,b] = |mask|, bytes at `bits` per parameter = sum_l U[l,b] * P * bits/8
 * with P = 3*H*I parameters per expert record.  Returns -1 on a bad ID.    */
int oracle_dedup(const int32_t *ids, int L, int Ttot, int k, int E, int B, int H, int I,
                 uint32_t *mask, int32_t *U, int64_t *bytes2, int64_t *bytes4) {
  const int nb = (Ttot + B - 1) / B;
  const int W = (E + 31) / 32;
  const int64_t P = 3LL * H * I;
  unsigned char *seen = (unsigned char *)malloc((size_t)E);
  for (int b = 0; b < nb; ++b) {
    int64_t usum = 0;
    for (int l = 0; l < L; ++l) {
      memset(seen, 0, (size_t)E);
      for (int t = b * B; t < Ttot && t < (b + 1) * B; ++t)
        for (int j = 0; j < k; ++j) {
          int e = ids[((size_t)l * Ttot + t) * k + j];
          if (e < 0 || e >= E) {
            free(seen);
            return -1;
          }
          seen[e] = 1;
        }
      int u = 0;
      for (int w = 0; w < W; ++w) {
        uint32_t m = 0;
        for (int bit = 0; bit < 32; ++bit)
          if (w * 32 + bit < E && seen[w * 32 + bit]) {
            m |= 1u << bit;
            ++u;
          }
        mask[((size_t)l * nb + b) * W + w] = m;
      }
      U[(size_t)l * nb + b] = u;
      usum += u;
    }
    bytes2[b] = usum * P * 2 / 8;
    bytes4[b] = usum * P * 4 / 8;
  }
  free(seen);
  return 0;
}

/* ---- expert cache plan ---------------------------------------------------
 * One call of the exact-miss expert cache (S slots over E experts).
 * State: slot_of [E] (slot or -1), expert_of [S] (expert or -1),
 * hand [2] = {FIFO hand, call counter}, score [E] (SCORE), last_use [S]
 * (LRU).  counts [E]: routes per expert in this call.
 *
 * Routed experts that hold a slot are hits; the others are misses, taken in
 * expert order.  A slot whose expert is routed in this call is pinned.  The
 * other slots are candidate victims, ordered by the policy:
 *   0 FIFO: rotation order starting at the hand (the oldest fill first);
 *   1 LRU: empty slots first, then the least recent call that used them;
 *   2 SCORE: empty slots first, then the lowest
 *        score(record) = P(use before eviction)
 *                        * expected exposed latency avoided / resident bytes.
 *     Readings: every record is a whole gate/up/down record of one size, so
 *     the latency a hit avoids (bytes / link bandwidth, the same for every
 *     record) divided by the resident bytes is one constant; P(use before
 *     eviction) over a common horizon grows with the per-call use rate p,
 *     estimated as p = (1 - decay) * f with f <- decay * f + [routed] (one
 *     fp32 fused multiply-add per call, the precision the device keeps).
 * Ties go to the lower slot.  Miss m takes the m-th candidate.  If there are
 * more misses than candidates the slots stay unchanged; returns 1 then
 * (CACHE_FULL), else 0.  The call counter and the use rates advance either
 * way.  stats = {hits, misses, running hits, running misses}.              */
typedef struct {
  double key;
  int empty;
  int slot;
} victim_t;

static int cmp_victim(const void *pa, const void *pb) {
  const victim_t *a = (const victim_t *)pa, *b = (const victim_t *)pb;
  if (a->empty != b->empty) return a->empty ? -1 : 1;
  if (a->key < b->key) return -1;
  if (a->key > b->key) return 1;
  return a->slot - b->slot;
}

int oracle_cache_plan(int policy, float decay, const int32_t *counts, int E, int32_t *slot_of,
                      int32_t *expert_of, int S, int32_t *hand, float *score, int32_t *last_use,
                      int32_t *miss_list, int32_t *miss_slot, int32_t *stats) {
  const int step = hand[1];
  const double link_bw = 1.0, record_bytes = 1.0; /* one size for every record */
  if (policy == 2)
    for (int e = 0; e < E; ++e) score[e] = fmaf(decay, score[e], counts[e] > 0 ? 1.0f : 0.0f);
  int hits = 0, nmiss = 0;
  int32_t *misses = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
  for (int e = 0; e < E; ++e) {
    if (counts[e] <= 0) continue;
    if (slot_of[e] >= 0)
      ++hits;
    else
      misses[nmiss++] = e;
  }
  victim_t *cand = (victim_t *)malloc(sizeof(victim_t) * (size_t)S);
  int nc = 0;
  const int h = ((hand[0] % S) + S) % S;
  for (int s = 0; s < S; ++s) {
    const int ex = expert_of[s];
    const int occupied = ex >= 0 && ex < E;
    if (occupied && counts[ex] > 0) continue; /* pinned by this call */
    victim_t v;
    v.slot = s;
    v.empty = 0;
    v.key = 0.0;
    if (policy == 0) {
      v.key = (double)((s - h + S) % S);
    } else if (!occupied) {
      v.empty = 1;
    } else if (policy == 1) {
      v.key = (double)last_use[s];
    } else {
      const double p_use = (1.0 - (double)decay) * (double)score[ex];
      v.key = p_use * (record_bytes / link_bw) / record_bytes;
    }
    cand[nc++] = v;
  }
  int full = 0;
  if (nmiss > nc) {
    full = 1;
    stats[0] = hits;
    stats[1] = 0;
    stats[2] += hits;
  } else {
    qsort(cand, (size_t)nc, sizeof(victim_t), cmp_victim);
    for (int m = 0; m < nmiss; ++m) {
      const int v = cand[m].slot;
      if (expert_of[v] >= 0 && expert_of[v] < E) slot_of[expert_of[v]] = -1;
    }
    for (int m = 0; m < nmiss; ++m) {
      const int e = misses[m], v = cand[m].slot;
      slot_of[e] = v;
      expert_of[v] = e;
      miss_list[m] = e;
      miss_slot[m] = v;
    }
    if (policy == 1)
      for (int e = 0; e < E; ++e)
        if (counts[e] > 0) last_use[slot_of[e]] = step;
    if (policy == 0 && nmiss > 0) hand[0] = (cand[nmiss - 1].slot + 1) % S;
    stats[0] = hits;
    stats[1] = nmiss;
    stats[2] += hits;
    stats[3] += nmiss;
  }
  hand[1] = step + 1;
  free(misses);
  free(cand);
  return full;
}

/* ---- route sidecar forward pass ------------------------------------------
 * feat [T,F], w_trunk [r,F], layer_emb [L,r], w_head [E,r], all bf16.
 * For position t and layer l:
 *   z      = w_trunk . feat[t]                 (the shared low-rank trunk)
 *   z_l    = z + layer_emb[l]                  (the target-layer embedding)
 *   s[e]   = w_head[e] . z_l                   (shared expert-head embeddings)
 * and the N experts with the largest s in rank order (ties to the lower ID).
 * Reading: no nonlinearity anywhere (the pages name none).  Everything in
 * fp64; scores [T,L,E] (optional) and cand_score are the fp64 values
 * (cand_score rounded to fp32).                                              */
static const double *sidecar_scores_for_sort;

static int cmp_sidecar(const void *pa, const void *pb) {
  const int a = *(const int *)pa, b = *(const int *)pb;
  const double sa = sidecar_scores_for_sort[a], sb = sidecar_scores_for_sort[b];
  if (sa > sb) return -1;
  if (sa < sb) return 1;
  return a - b;
}

void oracle_sidecar(const uint16_t *feat, const uint16_t *w_trunk, const uint16_t *layer_emb,
                    const uint16_t *w_head, int T, int F, int r, int E, int L, int N, int32_t *cand,
                    float *cand_score, double *scores) {
  double *z = (double *)malloc(sizeof(double) * (size_t)r);
  double *zl = (double *)malloc(sizeof(double) * (size_t)r);
  double *s = (double *)malloc(sizeof(double) * (size_t)E);
  int *order = (int *)malloc(sizeof(int) * (size_t)E);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int f = 0; f < F; ++f)
        acc += bf16_bits_to_f64(w_trunk[(size_t)j * F + f]) * bf16_bits_to_f64(feat[(size_t)t * F + f]);
      z[j] = acc;
    }
    for (int l = 0; l < L; ++l) {
      for (int j = 0; j < r; ++j) zl[j] = z[j] + bf16_bits_to_f64(layer_emb[(size_t)l * r + j]);
      for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int j = 0; j < r; ++j) acc += bf16_bits_to_f64(w_head[(size_t)e * r + j]) * zl[j];
        s[e] = acc;
        order[e] = e;
        if (scores) scores[((size_t)t * L + l) * E + e] = acc;
      }
      sidecar_scores_for_sort = s;
      qsort(order, (size_t)E, sizeof(int), cmp_sidecar);
      for (int n = 0; n < N; ++n) {
        cand[((size_t)t * L + l) * N + n] = order[n];
        cand_score[((size_t)t * L + l) * N + n] = (float)s[order[n]];
      }
    }
  }
  free(z);
  free(zl);
  free(s);
  free(order);
}
