/*
 * Host sanitizer lane for the oracle: TEST INFRASTRUCTURE ONLY.
 *
 * Built together with moe_oracle.c under -fsanitize=address,undefined (no
 * OpenMP) by tests/test_oracle_sanitize.py, this driver runs every oracle
 * entry point once on small deterministic inputs so that an out-of-bounds
 * access, a use after free, a leak or undefined behaviour stops the run.  It
 * checks no values (the pin tests do that); it prints a checksum.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

void oracle_router_logits(const uint16_t *x, const uint16_t *wr, const float *bias, int T, int H, int E,
                          float *logits);
void oracle_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w, float *gap);
int oracle_permute(const int32_t *ids, int T, int k, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                   int32_t *inv);
void oracle_dequant_int4(const uint8_t *q, const uint16_t *s, int rows, int K, float *w);
void oracle_experts_combine(const float *xin, int n, int H, int I, int k, const int32_t *ids, const float *w,
                            const uint16_t *wgu, const uint16_t *wd, const uint8_t *wgu_q, const uint16_t *sgu,
                            const uint8_t *wd_q, const uint16_t *sd, float *out);
void oracle_expert_rows(const float *xin, int n, int H, int I, const uint16_t *wgu, const uint16_t *wd, int e,
                        float *y);
void oracle_combine(const float *y, const int32_t *inv, const float *w, int T, int k, int H,
                    const float *residual, float *out);
void oracle_recall(const int32_t *pred, const int32_t *ref, int T, int k, int32_t *hits);
void oracle_round_bf16(const float *x, size_t n, uint16_t *out);
void oracle_rmsnorm(const float *x, const float *gamma, int T, int H, double eps, float *out);
int oracle_dedup(const int32_t *ids, int L, int Ttot, int k, int E, int B, int H, int I, uint32_t *mask,
                 int32_t *U, int64_t *bytes2, int64_t *bytes4);
int oracle_cache_plan(int policy, float decay, const int32_t *counts, int E, int32_t *slot_of,
                      int32_t *expert_of, int S, int32_t *hand, float *score, int32_t *last_use,
                      int32_t *miss_list, int32_t *miss_slot, int32_t *stats);
void oracle_sidecar(const uint16_t *feat, const uint16_t *w_trunk, const uint16_t *layer_emb,
                    const uint16_t *w_head, int T, int F, int r, int E, int L, int N, int32_t *cand,
                    float *cand_score, double *scores);

static uint32_t lcg_state = 12345u;
static uint32_t lcg(void) {
  lcg_state = lcg_state * 1664525u + 1013904223u;
  return lcg_state;
}
/* a bf16 value in about [-1, 1) */
static uint16_t rand_bf16(void) {
  const float f = ((float)(lcg() >> 8) / 16777216.0f) * 2.0f - 1.0f;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}
static void fill_bf16(uint16_t *p, size_t n) {
  for (size_t i = 0; i < n; ++i) p[i] = rand_bf16();
}

int main(void) {
  enum { T = 3, H = 64, E = 8, K = 3, I = 64, L = 2 };
  double check = 0.0;
  uint16_t *x = malloc(sizeof(uint16_t) * T * H), *wr = malloc(sizeof(uint16_t) * E * H);
  uint16_t *wgu = malloc(sizeof(uint16_t) * E * 2 * I * H), *wd = malloc(sizeof(uint16_t) * E * H * I);
  float *bias = malloc(sizeof(float) * E), *logits = malloc(sizeof(float) * T * E);
  fill_bf16(x, T * H);
  fill_bf16(wr, E * H);
  fill_bf16(wgu, (size_t)E * 2 * I * H);
  fill_bf16(wd, (size_t)E * H * I);
  for (int e = 0; e < E; ++e) bias[e] = -0.1f * e;
  oracle_router_logits(x, wr, bias, T, H, E, logits);
  int32_t ids[T * K], counts[E], offsets[E + 1], perm[T * K], inv[T * K];
  float w[T * K], gap[T];
  oracle_topk(logits, T, E, K, ids, w, gap);
  if (oracle_permute(ids, T, K, E, counts, offsets, perm, inv) != 0) return 2;
  float *xin = malloc(sizeof(float) * T * H), *out = malloc(sizeof(float) * T * H);
  for (int i = 0; i < T * H; ++i) {
    uint32_t u = (uint32_t)x[i] << 16;
    memcpy(&xin[i], &u, 4);
  }
  oracle_experts_combine(xin, T, H, I, K, ids, w, wgu, wd, NULL, NULL, NULL, NULL, out);
  for (int i = 0; i < T * H; ++i) check += out[i];
  /* int4 records: codes [E, 2I, H/2], scales [E, 2I, H/64]; down [E, H, I/2], [E, H, I/64] */
  uint8_t *qgu = malloc((size_t)E * 2 * I * H / 2), *qd = malloc((size_t)E * H * I / 2);
  uint16_t *sgu = malloc(sizeof(uint16_t) * E * 2 * I * (H / 64)), *sd = malloc(sizeof(uint16_t) * E * H * (I / 64));
  for (size_t i = 0; i < (size_t)E * 2 * I * H / 2; ++i) qgu[i] = (uint8_t)lcg();
  for (size_t i = 0; i < (size_t)E * H * I / 2; ++i) qd[i] = (uint8_t)lcg();
  fill_bf16(sgu, (size_t)E * 2 * I * (H / 64));
  fill_bf16(sd, (size_t)E * H * (I / 64));
  oracle_experts_combine(xin, T, H, I, K, ids, w, NULL, NULL, qgu, sgu, qd, sd, out);
  for (int i = 0; i < T * H; ++i) check += out[i];
  float *deq = malloc(sizeof(float) * 2 * I * H);
  oracle_dequant_int4(qgu, sgu, 2 * I, H, deq);
  check += deq[5];
  float *y = malloc(sizeof(float) * T * K * H), *res = malloc(sizeof(float) * T * H);
  oracle_expert_rows(xin, T, H, I, wgu, wd, 3, y);
  for (int i = 0; i < T * K * H; ++i) y[i] = (float)(i % 7) * 0.25f;
  for (int i = 0; i < T * H; ++i) res[i] = 1.0f;
  oracle_combine(y, inv, w, T, K, H, res, out);
  check += out[T * H - 1];
  int32_t hits[T];
  oracle_recall(ids, ids, T, K, hits);
  uint16_t rb[T * H];
  oracle_round_bf16(out, T * H, rb);
  oracle_rmsnorm(out, NULL, T, H, 1e-6, res);
  check += res[0] + hits[0] + rb[0];
  int32_t lids[L * T * K];
  for (int i = 0; i < L * T * K; ++i) lids[i] = ids[i % (T * K)];
  uint32_t mask[L * T * 1];
  int32_t U[L * T];
  int64_t b2[T], b4[T];
  if (oracle_dedup(lids, L, T, K, E, 1, H, I, mask, U, b2, b4) != 0) return 3;
  check += (double)b4[0];
  for (int policy = 0; policy < 3; ++policy) {
    const int S = 4;
    int32_t slot_of[E], expert_of[S], hand[2] = {0, 0}, last_use[S], ml[S], ms[S], stats[4] = {0, 0, 0, 0};
    float score[E];
    for (int e = 0; e < E; ++e) slot_of[e] = -1, score[e] = 0.0f;
    for (int s = 0; s < S; ++s) expert_of[s] = -1, last_use[s] = -1;
    for (int call = 0; call < 30; ++call) {
      int32_t c[E];
      for (int e = 0; e < E; ++e) c[e] = (lcg() >> 29) == 0 ? 1 : 0;
      oracle_cache_plan(policy, 0.8f, c, E, slot_of, expert_of, S, hand, score, last_use, ml, ms, stats);
    }
    check += stats[3];
  }
  {
    enum { F = 16, R = 8, LS = 3, N = 4 };
    uint16_t feat[T * F], trunk[R * F], emb[LS * R], head[E * R];
    fill_bf16(feat, T * F);
    fill_bf16(trunk, R * F);
    fill_bf16(emb, LS * R);
    fill_bf16(head, E * R);
    int32_t cand[T * LS * N];
    float cs[T * LS * N];
    double sc[T * LS * E];
    oracle_sidecar(feat, trunk, emb, head, T, F, R, E, LS, N, cand, cs, sc);
    check += cs[0] + cand[1];
  }
  printf("checksum %.6f\n", check);
  free(x), free(wr), free(wgu), free(wd), free(bias), free(logits), free(xin), free(out);
  free(qgu), free(qd), free(sgu), free(sd), free(deq), free(y), free(res);
  return isfinite(check) ? 0 : 4;
}
