/*
 * moe_route_sort_oracle.c -- plain, slow, single-threaded CPU oracle for MoE route-sort.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or call this
 * file: only the test suite, the smoke check and the CPU-baseline leg of the benchmark use it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff
 * (stack)", Summary: the route-sort kernel converts the logits to FP32, applies the
 * correction bias, runs grouped top-k and both sort phases, and hands the prepared
 * metadata to GEMM1; and "Summary -- general gfx1250 ordinary-TP route optimization"
 * (ROCm/aiter pull 7095), section "Dispatch and contracts": a negative expert id is a
 * dropped route that claims no slot).  Every step is written as its plain definition:
 * full sorts instead of partial selection, one token at a time, no blocking or fusion.
 *
 * Floating point: IEEE binary32 throughout, libm expf, IEEE division; build with
 * -ffp-contract=off and without -ffast-math so no operation is fused or reordered.
 *
 * Readings of points the pages leave open (each is stated where it is used):
 *   R1 score      s = 1 / (1 + expf(-x))                          (sigmoid scoring)
 *   R2 key        key = s + bias[e]   (one fp32 add; bias steers selection only)
 *   R3 group      group score = sum of the two largest keys of the group, largest first;
 *                 a group of one expert scores its single key
 *   R4 ties       larger value first; equal values -> lower index first (groups and experts)
 *   R5 slots      the K selected experts are listed in descending key order
 *   R6 weights    sum = s_0 + s_1 + ... + s_{K-1} in slot order; w_k = (s_k / sum) * R
 *   R7 sort       cnt_e over all routes, pad_e = ceil(cnt_e / B) * B (0 when cnt_e = 0),
 *                 off_e = exclusive prefix sum of pad over e ascending, npp = sum pad;
 *                 routes placed in flat order r = t*K + k (token-major, then slot);
 *                 padding rows hold the sentinel N = T*K with weight 0;
 *                 expert_ids[b] = owner of block b of size B
 *   R8 ids        in the sort step, id < 0 is a dropped route (no slot, not counted);
 *                 id >= E is invalid: flagged and dropped
 *   R13 softmax   the softmax variant (no bias, no groups): key = x; the K largest keys,
 *                 ties to the lower index; m = x of slot 0; s_k = expf(x_k - m) in slot
 *                 order; w_k = (s_k / (s_0 + ... + s_{K-1})) * R -- the softmax over all E
 *                 experts restricted to the selected ones and renormalised (the normaliser
 *                 over all E cancels), so selection and weights need no full-row sum
 *   R14 gate      the router gate projection ahead of the path: logits[t,e] = the bf16
 *                 nearest (ties to even) to the dot product of hidden row t and gate row e,
 *                 both bf16; one rounding of the exact sum (formed here as an exact
 *                 fixed-point integer, so no intermediate rounding happens at all)
 *
 * Parity pins: every function here is pinned by the tests in tests/test_oracle_pins.py
 * (bf16 decoding against a library conversion over all 65536 patterns, sigmoid against a
 * float64 evaluation, group selection against subset enumeration, top-k against an
 * independent full sort and a textbook argsort, sort phase against a stable sort and a
 * hand-worked example in tests/golden/).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARGS (-1)
#define ORACLE_ERR_NOMEM (-2)
#define ORACLE_FLAG_BAD_EXPERT_ID 0x1

/* ---------------------------------------------------------------- scalar steps */

/* O1. bf16 -> fp32: a bf16 value is the upper 16 bits of an IEEE binary32 pattern. */
float oracle_bf16_to_float(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

/* O2 / R1. sigmoid score with libm expf and an IEEE division. */
float oracle_sigmoid(float x) {
  float e = expf(-x);
  float d = 1.0f + e;
  return 1.0f / d;
}

/* Array forms of O1 and O2 (element by element), so that test code can read the
 * binary32 results without a round trip through a host double. */
void oracle_bf16_to_float_n(const uint16_t* h, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_float(h[i]);
}

void oracle_sigmoid_n(const float* x, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_sigmoid(x[i]);
}

/* ------------------------------------------------------------- sort helpers */

typedef struct {
  float value;
  int32_t index;
} oracle_item;

/* R4: larger value first; equal values -> lower index first.  A total order (indices are
 * unique), so qsort's lack of stability does not matter. */
static int oracle_item_desc(const void* pa, const void* pb) {
  const oracle_item* a = (const oracle_item*)pa;
  const oracle_item* b = (const oracle_item*)pb;
  if (a->value > b->value) return -1;
  if (a->value < b->value) return 1;
  if (a->index < b->index) return -1;
  if (a->index > b->index) return 1;
  return 0;
}

static int oracle_route_args_ok(int T, int E, int G, int Kg, int K) {
  if (T < 0 || E < 1 || G < 1 || E % G != 0) return 0;
  if (Kg < 1 || Kg > G) return 0;
  if (K < 1 || (int64_t)K > (int64_t)Kg * (E / G)) return 0;
  return 1;
}

/* ------------------------------------------------------- per-token steps (exposed) */

/* O1+O2+R2 for one row: s[e] and key[e]. */
void oracle_scores_row(const uint16_t* logits_row, const float* bias, int E, float* s,
                       float* key) {
  for (int e = 0; e < E; ++e) {
    float x = oracle_bf16_to_float(logits_row[e]);
    s[e] = oracle_sigmoid(x);
    key[e] = s[e] + bias[e];
  }
}

/* R3: group scores of one row from its keys.  Each group is fully sorted and its two
 * largest keys are added, largest first. */
int oracle_group_scores_row(const float* key, int E, int G, float* gs) {
  int g = E / G;
  oracle_item* tmp = (oracle_item*)malloc(sizeof(oracle_item) * (size_t)g);
  if (!tmp) return ORACLE_ERR_NOMEM;
  for (int j = 0; j < G; ++j) {
    for (int i = 0; i < g; ++i) {
      tmp[i].value = key[j * g + i];
      tmp[i].index = j * g + i;
    }
    qsort(tmp, (size_t)g, sizeof(oracle_item), oracle_item_desc);
    gs[j] = (g >= 2) ? (tmp[0].value + tmp[1].value) : tmp[0].value;
  }
  free(tmp);
  return ORACLE_OK;
}

/* R4: the Kg kept groups of one row, by a full sort of (score desc, index asc).
 * kept_flag[j] = 1 for kept groups, 0 otherwise. */
int oracle_kept_groups_row(const float* gs, int G, int Kg, int32_t* kept_flag) {
  oracle_item* tmp = (oracle_item*)malloc(sizeof(oracle_item) * (size_t)G);
  if (!tmp) return ORACLE_ERR_NOMEM;
  for (int j = 0; j < G; ++j) {
    tmp[j].value = gs[j];
    tmp[j].index = j;
    kept_flag[j] = 0;
  }
  qsort(tmp, (size_t)G, sizeof(oracle_item), oracle_item_desc);
  for (int r = 0; r < Kg; ++r) kept_flag[tmp[r].index] = 1;
  free(tmp);
  return ORACLE_OK;
}

/* R5: top-K experts of one row among the experts of kept groups, by a full sort of the
 * candidates on (key desc, index asc).  ids[k] in slot order. */
int oracle_topk_row(const float* key, int E, int G, const int32_t* kept_flag, int K,
                    int32_t* ids) {
  int g = E / G;
  oracle_item* cand = (oracle_item*)malloc(sizeof(oracle_item) * (size_t)E);
  if (!cand) return ORACLE_ERR_NOMEM;
  int n = 0;
  for (int e = 0; e < E; ++e) {
    if (kept_flag[e / g]) {
      cand[n].value = key[e];
      cand[n].index = e;
      ++n;
    }
  }
  qsort(cand, (size_t)n, sizeof(oracle_item), oracle_item_desc);
  for (int k = 0; k < K; ++k) ids[k] = cand[k].index;
  free(cand);
  return ORACLE_OK;
}

/* R6: renormalised routing weights of one row. */
void oracle_weights_row(const float* s, const int32_t* ids, int K, float routed_scale,
                        float* w) {
  float sum = 0.0f;
  for (int k = 0; k < K; ++k) sum = sum + s[ids[k]];
  for (int k = 0; k < K; ++k) {
    float q = s[ids[k]] / sum;
    w[k] = q * routed_scale;
  }
}

/* ------------------------------------------------------------------ whole steps */

/* Route step for all tokens: topk_ids [T,K] and topk_weights [T,K]. */
int oracle_route(const uint16_t* logits, const float* bias, int T, int E, int G, int Kg,
                 int K, float routed_scale, int32_t* topk_ids, float* topk_weights) {
  if (!oracle_route_args_ok(T, E, G, Kg, K)) return ORACLE_ERR_ARGS;
  float* s = (float*)malloc(sizeof(float) * (size_t)E);
  float* key = (float*)malloc(sizeof(float) * (size_t)E);
  float* gs = (float*)malloc(sizeof(float) * (size_t)G);
  int32_t* kept = (int32_t*)malloc(sizeof(int32_t) * (size_t)G);
  int rc = ORACLE_OK;
  if (!s || !key || !gs || !kept) {
    rc = ORACLE_ERR_NOMEM;
    goto done;
  }
  for (int t = 0; t < T; ++t) {
    oracle_scores_row(logits + (size_t)t * E, bias, E, s, key);
    rc = oracle_group_scores_row(key, E, G, gs);
    if (rc) goto done;
    rc = oracle_kept_groups_row(gs, G, Kg, kept);
    if (rc) goto done;
    rc = oracle_topk_row(key, E, G, kept, K, topk_ids + (size_t)t * K);
    if (rc) goto done;
    oracle_weights_row(s, topk_ids + (size_t)t * K, K, routed_scale,
                       topk_weights + (size_t)t * K);
  }
done:
  free(s);
  free(key);
  free(gs);
  free(kept);
  return rc;
}

/* Worst-case padded length: every nonempty expert pads by at most B-1 rows, and at most
 * min(E, N) experts are nonempty. */
int64_t oracle_max_padded(int T, int E, int K, int B) {
  int64_t N = (int64_t)T * K;
  int64_t nz = N < E ? N : E;
  return N + nz * (B - 1);
}

/* Sort step (R7, R8).  Outputs are written on [0, npp) and expert_ids on [0, npp/B);
 * nothing past those is touched.  *flags gets ORACLE_FLAG_BAD_EXPERT_ID when an id >= E
 * was seen. */
int oracle_sort(const int32_t* topk_ids, const float* topk_weights, int T, int E, int K,
                int B, int32_t* sorted_token_ids, float* sorted_weights,
                int32_t* expert_ids, int32_t* num_tokens_post_pad, int32_t* flags) {
  if (T < 0 || E < 1 || K < 1 || B < 1) return ORACLE_ERR_ARGS;
  int64_t N = (int64_t)T * K;
  int64_t* cnt = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  int64_t* pad = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  int64_t* off = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  if (!cnt || !pad || !off || !fill) {
    free(cnt);
    free(pad);
    free(off);
    free(fill);
    return ORACLE_ERR_NOMEM;
  }
  int32_t bad = 0;
  /* phase 1: histogram */
  for (int64_t r = 0; r < N; ++r) {
    int32_t e = topk_ids[r];
    if (e < 0) continue;
    if (e >= E) {
      bad = 1;
      continue;
    }
    cnt[e] += 1;
  }
  /* phase 2a: padded exclusive prefix sum */
  int64_t total = 0;
  for (int e = 0; e < E; ++e) {
    pad[e] = ((cnt[e] + B - 1) / B) * B;
    off[e] = total;
    total += pad[e];
  }
  /* phase 2b: stable placement in flat (token, slot) order */
  for (int64_t r = 0; r < N; ++r) {
    int32_t e = topk_ids[r];
    if (e < 0 || e >= E) continue;
    int64_t pos = off[e] + fill[e];
    fill[e] += 1;
    sorted_token_ids[pos] = (int32_t)r;
    sorted_weights[pos] = topk_weights[r];
  }
  /* padding rows and block owners */
  for (int e = 0; e < E; ++e) {
    for (int64_t p = off[e] + cnt[e]; p < off[e] + pad[e]; ++p) {
      sorted_token_ids[p] = (int32_t)N;
      sorted_weights[p] = 0.0f;
    }
    for (int64_t b = off[e] / B; b < (off[e] + pad[e]) / B; ++b) expert_ids[b] = e;
  }
  *num_tokens_post_pad = (int32_t)total;
  if (flags) *flags = bad ? ORACLE_FLAG_BAD_EXPERT_ID : 0;
  free(cnt);
  free(pad);
  free(off);
  free(fill);
  return ORACLE_OK;
}

/* R13: route step of the softmax variant for all tokens: topk_ids [T,K], topk_weights [T,K].
 * Selection is a full sort of the row's logits on (x desc, index asc). */
int oracle_route_softmax(const uint16_t* logits, int T, int E, int K, float routed_scale,
                         int32_t* topk_ids, float* topk_weights) {
  if (T < 0 || E < 1 || K < 1 || K > E) return ORACLE_ERR_ARGS;
  float* x = (float*)malloc(sizeof(float) * (size_t)E);
  int32_t kept_all = 1;
  int rc = ORACLE_OK;
  if (!x) return ORACLE_ERR_NOMEM;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) x[e] = oracle_bf16_to_float(logits[(size_t)t * E + e]);
    int32_t* ids = topk_ids + (size_t)t * K;
    rc = oracle_topk_row(x, E, 1, &kept_all, K, ids);
    if (rc) break;
    float m = x[ids[0]];
    float sum = 0.0f;
    for (int k = 0; k < K; ++k) sum = sum + expf(x[ids[k]] - m);
    for (int k = 0; k < K; ++k) {
      float q = expf(x[ids[k]] - m) / sum;
      topk_weights[(size_t)t * K + k] = q * routed_scale;
    }
  }
  free(x);
  return rc;
}

/* The softmax variant's whole path: route step (R13) then the sort step. */
int oracle_route_sort_softmax(const uint16_t* logits, int T, int E, int K, float routed_scale,
                              int B, int32_t* topk_ids, float* topk_weights,
                              int32_t* sorted_token_ids, float* sorted_weights,
                              int32_t* expert_ids, int32_t* num_tokens_post_pad) {
  int rc = oracle_route_softmax(logits, T, E, K, routed_scale, topk_ids, topk_weights);
  if (rc) return rc;
  int32_t flags = 0;
  return oracle_sort(topk_ids, topk_weights, T, E, K, B, sorted_token_ids, sorted_weights,
                     expert_ids, num_tokens_post_pad, &flags);
}

/* ------------------------------------------------------------ gate projection */

/* R14, exactly: the dot product of a bf16 row pair as an exact integer.  A finite bf16 value is
 * m * 2^q with an integer |m| < 2^8 and q >= -133, so a product of two is m * 2^q with
 * |m| < 2^16 and q >= -266; scaled by 2^266 every product, and so the exact sum, is an
 * integer.  The sum is held in 32-bit limbs (kept in int64, carries settled at the end): bit
 * positions up to 266 + 240 + 16 plus 13 bits of headroom for H <= 8192 need 17 limbs. */
#define ORACLE_ACC_LIMBS 18
#define ORACLE_ACC_SHIFT 266

typedef struct {
  int64_t limb[ORACLE_ACC_LIMBS];
} oracle_acc;

/* Integer significand and exponent of a finite bf16 value: v = m * 2^q. */
static void oracle_bf16_split(uint16_t bits, int32_t* m, int* q) {
  int32_t mag = (int32_t)(bits & 0x7fu);
  int ex = (int)((bits >> 7) & 0xffu);
  if (ex == 0) {
    *q = -133; /* subnormal: 0.mag * 2^-126 = mag * 2^-133 */
  } else {
    mag |= 0x80; /* hidden bit: 1.mag * 2^(ex-127) = (128 + mag) * 2^(ex-134) */
    *q = ex - 134;
  }
  *m = (bits & 0x8000u) ? -mag : mag;
}

static void oracle_acc_add_product(oracle_acc* acc, uint16_t a, uint16_t b) {
  int32_t ma, mb;
  int qa, qb;
  oracle_bf16_split(a, &ma, &qa);
  oracle_bf16_split(b, &mb, &qb);
  int64_t m = (int64_t)ma * (int64_t)mb; /* |m| < 2^16 */
  if (m == 0) return;
  int pos = qa + qb + ORACLE_ACC_SHIFT; /* >= 0 */
  acc->limb[pos / 32] += m * ((int64_t)1 << (pos % 32)); /* |term| < 2^47 */
}

/* The bf16 nearest (ties to even) to the accumulated exact value; +0 for an exact zero. */
static uint16_t oracle_acc_to_bf16(const oracle_acc* acc) {
  /* settle the carries: limbs 0..n-2 in [0, 2^32), the top limb signed */
  int64_t l[ORACLE_ACC_LIMBS];
  memcpy(l, acc->limb, sizeof l);
  for (int i = 0; i + 1 < ORACLE_ACC_LIMBS; ++i) {
    int64_t carry = l[i] >> 32; /* floor division by 2^32 (arithmetic shift) */
    l[i] -= carry * ((int64_t)1 << 32);
    l[i + 1] += carry;
  }
  uint16_t sign = 0;
  if (l[ORACLE_ACC_LIMBS - 1] < 0) { /* negate: two's complement over the limbs */
    sign = 0x8000u;
    int64_t borrow = 0;
    for (int i = 0; i < ORACLE_ACC_LIMBS; ++i) {
      int64_t v = -l[i] - borrow;
      borrow = 0;
      if (i + 1 < ORACLE_ACC_LIMBS && v < 0) {
        v += (int64_t)1 << 32;
        borrow = 1;
      }
      l[i] = v;
    }
  }
  int top = -1; /* highest set bit of the magnitude N */
  for (int i = ORACLE_ACC_LIMBS - 1; i >= 0 && top < 0; --i)
    if (l[i] != 0)
      for (int b = 31; b >= 0; --b)
        if ((l[i] >> b) & 1) {
          top = 32 * i + b;
          break;
        }
  if (top < 0) return 0x0000; /* exact zero */
  /* keep 8 significant bits, but never below bf16's last subnormal bit (2^-133) */
  int lsb = top - 7;
  if (lsb < ORACLE_ACC_SHIFT - 133) lsb = ORACLE_ACC_SHIFT - 133;
  int64_t mant = 0;
  for (int p = top; p >= lsb; --p) mant = 2 * mant + ((l[p / 32] >> (p % 32)) & 1);
  /* remainder below lsb against half of the lsb weight */
  int half = (lsb >= 1) ? ((l[(lsb - 1) / 32] >> ((lsb - 1) % 32)) & 1) : 0;
  int rest = 0; /* any set bit below lsb - 1 */
  for (int p = lsb - 2; p >= 0 && !rest; --p) rest = (l[p / 32] >> (p % 32)) & 1;
  if (half && (rest || (mant & 1))) mant += 1;
  /* value = mant * 2^(lsb - 266), at most 9 significant bits (a carry into a power of two) */
  double v = ldexp((double)mant, lsb - ORACLE_ACC_SHIFT);
  float f = (v >= 0x1p128) ? INFINITY : (float)v; /* exact: few significant bits */
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  return (uint16_t)((bits >> 16) | sign);
}

/* R14: logits [T,E] (bf16) of hidden [T,H] (bf16) times gate weights [E,H] (bf16, one row per
 * expert): each entry the exact dot product (as an integer above), rounded once to bf16.
 * Inputs must be finite. */
int oracle_gate_logits(const uint16_t* hidden, const uint16_t* w, int T, int E, int H,
                       uint16_t* logits) {
  if (T < 0 || E < 1 || H < 1 || H > 8192) return ORACLE_ERR_ARGS;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      oracle_acc acc;
      memset(&acc, 0, sizeof acc);
      for (int h = 0; h < H; ++h)
        oracle_acc_add_product(&acc, hidden[(size_t)t * H + h], w[(size_t)e * H + h]);
      logits[(size_t)t * E + e] = oracle_acc_to_bf16(&acc);
    }
  }
  return ORACLE_OK;
}

/* The whole path: route step then sort step. */
int oracle_route_sort(const uint16_t* logits, const float* bias, int T, int E, int G,
                      int Kg, int K, float routed_scale, int B, int32_t* topk_ids,
                      float* topk_weights, int32_t* sorted_token_ids,
                      float* sorted_weights, int32_t* expert_ids,
                      int32_t* num_tokens_post_pad) {
  int rc = oracle_route(logits, bias, T, E, G, Kg, K, routed_scale, topk_ids, topk_weights);
  if (rc) return rc;
  int32_t flags = 0;
  return oracle_sort(topk_ids, topk_weights, T, E, K, B, sorted_token_ids, sorted_weights,
                     expert_ids, num_tokens_post_pad, &flags);
}

/* ------------------------------------------------------------ near-tie margins */

/* Smallest decision gap of each token, used by the test-input generator to redraw tokens
 * whose selection would hinge on one-ulp differences between two correct sigmoid
 * evaluations.  margin[t] = min of
 *   (a) key_(K) - key_(K+1) among the candidates of the kept groups,
 *   (b) gs_(Kg) - gs_(Kg+1) among the groups,
 *   (c) key_(k) - key_(k+1) for adjacent selected slots k = 1..K-1,
 * each term present only when both of its values exist (+inf otherwise). */
int oracle_margins(const uint16_t* logits, const float* bias, int T, int E, int G, int Kg,
                   int K, float* margin) {
  if (!oracle_route_args_ok(T, E, G, Kg, K)) return ORACLE_ERR_ARGS;
  int g = E / G;
  float* s = (float*)malloc(sizeof(float) * (size_t)E);
  float* key = (float*)malloc(sizeof(float) * (size_t)E);
  float* gs = (float*)malloc(sizeof(float) * (size_t)G);
  int32_t* kept = (int32_t*)malloc(sizeof(int32_t) * (size_t)G);
  oracle_item* items = (oracle_item*)malloc(sizeof(oracle_item) * (size_t)E);
  int rc = ORACLE_OK;
  if (!s || !key || !gs || !kept || !items) {
    rc = ORACLE_ERR_NOMEM;
    goto done;
  }
  for (int t = 0; t < T; ++t) {
    float m = INFINITY;
    oracle_scores_row(logits + (size_t)t * E, bias, E, s, key);
    rc = oracle_group_scores_row(key, E, G, gs);
    if (rc) goto done;
    /* (b) */
    for (int j = 0; j < G; ++j) {
      items[j].value = gs[j];
      items[j].index = j;
    }
    qsort(items, (size_t)G, sizeof(oracle_item), oracle_item_desc);
    if (Kg < G) {
      float d = fabsf(items[Kg - 1].value - items[Kg].value);
      if (d < m) m = d;
    }
    rc = oracle_kept_groups_row(gs, G, Kg, kept);
    if (rc) goto done;
    /* (a), (c) */
    int n = 0;
    for (int e = 0; e < E; ++e) {
      if (kept[e / g]) {
        items[n].value = key[e];
        items[n].index = e;
        ++n;
      }
    }
    qsort(items, (size_t)n, sizeof(oracle_item), oracle_item_desc);
    if (K < n) {
      float d = fabsf(items[K - 1].value - items[K].value);
      if (d < m) m = d;
    }
    for (int k = 0; k + 1 < K; ++k) {
      float d = fabsf(items[k].value - items[k + 1].value);
      if (d < m) m = d;
    }
    margin[t] = m;
  }
done:
  free(s);
  free(key);
  free(gs);
  free(kept);
  free(items);
  return rc;
}
