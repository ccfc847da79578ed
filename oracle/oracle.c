/*
 * ORACLE — test infrastructure only.  A plain, slow, fp64 CPU statement of
 * what the routed MoE FFN layer computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it; the CUDA library never
 * does, and this file includes nothing of the library's.
 *
 * What the pages fix, and where:
 *  - An MoE layer runs only a few of its experts per token, chosen by a
 *    router kept on the GPU, plus an always-on shared expert
 *    ("nano-cuda-moe-qwen38" page, memory-hierarchy section; Strata/Project
 *    Maya page, "MoE architecture and hierarchical caching" and "Strata
 *    tiers" sections; "cyber-on-strata" page: 8 of 256 experts per token).
 *  - Every expert is reached through a resident table of cache slots (the
 *    VRAM expert cache of those pages), here sized to hold all experts.
 *  - Block-scaled low-bit storage with one scale per 32 values (the int8 KV
 *    cache paragraph of the "nano-cuda-moe-qwen38" page).
 * The pages give no formulas.  Readings taken where they are silent:
 *  - router logits z = W_r x + b in fp32 weights, computed here in fp64;
 *  - top-k by value, ties to the lower expert id, in descending order;
 *  - routing weights = softmax over the k selected logits (equal to a full
 *    softmax renormalised over the selection; both are implemented);
 *  - expert FFN = SwiGLU: h = silu(W_g x) * (W_u x), y_e = W_d h,
 *    silu(g) = g / (1 + exp(-g));
 *  - weight (n - 8) * scale for the 4-bit code n and its block's binary16
 *    scale; byte i of a row holds element 2i (low nibble), 2i+1 (high);
 *  - layer output y = sum_j w_j y_{e_j} + y_shared, shared weight 1,
 *    rounded to bf16 only at the output;
 *  - routing variants, each off unless its flag is set (the pages give no
 *    routing formulas, so these follow the common MoE conventions):
 *      no renormalisation (1): w_j = softmax over all E logits, read at
 *        the selected experts (the weights sum to less than 1);
 *      bias for selection only (2): the selection ranks z = W_r x + b, the
 *        weights use W_r x without b (over the selection, or over all E
 *        with flag 1);
 *      gated shared expert (4): the shared term is scaled per token by
 *        sigmoid(g . x) for a gate vector g [H];
 *  - stack (pre-norm residual, RMSNorm with unit gain; a plain residual
 *    stack of these layers diverges -- the SwiGLU output grows with the
 *    square of its input): u_l = bf16(h_l / sqrt(mean(h_l^2) + 1e-6)),
 *    h_{l+1} = bf16(h_l + bf16(MoE_l(u_l))).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------ scalars */

/* binary16 bits -> double (exact). */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);
  return sign ? -v : v;
}

/* bfloat16 bits -> double (exact). */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* double -> bfloat16 bits, one rounding to nearest even. */
uint16_t oracle_double_to_bf16(double v) {
  if (v != v) return 0x7fc0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7f80;
  int e;
  frexp(a, &e); /* a = m 2^e, m in [0.5, 1) -> a = 1.f 2^(e-1) */
  int E = e - 1;
  if (E < -126) { /* bf16 subnormal: multiples of 2^-133 */
    double r = rint(ldexp(a, 133));
    return sign | (uint16_t)r; /* r == 128 gives the smallest normal */
  }
  double r = rint(ldexp(a, 7 - E)); /* significand in [128, 256] */
  if (r == 256.0) {
    r = 128.0;
    E += 1;
  }
  if (E > 127) return sign | 0x7f80;
  return sign | (uint16_t)((E + 127) << 7) | (uint16_t)(r - 128.0);
}

void oracle_round_bf16(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_bf16(in[i]);
}

double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------ dequant */

/* One packed row of K weights -> fp64 (exact: a 4-bit integer times a
 * binary16 scale fits in 15 significant bits). */
void oracle_dequant_row(const uint8_t* q, const uint16_t* s, int K, double* w) {
  for (int k = 0; k < K; ++k) {
    uint8_t byte = q[k / 2];
    int nib = (k % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
    w[k] = (double)(nib - 8) * oracle_half_to_double(s[k / 32]);
  }
}

/* y[r] = sum_k W[r][k] x[k] for a packed [rows][K] matrix. */
static void qmatvec(const uint8_t* q, const uint16_t* s, int rows, int K, const double* x,
                    double* y, double* rowbuf) {
  for (int r = 0; r < rows; ++r) {
    oracle_dequant_row(q + (size_t)r * (K / 2), s + (size_t)r * (K / 32), K, rowbuf);
    double acc = 0.0;
    for (int k = 0; k < K; ++k) acc += rowbuf[k] * x[k];
    y[r] = acc;
  }
}

/* ------------------------------------------------------------ routing */

/* z[t][e] = sum_h W[e][h] x[t][h] + b[e]. */
void oracle_router_logits(int T, int H, int E, const float* W, const float* b,
                          const uint16_t* x_bf16, double* z) {
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += (double)W[(size_t)e * H + h] * oracle_bf16_to_double(x_bf16[(size_t)t * H + h]);
      z[(size_t)t * E + e] = acc + (b ? (double)b[e] : 0.0);
    }
}

typedef struct {
  double z;
  int e;
} zid;

static int cmp_zid(const void* a, const void* b) {
  const zid* x = (const zid*)a;
  const zid* y = (const zid*)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->e > y->e) - (x->e < y->e);
}

/* Full sort of the E logits (value descending, id ascending); the first k
 * are the selection.  w = softmax over the selected logits (max subtracted).
 * margin[t] = z_(k) - z_(k+1) (INFINITY when k == E). */
void oracle_topk_softmax(int T, int E, int k, const double* z, int32_t* ids, double* w,
                         double* margin) {
  zid* buf = (zid*)malloc(sizeof(zid) * (size_t)E);
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      buf[e].z = z[(size_t)t * E + e];
      buf[e].e = e;
    }
    qsort(buf, (size_t)E, sizeof(zid), cmp_zid);
    double zmax = buf[0].z, den = 0.0;
    for (int j = 0; j < k; ++j) den += exp(buf[j].z - zmax);
    for (int j = 0; j < k; ++j) {
      ids[(size_t)t * k + j] = buf[j].e;
      if (w) w[(size_t)t * k + j] = exp(buf[j].z - zmax) / den;
    }
    if (margin) margin[t] = (k < E) ? buf[k - 1].z - buf[k].z : INFINITY;
  }
  free(buf);
}

/* Routing weights of a given selection ids [T][k] under the variant flags
 * (1: no renormalisation, 2: bias for selection only).  zsel [T][E] are the
 * selection logits W_r x + b; b [E] (may be NULL = 0) is removed from the
 * weights' logits with flag 2.  Without flag 1: softmax over the k selected
 * weight logits; with it: softmax over all E weight logits, taken at the
 * selection. */
void oracle_route_weights(int T, int E, int k, int flags, const double* zsel, const float* b,
                          const int32_t* ids, double* w) {
  for (int t = 0; t < T; ++t) {
    const double* zt = zsel + (size_t)t * E;
    const int32_t* it = ids + (size_t)t * k;
    double* wt = w + (size_t)t * k;
    const int strip = (flags & 2) && b;
    if (flags & 1) {
      double m = -INFINITY, den = 0.0;
      for (int e = 0; e < E; ++e) {
        double v = zt[e] - (strip ? (double)b[e] : 0.0);
        m = v > m ? v : m;
      }
      for (int e = 0; e < E; ++e) den += exp(zt[e] - (strip ? (double)b[e] : 0.0) - m);
      for (int j = 0; j < k; ++j) wt[j] = exp(zt[it[j]] - (strip ? (double)b[it[j]] : 0.0) - m) / den;
    } else {
      double m = -INFINITY, den = 0.0;
      for (int j = 0; j < k; ++j) {
        double v = zt[it[j]] - (strip ? (double)b[it[j]] : 0.0);
        m = v > m ? v : m;
      }
      for (int j = 0; j < k; ++j) den += exp(zt[it[j]] - (strip ? (double)b[it[j]] : 0.0) - m);
      for (int j = 0; j < k; ++j) wt[j] = exp(zt[it[j]] - (strip ? (double)b[it[j]] : 0.0) - m) / den;
    }
  }
}

/* The other order of the same reading: softmax over all E logits, then the
 * same selection, then renormalise the k selected probabilities. */
void oracle_topk_softmax_full(int T, int E, int k, const double* z, int32_t* ids, double* w) {
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  oracle_topk_softmax(T, E, k, z, ids, NULL, NULL);
  for (int t = 0; t < T; ++t) {
    const double* zt = z + (size_t)t * E;
    double zmax = zt[0], den = 0.0, sel = 0.0;
    for (int e = 1; e < E; ++e) zmax = zt[e] > zmax ? zt[e] : zmax;
    for (int e = 0; e < E; ++e) den += (p[e] = exp(zt[e] - zmax));
    for (int e = 0; e < E; ++e) p[e] /= den;
    for (int j = 0; j < k; ++j) sel += p[ids[(size_t)t * k + j]];
    for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = p[ids[(size_t)t * k + j]] / sel;
  }
  free(p);
}

/* ------------------------------------------------------------ bucketing */

/* Group the T*k (token, j) assignments by expert: counts[E], exclusive
 * offsets[E+1], and the assignments sorted by expert then token then j
 * (a stable counting sort). */
void oracle_bucket(int T, int k, int E, const int32_t* ids, int32_t* counts, int32_t* offsets,
                   int32_t* perm_token, int32_t* perm_j) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int i = 0; i < T * k; ++i) counts[ids[i]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = ids[t * k + j];
      int p = fill[e]++;
      perm_token[p] = t;
      perm_j[p] = j;
    }
  free(fill);
}

/* ------------------------------------------------------------ expert FFN */

/* y[H] = W_d (silu(W_g x) * (W_u x)) for one token; x is fp64 [H]. */
void oracle_expert_ffn(int H, int F, const uint8_t* gq, const uint16_t* gs, const uint8_t* uq,
                       const uint16_t* us, const uint8_t* dq, const uint16_t* ds, const double* x,
                       double* y) {
  int kmax = H > F ? H : F;
  double* g = (double*)malloc(sizeof(double) * (size_t)F);
  double* u = (double*)malloc(sizeof(double) * (size_t)F);
  double* row = (double*)malloc(sizeof(double) * (size_t)kmax);
  qmatvec(gq, gs, F, H, x, g, row);
  qmatvec(uq, us, F, H, x, u, row);
  for (int f = 0; f < F; ++f) g[f] = oracle_silu(g[f]) * u[f];
  qmatvec(dq, ds, H, F, g, y, row);
  free(g);
  free(u);
  free(row);
}

/* One token through the layer, given the selected experts' weights:
 * y = sum_j w[j] FFN(expert j) + sh_w FFN(shared).  Pointer arrays hold the
 * k selected experts' tensors; sh_* may be NULL (no shared expert). */
static void combine_token_w(int H, int F, int Fs, int k, const double* w,
                            const uint8_t* const* gq, const uint16_t* const* gs,
                            const uint8_t* const* uq, const uint16_t* const* us,
                            const uint8_t* const* dq, const uint16_t* const* ds,
                            const uint8_t* sh_gq, const uint16_t* sh_gs, const uint8_t* sh_uq,
                            const uint16_t* sh_us, const uint8_t* sh_dq, const uint16_t* sh_ds,
                            double sh_w, const uint16_t* x_bf16, double* y) {
  double* x = (double*)malloc(sizeof(double) * (size_t)H);
  double* ye = (double*)malloc(sizeof(double) * (size_t)H);
  for (int h = 0; h < H; ++h) {
    x[h] = oracle_bf16_to_double(x_bf16[h]);
    y[h] = 0.0;
  }
  for (int j = 0; j < k; ++j) {
    oracle_expert_ffn(H, F, gq[j], gs[j], uq[j], us[j], dq[j], ds[j], x, ye);
    for (int h = 0; h < H; ++h) y[h] += w[j] * ye[h];
  }
  if (Fs > 0 && sh_gq) {
    oracle_expert_ffn(H, Fs, sh_gq, sh_gs, sh_uq, sh_us, sh_dq, sh_ds, x, ye);
    for (int h = 0; h < H; ++h) y[h] += sh_w * ye[h];
  }
  free(x);
  free(ye);
}

/* The same with the shared expert's weight 1 (the default routing). */
void oracle_combine_token(int H, int F, int Fs, int k, const double* w,
                          const uint8_t* const* gq, const uint16_t* const* gs,
                          const uint8_t* const* uq, const uint16_t* const* us,
                          const uint8_t* const* dq, const uint16_t* const* ds,
                          const uint8_t* sh_gq, const uint16_t* sh_gs, const uint8_t* sh_uq,
                          const uint16_t* sh_us, const uint8_t* sh_dq, const uint16_t* sh_ds,
                          const uint16_t* x_bf16, double* y) {
  combine_token_w(H, F, Fs, k, w, gq, gs, uq, us, dq, ds, sh_gq, sh_gs, sh_uq, sh_us, sh_dq, sh_ds,
                  1.0, x_bf16, y);
}

/* Gate of a gated shared expert for one token: sigmoid(sum_h g[h] x[h]). */
double oracle_shared_gate(int H, const float* g, const uint16_t* x_bf16) {
  double acc = 0.0;
  for (int h = 0; h < H; ++h) acc += (double)g[h] * oracle_bf16_to_double(x_bf16[h]);
  return 1.0 / (1.0 + exp(-acc));
}

/* ------------------------------------------------------------ whole layer */

typedef struct {
  int hidden, n_experts, top_k, ffn, shared_ffn, n_slots;
  const float* router_w;          /* [E][H] */
  const float* router_b;          /* [E] or NULL */
  const int32_t* slot_of_expert;  /* [E] */
  const uint8_t* gate_q;          /* [S][F][H/2] */
  const uint16_t* gate_s;         /* [S][F][H/32] */
  const uint8_t* up_q;
  const uint16_t* up_s;
  const uint8_t* down_q;          /* [S][H][F/2] */
  const uint16_t* down_s;         /* [S][H][F/32] */
  const uint8_t* sh_gate_q;       /* [Fs][H/2] or NULL */
  const uint16_t* sh_gate_s;
  const uint8_t* sh_up_q;
  const uint16_t* sh_up_s;
  const uint8_t* sh_down_q;       /* [H][Fs/2] */
  const uint16_t* sh_down_s;
  int routing_flags;              /* 1 no renormalisation, 2 bias selects only, 4 gated shared */
  const float* sh_gate_w;         /* [H], read with flag 4 */
} oracle_layer;

/* T tokens through one layer.  Outputs: y [T][H] fp64, and optionally the
 * selection ids/w [T][k] and margins [T].  If forced_ids is given, those
 * (logical) ids are used instead of the layer's own top-k, with weights from
 * the softmax over their logits (the tie-adoption rule of the parity tests). */
int oracle_moe_forward(const oracle_layer* L, int T, const uint16_t* x_bf16,
                       const int32_t* forced_ids, double* y, int32_t* ids_out, double* w_out,
                       double* margin_out) {
  const int H = L->hidden, E = L->n_experts, k = L->top_k, F = L->ffn, Fs = L->shared_ffn;
  if (k < 1 || k > E || H % 32 || F % 32 || (Fs % 32)) return -1;
  double* z = (double*)malloc(sizeof(double) * (size_t)T * E);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
  double* margin = (double*)malloc(sizeof(double) * (size_t)T);
  const int flags = L->routing_flags;
  if ((flags & ~7) || ((flags & 4) && (Fs == 0 || !L->sh_gate_w))) {
    free(z); free(ids); free(w); free(margin);
    return -1;
  }
  oracle_router_logits(T, H, E, L->router_w, L->router_b, x_bf16, z);
  oracle_topk_softmax(T, E, k, z, ids, w, margin);
  if (forced_ids) {
    for (int i = 0; i < T * k; ++i) {
      if (forced_ids[i] < 0 || forced_ids[i] >= E) {
        free(z); free(ids); free(w); free(margin);
        return -2;
      }
      ids[i] = forced_ids[i];
    }
  }
  /* the default weights (softmax over the selection) came with the top-k;
     the variants and forced selections recompute them */
  if (flags || forced_ids) oracle_route_weights(T, E, k, flags, z, L->router_b, ids, w);
  const size_t gsz = (size_t)F * (H / 2), gss = (size_t)F * (H / 32);
  const size_t dsz = (size_t)H * (F / 2), dss = (size_t)H * (F / 32);
  const uint8_t** pg = (const uint8_t**)malloc(sizeof(void*) * k);
  const uint16_t** pgs = (const uint16_t**)malloc(sizeof(void*) * k);
  const uint8_t** pu = (const uint8_t**)malloc(sizeof(void*) * k);
  const uint16_t** pus = (const uint16_t**)malloc(sizeof(void*) * k);
  const uint8_t** pd = (const uint8_t**)malloc(sizeof(void*) * k);
  const uint16_t** pds = (const uint16_t**)malloc(sizeof(void*) * k);
  int rc = 0;
  for (int t = 0; t < T && rc == 0; ++t) {
    for (int j = 0; j < k; ++j) {
      int slot = L->slot_of_expert[ids[t * k + j]];
      if (slot < 0 || slot >= L->n_slots) {
        rc = -3;
        break;
      }
      pg[j] = L->gate_q + slot * gsz;
      pgs[j] = L->gate_s + slot * gss;
      pu[j] = L->up_q + slot * gsz;
      pus[j] = L->up_s + slot * gss;
      pd[j] = L->down_q + slot * dsz;
      pds[j] = L->down_s + slot * dss;
    }
    if (rc) break;
    const double sh_w = (flags & 4) ? oracle_shared_gate(H, L->sh_gate_w, x_bf16 + (size_t)t * H) : 1.0;
    combine_token_w(H, F, Fs, k, w + (size_t)t * k, pg, pgs, pu, pus, pd, pds, L->sh_gate_q,
                    L->sh_gate_s, L->sh_up_q, L->sh_up_s, L->sh_down_q, L->sh_down_s, sh_w,
                    x_bf16 + (size_t)t * H, y + (size_t)t * H);
  }
  if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)T * k);
  if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)T * k);
  if (margin_out) memcpy(margin_out, margin, sizeof(double) * (size_t)T);
  free(pg); free(pgs); free(pu); free(pus); free(pd); free(pds);
  free(z); free(ids); free(w); free(margin);
  return rc;
}

/* Residual step of the stack: h_next = bf16(h + bf16(y)). */
void oracle_residual(const uint16_t* h_bf16, const double* y, uint16_t* h_next, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    double yb = oracle_bf16_to_double(oracle_double_to_bf16(y[i]));
    h_next[i] = oracle_double_to_bf16(oracle_bf16_to_double(h_bf16[i]) + yb);
  }
}

/* RMS normalisation with unit gain, per row of H: one rounding to bf16 of
 * h / sqrt(mean(h^2) + eps). */
void oracle_rmsnorm(const uint16_t* h_bf16, int T, int H, double eps, uint16_t* out) {
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int i = 0; i < H; ++i) {
      double v = oracle_bf16_to_double(h_bf16[(size_t)t * H + i]);
      ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / H + eps);
    for (int i = 0; i < H; ++i)
      out[(size_t)t * H + i] = oracle_double_to_bf16(oracle_bf16_to_double(h_bf16[(size_t)t * H + i]) * inv);
  }
}

/* L layers of the pre-norm residual stack: h_0 = x, u_l = rmsnorm(h_l),
 * h_{l+1} = bf16(h_l + bf16(MoE_l(u_l))).  Writes h_L to out; h_trace
 * (optional) receives h_1..h_L [L][T][H], ids_trace the selections. */
int oracle_stack_forward(const oracle_layer* layers, int n_layers, int T, const uint16_t* x_bf16,
                         uint16_t* out, uint16_t* h_trace, int32_t* ids_trace) {
  const int H = layers[0].hidden;
  const size_t n = (size_t)T * H;
  uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * n);
  uint16_t* u = (uint16_t*)malloc(sizeof(uint16_t) * n);
  double* y = (double*)malloc(sizeof(double) * n);
  memcpy(h, x_bf16, sizeof(uint16_t) * n);
  int rc = 0;
  for (int l = 0; l < n_layers && rc == 0; ++l) {
    int32_t* ids = ids_trace ? ids_trace + (size_t)l * T * layers[l].top_k : NULL;
    oracle_rmsnorm(h, T, H, 1e-6, u);
    rc = oracle_moe_forward(&layers[l], T, u, NULL, y, ids, NULL, NULL);
    oracle_residual(h, y, h, (int64_t)n);
    if (h_trace) memcpy(h_trace + (size_t)l * n, h, sizeof(uint16_t) * n);
  }
  memcpy(out, h, sizeof(uint16_t) * n);
  free(h);
  free(u);
  free(y);
  return rc;
}
