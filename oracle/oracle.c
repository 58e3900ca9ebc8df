/*
 * oracle.c -- plain, slow CPU reference of the FSDP / ZeRO-3 sharded-state step.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  The product path (the CUDA library and
 * its Python binding) never links, imports or calls it, and this file includes no
 * header of the product.
 *
 * Sources (the pages this restates; no code is taken from them):
 *   [FSDP-ch18]  "第18章 FSDP：ZeRO 风格的参数分片", yangyitao.com PyTorch book,
 *                §18.2 (strategies), §18.3 (unshard/reshard), §18.6 (mixed precision),
 *                §18.12 (FlatParameter), §18.14 (Shard(0) local shape), §18.21 (SHARD_GRAD_OP).
 *   [ZeRO-state] "NCCL ZeRO/FSDP state sharding", blog.cptz.space: sections
 *                "Canonical ZeRO 状态公式", "ZeRO-2 方向：Gradient Sharding",
 *                "ZeRO-3 方向：Parameter Sharding", "FlatParameter 与 Padding",
 *                "Optimizer Step 的所有权", "全模式性能结果与限制".
 *   [FSDP2-doc]  "PyTorch FSDP2 后端特性介绍" (MindSpeed-LLM), sections "DTensor", "混合精度".
 *   [titan]      gsyq.cn torchtitan FSDP2 article, §2.3 (dim-0 shards, 12 B/param state).
 *
 * Arithmetic: fp32 where the pages fix it (reduce_dtype=float32, fp32 master and
 * moments; [FSDP-ch18] §18.6, [FSDP2-doc] "混合精度"), bf16 for the low-precision
 * parameter copy.  Compile with -ffp-contract=off and no fast-math: every float
 * operation below is one IEEE-754 binary32 operation rounded to nearest-even, and
 * fmaf() is the correctly rounded fused multiply-add.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - reduce op is the MEAN over ranks (sum in rank order 0..N-1, then one IEEE
 *     division by N): the sharded result must equal DDP, whose gradient is the
 *     global average ([ZeRO-state] "全模式性能结果与限制", [FSDP-ch18] §18.18).
 *   - AdamW is the published decoupled-weight-decay Adam with bias correction,
 *     eps outside the square root; the operation order in adamw_elem() is the
 *     contract.
 *   - DIM0 placement for d0 % N != 0: c = ceil(d0/N) rows per rank slot, rank r
 *     owns rows [min(rc,d0), min((r+1)c,d0)), the rest of its slot is zero padding.
 *     The pages show only divisible examples; this reading is pinned by torch's
 *     own fully_shard on gloo (tests), not by the pages.
 *
 * Parity pins (tests/): page worked examples and closed forms, brute-force layout
 * enumeration, torch FSDP1/FSDP2 on gloo, torch.optim.AdamW (band), the DDP
 * equivalence of the sharded step, the exact fp64 value of single elements.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_FLAT 0
#define OR_DIM0 1
#define OR_F32 0
#define OR_BF16 1

/* ------------------------------------------------------------------------- */
/* Layout                                                                     */
/* ------------------------------------------------------------------------- */

typedef struct {
    int32_t mode, N, T, U;
    int64_t P;          /* logical elements (sum of tensor numels)                  */
    int64_t S;          /* per-rank shard elements (sum over units)                 */
    int64_t F;          /* elements of the full (unsharded) layout                  */
    int64_t *numel, *d0, *inner, *rows, *slot, *t_shard_off, *t_full_off, *t_unit_off;
    int32_t *unit;
    int64_t *u_numel, *u_S, *u_shard_off, *u_full_off;
} olayout;

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static void ol_free(olayout* L) {
    free(L->numel); free(L->d0); free(L->inner); free(L->rows); free(L->slot);
    free(L->t_shard_off); free(L->t_full_off); free(L->t_unit_off); free(L->unit);
    free(L->u_numel); free(L->u_S); free(L->u_shard_off); free(L->u_full_off);
}

/* Builds the layout.  Returns 0, or -1 on an invalid description.
 * FLAT: the tensors of one unit are flattened and concatenated into one flat
 *   parameter of P_u elements, padded at the end to N*ceil(P_u/N); rank r owns
 *   flat positions [r*S_u, (r+1)*S_u) ([FSDP-ch18] §18.12; [ZeRO-state]
 *   "FlatParameter 与 Padding": P_physical = N*ceil(P_logical/N), and the
 *   gathered buffer holds shard numel * world size elements).  The full layout of
 *   a unit is that padded flat parameter, so F = N*S.
 * DIM0: every tensor is split along dim 0 ([FSDP2-doc] "DTensor": [4096,4096] on
 *   8 ranks -> [512,4096]; [titan] §2.3: (C_out, C_in) -> (C_out/N, C_in)); each
 *   rank's slot holds c = ceil(d0/N) rows; the full layout is the plain
 *   concatenation of the tensors, F = P.  A 0-d tensor counts as [1]. */
static int ol_build(olayout* L, int32_t T, const int32_t* ndim, const int64_t* dims,
                    const int32_t* unit_id, int32_t N, int32_t mode) {
    memset(L, 0, sizeof *L);
    if (T < 1 || N < 1 || (mode != OR_FLAT && mode != OR_DIM0)) return -1;
    if (unit_id[0] != 0) return -1;
    for (int32_t t = 1; t < T; ++t)
        if (unit_id[t] != unit_id[t - 1] && unit_id[t] != unit_id[t - 1] + 1) return -1;
    L->mode = mode; L->N = N; L->T = T; L->U = unit_id[T - 1] + 1;
    L->numel = calloc(T, 8); L->d0 = calloc(T, 8); L->inner = calloc(T, 8);
    L->rows = calloc(T, 8); L->slot = calloc(T, 8); L->t_shard_off = calloc(T, 8);
    L->t_full_off = calloc(T, 8); L->t_unit_off = calloc(T, 8); L->unit = calloc(T, 4);
    L->u_numel = calloc(L->U, 8); L->u_S = calloc(L->U, 8);
    L->u_shard_off = calloc(L->U, 8); L->u_full_off = calloc(L->U, 8);

    int64_t dpos = 0;
    for (int32_t t = 0; t < T; ++t) {
        if (ndim[t] < 0) { ol_free(L); return -1; }
        int64_t n = 1;
        for (int32_t k = 0; k < ndim[t]; ++k) {
            if (dims[dpos + k] < 0) { ol_free(L); return -1; }
            n *= dims[dpos + k];
        }
        L->numel[t] = n;
        L->d0[t] = ndim[t] == 0 ? 1 : dims[dpos];
        L->inner[t] = L->d0[t] == 0 ? 0 : n / L->d0[t];
        if (L->d0[t] == 0) {           /* [0, a, b]: inner is the product of the rest */
            int64_t in = 1;
            for (int32_t k = 1; k < ndim[t]; ++k) in *= dims[dpos + k];
            L->inner[t] = in;
        }
        L->unit[t] = unit_id[t];
        dpos += ndim[t];
    }

    int64_t P = 0;
    for (int32_t t = 0; t < T; ++t) {
        int32_t u = L->unit[t];
        L->t_unit_off[t] = L->u_numel[u];       /* offset of the tensor inside its unit */
        L->u_numel[u] += L->numel[t];
        P += L->numel[t];
    }
    L->P = P;

    if (mode == OR_FLAT) {
        int64_t so = 0, fo = 0;
        for (int32_t u = 0; u < L->U; ++u) {
            L->u_S[u] = ceil_div(L->u_numel[u], N);
            L->u_shard_off[u] = so; L->u_full_off[u] = fo;
            so += L->u_S[u]; fo += (int64_t)N * L->u_S[u];
        }
        L->S = so; L->F = fo;
        for (int32_t t = 0; t < T; ++t) {
            L->t_full_off[t] = L->u_full_off[L->unit[t]] + L->t_unit_off[t];
            L->t_shard_off[t] = -1;       /* depends on the rank in FLAT mode */
            L->rows[t] = 0; L->slot[t] = 0;
        }
    } else {
        int64_t so = 0, fo = 0;
        for (int32_t t = 0; t < T; ++t) {
            L->rows[t] = ceil_div(L->d0[t], N);
            L->slot[t] = L->rows[t] * L->inner[t];
            L->t_shard_off[t] = so; L->t_full_off[t] = fo;
            so += L->slot[t]; fo += L->numel[t];
        }
        L->S = so; L->F = fo;
        for (int32_t u = 0; u < L->U; ++u) L->u_S[u] = 0;
        for (int32_t t = 0; t < T; ++t) {
            int32_t u = L->unit[t];
            if (t == 0 || L->unit[t - 1] != u) {      /* first tensor of unit u */
                L->u_shard_off[u] = L->t_shard_off[t];
                L->u_full_off[u] = L->t_full_off[t];
            }
            L->u_S[u] += L->slot[t];
        }
    }
    return 0;
}

/* Where shard element j of rank r lives in the full layout.
 * Returns the full index, or -1 when (r, j) is padding (no logical element).
 * For FLAT, *flatpos receives the position in the unit's padded flat parameter
 * (valid for padding too), so that the all-gather can copy padding verbatim. */
static int64_t ol_full_index(const olayout* L, int32_t r, int64_t j, int64_t* flatpos) {
    int32_t u = -1;
    for (int32_t w = 0; w < L->U; ++w)
        if (j >= L->u_shard_off[w] && j < L->u_shard_off[w] + L->u_S[w]) { u = w; break; }
    if (u < 0) { if (flatpos) *flatpos = -1; return -1; }
    int64_t k = j - L->u_shard_off[u];
    if (L->mode == OR_FLAT) {
        int64_t q = (int64_t)r * L->u_S[u] + k;
        if (flatpos) *flatpos = L->u_full_off[u] + q;
        return q < L->u_numel[u] ? L->u_full_off[u] + q : -1;
    }
    if (flatpos) *flatpos = -1;
    for (int32_t t = 0; t < L->T; ++t) {
        if (L->unit[t] != u) continue;
        if (j >= L->t_shard_off[t] && j < L->t_shard_off[t] + L->slot[t]) {
            int64_t kk = j - L->t_shard_off[t];
            int64_t row_in_slot = kk / L->inner[t];
            int64_t col = kk % L->inner[t];
            int64_t row = (int64_t)r * L->rows[t] + row_in_slot;
            if (row >= L->d0[t]) return -1;
            return L->t_full_off[t] + row * L->inner[t] + col;
        }
    }
    return -1;
}

/* ------------------------------------------------------------------------- */
/* Scalar helpers                                                             */
/* ------------------------------------------------------------------------- */

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* fp32 -> bf16, round to nearest, ties to even, on the binary32 bit pattern.
 * NaN becomes a quiet NaN with the sign and the top payload bits kept. */
uint16_t oracle_bf16_rne(float x) {
    uint32_t u = f2u(x);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

float oracle_bf16_to_f32(uint16_t h) { return u2f((uint32_t)h << 16); }

void oracle_bf16_rne_array(int64_t n, const float* x, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(x[i]);
}

static float load_grad(const void* g, int32_t dtype, int64_t i) {
    if (dtype == OR_F32) return ((const float*)g)[i];
    return oracle_bf16_to_f32(((const uint16_t*)g)[i]);
}

/* ------------------------------------------------------------------------- */
/* AdamW                                                                      */
/* ------------------------------------------------------------------------- */

typedef struct { float decay, om1, om2, step_size, bc2s, beta1, beta2, eps; } oscal;

/* Per-step scalars, each formed in double from the fp32 hyper-parameters and
 * rounded to fp32 once: decay = 1 - lr*wd, om1 = 1 - beta1, om2 = 1 - beta2,
 * step_size = lr / (1 - beta1^t), bc2s = sqrt(1 - beta2^t). */
static oscal scalars(float lr, float b1, float b2, float eps, float wd, int64_t t) {
    oscal s;
    double bc1 = 1.0 - pow((double)b1, (double)t);
    double bc2 = 1.0 - pow((double)b2, (double)t);
    s.decay = (float)(1.0 - (double)lr * (double)wd);
    s.om1 = (float)(1.0 - (double)b1);
    s.om2 = (float)(1.0 - (double)b2);
    s.step_size = (float)((double)lr / bc1);
    s.bc2s = (float)sqrt(bc2);
    s.beta1 = b1; s.beta2 = b2; s.eps = eps;
    return s;
}

/* One AdamW update of one element with the averaged gradient g (decoupled
 * weight decay, Adam moments, bias correction).  Operation order is the
 * contract: p *= decay; m = fma(b1, m, om1*g); v = fma(b2, v, (om2*g)*g);
 * den = sqrt(v)/bc2s + eps; p = fma(-step_size, m/den, p). */
static void adamw_elem(const oscal* s, float g, float* p, float* m, float* v) {
    float pp = *p * s->decay;
    float mm = fmaf(s->beta1, *m, s->om1 * g);
    float gg = s->om2 * g;
    float vv = fmaf(s->beta2, *v, gg * g);
    float den = sqrtf(vv) / s->bc2s + s->eps;
    float upd = mm / den;
    pp = fmaf(-s->step_size, upd, pp);
    *p = pp; *m = mm; *v = vv;
}

/* Reduce-scatter of one element: fp32 sum over the N replicas in rank order,
 * then the mean by one division ([ZeRO-state] "ZeRO-2 方向": reduce the matching
 * chunks across ranks, each rank keeps its chunk; fp32 reduce_dtype). */
static float reduce_mean(const void* const* grads, int32_t dtype, int32_t N, int64_t i) {
    float acc = 0.0f;
    for (int32_t q = 0; q < N; ++q) acc = acc + load_grad(grads[q], dtype, i);
    return acc / (float)N;
}

/* ------------------------------------------------------------------------- */
/* Exported entry points                                                      */
/* ------------------------------------------------------------------------- */

/* Layout description.  scal[0..4] = P, S, F, U, N.
 * Per tensor (T entries): t_full_off, t_shard_off (-1 in FLAT), t_rows (c, DIM0),
 * t_slot (c*inner, DIM0).  Per unit (U entries, arrays sized >= T): u_S,
 * u_shard_off, u_full_off, u_numel. */
int oracle_layout(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                  int32_t N, int32_t mode, int64_t* scal,
                  int64_t* t_full_off, int64_t* t_shard_off, int64_t* t_rows, int64_t* t_slot,
                  int64_t* u_S, int64_t* u_shard_off, int64_t* u_full_off, int64_t* u_numel) {
    olayout L;
    if (ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    scal[0] = L.P; scal[1] = L.S; scal[2] = L.F; scal[3] = L.U; scal[4] = L.N;
    for (int32_t t = 0; t < T; ++t) {
        t_full_off[t] = L.t_full_off[t]; t_shard_off[t] = L.t_shard_off[t];
        t_rows[t] = L.rows[t]; t_slot[t] = L.slot[t];
    }
    for (int32_t u = 0; u < L.U; ++u) {
        u_S[u] = L.u_S[u]; u_shard_off[u] = L.u_shard_off[u];
        u_full_off[u] = L.u_full_off[u]; u_numel[u] = L.u_numel[u];
    }
    ol_free(&L);
    return 0;
}

/* Full index of (rank, shard element j) for many j at once; -1 = padding. */
int oracle_full_index(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                      int32_t N, int32_t mode, int32_t rank, int64_t n, const int64_t* j,
                      int64_t* out) {
    olayout L;
    if (ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = ol_full_index(&L, rank, j[i], NULL);
    ol_free(&L);
    return 0;
}

/* Initial sharding / summon_full_params(writeback): full -> rank shards.
 * master: [N][stride] fp32 (or NULL); param: [N][stride] bf16 (or NULL).
 * Every element of every row is written: data, padding (+0) and the row tail
 * [S, stride) (+0).  full_dtype is OR_F32 or OR_BF16.  ([FSDP-ch18] §18.17
 * writeback; [ZeRO-state] "FlatParameter 与 Padding".) */
int oracle_reshard(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                   int32_t N, int32_t mode, const void* full, int32_t full_dtype, int64_t stride,
                   float* master, uint16_t* param) {
    olayout L;
    if (ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    if (stride < L.S) { ol_free(&L); return -1; }
    for (int32_t r = 0; r < N; ++r) {
        for (int64_t j = 0; j < stride; ++j) {
            float x = 0.0f;
            if (j < L.S) {
                int64_t fi = ol_full_index(&L, r, j, NULL);
                if (fi >= 0) x = load_grad(full, full_dtype, fi);
            }
            if (master) master[(int64_t)r * stride + j] = x;
            if (param) param[(int64_t)r * stride + j] = oracle_bf16_rne(x);
        }
    }
    ol_free(&L);
    return 0;
}

/* Unshard (all-gather) of units [ub, ue): rank shards -> full buffer.
 * FLAT: all_gather_into_tensor of the padded flat parameter -- every shard
 * element, padding included, lands at u_full_off + r*S_u + k ([ZeRO-state]
 * "ZeRO-3 方向：Parameter Sharding").  DIM0: copy-out of the owned rows only
 * ([FSDP-ch18] §18.8: copy-in, one all-gather, copy-out).
 * elem_bytes is 2 (bf16) or 4 (fp32): the copy is bitwise. */
int oracle_unshard(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                   int32_t N, int32_t mode, int32_t ub, int32_t ue, const void* shards,
                   int32_t elem_bytes, int64_t stride, void* full) {
    olayout L;
    if (ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    if (ub < 0 || ue > L.U || ub > ue || stride < L.S) { ol_free(&L); return -1; }
    const char* src = (const char*)shards;
    char* dst = (char*)full;
    for (int32_t u = ub; u < ue; ++u) {
        for (int32_t r = 0; r < N; ++r) {
            for (int64_t k = 0; k < L.u_S[u]; ++k) {
                int64_t j = L.u_shard_off[u] + k;
                int64_t flatpos;
                int64_t fi = ol_full_index(&L, r, j, &flatpos);
                int64_t dst_i = L.mode == OR_FLAT ? flatpos : fi;
                if (dst_i < 0) continue;
                memcpy(dst + dst_i * elem_bytes, src + ((int64_t)r * stride + j) * elem_bytes,
                       (size_t)elem_bytes);
            }
        }
    }
    ol_free(&L);
    return 0;
}

/* Fused reduce-scatter + AdamW + bf16 recast for units [ub, ue), in the pages'
 * order: (1) reduce-scatter: each rank's shard element gets the mean of the N
 * replicas' gradients at its full index (padding: g = 0, as the zero-padded
 * gradient of [ZeRO-state] "ZeRO-2 方向"); (2) AdamW on that rank's fp32
 * master/exp_avg/exp_avg_sq shard ([ZeRO-state] "Optimizer Step 的所有权");
 * (3) if param != NULL, the bf16 copy of the updated master ([FSDP-ch18] §18.6).
 * grads: N pointers, each a full-layout buffer (F elements) of grad_dtype.
 * grad_out (optional): the fp32 reduced gradient shard.  step is 1-based. */
int oracle_rs_adamw(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                    int32_t N, int32_t mode, int32_t ub, int32_t ue,
                    const void* const* grads, int32_t grad_dtype, int64_t stride,
                    float* master, float* m, float* v, uint16_t* param, float* grad_out,
                    float lr, float beta1, float beta2, float eps, float wd, int64_t step) {
    olayout L;
    if (ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    if (ub < 0 || ue > L.U || ub > ue || stride < L.S || step < 1) { ol_free(&L); return -1; }
    oscal s = scalars(lr, beta1, beta2, eps, wd, step);
    for (int32_t u = ub; u < ue; ++u) {
        for (int32_t r = 0; r < N; ++r) {
            for (int64_t k = 0; k < L.u_S[u]; ++k) {
                int64_t j = L.u_shard_off[u] + k;
                int64_t fi = ol_full_index(&L, r, j, NULL);
                float g = fi >= 0 ? reduce_mean(grads, grad_dtype, N, fi) : 0.0f;
                int64_t e = (int64_t)r * stride + j;
                adamw_elem(&s, g, &master[e], &m[e], &v[e]);
                if (param) param[e] = oracle_bf16_rne(master[e]);
                if (grad_out) grad_out[e] = g;
            }
        }
    }
    ol_free(&L);
    return 0;
}

/* The replicated (ZeRO-0 / DDP) step on the full layout: the averaged gradient
 * (same rank order, same division) and AdamW on full fp32 state.  n = number of
 * full-layout elements; skip (optional, n entries) marks positions that hold no
 * logical element (FLAT padding) -- they get g = 0 like the sharded path. */
int oracle_ddp_adamw(int64_t n, int32_t N, const void* const* grads, int32_t grad_dtype,
                     const uint8_t* skip, float* p, float* m, float* v,
                     float lr, float beta1, float beta2, float eps, float wd, int64_t step) {
    if (N < 1 || step < 1) return -1;
    oscal s = scalars(lr, beta1, beta2, eps, wd, step);
    for (int64_t i = 0; i < n; ++i) {
        float g = (skip && skip[i]) ? 0.0f : reduce_mean(grads, grad_dtype, N, i);
        adamw_elem(&s, g, &p[i], &m[i], &v[i]);
    }
    return 0;
}

/* The same update on a list of independent points: g_rows holds, per point,
 * the N replica gradients (already widened to fp32; bf16 -> fp32 is exact).
 * Used for sampled checks of large layouts. */
int oracle_adamw_points(int64_t n, int32_t N, const float* g_rows, float* p, float* m, float* v,
                        uint16_t* param, float* grad_out,
                        float lr, float beta1, float beta2, float eps, float wd, int64_t step) {
    if (N < 1 || step < 1) return -1;
    oscal s = scalars(lr, beta1, beta2, eps, wd, step);
    for (int64_t i = 0; i < n; ++i) {
        float acc = 0.0f;
        for (int32_t q = 0; q < N; ++q) acc = acc + g_rows[i * N + q];
        float g = acc / (float)N;
        adamw_elem(&s, g, &p[i], &m[i], &v[i]);
        if (param) param[i] = oracle_bf16_rne(p[i]);
        if (grad_out) grad_out[i] = g;
    }
    return 0;
}

/* Per-rank model-state bytes for ZeRO stage 0..3 ([ZeRO-state] "Canonical ZeRO
 * 状态公式": per rank P, P, 2P at stage 0; optimizer 2P/N from stage 1, gradient
 * P/N from stage 2, parameter P/N at stage 3; stages are cumulative).
 * pb, gb = bytes per parameter / gradient element; ob = optimizer-state bytes per
 * element (8 for fp32 exp_avg + exp_avg_sq, 12 with an fp32 master copy).
 * physical = 1 counts the rank's padded slot (S per rank); 0 counts only the
 * logical elements the rank owns.  step_bytes: optimizer metadata per tensor
 * (Adam's step scalar), counted once per tensor the rank's optimizer holds.
 * out[0..2] = parameter, gradient, optimizer bytes of this rank. */
int oracle_state_bytes(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                       int32_t N, int32_t mode, int32_t stage, int32_t rank, int32_t physical,
                       int64_t pb, int64_t gb, int64_t ob, int64_t step_bytes, int64_t* out) {
    olayout L;
    if (stage < 0 || stage > 3) return -1;
    if (ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    if (rank < 0 || rank >= N) { ol_free(&L); return -1; }
    int64_t own = 0;
    if (physical) {
        own = L.S;
    } else {
        for (int64_t j = 0; j < L.S; ++j)
            if (ol_full_index(&L, rank, j, NULL) >= 0) ++own;
    }
    int64_t P = L.P;
    out[0] = (stage >= 3 ? own : P) * pb;
    out[1] = (stage >= 2 ? own : P) * gb;
    out[2] = (stage >= 1 ? own : P) * ob + (int64_t)T * step_bytes;
    ol_free(&L);
    return 0;
}

/* Collective payload of one training step, per rank ([ZeRO-state] "Logical Payload
 * 模型": the logical total of each collective's input buffer, in elements, not the
 * bytes a ring algorithm moves over links).  strategy: 0 NO_SHARD (DDP: one all-reduce
 * of the gradient), 1 ZeRO-1 (ZeroRedundancyOptimizer: the same all-reduce, then the
 * updated parameters synchronised by broadcast, about P), 2 SHARD_GRAD_OP (forward
 * all-gather, gradient reduce-scatter), 3 FULL_SHARD (forward and backward all-gather,
 * reduce-scatter), 4 HYBRID_SHARD with R replica groups of N ranks ([FSDP-ch18] §18.9:
 * the FULL_SHARD collectives inside a group, then one all-reduce of the reduced shard,
 * S elements, across the groups).  R must be 1 for the other strategies.
 * elems[0..4] = all-reduce input, forward all-gather, backward all-gather,
 * reduce-scatter input, broadcast.
 * *bus = elements one rank sends (and receives) under ring algorithms: an all-reduce
 * over n ranks 2(n-1)/n times its input (the same page section); an all-gather or a
 * reduce-scatter over N ranks (N-1)/N times the full buffer (each rank passes on N-1 of
 * the N chunks); the broadcast: each rank receives the parameters it does not own,
 * (N-1)/N of P when owners hold equal shares (a reading: the page gives only the
 * logical size). */
int oracle_collective_payload(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                              int32_t N, int32_t mode, int32_t strategy, int32_t R, int64_t* elems, double* bus) {
    olayout L;
    if (strategy < 0 || strategy > 4 || R < 1 || (strategy != 4 && R != 1)) return -1;
    if (ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    int64_t P = L.P, S = L.S;
    for (int k = 0; k < 5; ++k) elems[k] = 0;
    if (strategy == 0 || strategy == 1) elems[0] = P;
    if (strategy == 1) elems[4] = P;
    if (strategy >= 2) { elems[1] = P; elems[3] = P; }
    if (strategy >= 3) elems[2] = P;
    double chunk = (double)(N - 1) / (double)N;            /* ring share over the N ranks */
    double b = chunk * (double)(elems[1] + elems[2] + elems[3] + elems[4]);
    if (strategy == 4) {
        elems[0] = S;
        b += 2.0 * (double)(R - 1) / (double)R * (double)S;
    } else {
        b += 2.0 * chunk * (double)elems[0];
    }
    *bus = b;
    ol_free(&L);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Rows beyond the core step                                                  */
/* ------------------------------------------------------------------------- */

/* Sharded clip_grad_norm_ between the reduce-scatter and AdamW
 * ([FSDP-ch18] §18.18: each rank's local sum of squares, an all-reduce of the
 * sums, the square root, every rank scales its own gradient slice).  Reading of
 * the constants the page leaves to torch's clip_grad_norm_: L2 norm,
 * coef = min(1, max_norm / (norm + 1e-6)).  The sum of squares is accumulated in
 * double over every rank's logical shard elements; coef is rounded to fp32 once
 * and each reduced gradient is scaled by it (one fp32 multiply) before AdamW.
 * grad_out (optional) receives the clipped gradient; *total_norm the norm. */
int oracle_rs_clip_adamw(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                         int32_t N, int32_t mode, int32_t ub, int32_t ue,
                         const void* const* grads, int32_t grad_dtype, int64_t stride,
                         float* master, float* m, float* v, uint16_t* param, float* grad_out, float max_norm,
                         float lr, float beta1, float beta2, float eps, float wd, int64_t step,
                         double* total_norm) {
    olayout L;
    if (ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    if (ub < 0 || ue > L.U || ub > ue || stride < L.S || step < 1) { ol_free(&L); return -1; }
    float* g = calloc((size_t)N * (size_t)stride + 1, sizeof(float));
    if (!g) { ol_free(&L); return -1; }
    /* (1) reduce-scatter, (2) the sum of squares over all ranks */
    double ss = 0.0;
    for (int32_t u = ub; u < ue; ++u)
        for (int32_t r = 0; r < N; ++r)
            for (int64_t k = 0; k < L.u_S[u]; ++k) {
                int64_t j = L.u_shard_off[u] + k;
                int64_t fi = ol_full_index(&L, r, j, NULL);
                float x = fi >= 0 ? reduce_mean(grads, grad_dtype, N, fi) : 0.0f;
                g[(int64_t)r * stride + j] = x;
                ss += (double)x * (double)x;
            }
    /* (3) the norm and the clip coefficient */
    double norm = sqrt(ss);
    double c = (double)max_norm / (norm + 1e-6);
    if (c > 1.0) c = 1.0;
    float coef = (float)c;
    if (total_norm) *total_norm = norm;
    /* (4) each rank's slice scaled, then AdamW */
    oscal s = scalars(lr, beta1, beta2, eps, wd, step);
    for (int32_t u = ub; u < ue; ++u)
        for (int32_t r = 0; r < N; ++r)
            for (int64_t k = 0; k < L.u_S[u]; ++k) {
                int64_t e = (int64_t)r * stride + L.u_shard_off[u] + k;
                float gc = g[e] * coef;
                adamw_elem(&s, gc, &master[e], &m[e], &v[e]);
                if (param) param[e] = oracle_bf16_rne(master[e]);
                if (grad_out) grad_out[e] = gc;
            }
    free(g);
    ol_free(&L);
    return 0;
}

/* Gradient accumulation without synchronisation ([FSDP-ch18] §18.26: no_sync /
 * set_requires_gradient_sync(False) -- the unsharded gradient accumulates
 * locally, the reduce-scatter runs once on the last micro-batch).  One replica:
 * acc = micro on the first micro-batch (first != 0), else acc = acc + micro, in
 * fp32, over n full-layout elements. */
int oracle_accumulate(int64_t n, float* acc, const void* micro, int32_t micro_dtype, int32_t first) {
    for (int64_t i = 0; i < n; ++i) {
        float x = load_grad(micro, micro_dtype, i);
        acc[i] = first ? x : acc[i] + x;
    }
    return 0;
}

/* HSDP ([FSDP-ch18] §18.9: shard within the group, replicate across groups; the
 * reduce-scatter runs in the shard dimension, then one all-reduce across the
 * replica groups).  R groups of N ranks; grads[rho*N + q] is rank q of group
 * rho.  Per shard element: g_rho = (sum_q G[rho][q]) / N (rank order), then
 * g = (sum_rho g_rho) / R (group order); every group's state copy gets the same
 * AdamW update.  master/m/v/param: R copies of [N][stride], copy rho at
 * rho*N*stride.  (The torchtitan article §3.4 orders the two collectives the
 * other way round; this follows the book chapter.) */
int oracle_hsdp_adamw(int32_t T, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                      int32_t N, int32_t mode, int32_t R, const void* const* grads, int32_t grad_dtype,
                      int64_t stride, float* master, float* m, float* v, uint16_t* param,
                      float lr, float beta1, float beta2, float eps, float wd, int64_t step) {
    olayout L;
    if (R < 1 || ol_build(&L, T, ndim, dims, unit_id, N, mode)) return -1;
    if (stride < L.S || step < 1) { ol_free(&L); return -1; }
    oscal s = scalars(lr, beta1, beta2, eps, wd, step);
    const int64_t copy = (int64_t)N * stride;
    for (int32_t r = 0; r < N; ++r)
        for (int64_t j = 0; j < L.S; ++j) {
            int64_t fi = ol_full_index(&L, r, j, NULL);
            float g = 0.0f;
            if (fi >= 0) {
                float outer = 0.0f;
                for (int32_t rho = 0; rho < R; ++rho)
                    outer = outer + reduce_mean(grads + (int64_t)rho * N, grad_dtype, N, fi);
                g = outer / (float)R;
            }
            for (int32_t rho = 0; rho < R; ++rho) {
                int64_t e = rho * copy + (int64_t)r * stride + j;
                adamw_elem(&s, g, &master[e], &m[e], &v[e]);
                if (param) param[e] = oracle_bf16_rne(master[e]);
            }
        }
    ol_free(&L);
    return 0;
}

/* ZeRO-1 owner partition ([ZeRO-state] "ZeRO-1：Optimizer State Sharding": each
 * rank updates about 1/N of the parameters -- whole parameters -- and
 * broadcasts them; "常见错误" warns against balancing owners by parameter count
 * instead of bytes).  Reading, after torch's ZeroRedundancyOptimizer: tensors
 * sorted by size, largest first (stable), each given to the rank with the
 * fewest elements so far (lowest rank on ties).  owner[t] receives the rank. */
int oracle_zero1_owners(int32_t T, const int32_t* ndim, const int64_t* dims, int32_t N, int32_t* owner) {
    if (T < 1 || N < 1) return -1;
    int64_t* numel = calloc((size_t)T, 8);
    int32_t* order = calloc((size_t)T, 4);
    int64_t* load = calloc((size_t)N, 8);
    int64_t pos = 0;
    for (int32_t t = 0; t < T; ++t) {
        int64_t n = 1;
        for (int32_t k = 0; k < ndim[t]; ++k) n *= dims[pos + k];
        pos += ndim[t];
        numel[t] = n;
        order[t] = t;
    }
    /* stable insertion sort by size, largest first */
    for (int32_t i = 1; i < T; ++i) {
        int32_t x = order[i], j = i - 1;
        while (j >= 0 && numel[order[j]] < numel[x]) { order[j + 1] = order[j]; --j; }
        order[j + 1] = x;
    }
    for (int32_t i = 0; i < T; ++i) {
        int32_t best = 0;
        for (int32_t r = 1; r < N; ++r) if (load[r] < load[best]) best = r;
        owner[order[i]] = best;
        load[best] += numel[order[i]];
    }
    free(numel); free(order); free(load);
    return 0;
}

/* ZeRO-1 step ([ZeRO-state] "ZeRO-1：Optimizer State Sharding": the gradient is
 * all-reduced (averaged), the owner updates its parameters with its optimizer
 * state, then broadcasts the updated parameters to every rank).  params[q] is
 * rank q's full replica of all parameters (P elements, tensors concatenated;
 * fp32, or bf16 when master != NULL).  Owner state for tensor t lives in the
 * owner's row at the tensor's place among the owner's tensors (tensor order):
 * master/m/v are [N][stride].  For fp32 parameters (master == NULL) the owner's
 * own replica is the parameter AdamW updates. */
int oracle_zero1_adamw(int32_t T, const int32_t* ndim, const int64_t* dims, int32_t N,
                       const void* const* grads, int32_t grad_dtype, int64_t stride,
                       float* master, float* m, float* v, void* const* params,
                       float lr, float beta1, float beta2, float eps, float wd, int64_t step) {
    if (T < 1 || N < 1 || step < 1) return -1;
    int32_t* owner = calloc((size_t)T, 4);
    int64_t* off_in_row = calloc((size_t)N, 8);
    oracle_zero1_owners(T, ndim, dims, N, owner);
    oscal s = scalars(lr, beta1, beta2, eps, wd, step);
    int64_t pos = 0, full = 0;
    for (int32_t t = 0; t < T; ++t) {
        int64_t n = 1;
        for (int32_t k = 0; k < ndim[t]; ++k) n *= dims[pos + k];
        pos += ndim[t];
        int32_t o = owner[t];
        int64_t row = (int64_t)o * stride + off_in_row[o];
        if (off_in_row[o] + n > stride) { free(owner); free(off_in_row); return -1; }
        for (int64_t k = 0; k < n; ++k) {
            float g = reduce_mean(grads, grad_dtype, N, full + k);
            float p = master ? master[row + k] : ((float*)params[o])[full + k];
            adamw_elem(&s, g, &p, &m[row + k], &v[row + k]);
            if (master) master[row + k] = p;
            for (int32_t q = 0; q < N; ++q) {          /* the broadcast */
                if (master) ((uint16_t*)params[q])[full + k] = oracle_bf16_rne(p);
                else ((float*)params[q])[full + k] = p;
            }
        }
        off_in_row[o] += n;
        full += n;
    }
    free(owner); free(off_in_row);
    return 0;
}
