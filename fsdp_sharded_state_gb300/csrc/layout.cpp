// layout.cpp -- host-side layout engine of libfsdpstate (no CUDA calls).
//
// FLAT ("第18章 FSDP：ZeRO 风格的参数分片" §18.12; "NCCL ZeRO/FSDP state sharding",
// section "FlatParameter 与 Padding"): the tensors of one unit are flattened and
// concatenated into P_u elements, padded at the end to N*S_u with
// S_u = ceil(P_u/N); rank r owns flat elements [r*S_u, (r+1)*S_u).
// DIM0 ("PyTorch FSDP2 后端特性介绍", section "DTensor"; torchtitan FSDP2 article
// §2.3): each tensor with d0 rows of `inner` elements gets a slot of c = ceil(d0/N)
// rows on every rank; rank r owns rows [min(rc,d0), min((r+1)c,d0)).
#include "layout.hpp"

#include <algorithm>

#include "../../include/fsdp_state.h"

namespace fsdp {
namespace {

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

void push(SegList& l, int64_t shard, int64_t full, int64_t len) {
    if (len <= 0) return;
    l.segs.push_back(Seg{shard, full, len, 0});
}

// Also files the piece under its alignment class.
void push2(SegList& all, SegList& al, SegList& sh, int64_t shard, int64_t full, int64_t len) {
    push(all, shard, full, len);
    push(((full - shard) & (kVec - 1)) == 0 ? al : sh, shard, full, len);
}

void finish(SegList& l) {
    int64_t t = 0;
    for (Seg& s : l.segs) {
        s.tile0 = t;
        t += seg_tiles(s.shard, s.len);
    }
    l.segs.push_back(Seg{0, -1, 0, t});   // sentinel: tile0 = total tiles
}

}  // namespace

int build_layout(fsdp_layout* L, int32_t T, const int32_t* ndim, const int64_t* dims,
                 const int32_t* unit_id, const int32_t* dtype, int32_t N, int32_t mode) {
    if (T < 1 || !ndim || !dims || !unit_id) return FSDP_EINVAL;
    if (N < 1 || N > FSDP_MAX_RANKS) return FSDP_EINVAL;
    if (mode != FSDP_FLAT && mode != FSDP_DIM0 && mode != FSDP_ZERO1) return FSDP_EINVAL;
    if (unit_id[0] != 0) return FSDP_ESHAPE;
    for (int32_t t = 1; t < T; ++t)
        if (unit_id[t] != unit_id[t - 1] && unit_id[t] != unit_id[t - 1] + 1) return FSDP_ESHAPE;
    if (dtype)
        for (int32_t t = 0; t < T; ++t)
            if (dtype[t] != FSDP_F32 && dtype[t] != FSDP_BF16) return FSDP_EDTYPE;

    L->T = T; L->N = N; L->mode = mode; L->U = unit_id[T - 1] + 1;
    const int32_t U = L->U;
    L->numel.assign(T, 0); L->d0.assign(T, 0); L->inner.assign(T, 0); L->rows.assign(T, 0);
    L->t_full_off.assign(T, 0); L->t_shard_off.assign(T, -1); L->t_unit_off.assign(T, 0);
    L->unit.assign(unit_id, unit_id + T);
    L->dtype.assign(T, FSDP_F32);
    if (dtype) L->dtype.assign(dtype, dtype + T);
    L->u_numel.assign(U, 0); L->u_S.assign(U, 0); L->u_shard_off.assign(U, 0); L->u_full_off.assign(U, 0);

    // Shapes.
    int64_t pos = 0;
    for (int32_t t = 0; t < T; ++t) {
        if (ndim[t] < 0 || ndim[t] > 16) return FSDP_ESHAPE;
        int64_t n = 1, in = 1;
        for (int32_t k = 0; k < ndim[t]; ++k) {
            const int64_t d = dims[pos + k];
            if (d < 0) return FSDP_ESHAPE;
            if (!mul_ok(n, d, &n)) return FSDP_EOVERFLOW;
            if (k > 0 && !mul_ok(in, d, &in)) return FSDP_EOVERFLOW;
        }
        L->numel[t] = n;
        L->d0[t] = ndim[t] == 0 ? 1 : dims[pos];
        L->inner[t] = ndim[t] == 0 ? 1 : in;
        pos += ndim[t];
    }

    // FlatParameter requires one dtype per unit.
    if (mode == FSDP_FLAT)
        for (int32_t t = 1; t < T; ++t)
            if (L->unit[t] == L->unit[t - 1] && L->dtype[t] != L->dtype[t - 1]) return FSDP_EDTYPE;

    int64_t P = 0;
    for (int32_t t = 0; t < T; ++t) {
        const int32_t u = L->unit[t];
        L->t_unit_off[t] = L->u_numel[u];
        if (!add_ok(L->u_numel[u], L->numel[t], &L->u_numel[u])) return FSDP_EOVERFLOW;
        if (!add_ok(P, L->numel[t], &P)) return FSDP_EOVERFLOW;
    }
    L->P = P;

    if (mode == FSDP_FLAT) {
        int64_t so = 0, fo = 0;
        for (int32_t u = 0; u < U; ++u) {
            L->u_S[u] = (L->u_numel[u] + N - 1) / N;
            L->u_shard_off[u] = so;
            L->u_full_off[u] = fo;
            int64_t slot;
            if (!mul_ok(L->u_S[u], N, &slot)) return FSDP_EOVERFLOW;
            if (!add_ok(so, L->u_S[u], &so) || !add_ok(fo, slot, &fo)) return FSDP_EOVERFLOW;
        }
        L->S = so; L->F = fo;
        for (int32_t t = 0; t < T; ++t)
            L->t_full_off[t] = L->u_full_off[L->unit[t]] + L->t_unit_off[t];
    } else if (mode == FSDP_ZERO1) {
        // Whole tensors on owner ranks: largest first (stable), each to the rank
        // holding the fewest elements so far, lowest rank on ties.  In its owner's
        // row a tensor sits at an offset congruent to its full offset mod 8.
        std::vector<int32_t> order(T);
        for (int32_t t = 0; t < T; ++t) order[t] = t;
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t a, int32_t b) { return L->numel[a] > L->numel[b]; });
        std::vector<int64_t> load(N, 0);
        L->owner.assign(T, 0);
        for (int32_t t : order) {
            int32_t best = 0;
            for (int32_t r = 1; r < N; ++r)
                if (load[r] < load[best]) best = r;
            L->owner[t] = best;
            load[best] += L->numel[t];
        }
        int64_t fo = 0;
        std::vector<int64_t> fill(N, 0);
        for (int32_t t = 0; t < T; ++t) {
            L->t_full_off[t] = fo;
            const int32_t o = L->owner[t];
            const int64_t at = fill[o] + ((fo - fill[o]) & (kVec - 1));   // == fo (mod 8)
            L->t_shard_off[t] = at;
            fill[o] = at + L->numel[t];
            if (!add_ok(fo, L->numel[t], &fo)) return FSDP_EOVERFLOW;
        }
        int64_t S = 0;
        for (int32_t r = 0; r < N; ++r) S = std::max(S, fill[r]);
        L->S = S; L->F = fo;
        for (int32_t t = 0; t < T; ++t) {
            const int32_t u = L->unit[t];
            if (t == 0 || L->unit[t - 1] != u) L->u_full_off[u] = L->t_full_off[t];
            L->u_shard_off[u] = 0;
            L->u_S[u] = S;                       // every unit spans the owner rows
        }
    } else {
        int64_t so = 0, fo = 0;
        for (int32_t t = 0; t < T; ++t) {
            L->rows[t] = (L->d0[t] + N - 1) / N;
            int64_t slot;
            if (!mul_ok(L->rows[t], L->inner[t], &slot)) return FSDP_EOVERFLOW;
            L->t_shard_off[t] = so;
            L->t_full_off[t] = fo;
            if (!add_ok(so, slot, &so) || !add_ok(fo, L->numel[t], &fo)) return FSDP_EOVERFLOW;
        }
        L->S = so; L->F = fo;
        for (int32_t t = 0; t < T; ++t) {
            const int32_t u = L->unit[t];
            if (t == 0 || L->unit[t - 1] != u) {
                L->u_shard_off[u] = L->t_shard_off[t];
                L->u_full_off[u] = L->t_full_off[t];
            }
            L->u_S[u] += L->rows[t] * L->inner[t];
        }
    }

    // Physical row stride.  Rank r's piece of unit/tensor x sits at shard index
    // r*stride + off_x and at full index full_x + r*len_x; 16-byte vectors line up on
    // both sides when the two are congruent mod 8.  That depends on stride mod 8
    // only, so pick the residue that keeps the most logical elements congruent and
    // prefer 0 (then stride = S rounded up to 64: rows 128/256-byte aligned).  A
    // single FLAT unit with S odd, say, gets stride = S and every rank lines up.
    int64_t aligned_elems[kVec] = {0};
    for (int32_t u = 0; u < U; ++u) {
        for (int32_t r = 0; r < N; ++r) {
            if (mode == FSDP_ZERO1) {
                break;
            } else if (mode == FSDP_FLAT) {
                const int64_t own = std::max<int64_t>(0, std::min(L->u_S[u], L->u_numel[u] - int64_t(r) * L->u_S[u]));
                for (int sig = 0; sig < kVec; ++sig) {
                    const int64_t dlt = L->u_full_off[u] + int64_t(r) * L->u_S[u] - int64_t(r) * sig - L->u_shard_off[u];
                    if ((dlt & (kVec - 1)) == 0) aligned_elems[sig] += own;
                }
            } else {
                for (int32_t t = 0; t < T; ++t) {
                    if (L->unit[t] != u) continue;
                    const int64_t c = L->rows[t];
                    const int64_t rb = std::min<int64_t>(int64_t(r) * c, L->d0[t]);
                    const int64_t re = std::min<int64_t>(int64_t(r + 1) * c, L->d0[t]);
                    const int64_t own = (re - rb) * L->inner[t];
                    for (int sig = 0; sig < kVec; ++sig) {
                        const int64_t dlt = L->t_full_off[t] + rb * L->inner[t] - int64_t(r) * sig - L->t_shard_off[t];
                        if ((dlt & (kVec - 1)) == 0) aligned_elems[sig] += own;
                    }
                }
            }
        }
    }
    int best = 0;
    for (int sig = 1; sig < kVec && mode != FSDP_ZERO1; ++sig)
        if (aligned_elems[sig] > aligned_elems[best]) best = sig;
    int64_t stride;
    if (best == 0) {
        if (!add_ok(L->S, 63, &stride)) return FSDP_EOVERFLOW;
        stride = stride / 64 * 64;
    } else {
        const int64_t rem = ((best - L->S) % kVec + kVec) % kVec;     // stride = S + rem = best (mod 8)
        if (!add_ok(L->S, rem, &stride)) return FSDP_EOVERFLOW;
    }
    int64_t total;
    if (!mul_ok(stride, N, &total)) return FSDP_EOVERFLOW;
    if (!mul_ok(total, 4, &total)) return FSDP_EOVERFLOW;   // fp32 byte size must fit too
    if (!mul_ok(L->F, 4, &total)) return FSDP_EOVERFLOW;
    L->stride = stride;

    // Segment lists, per unit: rank-major, then tensor order.
    SegList* lists[] = {&L->data, &L->gather, &L->pad, &L->data_al, &L->data_sh, &L->gather_al, &L->gather_sh,
                        &L->fullr};
    for (SegList* l : lists) {
        l->segs.clear();
        l->unit_begin.assign(U + 1, 0);
    }
    int64_t n_data = 0;
    for (int32_t u = 0; u < U; ++u) {
        for (SegList* l : lists) l->unit_begin[u] = int32_t(l->segs.size());
        // logical full-layout ranges of the unit
        if (mode == FSDP_FLAT) {
            push(L->fullr, L->u_full_off[u], L->u_full_off[u], L->u_numel[u]);
        } else {
            for (int32_t t = 0; t < T; ++t)
                if (L->unit[t] == u) push(L->fullr, L->t_full_off[t], L->t_full_off[t], L->numel[t]);
        }
        if (mode == FSDP_ZERO1) {
            for (int32_t t = 0; t < T; ++t) {
                if (L->unit[t] != u) continue;
                const int64_t sh = int64_t(L->owner[t]) * stride + L->t_shard_off[t];
                push2(L->data, L->data_al, L->data_sh, sh, L->t_full_off[t], L->numel[t]);
                if (L->numel[t] > 0) ++n_data;
            }
            if (u == U - 1) {                       // each row's unused tail: zero at reshard
                std::vector<std::pair<int64_t, int64_t>> used;
                for (int32_t r = 0; r < N; ++r) {
                    int64_t at = 0;
                    for (int32_t t = 0; t < T; ++t) {
                        if (L->owner[t] != r) continue;
                        push(L->pad, int64_t(r) * stride + at, -1, L->t_shard_off[t] - at);   // alignment gap
                        at = L->t_shard_off[t] + L->numel[t];
                    }
                    push(L->pad, int64_t(r) * stride + at, -1, stride - at);
                }
            }
            continue;
        }
        for (int32_t r = 0; r < N; ++r) {
            const int64_t row = int64_t(r) * stride;
            if (mode == FSDP_FLAT) {
                const int64_t Su = L->u_S[u];
                const int64_t first = int64_t(r) * Su;                     // flat position
                const int64_t own = std::max<int64_t>(0, std::min(Su, L->u_numel[u] - first));
                const int64_t sh = row + L->u_shard_off[u];
                const int64_t fu = L->u_full_off[u] + first;
                push2(L->data, L->data_al, L->data_sh, sh, fu, own);
                push2(L->gather, L->gather_al, L->gather_sh, sh, fu, Su);
                push(L->pad, sh + own, -1, Su - own);
                if (own > 0) ++n_data;
            } else {
                for (int32_t t = 0; t < T; ++t) {
                    if (L->unit[t] != u) continue;
                    const int64_t c = L->rows[t];
                    const int64_t rb = std::min<int64_t>(int64_t(r) * c, L->d0[t]);
                    const int64_t re = std::min<int64_t>(int64_t(r + 1) * c, L->d0[t]);
                    const int64_t own = (re - rb) * L->inner[t];
                    const int64_t sh = row + L->t_shard_off[t];
                    const int64_t fu = L->t_full_off[t] + rb * L->inner[t];
                    push2(L->data, L->data_al, L->data_sh, sh, fu, own);
                    push2(L->gather, L->gather_al, L->gather_sh, sh, fu, own);
                    push(L->pad, sh + own, -1, c * L->inner[t] - own);
                    if (own > 0) ++n_data;
                }
            }
            if (u == U - 1) push(L->pad, row + L->S, -1, stride - L->S);   // row tail
        }
    }
    int64_t off = 0;
    for (SegList* l : lists) {
        l->unit_begin[U] = int32_t(l->segs.size());
        finish(*l);
        l->dev_off = off;                       // position in the device table
        off += int64_t(l->segs.size());
    }
    L->n_data_segments = n_data;
    return FSDP_OK;
}

}  // namespace fsdp
