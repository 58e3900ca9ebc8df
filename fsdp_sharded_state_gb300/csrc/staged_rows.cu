// staged_rows.cu -- the rows beyond the core step on the bulk-copy pipeline
// (pipeline.cuh), sm_103a:
//
//   k_hsdp_adamw_staged   HSDP ("第18章 FSDP" §18.9): R replica groups of N shard
//                         ranks; mean within each group, mean over the groups, AdamW
//                         on each group's copy of the state.
//   k_accumulate_staged   fp32 accumulation of one micro-batch into each replica's
//                         gradient buffer ("第18章 FSDP" §18.26, no_sync).
//   k_rs_norm_staged      pass 1 of the sharded clip_grad_norm_ ("第18章 FSDP"
//                         §18.18): the reduce-scatter into the fp32 gradient shard
//                         plus the sum of squares, one partial per consumer warp.
//   k_adamw_scaled_staged pass 3 of it: the clip coefficient times the gradient
//                         shard, then AdamW and the cast.
//   k_zero1_adamw_staged  the ZeRO-1 owner step ("NCCL ZeRO/FSDP state sharding",
//                         "ZeRO-1"): mean over the N replicas, AdamW on the owner's
//                         state, the result stored into all N parameter replicas.
//   k_acc_rs_adamw_staged the last micro-batch of a no_sync accumulation ("第18章
//                         FSDP" §18.26) fused with the reduce-scatter + AdamW + cast.
//
// Arithmetic and its order are those of the direct kernels (rows.cu), bit for bit
// (the clip norm's double sum is grouped per warp instead of per CTA).
#include <type_traits>

#include "pipeline.cuh"
#include "staged.hpp"

namespace fsdp {
namespace {

// ---- HSDP: R replica groups x N shard ranks -----------------------------------------
// g = (sum over groups rho of (sum over q of G[rho*N + q]) / N) / R, then AdamW on
// each group's copy of the state (copy rho at element offset rho * copy).
template <typename GT, bool PARAM>
struct HsdpAdamw {
    static constexpr bool kGeomFirst = false;
    static constexpr int kMaxR = 3;
    const Seg* segs;
    int64_t tile_base;
    GradPtrs gp;
    int N, R;
    int64_t copy;
    float *master, *exp_avg, *exp_avg_sq;
    uint16_t* param;
    AdamScal sc;
    float rf;

    using Carry = NoCarry;
    __device__ int groups() const { return 1; }
    __device__ TileGeom geom(int64_t u, int, int& cur) const {
        const int64_t gt = tile_base + u;
        cur = advance_seg(segs, cur, gt);
        return tile_geom<GT>(segs[cur], gt);
    }
    __device__ uint32_t bytes(const TileGeom& g) const {
        const uint32_t sb = g.bs > g.as ? uint32_t(g.bs - g.as) * 4u : 0u;
        const uint32_t gb = g.bg > g.ag ? uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT)) : 0u;
        return 3u * uint32_t(R) * sb + uint32_t(R * N) * gb;
    }
    __device__ void issue(const TileGeom& g, uint32_t sbase, uint32_t bar, int lane) const {
        const uint32_t sb = g.bs > g.as ? uint32_t(g.bs - g.as) * 4u : 0u;
        const uint32_t gb = g.bg > g.ag ? uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT)) : 0u;
        const int ns = 3 * R;
        for (int k = lane; k < ns + R * N; k += 32) {
            if (k < ns) {
                const int arr_i = k % 3, rho = k / 3;
                const float* arr = arr_i == 0 ? master : (arr_i == 1 ? exp_avg : exp_avg_sq);
                if (sb) bulk_g2s(sbase + k * kStateBytes + uint32_t(g.as - g.t0) * 4u, arr + rho * copy + g.as, sb, bar);
            } else if (gb) {
                const int q = k - ns;
                bulk_g2s(sbase + ns * kStateBytes + q * grank_bytes<GT>() + uint32_t(g.ag - g.gbase) * uint32_t(sizeof(GT)),
                         static_cast<const GT*>(gp.p[q]) + g.ag, gb, bar);
            }
        }
    }
    template <class Release>
    __device__ double consume(const TileGeom& g, const unsigned char* sb, int tid, Carry& carry, Release release) const {
        const int c = tid * 4;
        const int64_t x = g.t0 + c, f = x + g.delta;
        const bool live = x + 4 > g.s0 && x < g.s1;
        const bool fast = x >= g.s0 && x + 4 <= g.s1 && f >= g.ag && f + 4 <= g.bg;
        float4 st[3 * kMaxR];
        float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f;
        if (fast) {
#pragma unroll
            for (int k = 0; k < 3 * kMaxR; ++k)
                if (k < 3 * R) st[k] = lds4(sb + k * kStateBytes + c * 4);
            const int o = int(f - g.gbase);
            const unsigned char* gs = sb + 3 * R * kStateBytes;
            for (int rho = 0; rho < R; ++rho) {
                float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll 4
                for (int q = 0; q < N; ++q) {
                    const float4 x4 = grad4<GT>(gs + (rho * N + q) * grank_bytes<GT>(), o);
                    a0 = __fadd_rn(a0, x4.x); a1 = __fadd_rn(a1, x4.y);
                    a2 = __fadd_rn(a2, x4.z); a3 = __fadd_rn(a3, x4.w);
                }
                o0 = __fadd_rn(o0, mean_div(a0, sc.nf)); o1 = __fadd_rn(o1, mean_div(a1, sc.nf));
                o2 = __fadd_rn(o2, mean_div(a2, sc.nf)); o3 = __fadd_rn(o3, mean_div(a3, sc.nf));
            }
        }
        release();
        if (fast) {
            const float gg[4] = {mean_div(o0, rf), mean_div(o1, rf), mean_div(o2, rf), mean_div(o3, rf)};
#pragma unroll
            for (int rho = 0; rho < kMaxR; ++rho) {
                if (rho >= R) break;
                float p[4] = {st[3 * rho].x, st[3 * rho].y, st[3 * rho].z, st[3 * rho].w};
                float m[4] = {st[3 * rho + 1].x, st[3 * rho + 1].y, st[3 * rho + 1].z, st[3 * rho + 1].w};
                float v[4] = {st[3 * rho + 2].x, st[3 * rho + 2].y, st[3 * rho + 2].z, st[3 * rho + 2].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) adamw1(sc, gg[k], p[k], m[k], v[k]);
                const int64_t e = rho * copy + x;
                // streaming stores (st.global.cs, evict-first in L2): fewer of this call's
                // dirty lines are left in L2 for the next call to write back (measured on
                // GB300, calls back to back on the 128 MiB fp32 layout, R = 2: 430 -> 413 us;
                // the 4-block Llama unchanged)
                __stcs(reinterpret_cast<float4*>(master + e), make_float4(p[0], p[1], p[2], p[3]));
                __stcs(reinterpret_cast<float4*>(exp_avg + e), make_float4(m[0], m[1], m[2], m[3]));
                __stcs(reinterpret_cast<float4*>(exp_avg_sq + e), make_float4(v[0], v[1], v[2], v[3]));
                if (PARAM)
                    __stcs(reinterpret_cast<uint2*>(param + e), make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3])));
            }
        } else if (live) {
            const int64_t a = x > g.s0 ? x : g.s0;
            const int64_t b = (x + 4) < g.s1 ? (x + 4) : g.s1;
            for (int64_t e = a; e < b; ++e) {
                float outer = 0.0f;
                for (int rho = 0; rho < R; ++rho) {
                    float acc = 0.0f;
                    for (int q = 0; q < N; ++q)
                        acc = __fadd_rn(acc, GradIO<GT>::load1(gp.p[rho * N + q], e + g.delta));
                    outer = __fadd_rn(outer, mean_div(acc, sc.nf));
                }
                const float gg = mean_div(outer, rf);
                for (int rho = 0; rho < R; ++rho) {
                    const int64_t y = rho * copy + e;
                    float pp = master[y], mm = exp_avg[y], vv = exp_avg_sq[y];
                    adamw1(sc, gg, pp, mm, vv);
                    master[y] = pp; exp_avg[y] = mm; exp_avg_sq[y] = vv;
                    if (PARAM) param[y] = to_bf16(pp);
                }
            }
        }
        return 0.0;
    }
    __device__ void finish(int, double) const {}
};

// ---- ZeRO-1: owner update + broadcast ------------------------------------------------
// Parameters are whole and replicated; each tensor's optimizer state lives in its
// owner's row.  g = mean over the N replicas; the owner's AdamW on its state (p from
// the fp32 master in the row when the replicas are bf16, else from the owner's own
// fp32 replica); the updated parameter goes to all N replicas, stored straight from
// the consumers' registers (16-byte fp32 or 8-byte bf16 stores, a warp covering 512
// contiguous bytes of each replica).  Owner rows keep every tensor congruent to its
// full offset mod 8 (delta = 0 mod 8); anything else, and the at most 7 elements at
// each end that 16-byte copies leave out, is stored element by element.  (A form that
// wrote each tile's result once into a shared-memory output slot and broadcast it with
// one cp.async.bulk per replica from a store warp measured slower on GB300: 0.89 of the
// copy peak on the 128 MiB fp32 layout, 0.93-0.96 on the 4-block Llama.)
struct ParamReplicas {
    void* p[kMaxRanks];
};

template <typename GT, bool MASTER>
struct Zero1Adamw {
    static constexpr bool kGeomFirst = true;
    const Seg* segs;
    int64_t tile_base;
    GradPtrs gp;
    ParamReplicas pr;
    int N;
    int64_t stride;
    float *master, *exp_avg, *exp_avg_sq;
    AdamScal sc;

    using Carry = NoCarry;
    __device__ int groups() const { return 1; }
    __device__ TileGeom geom(int64_t u, int, int& cur) const {
        const int64_t gt = tile_base + u;
        cur = advance_seg(segs, cur, gt);
        const Seg sg = segs[cur];
        TileGeom g = tile_geom<GT>(sg, gt);
        g.q = int32_t(sg.shard / stride);            // the owner
        return g;
    }
    __device__ uint32_t bytes(const TileGeom& g) const {
        const uint32_t sb = g.bs > g.as ? uint32_t(g.bs - g.as) * 4u : 0u;
        const uint32_t gb = g.bg > g.ag ? uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT)) : 0u;
        const uint32_t pb = g.bg > g.ag && (g.delta & 7) == 0 ? uint32_t(g.bg - g.ag) * 4u : 0u;   // owner's replica
        return (MASTER ? 3u * sb : 2u * sb + pb) + uint32_t(N) * gb;
    }
    __device__ void issue(const TileGeom& g, uint32_t sbase, uint32_t bar, int lane) const {
        const uint32_t sb = g.bs > g.as ? uint32_t(g.bs - g.as) * 4u : 0u;
        const uint32_t gb = g.bg > g.ag ? uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT)) : 0u;
        for (int k = lane; k < N + 3; k += 32) {
            if (k == 0) {
                if (MASTER) {
                    if (sb) bulk_g2s(sbase + uint32_t(g.as - g.t0) * 4u, master + g.as, sb, bar);
                } else if (g.bg > g.ag && (g.delta & 7) == 0) {
                    // delta = 0 mod 8: gbase = t0 + delta, the slice fills the slot from its start
                    bulk_g2s(sbase + uint32_t(g.ag - g.gbase) * 4u, static_cast<const float*>(pr.p[g.q]) + g.ag,
                             uint32_t(g.bg - g.ag) * 4u, bar);
                }
            } else if (k < 3) {
                const float* arr = k == 1 ? exp_avg : exp_avg_sq;
                if (sb) bulk_g2s(sbase + k * kStateBytes + uint32_t(g.as - g.t0) * 4u, arr + g.as, sb, bar);
            } else if (gb) {
                const int q = k - 3;
                bulk_g2s(sbase + 3 * kStateBytes + q * grank_bytes<GT>() + uint32_t(g.ag - g.gbase) * uint32_t(sizeof(GT)),
                         static_cast<const GT*>(gp.p[q]) + g.ag, gb, bar);
            }
        }
    }
    template <class Release>
    __device__ double consume(const TileGeom& g, const unsigned char* sb, int tid, NoCarry&, Release release) const {
        const int c = tid * 4;
        const int64_t x = g.t0 + c, f = x + g.delta;
        const bool live = x + 4 > g.s0 && x < g.s1;
        const bool al = (g.delta & 7) == 0;              // owner rows keep delta = 0 mod 8
        const bool fast = x >= g.s0 && x + 4 <= g.s1 && f >= g.ag && f + 4 <= g.bg && al;
        float4 pv, mv, vv;
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        if (fast) {
            pv = lds4(sb + c * 4);
            mv = lds4(sb + 1 * kStateBytes + c * 4);
            vv = lds4(sb + 2 * kStateBytes + c * 4);
            const int o = int(f - g.gbase);
            const unsigned char* gs = sb + 3 * kStateBytes;
#pragma unroll 4
            for (int q = 0; q < N; ++q) {
                const float4 x4 = grad4<GT>(gs + q * grank_bytes<GT>(), o);
                a0 = __fadd_rn(a0, x4.x); a1 = __fadd_rn(a1, x4.y);
                a2 = __fadd_rn(a2, x4.z); a3 = __fadd_rn(a3, x4.w);
            }
        }
        release();
        if (fast) {
            float p[4] = {pv.x, pv.y, pv.z, pv.w};
            float m[4] = {mv.x, mv.y, mv.z, mv.w};
            float v[4] = {vv.x, vv.y, vv.z, vv.w};
            const float gg[4] = {mean_div(a0, sc.nf), mean_div(a1, sc.nf), mean_div(a2, sc.nf), mean_div(a3, sc.nf)};
#pragma unroll
            for (int k = 0; k < 4; ++k) adamw1(sc, gg[k], p[k], m[k], v[k]);
            if (MASTER) st4(master + x, make_float4(p[0], p[1], p[2], p[3]));
            st4(exp_avg + x, make_float4(m[0], m[1], m[2], m[3]));
            st4(exp_avg_sq + x, make_float4(v[0], v[1], v[2], v[3]));
            if (MASTER) {
                const uint2 w = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
#pragma unroll 1
                for (int q = 0; q < N; ++q) *reinterpret_cast<uint2*>(static_cast<uint16_t*>(pr.p[q]) + f) = w;
            } else {
                const float4 w = make_float4(p[0], p[1], p[2], p[3]);
#pragma unroll 1
                for (int q = 0; q < N; ++q) st4(static_cast<float*>(pr.p[q]) + f, w);
            }
        } else if (live) {
            const int64_t a = x > g.s0 ? x : g.s0;
            const int64_t b = (x + 4) < g.s1 ? (x + 4) : g.s1;
            for (int64_t e = a; e < b; ++e) {
                const int64_t fe = e + g.delta;
                float pp = MASTER ? master[e] : static_cast<const float*>(pr.p[g.q])[fe];
                float mm = exp_avg[e], vv2 = exp_avg_sq[e];
                adamw1(sc, mean_div(reduce1<GT>(gp, N, fe), sc.nf), pp, mm, vv2);
                if (MASTER) master[e] = pp;
                exp_avg[e] = mm; exp_avg_sq[e] = vv2;
                for (int q = 0; q < N; ++q) {
                    if (MASTER) static_cast<uint16_t*>(pr.p[q])[fe] = to_bf16(pp);
                    else static_cast<float*>(pr.p[q])[fe] = pp;
                }
            }
        }
        return 0.0;
    }
    __device__ void finish(int, double) const {}
};

// ---- clip pass 3: AdamW on the clipped fp32 gradient shard ----------------------------
// g = gshard * coef (one fp32 multiplication; coef from device memory, written by the
// norm pass), written back as the clipped gradient, then the AdamW and cast of the
// fused step.  The gradient shard shares the state's (shard) index: four slices of
// one tile per stage, no shift.
template <bool PARAM>
struct ScaledAdamw {
    static constexpr bool kGeomFirst = true;
    const Seg* segs;
    int64_t tile_base;
    float* gshard;
    const float* coef_p;
    float *master, *exp_avg, *exp_avg_sq;
    uint16_t* param;
    AdamScal sc;

    using Carry = NoCarry;
    __device__ int groups() const { return 1; }
    __device__ TileGeom geom(int64_t u, int, int& cur) const {
        const int64_t gt = tile_base + u;
        cur = advance_seg(segs, cur, gt);
        TileGeom g = tile_geom<float>(segs[cur], gt);
        g.q = __float_as_int(*coef_p);                 // the clip coefficient, once per item
        return g;
    }
    __device__ uint32_t bytes(const TileGeom& g) const {
        return g.bs > g.as ? 4u * uint32_t(g.bs - g.as) * 4u : 0u;
    }
    __device__ void issue(const TileGeom& g, uint32_t sbase, uint32_t bar, int lane) const {
        if (g.bs <= g.as || lane >= 4) return;
        const float* arr = lane == 0 ? master : (lane == 1 ? exp_avg : (lane == 2 ? exp_avg_sq : gshard));
        bulk_g2s(sbase + lane * kStateBytes + uint32_t(g.as - g.t0) * 4u, arr + g.as, uint32_t(g.bs - g.as) * 4u, bar);
    }
    template <class Release>
    __device__ double consume(const TileGeom& g, const unsigned char* sb, int tid, Carry&, Release release) const {
        const int c = tid * 4;
        const int64_t x = g.t0 + c;
        const bool live = x + 4 > g.s0 && x < g.s1;
        const bool fast = x >= g.s0 && x + 4 <= g.s1;
        const float coef = __int_as_float(g.q);
        float4 pv, mv, vv, gv;
        if (fast) {
            pv = lds4(sb + 0 * kStateBytes + c * 4);
            mv = lds4(sb + 1 * kStateBytes + c * 4);
            vv = lds4(sb + 2 * kStateBytes + c * 4);
            gv = lds4(sb + 3 * kStateBytes + c * 4);
        }
        release();
        if (fast) {
            float p[4] = {pv.x, pv.y, pv.z, pv.w};
            float m[4] = {mv.x, mv.y, mv.z, mv.w};
            float v[4] = {vv.x, vv.y, vv.z, vv.w};
            const float gg[4] = {__fmul_rn(gv.x, coef), __fmul_rn(gv.y, coef), __fmul_rn(gv.z, coef),
                                 __fmul_rn(gv.w, coef)};
#pragma unroll
            for (int k = 0; k < 4; ++k) adamw1(sc, gg[k], p[k], m[k], v[k]);
            st4(gshard + x, make_float4(gg[0], gg[1], gg[2], gg[3]));
            st4(master + x, make_float4(p[0], p[1], p[2], p[3]));
            st4(exp_avg + x, make_float4(m[0], m[1], m[2], m[3]));
            st4(exp_avg_sq + x, make_float4(v[0], v[1], v[2], v[3]));
            if (PARAM)
                *reinterpret_cast<uint2*>(param + x) = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
        } else if (live) {
            const int64_t a = x > g.s0 ? x : g.s0;
            const int64_t b = (x + 4) < g.s1 ? (x + 4) : g.s1;
            for (int64_t e = a; e < b; ++e) {
                const float gg = __fmul_rn(gshard[e], coef);
                float pp = master[e], mm = exp_avg[e], vv2 = exp_avg_sq[e];
                adamw1(sc, gg, pp, mm, vv2);
                gshard[e] = gg; master[e] = pp; exp_avg[e] = mm; exp_avg_sq[e] = vv2;
                if (PARAM) param[e] = to_bf16(pp);
            }
        }
        return 0.0;
    }
    __device__ void finish(int, double) const {}
};

// ---- clip pass 1: reduce-scatter into the fp32 shard + sums of squares ---------------
// Each 4-element chunk's squares are summed in fp32 (fma), the chunks in double; one
// partial per consumer warp (warp tree, lane order), written to part[CTA * 16 + warp].
template <typename GT>
struct RsNorm {
    static constexpr bool kGeomFirst = false;
    const Seg* segs;
    int64_t tile_base;
    GradPtrs gp;
    int N;
    float* gout;
    float nf;
    double* part;

    using Carry = NoCarry;
    __device__ int groups() const { return 1; }
    __device__ TileGeom geom(int64_t u, int, int& cur) const {
        const int64_t gt = tile_base + u;
        cur = advance_seg(segs, cur, gt);
        return tile_geom<GT>(segs[cur], gt);
    }
    __device__ uint32_t bytes(const TileGeom& g) const {
        return g.bg > g.ag ? uint32_t(N) * uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT)) : 0u;
    }
    __device__ void issue(const TileGeom& g, uint32_t sbase, uint32_t bar, int lane) const {
        if (g.bg <= g.ag) return;
        const uint32_t gb = uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT));
        for (int q = lane; q < N; q += 32)
            bulk_g2s(sbase + q * grank_bytes<GT>() + uint32_t(g.ag - g.gbase) * uint32_t(sizeof(GT)),
                     static_cast<const GT*>(gp.p[q]) + g.ag, gb, bar);
    }
    template <class Release>
    __device__ double consume(const TileGeom& g, const unsigned char* sb, int tid, Carry& carry, Release release) const {
        const int c = tid * 4;
        const int64_t x = g.t0 + c, f = x + g.delta;
        const bool live = x + 4 > g.s0 && x < g.s1;
        const bool fast = x >= g.s0 && x + 4 <= g.s1 && f >= g.ag && f + 4 <= g.bg;
        double ss = 0.0;
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        if (fast) {
            const int o = int(f - g.gbase);
#pragma unroll 4
            for (int q = 0; q < N; ++q) {
                const float4 x4 = grad4<GT>(sb + q * grank_bytes<GT>(), o);
                a0 = __fadd_rn(a0, x4.x); a1 = __fadd_rn(a1, x4.y);
                a2 = __fadd_rn(a2, x4.z); a3 = __fadd_rn(a3, x4.w);
            }
        }
        release();
        if (fast) {
            const float g0 = mean_div(a0, nf), g1 = mean_div(a1, nf), g2 = mean_div(a2, nf), g3 = mean_div(a3, nf);
            st4(gout + x, make_float4(g0, g1, g2, g3));
            float sq = __fmul_rn(g0, g0);
            sq = __fmaf_rn(g1, g1, sq);
            sq = __fmaf_rn(g2, g2, sq);
            sq = __fmaf_rn(g3, g3, sq);
            ss += double(sq);
        } else if (live) {
            const int64_t a = x > g.s0 ? x : g.s0;
            const int64_t b = (x + 4) < g.s1 ? (x + 4) : g.s1;
            for (int64_t e = a; e < b; ++e) {
                const float gg = mean_div(reduce1<GT>(gp, N, e + g.delta), nf);
                gout[e] = gg;
                ss += double(gg) * double(gg);
            }
        }
        return ss;
    }
    __device__ void finish(int tid, double x) const {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xffffffffu, x, o);
        if ((tid & 31) == 0) part[int64_t(blockIdx.x) * kConsumerWarps + (tid >> 5)] = x;
    }
};

// ---- accumulation of one micro-batch into each replica's fp32 buffer ----------------
// Items are (tile of the full layout, group of Q consecutive replicas): the stage
// holds the group's micro-batch slices, then (unless FIRST) its accumulator slices,
// so that one item moves about as many bytes as a tile of the fused step.  For
// each replica q of the group, acc[q] = micro[q] (FIRST) or acc[q] + micro[q], one
// fp32 addition per element.
template <typename MT, bool FIRST>
struct Accumulate {
    static constexpr bool kGeomFirst = false;
    static constexpr int kMaxQ = 8;
    const Seg* segs;                   // logical full-layout ranges (shard field = full index)
    int64_t tile_base;
    int N, Q, NG;                      // replicas, replicas per item, groups (ceil(N / Q))
    float* acc[kMaxRanks];
    const void* micro[kMaxRanks];

    static constexpr int kMicroBytes = int(kTileElems * sizeof(MT));
    __device__ int nq(const TileGeom& g) const { return (N - g.q) < Q ? (N - g.q) : Q; }
    using Carry = NoCarry;
    __device__ int groups() const { return 1; }
    __device__ TileGeom geom(int64_t i, int, int& cur) const {
        const int64_t gt = tile_base + i / NG;
        cur = advance_seg(segs, cur, gt);
        TileGeom g = tile_geom<MT>(segs[cur], gt);     // delta = 0: micro and acc share the index
        g.as = g.ag; g.bs = g.bg;                        // one aligned interior for both arrays
        g.q = int32_t(i % NG) * Q;
        return g;
    }
    __device__ uint32_t bytes(const TileGeom& g) const {
        if (g.bg <= g.ag) return 0u;
        const uint32_t n = uint32_t(g.bg - g.ag);
        return uint32_t(nq(g)) * (n * uint32_t(sizeof(MT)) + (FIRST ? 0u : n * 4u));
    }
    __device__ void issue(const TileGeom& g, uint32_t sbase, uint32_t bar, int lane) const {
        if (g.bg <= g.ag) return;
        const uint32_t n = uint32_t(g.bg - g.ag);
        const int k = nq(g);
        for (int c = lane; c < (FIRST ? k : 2 * k); c += 32) {
            if (c < k)
                bulk_g2s(sbase + c * kMicroBytes + uint32_t(g.ag - g.t0) * uint32_t(sizeof(MT)),
                         static_cast<const MT*>(micro[g.q + c]) + g.ag, n * uint32_t(sizeof(MT)), bar);
            else
                bulk_g2s(sbase + Q * kMicroBytes + (c - k) * kStateBytes + uint32_t(g.ag - g.t0) * 4u,
                         acc[g.q + c - k] + g.ag, n * 4u, bar);
        }
    }
    template <class Release>
    __device__ double consume(const TileGeom& g, const unsigned char* sb, int tid, Carry& carry, Release release) const {
        const int c = tid * 4;
        const int64_t x = g.t0 + c;
        const bool live = x + 4 > g.s0 && x < g.s1;
        const bool fast = x >= g.ag && x + 4 <= g.bg;
        const int k = nq(g);
        float4 out[kMaxQ];
        if (fast) {
#pragma unroll
            for (int r = 0; r < kMaxQ; ++r) {
                if (r >= k) break;
                float4 mv = grad4<MT>(sb + r * kMicroBytes, c);
                if (!FIRST) {
                    const float4 av = lds4(sb + Q * kMicroBytes + r * kStateBytes + c * 4);
                    mv.x = __fadd_rn(av.x, mv.x); mv.y = __fadd_rn(av.y, mv.y);
                    mv.z = __fadd_rn(av.z, mv.z); mv.w = __fadd_rn(av.w, mv.w);
                }
                out[r] = mv;
            }
        }
        release();
        if (fast) {
            // streaming stores (st.global.cs): measured on GB300, accumulation calls back to
            // back on the 128 MiB fp32 layout 246 -> 242 us, the 4-block Llama unchanged
#pragma unroll
            for (int r = 0; r < kMaxQ; ++r) {
                if (r >= k) break;
                __stcs(reinterpret_cast<float4*>(acc[g.q + r] + x), out[r]);
            }
        } else if (live) {
            const int64_t lo = x > g.s0 ? x : g.s0;
            const int64_t hi = (x + 4) < g.s1 ? (x + 4) : g.s1;
            for (int r = 0; r < k; ++r)
                for (int64_t e = lo; e < hi; ++e) {
                    const float v = GradIO<MT>::load1(micro[g.q + r], e);
                    acc[g.q + r][e] = FIRST ? v : __fadd_rn(acc[g.q + r][e], v);
                }
        }
        return 0.0;
    }
    __device__ void finish(int, double) const {}
};

template <typename GT, bool PARAM>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_hsdp_adamw_staged(HsdpAdamw<GT, PARAM> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns,
                  unsigned int* claim, int claim_batch) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns, claim, claim_batch);
}

template <typename GT, bool MASTER>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_zero1_adamw_staged(Zero1Adamw<GT, MASTER> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns,
                 unsigned int* claim, int claim_batch) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns, claim, claim_batch);
}

template <bool PARAM>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_adamw_scaled_staged(ScaledAdamw<PARAM> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns,
                  unsigned int* claim, int claim_batch) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns, claim, claim_batch);
}

template <typename GT>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_rs_norm_staged(RsNorm<GT> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns,
                  unsigned int* claim, int claim_batch) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns, claim, claim_batch);
}

template <typename MT, bool FIRST>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_accumulate_staged(Accumulate<MT, FIRST> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns,
                  unsigned int* claim, int claim_batch) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns, claim, claim_batch);
}

// Running sums of a thread's four elements, carried from one replica group to the next.
struct AccSum4 {
    float a0, a1, a2, a3;
};

// ---- the last micro-batch of a no_sync accumulation, fused with the step -----------
// ("第18章 FSDP" §18.26.)  Replica q contributes acc_q + micro_q: its fp32 accumulator
// and its micro-batch gradient (MT) at the same full-layout element, added in fp32 --
// the accumulation's own addition -- and the sums join the running mean's sum in rank
// order, as the fused step would read accumulators that had been updated first.  The
// accumulators are read only.  A stage holds the three state slices and, per replica of
// the group, its accumulator slice then its micro-batch slice; each slice is the
// 16-byte-aligned window of its own element size around the tile's full-layout range.
template <typename MT, bool PARAM, bool GOUT>
struct AccRsAdamw {
    static constexpr bool kGeomFirst = true;
    static constexpr int kPair = grank_bytes<float>() + grank_bytes<MT>();   // one replica's slices
    const Seg* segs;
    int64_t tile_base;
    GradPtrs acc, micro;
    int N, Q, NG;
    float *master, *exp_avg, *exp_avg_sq;
    uint16_t* param;
    float* gout;
    AdamScal sc;

    using Carry = AccSum4;
    __device__ int groups() const { return NG; }
    __device__ int q0(const TileGeom& g) const { return g.q * Q; }
    __device__ int nq(const TileGeom& g) const { return (N - g.q * Q) < Q ? (N - g.q * Q) : Q; }
    __device__ bool last(const TileGeom& g) const { return g.q == NG - 1; }
    // the fp32 accumulators' window is the geometry's (ag, bg, gbase); the micro-batch's
    // window, for MT elements, is formed here
    __device__ static void mwin(const TileGeom& g, int64_t& a, int64_t& b, int64_t& base) {
        constexpr int64_t E = 16 / sizeof(MT);
        a = ceil_to(g.s0 + g.delta, E);
        b = floor_to(g.s1 + g.delta, E);
        base = floor_to(g.t0 + g.delta, E);
    }
    __device__ TileGeom geom(int64_t u, int k, int& cur) const {
        const int64_t gt = tile_base + u;
        cur = advance_seg(segs, cur, gt);
        TileGeom g = tile_geom<float>(segs[cur], gt);
        g.q = k;
        return g;
    }
    __device__ uint32_t bytes(const TileGeom& g) const {
        int64_t ma, mb, mbase;
        mwin(g, ma, mb, mbase);
        const uint32_t sb = g.bs > g.as && last(g) ? uint32_t(g.bs - g.as) * 4u : 0u;
        const uint32_t ab = g.bg > g.ag ? uint32_t(g.bg - g.ag) * 4u : 0u;
        const uint32_t mbytes = mb > ma ? uint32_t(mb - ma) * uint32_t(sizeof(MT)) : 0u;
        return 3u * sb + uint32_t(nq(g)) * (ab + mbytes);
    }
    __device__ void issue(const TileGeom& g, uint32_t sbase, uint32_t bar, int lane) const {
        int64_t ma, mb, mbase;
        mwin(g, ma, mb, mbase);
        const uint32_t sb = g.bs > g.as && last(g) ? uint32_t(g.bs - g.as) * 4u : 0u;
        const uint32_t ab = g.bg > g.ag ? uint32_t(g.bg - g.ag) * 4u : 0u;
        const uint32_t mbytes = mb > ma ? uint32_t(mb - ma) * uint32_t(sizeof(MT)) : 0u;
        const int k0 = q0(g), n = nq(g);
        for (int k = lane; k < 3 + 2 * n; k += 32) {
            if (k < 3) {
                const float* arr = k == 0 ? master : (k == 1 ? exp_avg : exp_avg_sq);
                if (sb) bulk_g2s(sbase + k * kStateBytes + uint32_t(g.as - g.t0) * 4u, arr + g.as, sb, bar);
            } else {
                const int q = (k - 3) >> 1;
                const uint32_t slot = sbase + 3 * kStateBytes + q * kPair;
                if ((k - 3) & 1) {
                    if (mbytes)
                        bulk_g2s(slot + grank_bytes<float>() + uint32_t(ma - mbase) * uint32_t(sizeof(MT)),
                                 static_cast<const MT*>(micro.p[k0 + q]) + ma, mbytes, bar);
                } else if (ab) {
                    bulk_g2s(slot + uint32_t(g.ag - g.gbase) * 4u, static_cast<const float*>(acc.p[k0 + q]) + g.ag,
                             ab, bar);
                }
            }
        }
    }
    template <class Release>
    __device__ double consume(const TileGeom& g, const unsigned char* sb, int tid, Carry& carry, Release release) const {
        int64_t ma, mb, mbase;
        mwin(g, ma, mb, mbase);
        const int c = tid * 4;
        const int64_t x = g.t0 + c, f = x + g.delta;
        const bool live = x + 4 > g.s0 && x < g.s1;
        const bool fast = x >= g.s0 && x + 4 <= g.s1 && f >= g.ag && f + 4 <= g.bg && f >= ma && f + 4 <= mb;
        const bool fin = last(g);
        float4 pv, mv, vv;
        if (g.q == 0) carry = AccSum4{0.0f, 0.0f, 0.0f, 0.0f};
        if (fast) {
            if (fin) {
                pv = lds4(sb + 0 * kStateBytes + c * 4);
                mv = lds4(sb + 1 * kStateBytes + c * 4);
                vv = lds4(sb + 2 * kStateBytes + c * 4);
            }
            const int oa = int(f - g.gbase), om = int(f - mbase), n = nq(g);
            const unsigned char* gs = sb + 3 * kStateBytes;
            float a0 = carry.a0, a1 = carry.a1, a2 = carry.a2, a3 = carry.a3;
#pragma unroll 2
            for (int q = 0; q < n; ++q) {            // rank order, continued from the last group
                const float4 y = grad4<float>(gs + q * kPair, oa);
                const float4 z = grad4<MT>(gs + q * kPair + grank_bytes<float>(), om);
                a0 = __fadd_rn(a0, __fadd_rn(y.x, z.x)); a1 = __fadd_rn(a1, __fadd_rn(y.y, z.y));
                a2 = __fadd_rn(a2, __fadd_rn(y.z, z.z)); a3 = __fadd_rn(a3, __fadd_rn(y.w, z.w));
            }
            carry = AccSum4{a0, a1, a2, a3};
        }
        release();
        if (!fin) return 0.0;
        if (fast) {
            float p[4] = {pv.x, pv.y, pv.z, pv.w};
            float m[4] = {mv.x, mv.y, mv.z, mv.w};
            float v[4] = {vv.x, vv.y, vv.z, vv.w};
            float gg[4] = {mean_div(carry.a0, sc.nf), mean_div(carry.a1, sc.nf), mean_div(carry.a2, sc.nf),
                           mean_div(carry.a3, sc.nf)};
#pragma unroll
            for (int k = 0; k < 4; ++k) adamw1(sc, gg[k], p[k], m[k], v[k]);
            st4(master + x, make_float4(p[0], p[1], p[2], p[3]));
            st4(exp_avg + x, make_float4(m[0], m[1], m[2], m[3]));
            st4(exp_avg_sq + x, make_float4(v[0], v[1], v[2], v[3]));
            if (PARAM)
                *reinterpret_cast<uint2*>(param + x) = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
            if (GOUT) st4(gout + x, make_float4(gg[0], gg[1], gg[2], gg[3]));
        } else if (live) {
            // segment edge, or a window edge: element by element from global memory
            const int64_t a = x > g.s0 ? x : g.s0;
            const int64_t b = (x + 4) < g.s1 ? (x + 4) : g.s1;
            for (int64_t e = a; e < b; ++e) {
                const int64_t fe = e + g.delta;
                float sum = 0.0f;
                for (int q = 0; q < N; ++q)
                    sum = __fadd_rn(sum, __fadd_rn(static_cast<const float*>(acc.p[q])[fe],
                                                   GradIO<MT>::load1(micro.p[q], fe)));
                const float gg = mean_div(sum, sc.nf);
                float pp = master[e], mm = exp_avg[e], vv2 = exp_avg_sq[e];
                adamw1(sc, gg, pp, mm, vv2);
                master[e] = pp; exp_avg[e] = mm; exp_avg_sq[e] = vv2;
                if (PARAM) param[e] = to_bf16(pp);
                if (GOUT) gout[e] = gg;
            }
        }
        return 0.0;
    }
    __device__ void finish(int, double) const {}
};

template <typename MT, bool PARAM, bool GOUT>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_acc_rs_adamw_staged(AccRsAdamw<MT, PARAM, GOUT> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns,
                  unsigned int* claim, int claim_batch) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns, claim, claim_batch);
}

// Accumulation items: as many replicas (up to 8) as keep an item near 96 KB of stage.
constexpr int kAccItemBytes = 96 * 1024;
// ZeRO-1 aims at 96 KB in flight (2 stages of 57 KB): measured 0.5 % faster than 3; the
// accumulation at 128 KB (3 stages of 64 KB): 0.4 % faster than 2.
constexpr int kZero1InFlightBytes = 96 * 1024;
constexpr int kAccInFlightBytes = 128 * 1024;
// The last micro-batch fused with the step aims at 160 KB: 3 stages where they fit (the
// 4-block Llama's two replica groups, 74 KB stages: 8.71 against 8.87 ms with 2).
constexpr int kAccStepInFlightBytes = 160 * 1024;

int hsdp_stage_bytes(int N, int R, bool bf16) {
    return 3 * R * kStateBytes + R * N * (bf16 ? grank_bytes<uint16_t>() : grank_bytes<float>());
}
int norm_stage_bytes(int N, bool bf16) { return N * (bf16 ? grank_bytes<uint16_t>() : grank_bytes<float>()); }
int acc_stage_bytes(int Q, bool bf16, bool first) { return Q * (int(kTileElems) * (bf16 ? 2 : 4) + (first ? 0 : kStateBytes)); }

}  // namespace

cudaError_t launch_acc_rs_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool micro_bf16,
                                       const GradPtrs& acc, const GradPtrs& micro, int N, float* master, float* m,
                                       float* v, uint16_t* param, float* gout, const AdamScal& sc, uint64_t wait_ns,
                                       cudaStream_t st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int pair = micro_bf16 ? AccRsAdamw<uint16_t, false, false>::kPair : AccRsAdamw<float, false, false>::kPair;
    auto stage = [&](int q) { return 3 * kStateBytes + q * pair; };
    int NG = 1;                          // the fewest equal groups whose stage fits twice
    while (NG < N && stage_count(stage((N + NG - 1) / NG), dev) < 2) ++NG;
    const int Q = (N + NG - 1) / NG;
    if (stage_count(stage(Q), dev) < 2) return cudaErrorInvalidValue;
    auto go = [&](auto tag_mt, auto tag_p, auto tag_g) {
        using MT = decltype(tag_mt);
        constexpr bool P = decltype(tag_p)::value, O = decltype(tag_g)::value;
        AccRsAdamw<MT, P, O> pol{segs, tile_base, acc, micro, N, Q, NG, master, m, v, param, gout, sc};
        return launch_pipeline(k_acc_rs_adamw_staged<MT, P, O>, pol, n_tiles, stage(Q), wait_ns, st, nullptr, true,
                               kAccStepInFlightBytes);
    };
    using T = std::true_type;
    using F = std::false_type;
    if (micro_bf16) {
        if (param) return gout ? go(uint16_t{}, T{}, T{}) : go(uint16_t{}, T{}, F{});
        return gout ? go(uint16_t{}, F{}, T{}) : go(uint16_t{}, F{}, F{});
    }
    if (param) return gout ? go(float{}, T{}, T{}) : go(float{}, T{}, F{});
    return gout ? go(float{}, F{}, T{}) : go(float{}, F{}, F{});
}

bool acc_rs_staged_fits(bool micro_bf16) {
    const int pair = micro_bf16 ? AccRsAdamw<uint16_t, false, false>::kPair : AccRsAdamw<float, false, false>::kPair;
    return fits(3 * kStateBytes + pair);
}

bool hsdp_staged_fits(int N, int R, bool grad_bf16, int64_t copy) {
    return R <= HsdpAdamw<float, false>::kMaxR && (copy & 3) == 0 && fits(hsdp_stage_bytes(N, R, grad_bf16));
}

bool norm_staged_fits(int N, bool grad_bf16) { return fits(norm_stage_bytes(N, grad_bf16)); }

bool zero1_staged_fits(int N, bool grad_bf16) { return fits(rs_stage_bytes(N, grad_bf16)); }

cudaError_t launch_adamw_scaled_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, float* gshard,
                                       const float* coef, float* master, float* m, float* v, uint16_t* param,
                                       const AdamScal& sc, uint64_t wait_ns, cudaStream_t st) {
    const int sb = 4 * kStateBytes;
    if (param) {
        ScaledAdamw<true> pol{segs, tile_base, gshard, coef, master, m, v, param, sc};
        return launch_pipeline(k_adamw_scaled_staged<true>, pol, n_tiles, sb, wait_ns, st, nullptr, true);
    }
    ScaledAdamw<false> pol{segs, tile_base, gshard, coef, master, m, v, param, sc};
    return launch_pipeline(k_adamw_scaled_staged<false>, pol, n_tiles, sb, wait_ns, st, nullptr, true);
}

int norm_staged_partials(int64_t n_tiles) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = n_tiles < sms ? n_tiles : sms;
    return int(blocks) * kConsumerWarps;
}

cudaError_t launch_hsdp_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                     const GradPtrs& gp, int N, int R, int64_t copy, float* master, float* m,
                                     float* v, uint16_t* param, const AdamScal& sc, float rf, uint64_t wait_ns,
                                     cudaStream_t st) {
    const int sb = hsdp_stage_bytes(N, R, grad_bf16);
    auto go = [&](auto tag_gt, auto tag_p) {
        using GT = decltype(tag_gt);
        constexpr bool P = decltype(tag_p)::value;
        HsdpAdamw<GT, P> pol{segs, tile_base, gp, N, R, copy, master, m, v, param, sc, rf};
        return launch_pipeline(k_hsdp_adamw_staged<GT, P>, pol, n_tiles, sb, wait_ns, st, nullptr, true);
    };
    if (grad_bf16) return param ? go(uint16_t{}, std::true_type{}) : go(uint16_t{}, std::false_type{});
    return param ? go(float{}, std::true_type{}) : go(float{}, std::false_type{});
}

cudaError_t launch_rs_norm_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                  const GradPtrs& gp, int N, float* gout, double* part, int* n_part, uint64_t wait_ns,
                                  cudaStream_t st) {
    const int sb = norm_stage_bytes(N, grad_bf16);
    int grid = 0;
    cudaError_t e;
    if (grad_bf16) {
        RsNorm<uint16_t> pol{segs, tile_base, gp, N, gout, float(N), part};
        e = launch_pipeline(k_rs_norm_staged<uint16_t>, pol, n_tiles, sb, wait_ns, st, &grid);
    } else {
        RsNorm<float> pol{segs, tile_base, gp, N, gout, float(N), part};
        e = launch_pipeline(k_rs_norm_staged<float>, pol, n_tiles, sb, wait_ns, st, &grid);
    }
    *n_part = grid * kConsumerWarps;
    return e;
}

cudaError_t launch_accumulate_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, int N, float* const* acc,
                                     const void* const* micro, bool micro_bf16, bool first, uint64_t wait_ns,
                                     cudaStream_t st) {
    // replicas per item: as many as keep a stage near the in-flight target (at most 8)
    const int per = acc_stage_bytes(1, micro_bf16, first);
    int Q = kAccItemBytes / per;
    Q = Q < 1 ? 1 : (Q > Accumulate<float, false>::kMaxQ ? Accumulate<float, false>::kMaxQ : Q);
    if (Q > N) Q = N;
    const int NG = (N + Q - 1) / Q;
    const int sb = acc_stage_bytes(Q, micro_bf16, first);
    const int64_t n_items = n_tiles * NG;
    auto go = [&](auto tag_mt, auto tag_first) {
        using MT = decltype(tag_mt);
        constexpr bool FIRST = decltype(tag_first)::value;
        Accumulate<MT, FIRST> pol{};
        pol.segs = segs;
        pol.tile_base = tile_base;
        pol.N = N;
        pol.Q = Q;
        pol.NG = NG;
        for (int q = 0; q < N; ++q) {
            pol.acc[q] = acc[q];
            pol.micro[q] = micro[q];
        }
        return launch_pipeline(k_accumulate_staged<MT, FIRST>, pol, n_items, sb, wait_ns, st, nullptr, true,
                               kAccInFlightBytes);
    };
    if (micro_bf16) return first ? go(uint16_t{}, std::true_type{}) : go(uint16_t{}, std::false_type{});
    return first ? go(float{}, std::true_type{}) : go(float{}, std::false_type{});
}

cudaError_t launch_zero1_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                      const GradPtrs& gp, void* const* replicas, int N, int64_t stride,
                                      float* master, float* m, float* v, const AdamScal& sc, uint64_t wait_ns,
                                      cudaStream_t st) {
    const int sb = rs_stage_bytes(N, grad_bf16);
    auto go = [&](auto tag_gt, auto tag_m) {
        using GT = decltype(tag_gt);
        constexpr bool M = decltype(tag_m)::value;
        Zero1Adamw<GT, M> pol{};
        pol.segs = segs;
        pol.tile_base = tile_base;
        pol.gp = gp;
        for (int q = 0; q < N; ++q) pol.pr.p[q] = replicas[q];
        pol.N = N;
        pol.stride = stride;
        pol.master = master;
        pol.exp_avg = m;
        pol.exp_avg_sq = v;
        pol.sc = sc;
        return launch_pipeline(k_zero1_adamw_staged<GT, M>, pol, n_tiles, sb, wait_ns, st, nullptr, true,
                               kZero1InFlightBytes);
    };
    if (grad_bf16) return master ? go(uint16_t{}, std::true_type{}) : go(uint16_t{}, std::false_type{});
    return master ? go(float{}, std::true_type{}) : go(float{}, std::false_type{});
}

cudaError_t take_wait_error_rows(unsigned int* flag) { return take_local_wait_error(flag); }

}  // namespace fsdp
