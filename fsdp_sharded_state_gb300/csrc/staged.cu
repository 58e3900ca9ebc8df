// staged.cu -- the fused reduce-scatter + AdamW + bf16 recast on the bulk-copy
// pipeline (pipeline.cuh), sm_103a.
//
// "NCCL ZeRO/FSDP state sharding", "ZeRO-2 方向"/"ZeRO-3 方向": each rank keeps only
// the 1/N slice of the reduce-scattered gradient and updates its own optimizer state
// with it; "第18章 FSDP" §18.6: fp32 reduce, AdamW on the fp32 master, cast to
// param_dtype.  Per tile the stage holds the three fp32 state slices and the N
// gradient slices; the arithmetic and its order are those of the direct kernel
// (kernels.cu), bit for bit.  Also here: the bounded-wait self-test and the reader
// of every staged translation unit's wait word.
#include <type_traits>

#include "pipeline.cuh"
#include "staged.hpp"

namespace fsdp {
namespace {

// ---- fused reduce-scatter + AdamW + cast ------------------------------------------
// A tile's N replicas come in NG groups of Q (the last may be shorter); the partial
// sums carry over in registers from group to group in rank order, and the last
// group also stages the three state slices and does the update.  NG = 1 unless N
// replicas and the state do not fit two stages.
struct Sum4 {
    float a0, a1, a2, a3;
};

// A consumer thread's carry when the step constants come from memory: the partial
// sums, and the constants, taken from shared memory at the thread's first item.
struct SumConsts {
    Sum4 sum;
    AdamScal s;
    int ready;
};

// The CTA's copy of the constants block (read by one consumer thread per CTA), in
// the pipeline's policy area of shared memory.
__device__ __forceinline__ AdamScal& consts_shared() {
    static_assert(sizeof(AdamScal) <= 64, "policy area");
    return *reinterpret_cast<AdamScal*>(policy_front());
}

// The constants block (16-byte aligned; device or page-locked host memory), read
// with .cv loads: no cached copy is used, so a replayed launch sees what the host
// wrote into a host block since the last one.
__device__ __forceinline__ AdamScal ld_consts_fresh(const AdamScal* p) {
    float v[12];
    const float* f = reinterpret_cast<const float*>(p);
    asm volatile("ld.global.cv.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "l"(f) : "memory");
    asm volatile("ld.global.cv.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                 : "l"(f + 4) : "memory");
    asm volatile("ld.global.cv.f32 %0, [%1];" : "=f"(v[8]) : "l"(f + 8) : "memory");
    AdamScal s;
    s.decay = v[0];
    s.om1 = v[1];
    s.om2 = v[2];
    s.step_size = v[3];
    s.bc2s = v[4];
    s.beta1 = v[5];
    s.beta2 = v[6];
    s.eps = v[7];
    s.nf = v[8];
    return s;
}

// DC: the step's AdamW constants are read from a block in memory (dsc: device or
// page-locked host memory), once per CTA into shared memory, instead of taken from
// the kernel argument (sc), so that a captured CUDA graph can replay the launch with
// the constants rewritten in between.
template <typename GT, bool PARAM, bool GOUT, bool DC = false>
struct RsAdamw {
    static constexpr bool kGeomFirst = true;
    const Seg* segs;
    int64_t tile_base;
    GradPtrs gp;
    int N, Q, NG;
    float *master, *exp_avg, *exp_avg_sq;
    uint16_t* param;
    float* gout;
    AdamScal sc;
    const AdamScal* dsc;

    using Carry = typename std::conditional<DC, SumConsts, Sum4>::type;
    static constexpr bool kPrologue = DC;
    __device__ void prologue(int tid) const {
        if (tid == 0) consts_shared() = ld_consts_fresh(dsc);   // one read of the block per CTA
    }
    __device__ int groups() const { return NG; }
    __device__ int q0(const TileGeom& g) const { return g.q * Q; }
    __device__ int nq(const TileGeom& g) const { return (N - g.q * Q) < Q ? (N - g.q * Q) : Q; }
    __device__ bool last(const TileGeom& g) const { return g.q == NG - 1; }
    __device__ TileGeom geom(int64_t u, int k, int& cur) const {
        const int64_t gt = tile_base + u;
        cur = advance_seg(segs, cur, gt);
        TileGeom g = tile_geom<GT>(segs[cur], gt);
        g.q = k;
        return g;
    }
    __device__ uint32_t bytes(const TileGeom& g) const {
        const uint32_t sb = g.bs > g.as && last(g) ? uint32_t(g.bs - g.as) * 4u : 0u;
        const uint32_t gb = g.bg > g.ag ? uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT)) : 0u;
        return 3u * sb + uint32_t(nq(g)) * gb;
    }
    __device__ void issue(const TileGeom& g, uint32_t sbase, uint32_t bar, int lane) const {
        const uint32_t sb = g.bs > g.as && last(g) ? uint32_t(g.bs - g.as) * 4u : 0u;
        const uint32_t gb = g.bg > g.ag ? uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT)) : 0u;
        const int k0 = q0(g), n = nq(g);
        for (int k = lane; k < n + 3; k += 32) {
            if (k < 3) {
                const float* arr = k == 0 ? master : (k == 1 ? exp_avg : exp_avg_sq);
                if (sb) bulk_g2s(sbase + k * kStateBytes + uint32_t(g.as - g.t0) * 4u, arr + g.as, sb, bar);
            } else if (gb) {
                const int q = k - 3;
                bulk_g2s(sbase + 3 * kStateBytes + q * grank_bytes<GT>() + uint32_t(g.ag - g.gbase) * uint32_t(sizeof(GT)),
                         static_cast<const GT*>(gp.p[k0 + q]) + g.ag, gb, bar);
            }
        }
    }
    template <class Release>
    __device__ double consume(const TileGeom& g, const unsigned char* sb, int tid, Carry& carry, Release release) const {
        if constexpr (DC) {
            if (!carry.ready) {
                carry.s = consts_shared();
                carry.ready = 1;
            }
            return consume_with(carry.s, g, sb, tid, carry.sum, release);
        } else {
            return consume_with(sc, g, sb, tid, carry, release);
        }
    }
    template <class Release>
    __device__ double consume_with(const AdamScal& sc, const TileGeom& g, const unsigned char* sb, int tid,
                                   Sum4& carry, Release release) const {
        const int c = tid * 4;
        const int64_t x = g.t0 + c, f = x + g.delta;
        const bool live = x + 4 > g.s0 && x < g.s1;
        const bool fast = x >= g.s0 && x + 4 <= g.s1 && f >= g.ag && f + 4 <= g.bg;
        const bool fin = last(g);
        float4 pv, mv, vv;
        if (g.q == 0) carry = Sum4{0.0f, 0.0f, 0.0f, 0.0f};
        if (fast) {
            if (fin) {
                pv = lds4(sb + 0 * kStateBytes + c * 4);
                mv = lds4(sb + 1 * kStateBytes + c * 4);
                vv = lds4(sb + 2 * kStateBytes + c * 4);
            }
            const int o = int(f - g.gbase), n = nq(g);
            const unsigned char* gs = sb + 3 * kStateBytes;
            float a0 = carry.a0, a1 = carry.a1, a2 = carry.a2, a3 = carry.a3;
#pragma unroll 4
            for (int q = 0; q < n; ++q) {            // fixed rank order, continued from the last group
                const float4 x4 = grad4<GT>(gs + q * grank_bytes<GT>(), o);
                a0 = __fadd_rn(a0, x4.x); a1 = __fadd_rn(a1, x4.y);
                a2 = __fadd_rn(a2, x4.z); a3 = __fadd_rn(a3, x4.w);
            }
            carry = Sum4{a0, a1, a2, a3};
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
            // segment edge: element by element from global memory, all N replicas at once
            const int64_t a = x > g.s0 ? x : g.s0;
            const int64_t b = (x + 4) < g.s1 ? (x + 4) : g.s1;
            for (int64_t e = a; e < b; ++e) {
                const float gg = mean_div(reduce1<GT>(gp, N, e + g.delta), sc.nf);
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

template <typename GT, bool PARAM, bool GOUT, bool DC>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_rs_adamw_staged(RsAdamw<GT, PARAM, GOUT, DC> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns,
                  unsigned int* claim, int claim_batch) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns, claim, claim_batch);
}

// A wait that nothing completes: one mbarrier expects 16 bytes that no copy
// delivers.  The bounded wait must give up, record the error and return.
__global__ void k_wait_selftest(uint64_t wait_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    mbar_fence_init();
    mbar_arrive_tx(b, 16);
    if (!mbar_wait_bounded(b, 0, wait_ns)) atomicOr(&g_wait_error, 1u);
}

// Replica groups of the fused step: one group when all N replicas and the state fit
// two stages, else the fewest groups (of equal size, rounded up) that do.
void rs_groups(int N, bool bf16, int dev, int* Q, int* NG) {
    int ng = 1;
    while (ng < N && stage_count(rs_stage_bytes((N + ng - 1) / ng, bf16), dev) < 2) ++ng;
    *NG = ng;
    *Q = (N + ng - 1) / ng;
}

}  // namespace

bool staged_fits(int N, bool grad_bf16) {
    // with replica groups, any N whose single-replica stage fits two stages
    return N >= 1 && N <= kMaxRanks && fits(rs_stage_bytes(1, grad_bf16));
}

cudaError_t launch_rs_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                   const GradPtrs& gp, int N, float* master, float* m, float* v, uint16_t* param,
                                   float* gout, const AdamScal& sc, uint64_t wait_ns, cudaStream_t st,
                                   const AdamScal* dsc, bool claims) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int Q = N, NG = 1;
    rs_groups(N, grad_bf16, dev, &Q, &NG);
    const int sb = rs_stage_bytes(Q, grad_bf16);
    auto go = [&](auto tag_gt, auto tag_p, auto tag_g) {
        using GT = decltype(tag_gt);
        constexpr bool P = decltype(tag_p)::value, O = decltype(tag_g)::value;
        if (dsc) {
            RsAdamw<GT, P, O, true> pol{segs, tile_base, gp, N, Q, NG, master, m, v, param, gout, sc, dsc};
            return launch_pipeline(k_rs_adamw_staged<GT, P, O, true>, pol, n_tiles, sb, wait_ns, st, nullptr,
                                   claims);
        }
        RsAdamw<GT, P, O, false> pol{segs, tile_base, gp, N, Q, NG, master, m, v, param, gout, sc, nullptr};
        return launch_pipeline(k_rs_adamw_staged<GT, P, O, false>, pol, n_tiles, sb, wait_ns, st, nullptr, claims);
    };
    using T = std::true_type;
    using F = std::false_type;
    if (grad_bf16) {
        if (param) return gout ? go(uint16_t{}, T{}, T{}) : go(uint16_t{}, T{}, F{});
        return gout ? go(uint16_t{}, F{}, T{}) : go(uint16_t{}, F{}, F{});
    }
    if (param) return gout ? go(float{}, T{}, T{}) : go(float{}, T{}, F{});
    return gout ? go(float{}, F{}, T{}) : go(float{}, F{}, F{});
}

cudaError_t launch_wait_selftest(uint64_t wait_ns, cudaStream_t st) {
    k_wait_selftest<<<1, 32, 0, st>>>(wait_ns);
    return cudaGetLastError();
}

cudaError_t take_wait_error(unsigned int* flag) {
    unsigned int a = 0, b = 0, c = 0, d = 0;
    cudaError_t e = take_local_wait_error(&a);
    if (e == cudaSuccess) e = take_wait_error_allgather(&b);
    if (e == cudaSuccess) e = take_wait_error_rows(&c);
    if (e == cudaSuccess) e = take_wait_error_coop(&d);
    *flag = a | b | c | d;
    return e;
}

}  // namespace fsdp
