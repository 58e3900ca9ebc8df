// staged.cu -- kernels whose inputs the bulk-copy (TMA) engine stages in shared
// memory (sm_103a).
//
// One pipeline, six uses.  A persistent CTA per SM walks its work items (a tile of
// 2048 elements of one segment, or of one segment and one replica); per item, a
// producer warp issues one cp.async.bulk global -> shared per input array into a
// free stage and writes the item's geometry into the stage header, and a "full"
// mbarrier per stage counts the bytes in (complete_tx).  16 consumer warps wait on
// it, read their 4 elements of every staged array into registers, release the
// stage on an "empty" mbarrier (one arrive per warp) and only then compute and
// store, so the next copies go out while they do.  No CTA-wide barrier in the loop;
// the bytes in flight per SM do not depend on registers.  The uses:
//
//   k_rs_adamw_staged    the fused reduce-scatter (fp32 mean over the N replicas,
//                        fixed rank order) + AdamW + bf16 recast ("NCCL ZeRO/FSDP
//                        state sharding", "ZeRO-2 方向"/"ZeRO-3 方向"; "第18章 FSDP"
//                        §18.6): stage = 3 fp32 state slices + N gradient slices.
//   k_hsdp_adamw_staged  the same step for R replica groups of N shard ranks ("第18章
//                        FSDP" §18.9): mean within each group, mean over the groups,
//                        AdamW on each group's copy of the state.
//   k_rs_norm_staged     pass 1 of the sharded clip_grad_norm_ ("第18章 FSDP" §18.18):
//                        the reduce-scatter into the fp32 gradient shard plus the sum
//                        of squares, one partial per consumer warp.
//   k_adamw_scaled_staged  pass 3 of it: the clip coefficient times the gradient
//                        shard, then AdamW and the cast.
//   k_accumulate_staged  fp32 accumulation of one micro-batch into each replica's
//                        gradient buffer ("第18章 FSDP" §18.26, no_sync).
//   k_zero1_adamw_staged the ZeRO-1 owner step ("NCCL ZeRO/FSDP state sharding",
//                        "ZeRO-1"): mean over the N replicas, AdamW on the owner's
//                        state, the result stored into all N parameter replicas.
//
// Arithmetic and its order are those of the direct kernels (kernels.cu, rows.cu),
// bit for bit.  A gradient piece whose full-layout offset is not congruent to its
// shard offset mod 8 is copied as the 16-byte-aligned window around it and read
// from shared memory at its offset: no warp shuffle, one launch for both alignment
// classes.  Each consumer thread owns 4 consecutive elements of an item: 16-byte
// shared-memory reads, 16-byte (fp32) and 8-byte (bf16) global stores that cover
// whole sectors per warp.  The at most 7 elements at each end of a segment that
// the 16-byte copies leave out go element by element from global memory.
//
// The all-gather of the aligned class (k_unshard_bulk, further down) moves whole
// tiles global -> shared -> global with bulk copies and no thread touching them.
//
// Every wait on an mbarrier is bounded in time; a warp that gives up records
// FSDP_ETIMEOUT in a device word that fsdp_check_status reads and returns (a
// producer first waits, bounded, for the copies it has in flight), after which the
// CTA's other waits run out in turn.  Nothing else in these kernels waits.
#include <atomic>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "device_ops.cuh"
#include "staged.hpp"

namespace fsdp {

// Nonzero once a bounded wait on this device gave up; read and cleared by the host.
__device__ unsigned int g_wait_error = 0;

namespace {

constexpr int kStThreads = 512;                 // consumer threads: 4 elements each per item
constexpr int kConsumerWarps = kStThreads / 32;
constexpr int kMaxStages = 8;
constexpr int kInFlightBytes = 96 * 1024;       // stage bytes in flight per SM to aim for
constexpr int kFrontBytes = 1024;               // mbarriers + per-stage item geometry
constexpr int kStateBytes = int(kTileElems) * 4;

// ---- PTX wrappers: mbarrier, bulk copy, timer ------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    // make the initialised barriers visible to the async proxy (the bulk-copy engine)
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for phase `parity` of the barrier to complete, for at most about limit_ns
// nanoseconds (and at most 2^24 polls); false if it gave up.  The clock is read
// once every 64 polls, starting at the 64th: a read of %globaltimer is slow, and
// most waits end within the first polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    uint64_t t0 = 0;
#pragma unroll 1
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 63) {
            const uint64_t now = global_ns();
            if (i == 63) t0 = now;
            else if (now - t0 > limit_ns) return false;
        }
    }
    return false;
}
// Global -> shared bulk copy whose completion is counted on the barrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ int64_t floor_to(int64_t x, int64_t a) { return x & ~(a - 1); }   // a: power of 2
__device__ __forceinline__ int64_t ceil_to(int64_t x, int64_t a) { return (x + a - 1) & ~(a - 1); }

// Geometry of one tile: its shard range [s0, s1) (inside the 2048-element block
// at t0), the full-layout shift delta, and the 16-byte-aligned sub-ranges the
// bulk copies bring in: state [as, bs) (shard side), gradients [ag, bg) (full
// side), staged at shared offset (x - t0) and (f - gbase) respectively.  q is the
// first replica of a per-replica item.
struct TileGeom {
    int64_t t0, s0, s1, delta, as, bs, ag, bg, gbase;
    int32_t q;
};

template <typename GT>
__device__ __forceinline__ TileGeom tile_geom(const Seg& sg, int64_t gt) {
    constexpr int64_t E = 16 / sizeof(GT);      // gradient elements per 16 bytes
    TileGeom g;
    g.t0 = (seg_vec0(sg.shard) + (gt - sg.tile0) * kThreads) * kVec;
    const int64_t hi = sg.shard + sg.len;
    g.s0 = g.t0 > sg.shard ? g.t0 : sg.shard;
    g.s1 = (g.t0 + kTileElems) < hi ? (g.t0 + kTileElems) : hi;
    g.delta = sg.full - sg.shard;
    g.as = ceil_to(g.s0, 4);
    g.bs = floor_to(g.s1, 4);
    g.ag = ceil_to(g.s0 + g.delta, E);
    g.bg = floor_to(g.s1 + g.delta, E);
    g.gbase = floor_to(g.t0 + g.delta, E);
    g.q = 0;
    return g;
}

// Four gradient elements at shared element offset o (GT elements) of one staged
// slice, as fp32; r = o mod 4 is uniform over the item.
__device__ __forceinline__ float4 smem_grad4(const unsigned char* base, int o, const float*) {
    const float* p = reinterpret_cast<const float*>(base);
    const int r = o & 3;
    const float4 a = *reinterpret_cast<const float4*>(p + (o - r));
    if (r == 0) return a;
    const float4 b = *reinterpret_cast<const float4*>(p + (o - r) + 4);
    if (r == 1) return make_float4(a.y, a.z, a.w, b.x);
    if (r == 2) return make_float4(a.z, a.w, b.x, b.y);
    return make_float4(a.w, b.x, b.y, b.z);
}
__device__ __forceinline__ float4 smem_grad4(const unsigned char* base, int o, const uint16_t*) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(base);
    const int r = o & 3;
    const uint2 a = *reinterpret_cast<const uint2*>(p + (o - r));
    uint32_t w0, w1;
    if (r == 0) {
        w0 = a.x; w1 = a.y;
    } else {
        const uint2 b = *reinterpret_cast<const uint2*>(p + (o - r) + 4);
        if (r == 1) { w0 = __funnelshift_r(a.x, a.y, 16); w1 = __funnelshift_r(a.y, b.x, 16); }
        else if (r == 2) { w0 = a.y; w1 = b.x; }
        else { w0 = __funnelshift_r(a.y, b.x, 16); w1 = __funnelshift_r(b.x, b.y, 16); }
    }
    return make_float4(bf16lo(w0), bf16hi(w0), bf16lo(w1), bf16hi(w1));
}
template <typename GT>
__device__ __forceinline__ float4 grad4(const unsigned char* base, int o) {
    return smem_grad4(base, o, static_cast<const GT*>(nullptr));
}

__device__ __forceinline__ float4 lds4(const unsigned char* p) { return *reinterpret_cast<const float4*>(p); }

// Bytes of one staged gradient slice: a tile plus the 16 bytes a shifted window adds.
template <typename GT>
__host__ __device__ constexpr int grank_bytes() { return int(kTileElems * sizeof(GT)) + 16; }

// ----------------------------------------------------------------------------
// The pipeline.  A launch covers n_units units (tiles); CTA b takes units b, b + G,
// b + 2G, ... and, when Pol::groups() = NG > 1, every unit as NG consecutive items
// (group 0 .. NG-1), so that a unit's groups meet the same consumer threads in order
// and a per-thread Pol::Carry can hold partial results from one group to the next.
// Pol supplies, for unit u and group k:
//   geom(u, k, cursor)         the item's geometry (producer side, once per item), resolved
//                              before the producer waits for a free stage when
//                              Pol::kGeomFirst, else after (measured on GB300: the
//                              fused step gains 1-3 % from the first order, HSDP and
//                              accumulation lose 3-4 % with it)
//   bytes(g)                   the bytes its copies bring in
//   issue(g, stage, bar, lane) its copies (all producer lanes call it)
//   consume(g, stage, tid, carry, release)  the consumers' work; release() (all lanes
//                              of each consumer warp call it once) frees the stage;
//                              returns the thread's contribution to a sum
//   finish(tid, sum)           after the consumer's last item, with the thread's sum
// ----------------------------------------------------------------------------
struct NoCarry {};

template <class Pol>
__device__ __forceinline__ void run_pipeline(const Pol& pol, int64_t n_units, int S, int stage_bytes, uint64_t wait_ns) {
    extern __shared__ __align__(128) unsigned char smem[];
    static_assert(16 * kMaxStages + kMaxStages * sizeof(TileGeom) <= kFrontBytes, "front region");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t G = gridDim.x;
    const int NG = pol.groups();
    const int64_t n_mine = blockIdx.x < n_units ? (n_units - blockIdx.x + G - 1) / G * NG : 0;
    const uint32_t full0 = smem_addr(smem), empty0 = full0 + 8 * kMaxStages;
    TileGeom* geo = reinterpret_cast<TileGeom*>(smem + 16 * kMaxStages);
    unsigned char* stage0 = smem + kFrontBytes;

    if (tid == 0) {
        for (int k = 0; k < S; ++k) {
            mbar_init(full0 + 8 * k, 1);                      // the producer's arrive (+ bytes)
            mbar_init(empty0 + 8 * k, kConsumerWarps);        // one arrive per consumer warp
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---- producer warp: item j of this CTA into stage j mod S ----
        int cursor = 0;
        int64_t j = 0;
        for (; j < n_mine; ++j) {
            const int st = int(j % S);
            const int64_t use = j / S;
            // the item's geometry (segment-table reads) before or after the wait for a
            // free stage: Pol::kGeomFirst, chosen per use by measurement
            TileGeom g;
            if (Pol::kGeomFirst) g = pol.geom(blockIdx.x + (j / NG) * G, int(j % NG), cursor);
            if (use > 0 &&
                !__all_sync(0xffffffffu, mbar_wait_bounded(empty0 + 8 * st, uint32_t((use - 1) & 1), wait_ns))) {
                if (lane == 0) atomicOr(&g_wait_error, 1u);
                break;
            }
            if (!Pol::kGeomFirst) g = pol.geom(blockIdx.x + (j / NG) * G, int(j % NG), cursor);
            const uint32_t bar = full0 + 8 * st;
            if (lane == 0) {
                geo[st] = g;                                  // released by the arrive
                mbar_arrive_tx(bar, pol.bytes(g));
            }
            __syncwarp();
            pol.issue(g, smem_addr(stage0 + int64_t(st) * stage_bytes), bar, lane);
        }
        if (j < n_mine) {
            // gave up: let the copies already issued land before the shared memory goes away
            for (int64_t k = j - S > 0 ? j - S : 0; k < j; ++k)
                mbar_wait_bounded(full0 + 8 * int(k % S), uint32_t((k / S) & 1), wait_ns);
        }
        return;
    }

    // ---- consumer warps ----
    double sum = 0.0;
    typename Pol::Carry carry{};
    for (int64_t j = 0; j < n_mine; ++j) {
        const int st = int(j % S);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * st, uint32_t((j / S) & 1), wait_ns))) {
            if (lane == 0) atomicOr(&g_wait_error, 1u);
            return;
        }
        const TileGeom g = geo[st];
        const uint32_t empty = empty0 + 8 * st;
        sum += pol.consume(g, stage0 + int64_t(st) * stage_bytes, tid, carry, [&] {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty);
        });
    }
    pol.finish(tid, sum);
}

// ---- fused reduce-scatter + AdamW + cast ------------------------------------------
// A tile's N replicas come in NG groups of Q (the last may be shorter); the partial
// sums carry over in registers from group to group in rank order, and the last
// group also stages the three state slices and does the update.  NG = 1 unless N
// replicas and the state do not fit two stages.
struct Sum4 {
    float a0, a1, a2, a3;
};

template <typename GT, bool PARAM, bool GOUT>
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

    using Carry = Sum4;
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
            float gg[4] = {__fdiv_rn(carry.a0, sc.nf), __fdiv_rn(carry.a1, sc.nf), __fdiv_rn(carry.a2, sc.nf),
                           __fdiv_rn(carry.a3, sc.nf)};
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
                const float gg = __fdiv_rn(reduce1<GT>(gp, N, e + g.delta), sc.nf);
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
                o0 = __fadd_rn(o0, __fdiv_rn(a0, sc.nf)); o1 = __fadd_rn(o1, __fdiv_rn(a1, sc.nf));
                o2 = __fadd_rn(o2, __fdiv_rn(a2, sc.nf)); o3 = __fadd_rn(o3, __fdiv_rn(a3, sc.nf));
            }
        }
        release();
        if (fast) {
            const float gg[4] = {__fdiv_rn(o0, rf), __fdiv_rn(o1, rf), __fdiv_rn(o2, rf), __fdiv_rn(o3, rf)};
#pragma unroll
            for (int rho = 0; rho < kMaxR; ++rho) {
                if (rho >= R) break;
                float p[4] = {st[3 * rho].x, st[3 * rho].y, st[3 * rho].z, st[3 * rho].w};
                float m[4] = {st[3 * rho + 1].x, st[3 * rho + 1].y, st[3 * rho + 1].z, st[3 * rho + 1].w};
                float v[4] = {st[3 * rho + 2].x, st[3 * rho + 2].y, st[3 * rho + 2].z, st[3 * rho + 2].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) adamw1(sc, gg[k], p[k], m[k], v[k]);
                const int64_t e = rho * copy + x;
                st4(master + e, make_float4(p[0], p[1], p[2], p[3]));
                st4(exp_avg + e, make_float4(m[0], m[1], m[2], m[3]));
                st4(exp_avg_sq + e, make_float4(v[0], v[1], v[2], v[3]));
                if (PARAM)
                    *reinterpret_cast<uint2*>(param + e) = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
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
                    outer = __fadd_rn(outer, __fdiv_rn(acc, sc.nf));
                }
                const float gg = __fdiv_rn(outer, rf);
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
// fp32 replica); the updated parameter is stored into all N replicas.  Owner rows
// keep every tensor congruent to its full offset mod 8 (delta = 0 mod 8).
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
    __device__ double consume(const TileGeom& g, const unsigned char* sb, int tid, Carry&, Release release) const {
        const int c = tid * 4;
        const int64_t x = g.t0 + c, f = x + g.delta;
        const bool live = x + 4 > g.s0 && x < g.s1;
        // owner rows keep delta = 0 mod 8; anything else goes element by element
        const bool fast = x >= g.s0 && x + 4 <= g.s1 && f >= g.ag && f + 4 <= g.bg && (MASTER || (g.delta & 7) == 0);
        float4 pv, mv, vv;
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        if (fast) {
            // p at the shard offset (master) or at the full offset (the owner's replica; gbase = t0 + delta)
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
            const float gg[4] = {__fdiv_rn(a0, sc.nf), __fdiv_rn(a1, sc.nf), __fdiv_rn(a2, sc.nf), __fdiv_rn(a3, sc.nf)};
#pragma unroll
            for (int k = 0; k < 4; ++k) adamw1(sc, gg[k], p[k], m[k], v[k]);
            if (MASTER) st4(master + x, make_float4(p[0], p[1], p[2], p[3]));
            st4(exp_avg + x, make_float4(m[0], m[1], m[2], m[3]));
            st4(exp_avg_sq + x, make_float4(v[0], v[1], v[2], v[3]));
            if (MASTER) {                             // bf16 replicas
                const uint2 w = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
                for (int q = 0; q < N; ++q) *reinterpret_cast<uint2*>(static_cast<uint16_t*>(pr.p[q]) + f) = w;
            } else {                                  // fp32 replicas
                const float4 w = make_float4(p[0], p[1], p[2], p[3]);
                for (int q = 0; q < N; ++q) st4(static_cast<float*>(pr.p[q]) + f, w);
            }
        } else if (live) {
            const int64_t a = x > g.s0 ? x : g.s0;
            const int64_t b = (x + 4) < g.s1 ? (x + 4) : g.s1;
            for (int64_t e = a; e < b; ++e) {
                const int64_t fe = e + g.delta;
                float pp = MASTER ? master[e] : static_cast<const float*>(pr.p[g.q])[fe];
                float mm = exp_avg[e], vv2 = exp_avg_sq[e];
                adamw1(sc, __fdiv_rn(reduce1<GT>(gp, N, fe), sc.nf), pp, mm, vv2);
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
            const float g0 = __fdiv_rn(a0, nf), g1 = __fdiv_rn(a1, nf), g2 = __fdiv_rn(a2, nf), g3 = __fdiv_rn(a3, nf);
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
                const float gg = __fdiv_rn(reduce1<GT>(gp, N, e + g.delta), nf);
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
#pragma unroll
            for (int r = 0; r < kMaxQ; ++r) {
                if (r >= k) break;
                st4(acc[g.q + r] + x, out[r]);
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

// ---- the kernels ------------------------------------------------------------------
template <typename GT, bool PARAM, bool GOUT>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_rs_adamw_staged(RsAdamw<GT, PARAM, GOUT> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns);
}

template <typename GT, bool PARAM>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_hsdp_adamw_staged(HsdpAdamw<GT, PARAM> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns);
}

template <typename GT, bool MASTER>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_zero1_adamw_staged(Zero1Adamw<GT, MASTER> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns);
}

template <bool PARAM>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_adamw_scaled_staged(ScaledAdamw<PARAM> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns);
}

template <typename GT>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_rs_norm_staged(RsNorm<GT> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns);
}

template <typename MT, bool FIRST>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_accumulate_staged(Accumulate<MT, FIRST> pol, int64_t n_items, int S, int stage_bytes, uint64_t wait_ns) {
    run_pipeline(pol, n_items, S, stage_bytes, wait_ns);
}

// ----------------------------------------------------------------------------
// All-gather of the aligned class by bulk copies: global -> shared -> global.
// ----------------------------------------------------------------------------
// Pieces whose full-layout offset is congruent to their shard offset mod 8 start
// 16-byte aligned on both sides, so the bulk-copy engine can move them without a
// thread touching the data: per tile, one cp.async.bulk global->shared and one
// cp.async.bulk shared->global of its aligned interior.  Each CTA is one warp with
// a ring of 4 tile buffers and 2 loads ahead; 4 CTAs per SM.  Measured on GB300
// (bf16, 1-3 GB): as fast as a device copy of the same bytes; 1 or 3 loads ahead,
// 3, 5 or 8 CTAs per SM, or deeper rings were 2-8 % slower, and one CTA per SM
// with 8 loads ahead ran at 40 %.  Lane 0 issues the copies; the at most 7
// elements at each end of a segment that the copies leave out are copied by the
// warp's lanes with plain loads and stores.
constexpr int kURing = 4, kUAhead = 2, kUCtasPerSm = 4;

template <int ES>
__global__ void __launch_bounds__(32)
k_unshard_bulk(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles, const unsigned char* src,
               unsigned char* dst, uint64_t wait_ns) {
    constexpr int64_t E = 16 / ES;              // elements per 16 bytes
    using W = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
    __shared__ __align__(128) unsigned char buf[kURing][kTileElems * ES];
    __shared__ __align__(8) uint64_t bars[kURing];
    const int lane = threadIdx.x;
    const int64_t G = gridDim.x;
    const int64_t n_mine = blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + G - 1) / G : 0;
    const uint32_t bar0 = smem_addr(&bars[0]);
    if (lane == 0) {
        for (int k = 0; k < kURing; ++k) mbar_init(bar0 + 8 * k, 1);
        mbar_fence_init();
    }
    __syncwarp();

    struct Piece { int64_t t0, s0, s1, delta, a, b; };     // tile range, aligned interior [a, b)
    auto piece = [&](int& cur, int64_t j) {
        const int64_t gt = tile_base + blockIdx.x + j * G;
        cur = advance_seg(segs, cur, gt);
        const Seg sg = segs[cur];
        Piece p;
        p.t0 = (seg_vec0(sg.shard) + (gt - sg.tile0) * kThreads) * kVec;
        const int64_t hi = sg.shard + sg.len;
        p.s0 = p.t0 > sg.shard ? p.t0 : sg.shard;
        p.s1 = (p.t0 + kTileElems) < hi ? (p.t0 + kTileElems) : hi;
        p.delta = sg.full - sg.shard;
        p.a = ceil_to(p.s0, E);
        p.b = floor_to(p.s1, E);
        return p;
    };
    int load_cur = 0, store_cur = 0;             // segment cursors of the two sides
    auto load = [&](int64_t j) {
        const Piece p = piece(load_cur, j);
        if (lane == 0) {
            const int k = int(j % kURing);
            const uint32_t bytes = p.b > p.a ? uint32_t(p.b - p.a) * ES : 0u;
            mbar_arrive_tx(bar0 + 8 * k, bytes);
            if (bytes) bulk_g2s(smem_addr(&buf[k][(p.a - p.t0) * ES]), src + p.a * ES, bytes, bar0 + 8 * k);
        }
    };
    for (int64_t j = 0; j < n_mine && j < kUAhead; ++j) load(j);
    int64_t j = 0;
    bool ok = true;
    for (; j < n_mine; ++j) {
        if (j + kUAhead < n_mine) {
            // buffer (j + ahead) mod ring was last stored from by tile j + ahead - ring
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kURing - kUAhead - 1) : "memory");
            __syncwarp();
            load(j + kUAhead);
        }
        const int k = int(j % kURing);
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * k, uint32_t((j / kURing) & 1), wait_ns));
        if (!ok) break;
        const Piece p = piece(store_cur, j);
        if (lane == 0) {
            if (p.b > p.a) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                             ::"l"(dst + (p.a + p.delta) * ES), "r"(smem_addr(&buf[k][(p.a - p.t0) * ES])),
                               "r"(uint32_t(p.b - p.a) * ES)
                             : "memory");
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        // the ends the 16-byte copies leave out
        const int64_t lo_end = p.a < p.s1 ? (p.a > p.s0 ? p.a : p.s0) : p.s1;
        for (int64_t e = p.s0 + lane; e < lo_end; e += 32)
            reinterpret_cast<W*>(dst)[e + p.delta] = reinterpret_cast<const W*>(src)[e];
        for (int64_t e = (p.b > lo_end ? p.b : lo_end) + lane; e < p.s1; e += 32)
            reinterpret_cast<W*>(dst)[e + p.delta] = reinterpret_cast<const W*>(src)[e];
    }
    if (!ok && lane == 0) {
        atomicOr(&g_wait_error, 1u);
        // loads already issued must land before the shared memory goes away
        for (int64_t q = j + 1; q < n_mine && q < j + kUAhead; ++q)
            mbar_wait_bounded(bar0 + 8 * int(q % kURing), uint32_t((q / kURing) & 1), wait_ns);
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
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

// ---- host side ------------------------------------------------------------------
// Opt-in shared memory per block of each device, queried once.
std::atomic<int> g_optin[64];

int optin_smem(int dev) {
    if (dev < 0 || dev >= 64) return 0;
    int v = g_optin[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    g_optin[dev].store(v, std::memory_order_relaxed);
    return v;
}

// Stages for a stage of `stage_bytes`: as many as keep about 96 KB in flight (the
// stages beyond the one being consumed), between 2 and kMaxStages, within the
// opt-in shared memory; 0 if two do not fit.  Measured on GB300 (fused step): about
// 50-100 KB in flight per SM streams best; 3-4 stages of 57 KB lost up to 10 % of
// the bandwidth, fewer than 40 KB in flight lost 8 %.
int stage_count(int stage_bytes, int dev) {
    const int avail = optin_smem(dev) - kFrontBytes;
    const int fit = avail > 0 ? avail / stage_bytes : 0;
    int want = kInFlightBytes / stage_bytes + 1;
    want = want < 2 ? 2 : (want > kMaxStages ? kMaxStages : want);
    const int s = fit < want ? fit : want;
    return s >= 2 ? s : 0;
}

std::mutex g_st_mu;
std::map<std::pair<const void*, int>, std::pair<int, int>> g_st_cache;   // (kernel, dev) -> (SMs, smem set)

// One CTA of 544 threads per SM (at most one per item).
template <typename K, typename Pol>
cudaError_t launch_pipeline(K kernel, const Pol& pol, int64_t n_items, int stage_bytes, uint64_t wait_ns,
                            cudaStream_t st, int* grid_out = nullptr) {
    if (grid_out) *grid_out = 0;
    if (n_items <= 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int S = stage_count(stage_bytes, dev);
    if (S < 2) return cudaErrorInvalidValue;
    const int smem = kFrontBytes + S * stage_bytes;
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    int sms = 0, set = 0;
    {
        std::lock_guard<std::mutex> lk(g_st_mu);
        auto it = g_st_cache.find(key);
        if (it != g_st_cache.end()) { sms = it->second.first; set = it->second.second; }
    }
    if (set < smem) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lk(g_st_mu);
        g_st_cache[key] = std::make_pair(sms, smem);
    }
    const int64_t blocks = n_items < sms ? n_items : (sms > 0 ? sms : 1);
    kernel<<<int(blocks), kStThreads + 32, smem, st>>>(pol, n_items, S, stage_bytes, wait_ns);
    if (grid_out) *grid_out = int(blocks);
    return cudaGetLastError();
}

int rs_stage_bytes(int N, bool bf16) { return 3 * kStateBytes + N * (bf16 ? grank_bytes<uint16_t>() : grank_bytes<float>()); }

// Replica groups of the fused step: one group when all N replicas and the state fit
// two stages, else the fewest groups (of equal size, rounded up) that do.
void rs_groups(int N, bool bf16, int dev, int* Q, int* NG) {
    int ng = 1;
    while (ng < N && stage_count(rs_stage_bytes((N + ng - 1) / ng, bf16), dev) < 2) ++ng;
    *NG = ng;
    *Q = (N + ng - 1) / ng;
}
int hsdp_stage_bytes(int N, int R, bool bf16) {
    return 3 * R * kStateBytes + R * N * (bf16 ? grank_bytes<uint16_t>() : grank_bytes<float>());
}
int norm_stage_bytes(int N, bool bf16) { return N * (bf16 ? grank_bytes<uint16_t>() : grank_bytes<float>()); }
int acc_stage_bytes(int Q, bool bf16, bool first) { return Q * (int(kTileElems) * (bf16 ? 2 : 4) + (first ? 0 : kStateBytes)); }

bool fits(int stage_bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    return stage_count(stage_bytes, dev) >= 2;
}

}  // namespace

bool staged_fits(int N, bool grad_bf16) {
    // with replica groups, any N whose single-replica stage fits two stages
    return N >= 1 && N <= kMaxRanks && fits(rs_stage_bytes(1, grad_bf16));
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
        return launch_pipeline(k_adamw_scaled_staged<true>, pol, n_tiles, sb, wait_ns, st);
    }
    ScaledAdamw<false> pol{segs, tile_base, gshard, coef, master, m, v, param, sc};
    return launch_pipeline(k_adamw_scaled_staged<false>, pol, n_tiles, sb, wait_ns, st);
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
        return launch_pipeline(k_zero1_adamw_staged<GT, M>, pol, n_tiles, sb, wait_ns, st);
    };
    if (grad_bf16) return master ? go(uint16_t{}, std::true_type{}) : go(uint16_t{}, std::false_type{});
    return master ? go(float{}, std::true_type{}) : go(float{}, std::false_type{});
}

int norm_staged_partials(int64_t n_tiles) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = n_tiles < sms ? n_tiles : sms;
    return int(blocks) * kConsumerWarps;
}

cudaError_t launch_rs_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                   const GradPtrs& gp, int N, float* master, float* m, float* v, uint16_t* param,
                                   float* gout, const AdamScal& sc, uint64_t wait_ns, cudaStream_t st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int Q = N, NG = 1;
    rs_groups(N, grad_bf16, dev, &Q, &NG);
    const int sb = rs_stage_bytes(Q, grad_bf16);
    auto go = [&](auto tag_gt, auto tag_p, auto tag_g) {
        using GT = decltype(tag_gt);
        constexpr bool P = decltype(tag_p)::value, O = decltype(tag_g)::value;
        RsAdamw<GT, P, O> pol{segs, tile_base, gp, N, Q, NG, master, m, v, param, gout, sc};
        return launch_pipeline(k_rs_adamw_staged<GT, P, O>, pol, n_tiles, sb, wait_ns, st);
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

cudaError_t launch_hsdp_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                     const GradPtrs& gp, int N, int R, int64_t copy, float* master, float* m,
                                     float* v, uint16_t* param, const AdamScal& sc, float rf, uint64_t wait_ns,
                                     cudaStream_t st) {
    const int sb = hsdp_stage_bytes(N, R, grad_bf16);
    auto go = [&](auto tag_gt, auto tag_p) {
        using GT = decltype(tag_gt);
        constexpr bool P = decltype(tag_p)::value;
        HsdpAdamw<GT, P> pol{segs, tile_base, gp, N, R, copy, master, m, v, param, sc, rf};
        return launch_pipeline(k_hsdp_adamw_staged<GT, P>, pol, n_tiles, sb, wait_ns, st);
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
    int Q = kInFlightBytes / per;
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
        return launch_pipeline(k_accumulate_staged<MT, FIRST>, pol, n_items, sb, wait_ns, st);
    };
    if (micro_bf16) return first ? go(uint16_t{}, std::true_type{}) : go(uint16_t{}, std::false_type{});
    return first ? go(float{}, std::true_type{}) : go(float{}, std::false_type{});
}

cudaError_t launch_unshard_bulk(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool bf16, const void* src,
                                void* dst, uint64_t wait_ns, cudaStream_t st) {
    if (n_tiles <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int64_t blocks = int64_t(sms > 0 ? sms : 1) * kUCtasPerSm;
    if (blocks > n_tiles) blocks = n_tiles;
    const auto* s8 = static_cast<const unsigned char*>(src);
    auto* d8 = static_cast<unsigned char*>(dst);
    if (bf16) k_unshard_bulk<2><<<int(blocks), 32, 0, st>>>(segs, tile_base, n_tiles, s8, d8, wait_ns);
    else k_unshard_bulk<4><<<int(blocks), 32, 0, st>>>(segs, tile_base, n_tiles, s8, d8, wait_ns);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t wait_ns, cudaStream_t st) {
    k_wait_selftest<<<1, 32, 0, st>>>(wait_ns);
    return cudaGetLastError();
}

cudaError_t take_wait_error(unsigned int* flag) {
    *flag = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_wait_error, sizeof(unsigned int));
    if (e != cudaSuccess || *flag == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_wait_error, &zero, sizeof(unsigned int));
}

}  // namespace fsdp
