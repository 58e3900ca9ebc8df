// staged.cu -- kernels whose inputs the bulk-copy (TMA) engine stages in shared
// memory (sm_103a): the fused reduce-scatter + AdamW + bf16 recast, and the
// all-gather of the aligned class (k_unshard_bulk, further down).
//
// Same contract and arithmetic as k_rs_adamw in kernels.cu ("NCCL ZeRO/FSDP state
// sharding", "ZeRO-2 方向"/"ZeRO-3 方向": each rank keeps only the 1/N slice of
// the reduce-scattered gradient and updates its own optimizer state with it; "第18章
// FSDP" §18.16: fp32 reduce, AdamW on the fp32 master, cast to param_dtype).  What
// differs is how the bytes move:
//
//  * One CTA per SM, persistent over its tiles (a tile is 2048 shard elements of
//    one segment, the tiling of the segment tables), with 2 to 4 pipeline stages
//    in shared memory, as many as keep about 96 KB in flight; a stage holds the
//    tile's fp32 master/exp_avg/exp_avg_sq slices and its N gradient slices.
//  * Warp-specialised: one producer warp issues, per tile, one cp.async.bulk per
//    array (N + 3 copies) into a free stage and writes the tile's geometry into the
//    stage header; a "full" mbarrier per stage counts the bytes in (complete_tx).
//    16 consumer warps wait on it, read the stage into registers and release it on
//    an "empty" mbarrier before they compute, so the next copies go out while they
//    do.  No CTA-wide barrier in the loop; the bytes in flight per SM do not depend
//    on registers.
//  * A gradient piece whose full-layout offset is not congruent to its shard offset
//    mod 8 is copied as the 16-byte-aligned window around it and read from shared
//    memory at the offset: no warp shuffle, one kernel for both alignment classes.
//  * Each consumer thread owns 4 consecutive elements of the tile: 16-byte
//    shared-memory reads of the state, 16-byte (fp32) and 8-byte (bf16) global
//    stores that cover whole sectors per warp.  The at most 3 elements at each end
//    of a segment that the 16-byte copies leave out go element by element from
//    global memory.
//
// Every wait on an mbarrier is bounded in time; a warp that gives up records
// FSDP_ETIMEOUT in a device word that fsdp_check_status reads and returns (the
// producer first waits, bounded, for the copies it has in flight), after which the
// CTA's other waits run out in turn.  Nothing else in the kernel waits.
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

constexpr int kStThreads = 512;                 // consumer threads: 4 elements each per tile
constexpr int kConsumerWarps = kStThreads / 32;
constexpr int kMaxStages = 4;
constexpr int kInFlightBytes = 96 * 1024;       // stage bytes in flight per SM to aim for
constexpr int kFrontBytes = 512;                // mbarriers + per-stage tile geometry
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
// Waits for phase `parity` of the barrier to complete, for at most limit_ns
// nanoseconds (and at most 2^24 polls); false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
#pragma unroll 1
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
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
// side), staged at shared offset (x - t0) and (f - gbase) respectively.
struct TileGeom {
    int64_t t0, s0, s1, delta, as, bs, ag, bg, gbase;
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
    return g;
}

// Four gradient elements at shared element offset o (GT elements) of one staged
// slice, as fp32; r = o mod (elements per read) is uniform over the tile.
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

struct StageLayout {
    int n_stages;      // 2..4
    int grank_bytes;   // bytes of one staged gradient slice: 2048 elements + 16
    int stage_bytes;   // 3 * 8192 + N * grank_bytes
};

template <typename GT, bool PARAM, bool GOUT>
__global__ void __launch_bounds__(kStThreads + 32, 1)
k_rs_adamw_staged(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles, GradPtrs gp, int N,
                  float* master, float* exp_avg, float* exp_avg_sq, uint16_t* __restrict__ param,
                  float* __restrict__ gout, AdamScal sc, StageLayout sl, uint64_t wait_ns) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = sl.n_stages;
    const int64_t G = gridDim.x;
    const int64_t n_mine = blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + G - 1) / G : 0;
    // front region: full[S] and empty[S] mbarriers, then one TileGeom per stage
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
        // ---- producer warp: bring tile j of this CTA into stage j mod S ----
        int ps = 0;                                  // segment cursor
        int64_t j = 0;
        for (; j < n_mine; ++j) {
            const int st = int(j % S);
            const int64_t use = j / S;
            if (use > 0 && !__all_sync(0xffffffffu, mbar_wait_bounded(empty0 + 8 * st, uint32_t((use - 1) & 1), wait_ns))) {
                if (lane == 0) atomicOr(&g_wait_error, 1u);
                break;
            }
            const int64_t gt = tile_base + blockIdx.x + j * G;
            ps = advance_seg(segs, ps, gt);
            const TileGeom g = tile_geom<GT>(segs[ps], gt);
            const uint32_t bar = full0 + 8 * st;
            const uint32_t sbase = smem_addr(stage0 + int64_t(st) * sl.stage_bytes);
            const uint32_t sbytes = g.bs > g.as ? uint32_t(g.bs - g.as) * 4u : 0u;
            const uint32_t gbytes = g.bg > g.ag ? uint32_t(g.bg - g.ag) * uint32_t(sizeof(GT)) : 0u;
            if (lane == 0) {
                geo[st] = g;                                          // released by the arrive
                mbar_arrive_tx(bar, 3u * sbytes + uint32_t(N) * gbytes);
            }
            __syncwarp();
            for (int k = lane; k < N + 3; k += 32) {
                if (k < 3) {
                    const float* arr = k == 0 ? master : (k == 1 ? exp_avg : exp_avg_sq);
                    if (sbytes) bulk_g2s(sbase + k * kStateBytes + uint32_t(g.as - g.t0) * 4u, arr + g.as, sbytes, bar);
                } else if (gbytes) {
                    const int q = k - 3;
                    bulk_g2s(sbase + 3 * kStateBytes + q * sl.grank_bytes +
                                 uint32_t(g.ag - g.gbase) * uint32_t(sizeof(GT)),
                             static_cast<const GT*>(gp.p[q]) + g.ag, gbytes, bar);
                }
            }
        }
        if (j < n_mine) {
            // gave up: let the copies already issued land before the CTA's shared memory goes away
            for (int64_t k = j - S > 0 ? j - S : 0; k < j; ++k)
                mbar_wait_bounded(full0 + 8 * int(k % S), uint32_t((k / S) & 1), wait_ns);
        }
        return;
    }

    // ---- consumer warps: 4 elements per thread per tile ----
    const int c = tid * 4;
    for (int64_t j = 0; j < n_mine; ++j) {
        const int st = int(j % S);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * st, uint32_t((j / S) & 1), wait_ns))) {
            if (lane == 0) atomicOr(&g_wait_error, 1u);
            return;
        }
        const TileGeom g = geo[st];
        const unsigned char* sb = stage0 + int64_t(st) * sl.stage_bytes;
        const int64_t x = g.t0 + c;
        const int64_t f = x + g.delta;
        const bool live = x + 4 > g.s0 && x < g.s1;
        const bool fast = x >= g.s0 && x + 4 <= g.s1 && f >= g.ag && f + 4 <= g.bg;
        float4 pv, mv, vv;
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        if (fast) {
            // everything this thread needs from the stage, into registers
            pv = *reinterpret_cast<const float4*>(sb + 0 * kStateBytes + c * 4);
            mv = *reinterpret_cast<const float4*>(sb + 1 * kStateBytes + c * 4);
            vv = *reinterpret_cast<const float4*>(sb + 2 * kStateBytes + c * 4);
            const int o = int(f - g.gbase);
            const unsigned char* gs = sb + 3 * kStateBytes;
#pragma unroll 4
            for (int q = 0; q < N; ++q) {            // fixed rank order
                const float4 x4 = smem_grad4(gs + q * sl.grank_bytes, o, static_cast<const GT*>(nullptr));
                a0 = __fadd_rn(a0, x4.x); a1 = __fadd_rn(a1, x4.y);
                a2 = __fadd_rn(a2, x4.z); a3 = __fadd_rn(a3, x4.w);
            }
        }
        // the stage is free for the producer once the whole warp has read it
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
        if (fast) {
            float p[4] = {pv.x, pv.y, pv.z, pv.w};
            float m[4] = {mv.x, mv.y, mv.z, mv.w};
            float v[4] = {vv.x, vv.y, vv.z, vv.w};
            float gg[4] = {__fdiv_rn(a0, sc.nf), __fdiv_rn(a1, sc.nf), __fdiv_rn(a2, sc.nf), __fdiv_rn(a3, sc.nf)};
#pragma unroll
            for (int k = 0; k < 4; ++k) adamw1(sc, gg[k], p[k], m[k], v[k]);
            st4(master + x, make_float4(p[0], p[1], p[2], p[3]));
            st4(exp_avg + x, make_float4(m[0], m[1], m[2], m[3]));
            st4(exp_avg_sq + x, make_float4(v[0], v[1], v[2], v[3]));
            if (PARAM)
                *reinterpret_cast<uint2*>(param + x) = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
            if (GOUT) st4(gout + x, make_float4(gg[0], gg[1], gg[2], gg[3]));
        } else if (live) {
            // segment edge: element by element from global memory
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
    }
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
std::mutex g_st_mu;
std::map<std::pair<const void*, int>, std::pair<int, int>> g_st_cache;   // (kernel, dev) -> (SMs, smem set)

int optin_smem(int dev) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return v;
}

StageLayout stage_layout(int N, bool grad_bf16, int dev) {
    StageLayout sl{};
    const int gs = grad_bf16 ? 2 : 4;
    sl.grank_bytes = int(kTileElems) * gs + 16;
    sl.stage_bytes = 3 * kStateBytes + N * sl.grank_bytes;
    const int avail = optin_smem(dev) - kFrontBytes;
    const int fit = avail > 0 ? avail / sl.stage_bytes : 0;
    // Stages beyond the one being consumed are in flight.  Measured on GB300: about
    // 50-100 KB in flight per SM streams best; more (3-4 stages of 57 KB) lost up to
    // 10 % of the bandwidth, fewer than 40 KB lost 8 %.
    int want = kInFlightBytes / sl.stage_bytes + 1;
    want = want < 2 ? 2 : (want > kMaxStages ? kMaxStages : want);
    sl.n_stages = fit < want ? fit : want;
    return sl;
}

template <typename K>
cudaError_t launch_staged_k(K kernel, const Seg* segs, int64_t tile_base, int64_t n_tiles, const GradPtrs& gp,
                            int N, float* master, float* m, float* v, uint16_t* param, float* gout,
                            const AdamScal& sc, const StageLayout& sl, uint64_t wait_ns, int dev, cudaStream_t st) {
    const int smem = kFrontBytes + sl.n_stages * sl.stage_bytes;
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    int sms = 0, set = 0;
    {
        std::lock_guard<std::mutex> lk(g_st_mu);
        auto it = g_st_cache.find(key);
        if (it != g_st_cache.end()) { sms = it->second.first; set = it->second.second; }
    }
    if (set < smem) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        std::lock_guard<std::mutex> lk(g_st_mu);
        g_st_cache[key] = std::make_pair(sms, smem);
    }
    const int64_t blocks = n_tiles < sms ? n_tiles : (sms > 0 ? sms : 1);
    kernel<<<int(blocks), kStThreads + 32, smem, st>>>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc, sl,
                                                  wait_ns);
    return cudaGetLastError();
}

template <typename GT>
cudaError_t launch_staged_t(const Seg* segs, int64_t tile_base, int64_t n_tiles, const GradPtrs& gp, int N,
                            float* master, float* m, float* v, uint16_t* param, float* gout, const AdamScal& sc,
                            const StageLayout& sl, uint64_t wait_ns, int dev, cudaStream_t st) {
    if (param && gout)
        return launch_staged_k(k_rs_adamw_staged<GT, true, true>, segs, tile_base, n_tiles, gp, N, master, m, v, param,
                               gout, sc, sl, wait_ns, dev, st);
    if (param)
        return launch_staged_k(k_rs_adamw_staged<GT, true, false>, segs, tile_base, n_tiles, gp, N, master, m, v,
                               param, gout, sc, sl, wait_ns, dev, st);
    if (gout)
        return launch_staged_k(k_rs_adamw_staged<GT, false, true>, segs, tile_base, n_tiles, gp, N, master, m, v,
                               param, gout, sc, sl, wait_ns, dev, st);
    return launch_staged_k(k_rs_adamw_staged<GT, false, false>, segs, tile_base, n_tiles, gp, N, master, m, v, param,
                           gout, sc, sl, wait_ns, dev, st);
}

}  // namespace

bool staged_fits(int N, bool grad_bf16) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    return stage_layout(N, grad_bf16, dev).n_stages >= 2;
}

cudaError_t launch_rs_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                   const GradPtrs& gp, int N, float* master, float* m, float* v, uint16_t* param,
                                   float* gout, const AdamScal& sc, uint64_t wait_ns, cudaStream_t st) {
    if (n_tiles <= 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const StageLayout sl = stage_layout(N, grad_bf16, dev);
    if (sl.n_stages < 2) return cudaErrorInvalidValue;
    return grad_bf16 ? launch_staged_t<uint16_t>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc, sl,
                                                 wait_ns, dev, st)
                     : launch_staged_t<float>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc, sl,
                                              wait_ns, dev, st);
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
