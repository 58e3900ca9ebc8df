// pipeline.cuh -- the bulk-copy pipeline shared by the staged kernels (sm_103a).
//
// A persistent CTA per SM walks its work items (a tile of 2048 elements of one
// segment, or a tile and a group of replicas); per item, a producer warp issues one
// cp.async.bulk global -> shared per input array into a free stage and writes the
// item's geometry into the stage header, and a "full" mbarrier per stage counts the
// bytes in (complete_tx).  16 consumer warps wait on it, read their 4 elements of
// every staged array into registers, release the stage on an "empty" mbarrier (one
// arrive per warp) and only then compute and store, so the next copies go out while
// they do.  No CTA-wide barrier in the loop; the bytes in flight per SM do not
// depend on registers.  A gradient piece whose full-layout offset is not congruent
// to its shard offset mod 8 is copied as the 16-byte-aligned window around it and
// read from shared memory at its offset: no warp shuffle.
//
// Every wait on an mbarrier is bounded in time; a warp that gives up records
// FSDP_ETIMEOUT in this translation unit's device word (g_wait_error, read and
// cleared through take_local_wait_error) and returns (a producer first waits,
// bounded, for the copies it has in flight), after which the CTA's other waits run
// out in turn.
//
// Everything here has internal linkage: each translation unit that includes it has
// its own copy, its own wait word and its own launch-attribute cache.
#pragma once

#include <atomic>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "device_ops.cuh"
#include "staged.hpp"

namespace fsdp {
namespace {

// Nonzero once a bounded wait of this translation unit's kernels gave up.
__device__ unsigned int g_wait_error = 0;

constexpr int kStThreads = 512;                 // consumer threads: 4 elements each per item
constexpr int kConsumerWarps = kStThreads / 32;
constexpr int kMaxStages = 8;
constexpr int kInFlightBytes = 116 * 1024;      // stage bytes in flight per SM to aim for
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

// Shared -> global bulk copy in the current bulk async-group (16-byte aligned both
// sides, bytes a multiple of 16), the group commit, and the waits on the groups.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ int64_t floor_to(int64_t x, int64_t a) { return x & ~(a - 1); }   // a: power of 2
__device__ __forceinline__ int64_t ceil_to(int64_t x, int64_t a) { return (x + a - 1) & ~(a - 1); }

// Geometry of one tile: its shard range [s0, s1) (inside the 2048-element block
// at t0), the full-layout shift delta, and the 16-byte-aligned sub-ranges the
// bulk copies bring in: state [as, bs) (shard side), gradients [ag, bg) (full
// side), staged at shared offset (x - t0) and (f - gbase) respectively.  q is the
// first replica of a per-replica item; end marks the item that tells the consumers
// a launch with claimed units has no more work for their CTA.
struct TileGeom {
    int64_t t0, s0, s1, delta, as, bs, ag, bg, gbase;
    int32_t q, end;
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
    g.end = 0;
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
// The pipeline.  A launch covers n_units units (tiles).  Without claim counters CTA b
// takes units b, b + G, b + 2G, ...  With them (claim = a zeroed pair of device words:
// units claimed, CTAs done) the producer of CTA b starts on the units [b B, b B + B)
// (B = claim_batch), then takes the next B consecutive units from G B + claim[0] whenever
// it has used up the last ones, so that the SMs that stream faster take more units
// (measured on GB300: with the static split, the CTAs of the accumulation and HSDP
// kernels on the same workload ended up to 22 % apart, the same SMs always first).  The
// producer asks for its next batch while it issues the current one's copies (a batch
// covers a microsecond of streaming or more, so the atomic's round trip stays hidden);
// after its last unit it queues an item marked end, which tells the consumers to stop,
// and the last producer to count itself out in claim[1] clears both words for the
// slot's next launch.  Either way, when Pol::groups() = NG > 1, every unit is NG
// consecutive items (group 0 .. NG-1), so that a unit's groups meet the same consumer
// threads in order and a per-thread Pol::Carry can hold partial results from one group
// to the next.
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

// A policy with `static constexpr bool kPrologue = true` gets prologue(tid) called by
// every consumer thread once, before its first item, followed by a barrier among the
// consumer warps only (the producer is not held): for per-launch data the consumers
// need, read once per CTA into shared memory.
template <class P, class = void>
struct PrologueOf {
    static constexpr bool value = false;
};
template <class P>
struct PrologueOf<P, std::void_t<decltype(P::kPrologue)>> {
    static constexpr bool value = P::kPrologue;
};

// Front region: stage barriers, stage geometry and, at its end, 64 bytes a policy may
// use for per-launch data (policy_front()).
constexpr int kGeoOff = 16 * kMaxStages;
constexpr int kPolicyFrontOff = kFrontBytes - 64;
static_assert(kGeoOff + kMaxStages * int(sizeof(TileGeom)) <= kPolicyFrontOff, "front region");

__device__ __forceinline__ unsigned char* policy_front() {
    extern __shared__ __align__(128) unsigned char smem[];
    return smem + kPolicyFrontOff;
}

template <class Pol>
__device__ __forceinline__ void run_pipeline(const Pol& pol, int64_t n_units, int S, int stage_bytes, uint64_t wait_ns,
                                             unsigned int* claim, int claim_batch) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t G = gridDim.x;
    const int NG = pol.groups();
    // items of this CTA: known with the static split, else until the end item
    const int64_t n_mine = claim ? INT64_MAX
                                 : (blockIdx.x < n_units ? (n_units - blockIdx.x + G - 1) / G * NG : 0);
    const uint32_t full0 = smem_addr(smem), empty0 = full0 + 8 * kMaxStages;
    TileGeom* geo = reinterpret_cast<TileGeom*>(smem + kGeoOff);
    unsigned char* stage0 = smem + kFrontBytes;

    if (tid == 0) {
        for (int k = 0; k < S; ++k) {
            mbar_init(full0 + 8 * k, 1);                      // the producer's arrive (+ bytes)
            mbar_init(empty0 + 8 * k, kConsumerWarps);        // one arrive per consumer warp
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();

    if (warp == kConsumerWarps) {
        // ---- producer warp: item j of this CTA into stage j mod S ----
        int cursor = 0;
        int64_t j = 0, u = -1, u_end = 0;                     // unit; end of the current batch
        // the first batch is the CTA's own, [b B, b B + B): no claim to wait for at the start;
        // the claims hand out the units from G B on
        int64_t first = int64_t(blockIdx.x) * claim_batch;
        unsigned int next = 0;                                // the claim in flight (lane 0)
        if (claim && lane == 0) next = atomicAdd(claim, unsigned(claim_batch));
        bool gave_up = false;
        for (;; ++j) {
            const int k = int(j % NG);
            bool end;
            if (claim) {
                if (k == 0 && ++u >= u_end) {                 // batch used up: the claim taken before
                    int64_t c = first;
                    if (first < 0) {
                        c = G * claim_batch + int64_t(__shfl_sync(0xffffffffu, next, 0));
                        if (c < n_units && lane == 0) next = atomicAdd(claim, unsigned(claim_batch));
                    }
                    first = -1;
                    u = c;
                    u_end = c + claim_batch < n_units ? c + claim_batch : n_units;
                }
                end = u >= n_units;
            } else {
                if (j >= n_mine) break;
                u = blockIdx.x + (j / NG) * G;
                end = false;
            }
            const int st = int(j % S);
            const int64_t use = j / S;
            // the item's geometry (segment-table reads) before or after the wait for a
            // free stage: Pol::kGeomFirst, chosen per use by measurement
            TileGeom g;
            if (Pol::kGeomFirst && !end) g = pol.geom(u, k, cursor);
            if (use > 0 &&
                !__all_sync(0xffffffffu, mbar_wait_bounded(empty0 + 8 * st, uint32_t((use - 1) & 1), wait_ns))) {
                gave_up = true;
                break;
            }
            const uint32_t bar = full0 + 8 * st;
            if (end) {                                        // no more units: tell the consumers
                if (lane == 0) {
                    geo[st].end = 1;                          // released by the arrive
                    mbar_arrive(bar);
                }
                __syncwarp();
                ++j;
                break;
            }
            if (!Pol::kGeomFirst) g = pol.geom(u, k, cursor);
            g.end = 0;
            if (lane == 0) {
                geo[st] = g;                                  // released by the arrive
                mbar_arrive_tx(bar, pol.bytes(g));
            }
            __syncwarp();
            pol.issue(g, smem_addr(stage0 + int64_t(st) * stage_bytes), bar, lane);
        }
        if (gave_up) {
            // let the copies already issued land before the shared memory goes away
            if (lane == 0) atomicOr(&g_wait_error, 1u);
            for (int64_t k = j - S > 0 ? j - S : 0; k < j; ++k)
                mbar_wait_bounded(full0 + 8 * int(k % S), uint32_t((k / S) & 1), wait_ns);
        }
        if (claim && lane == 0) {
            // done claiming (here on every path): the last CTA out leaves the pair at zero
            __threadfence();
            if (atomicAdd(claim + 1, 1u) == unsigned(G) - 1u) {
                atomicExch(claim, 0u);
                atomicExch(claim + 1, 0u);
            }
        }
        return;
    }

    // ---- consumer warps ----
    if constexpr (PrologueOf<Pol>::value) {
        pol.prologue(tid);
        asm volatile("bar.sync 1, %0;" ::"n"(kStThreads) : "memory");   // the consumer warps only
    }
    double sum = 0.0;
    typename Pol::Carry carry{};
    for (int64_t j = 0; j < n_mine; ++j) {
        const int st = int(j % S);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * st, uint32_t((j / S) & 1), wait_ns))) {
            if (lane == 0) atomicOr(&g_wait_error, 1u);
            return;
        }
        const TileGeom g = geo[st];
        if (g.end) break;                                     // only with claimed units
        const uint32_t empty = empty0 + 8 * st;
        auto release = [&] {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty);
        };
        sum += pol.consume(g, stage0 + int64_t(st) * stage_bytes, tid, carry, release);
    }
    pol.finish(tid, sum);
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

// Stages for a stage of `stage_bytes`: as many as keep about `in_flight` bytes in flight
// (the stages beyond the one being consumed), 4 for stages under 36 KB, between 2 and
// kMaxStages, within the opt-in shared memory; 0 if two do not fit.  Measured on GB300,
// with the tiles claimed from a counter: the fused step ran 1-3 % faster with 3 stages of
// 49-57 KB than with 2 (mlp128m 195.8 against 199.0 us, llama4 4.671 against 4.725 ms,
// dim0_n6 1.310 against 1.351 ms) and 0.9 % slower with 4 stages of 40 KB than with 3
// (fp32, N = 2); 41 KB stages (bf16, N = 4) ran the same with 3 or 4, stages of 33 KB
// (bf16, N = 2) best with 4.  The default target (116 KB) gives 3 stages from 40 to
// 57 KB; the accumulation passes 128 KB (3 stages of 64 KB: 0.4 % faster than 2), ZeRO-1
// 96 KB (2 stages of 57 KB: 0.5 % faster than 3).  (With the tiles split statically,
// 3-4 stages of 57 KB had lost up to 10 %.)
int stage_count(int stage_bytes, int dev, int extra_bytes = 0, int in_flight = kInFlightBytes) {
    const int avail = optin_smem(dev) - kFrontBytes - extra_bytes;
    const int fit = avail > 0 ? avail / stage_bytes : 0;
    int want = stage_bytes < 36 * 1024 ? 4 : in_flight / stage_bytes + 1;
    want = want < 2 ? 2 : (want > kMaxStages ? kMaxStages : want);
    const int s = fit < want ? fit : want;
    return s >= 2 ? s : 0;
}

std::mutex g_st_mu;
std::map<std::pair<const void*, int>, std::pair<int, int>> g_st_cache;   // (kernel, dev) -> (SMs, smem set)

// Threads of a pipeline CTA: the consumers and the producer warp.
constexpr int kPipelineThreads = kStThreads + 32;

// Launches with at least this many units per CTA claim their units (claims.cu); shorter
// ones split them statically (a claim costs an atomic, and the host an event).  A claim
// takes ceil(kClaimBytes / stage_bytes) consecutive units: about 96 KB of stage, which a
// CTA streams in 2 us or more, well over the atomic's round trip.
constexpr int64_t kClaimMinUnitsPerCta = 8;
constexpr int kClaimBytes = 96 * 1024;

// One CTA of 544 threads per SM (at most one per item).  With claims = true the units
// are claimed from a counter pair of the device's ring where one is free.
template <typename K, typename Pol>
cudaError_t launch_pipeline(K kernel, const Pol& pol, int64_t n_items, int stage_bytes, uint64_t wait_ns,
                            cudaStream_t st, int* grid_out = nullptr, bool claims = false,
                            int in_flight = kInFlightBytes) {
    if (grid_out) *grid_out = 0;
    if (n_items <= 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int S = stage_count(stage_bytes, dev, 0, in_flight);
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
    unsigned int* claim = nullptr;
    int slot = -1, cdev = -1;
    if (claims && n_items >= kClaimMinUnitsPerCta * blocks &&
        n_items < (int64_t(1) << 31))
        claim = claim_acquire(st, &slot, &cdev);
    const int batch = (kClaimBytes + stage_bytes - 1) / stage_bytes;
    e = launch(kernel, dim3(unsigned(blocks)), dim3(kPipelineThreads), size_t(smem), st, pol, n_items, S,
               stage_bytes, wait_ns, claim, batch);
    claim_release(slot, cdev, st, e == cudaSuccess);
    if (e == cudaSuccess && grid_out) *grid_out = int(blocks);
    return e;
}

int rs_stage_bytes(int N, bool bf16) { return 3 * kStateBytes + N * (bf16 ? grank_bytes<uint16_t>() : grank_bytes<float>()); }

bool fits(int stage_bytes, int extra_bytes = 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    return stage_count(stage_bytes, dev, extra_bytes) >= 2;
}

// Reads and clears this translation unit's wait word (synchronous).
cudaError_t take_local_wait_error(unsigned int* flag) {
    *flag = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_wait_error, sizeof(unsigned int));
    if (e != cudaSuccess || *flag == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_wait_error, &zero, sizeof(unsigned int));
}

}  // namespace
}  // namespace fsdp
