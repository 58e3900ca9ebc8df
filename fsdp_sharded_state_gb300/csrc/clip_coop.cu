// clip_coop.cu -- the sharded clip_grad_norm_ step ("第18章 FSDP：ZeRO 风格的参数分片"
// §18.18: every rank's sum of squares of its gradient shard, one all-reduce of the sums,
// the global norm, every rank scales its own shard) in one cooperative launch, for unit
// ranges whose pieces sit in the aligned class (rank view congruent to its full-layout
// position mod 8) but for a few tiles at most.
//
// The two-pass form (rows.cu) writes the whole fp32 gradient shard in pass 1 and reads
// it back in pass 3.  Here CTA b of G takes tiles b, b + G, b + 2G, ... of the range in
// phase 1 (reduce-scatter, sum of squares), spread over its four 256-thread groups, and
// keeps the reduced gradient of its last kKeepTotal tiles in shared memory instead of
// storing it (over the grid: the top kKeepTotal G tiles of the range); the kKeepTotal
// before those are stored with an L2 evict-last policy.  After a grid-wide barrier
// (bounded in time) every CTA forms the norm and the clip coefficient from the per-CTA
// partials, in one fixed order.  In phase 3 each group first updates its kept tiles
// from shared memory, then claims the other tiles one at a time from a grid-wide
// counter, from the top of the range down (the evict-last tiles first).  The kept
// tiles' gradient never makes the write-and-read-back round trip through DRAM, and the
// claims let the SMs that stream faster take more tiles: measured on GB300, a static
// split of phase 3 left the fastest SMs idle for up to 13 % of it.  Phase 1 stays a
// static split, so that the norm's grouping, and with it the norm, is the same in
// every run.
//
// The arithmetic per element is that of the two-pass kernels (rows.cu), operation for
// operation; the norm's double sum is grouped per CTA over other tile sets, so its last
// bits (and at most the coefficient's last bit) may differ from theirs.
#include <mutex>

#include "pipeline.cuh"
#include "staged.hpp"

namespace fsdp {
namespace {

constexpr int kCoopGroups = 4;                          // 256-thread tile groups per CTA
constexpr int kCoopThreads = kThreads * kCoopGroups;    // 1024
constexpr int kKeepSmem = 6;                            // tiles kept in shared memory per group
constexpr int kKeepTotal = kKeepSmem * kCoopGroups;     // per CTA; as many before them: evict-last stores
constexpr size_t kCoopSmem = size_t(kCoopGroups) * kKeepSmem * size_t(kTileElems) * sizeof(float);  // 192 KB

__device__ __forceinline__ int64_t coop_tile_x0(const Seg& sg, int64_t gt) {
    return (seg_vec0(sg.shard) + (gt - sg.tile0) * kThreads) * kVec;
}

// Index of the segment that holds tile gt (segs[n_segs] is the sentinel).
__device__ __forceinline__ int coop_find_seg(const Seg* __restrict__ segs, int n_segs, int64_t gt) {
    int a = 0, b = n_segs - 1;
    while (a < b) {                       // largest s with segs[s].tile0 <= gt
        const int m = (a + b + 1) >> 1;
        if (segs[m].tile0 <= gt) a = m;
        else b = m - 1;
    }
    return a;
}

__device__ __forceinline__ uint64_t coop_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void coop_st4(float* p, float4 x, bool hint, uint64_t pol) {
    if (hint)
        asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;"
                     ::"l"(p), "f"(x.x), "f"(x.y), "f"(x.z), "f"(x.w), "l"(pol) : "memory");
    else
        st4(p, x);
}

// Sum of a double over the CTA in one fixed order (warp trees, then warp 0's 32 partials
// in order); valid in thread 0.
__device__ __forceinline__ double coop_block_sum(double x, double* warp_part) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = x;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < kCoopThreads / 32; ++w) t += warp_part[w];
    __syncthreads();
    return t;
}

// All CTAs of the (cooperative, co-resident) grid meet here.  counter starts at 0 (the
// launcher clears it).  Thread 0 of every CTA publishes its CTA's writes, counts in and
// polls the count with acquire loads, for at most about wait_ns nanoseconds; on giving up
// it records FSDP_ETIMEOUT in this unit's wait word.  True when every CTA arrived.
__device__ __forceinline__ bool coop_grid_barrier(unsigned int* counter, uint64_t wait_ns, int* ok_sh) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1u);
        bool ok = false;
        const uint64_t t0 = global_ns();
#pragma unroll 1
        for (uint32_t i = 0; i < (1u << 28); ++i) {
            unsigned int v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
            if (v >= gridDim.x) {
                ok = true;
                break;
            }
            __nanosleep(64);
            if ((i & 63) == 63 && global_ns() - t0 > wait_ns) break;
        }
        __threadfence();
        if (!ok) atomicOr(&g_wait_error, 1u);
        *ok_sh = ok ? 1 : 0;
    }
    __syncthreads();
    return *ok_sh != 0;
}

// Sum of the N bf16 replicas at 8 consecutive full-layout elements from f (16-byte
// aligned), in rank order; four replicas' loads in flight at a time (the kernel runs
// 1024 threads on 64 registers).  Same sums as reduce8_vec: only the loads are batched.
__device__ __forceinline__ void coop_reduce8_bf16(const GradPtrs& gp, int N, int64_t f, float (&acc)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
#pragma unroll 1
    for (int q0 = 0; q0 < N; q0 += 4) {
        uint4 x[4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (q0 + b < N) x[b] = ld_once(static_cast<const uint16_t*>(gp.p[q0 + b]) + f);
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (q0 + b < N) {
                const uint32_t w[4] = {x[b].x, x[b].y, x[b].z, x[b].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc[2 * k] = __fadd_rn(acc[2 * k], bf16lo(w[k]));
                    acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], bf16hi(w[k]));
                }
            }
    }
}

// Phase 1 on one tile, by one 256-thread group (t = thread in the group): the fp32 mean
// of the N replicas into the gradient shard -- or, for a kept tile, into its shared-memory
// slot `keep` (2048 floats, indexed by element in the tile) -- and the thread's sum of
// squares (fp32 over a vector in order, then double, as the two-pass kernels).  A tile
// whose rank view is not congruent to its full-layout position mod 8 (the launcher lets
// through ranges where such tiles are rare) takes the per-element path throughout: its
// replicas cannot be read with aligned 16-byte loads.
template <typename GT>
__device__ __forceinline__ double coop_phase1(const Seg& sg, int64_t gt, const GradPtrs& gp, int N, float nf,
                                              float* __restrict__ gout, float* keep, bool hint, uint64_t pol,
                                              int t) {
    const int64_t base = coop_tile_x0(sg, gt);
    const int64_t lo = sg.shard, hi = sg.shard + sg.len, delta = sg.full - sg.shard;
    const bool al = (delta & (kVec - 1)) == 0;
    double ss = 0.0;
    if constexpr (std::is_same<GT, float>::value) {
        // split lane mapping: lane l owns [4l, 4l+4) and [128+4l, 128+4l+4) of its warp's 256
        const int64_t x0 = base + (t >> 5) * 256 + (t & 31) * 4, x1 = x0 + 128;
        if (x0 >= hi) return 0.0;
        if (al && x0 >= lo && x1 + 4 <= hi) {
            float acc[8], g[8], sq = 0.0f;
            reduce_split_f32(gp, N, x0 + delta, x1 + delta, acc);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                g[k] = mean_div(acc[k], nf);
                sq = __fmaf_rn(g[k], g[k], sq);
            }
            const float4 a = make_float4(g[0], g[1], g[2], g[3]), b = make_float4(g[4], g[5], g[6], g[7]);
            if (keep) {
                *reinterpret_cast<float4*>(keep + (x0 - base)) = a;
                *reinterpret_cast<float4*>(keep + (x1 - base)) = b;
            } else {
                coop_st4(gout + x0, a, hint, pol);
                coop_st4(gout + x1, b, hint, pol);
            }
            return double(sq);
        }
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {                       // a chunk at a segment edge, or misaligned
            const int64_t xc = c ? x1 : x0;
            const int64_t a = xc > lo ? xc : lo, b = (xc + 4) < hi ? (xc + 4) : hi;
            for (int64_t e = a; e < b; ++e) {
                const float g = mean_div(reduce1<float>(gp, N, e + delta), nf);
                if (keep) keep[e - base] = g;
                else gout[e] = g;
                ss += double(g) * double(g);
            }
        }
        return ss;
    } else {
        // bf16 replicas: thread t owns the 8 elements [8t, 8t+8) of the tile
        const int64_t e0 = base + int64_t(t) * kVec;
        if (e0 >= hi) return 0.0;
        if (al && e0 >= lo && e0 + kVec <= hi) {
            float acc[8], g[8], sq = 0.0f;
            coop_reduce8_bf16(gp, N, e0 + delta, acc);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                g[k] = mean_div(acc[k], nf);
                sq = __fmaf_rn(g[k], g[k], sq);
            }
            const float4 a = make_float4(g[0], g[1], g[2], g[3]), b = make_float4(g[4], g[5], g[6], g[7]);
            if (keep) {
                *reinterpret_cast<float4*>(keep + (e0 - base)) = a;
                *reinterpret_cast<float4*>(keep + (e0 - base) + 4) = b;
            } else {
                coop_st4(gout + e0, a, hint, pol);
                coop_st4(gout + e0 + 4, b, hint, pol);
            }
            return double(sq);
        }
        const int64_t a = e0 > lo ? e0 : lo, b = (e0 + kVec) < hi ? (e0 + kVec) : hi;
        for (int64_t e = a; e < b; ++e) {
            const float g = mean_div(reduce1<GT>(gp, N, e + delta), nf);
            if (keep) keep[e - base] = g;
            else gout[e] = g;
            ss += double(g) * double(g);
        }
        return ss;
    }
}

// Phase 3 on one tile (split lane mapping, as the two-pass kernel's pass 3): the clipped
// gradient g = shard * coef -- the shard read from the tile's shared-memory slot `keep`
// when it has one, else from L2 (another SM may have written it in phase 1) -- written
// back, then AdamW and the cast.
template <bool PARAM>
__device__ __forceinline__ void coop_phase3(const Seg& sg, int64_t gt, const float* keep, float coef,
                                            float* __restrict__ gshard, float* __restrict__ master,
                                            float* __restrict__ exp_avg, float* __restrict__ exp_avg_sq,
                                            uint16_t* __restrict__ param, const AdamScal& sc, int t) {
    const int64_t base = coop_tile_x0(sg, gt);
    const int64_t x0 = base + (t >> 5) * 256 + (t & 31) * 4;
    const int64_t lo = sg.shard, hi = sg.shard + sg.len;
    if (x0 >= hi) return;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int64_t xc = x0 + 128 * c;
        if (xc >= lo && xc + 4 <= hi) {
            const float4 gq = keep ? *reinterpret_cast<const float4*>(keep + (xc - base)) : __ldcg(reinterpret_cast<const float4*>(gshard + xc));
            const float4 pq = ld4(master + xc), mq = ld4(exp_avg + xc), vq = ld4(exp_avg_sq + xc);
            float g[4] = {gq.x, gq.y, gq.z, gq.w}, p[4] = {pq.x, pq.y, pq.z, pq.w};
            float m[4] = {mq.x, mq.y, mq.z, mq.w}, v[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                g[k] = __fmul_rn(g[k], coef);
                adamw1(sc, g[k], p[k], m[k], v[k]);
            }
            st4(gshard + xc, make_float4(g[0], g[1], g[2], g[3]));
            st4(master + xc, make_float4(p[0], p[1], p[2], p[3]));
            st4(exp_avg + xc, make_float4(m[0], m[1], m[2], m[3]));
            st4(exp_avg_sq + xc, make_float4(v[0], v[1], v[2], v[3]));
            if (PARAM)
                *reinterpret_cast<uint2*>(param + xc) = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
        } else {
            const int64_t a = xc > lo ? xc : lo, b = (xc + 4) < hi ? (xc + 4) : hi;
            for (int64_t e = a; e < b; ++e) {
                const float g = __fmul_rn(keep ? keep[e - base] : __ldcg(gshard + e), coef);
                float p = master[e], m = exp_avg[e], v = exp_avg_sq[e];
                adamw1(sc, g, p, m, v);
                gshard[e] = g; master[e] = p; exp_avg[e] = m; exp_avg_sq[e] = v;
                if (PARAM) param[e] = to_bf16(p);
            }
        }
    }
}

// The whole clip step.  counter[0] counts the CTAs in at the grid barrier, counter[1]
// hands out the phase-3 tiles; both start at 0 (the launcher clears them).
template <typename GT, bool PARAM>
__global__ void __launch_bounds__(kCoopThreads, 1)
k_clip_coop(const Seg* __restrict__ segs, int n_segs, int64_t tile_base, int64_t n_tiles, GradPtrs gp, int N,
            float nf, float* __restrict__ gshard, float* __restrict__ master, float* __restrict__ exp_avg,
            float* __restrict__ exp_avg_sq, uint16_t* __restrict__ param, double* __restrict__ part,
            unsigned int* counter, double* __restrict__ ws_norm, float* __restrict__ ws_coef,
            float* __restrict__ norm_out, float max_norm, AdamScal sc, uint64_t wait_ns) {
    extern __shared__ __align__(16) float keep_sm[];
    __shared__ double warp_part[kCoopThreads / 32];
    __shared__ int claim_sh[kCoopGroups][2];
    __shared__ float coef_sh;
    __shared__ int ok_sh;
    const int grp = threadIdx.x / kThreads, t = threadIdx.x % kThreads;
    const int64_t G = gridDim.x, b = blockIdx.x;
    // this CTA's list: tiles b + k G, k < n1 (a list length fits in an int: the launcher
    // takes ranges of fewer than 2^31 tiles); group grp takes k = grp, grp + 4, ...
    const int n1 = b < n_tiles ? int((n_tiles - b + G - 1) / G) : 0;
    const int keep_from = n1 - kKeepTotal;              // k >= keep_from: kept (slot (k - keep_from) / 4)
    const int hint_from = keep_from - kKeepTotal;       // k in [hint_from, keep_from): evict-last stores
    float* my_keep = keep_sm + size_t(grp) * kKeepSmem * size_t(kTileElems);
    const uint64_t pol = coop_policy_evict_last();

    // ---- phase 1: reduce-scatter and sums of squares, the group's tiles forward ----
    double ss = 0.0;
    if (grp < n1) {
        int s = coop_find_seg(segs, n_segs, tile_base + b + grp * G);
#pragma unroll 1
        for (int k = grp; k < n1; k += kCoopGroups) {
            const int64_t gt = tile_base + b + int64_t(k) * G;
            s = advance_seg(segs, s, gt);
            const Seg sg = segs[s];
            float* keep = k >= keep_from ? my_keep + ((k - keep_from) >> 2) * kTileElems : nullptr;
            ss += coop_phase1<GT>(sg, gt, gp, N, nf, gshard, keep, k >= hint_from, pol, t);
        }
    }
    const double tot = coop_block_sum(ss, warp_part);
    if (threadIdx.x == 0) part[b] = tot;

    // ---- the grid barrier, then the norm and the clip coefficient in every CTA ----
    if (!coop_grid_barrier(counter, wait_ns, &ok_sh)) return;
    double x = 0.0;
    for (int i = threadIdx.x; i < int(G); i += kCoopThreads) x += __ldcg(part + i);
    const double all = coop_block_sum(x, warp_part);
    if (threadIdx.x == 0) {
        const double norm = sqrt(all);
        double c = double(max_norm) / (norm + 1e-6);
        if (c > 1.0) c = 1.0;
        coef_sh = float(c);
        if (b == 0) {
            *ws_norm = norm;
            *ws_coef = float(c);
            if (norm_out) {
                norm_out[0] = float(norm);
                norm_out[1] = float(c);
            }
        }
    }
    __syncthreads();
    const float coef = coef_sh;

    // ---- phase 3 (a): the group's kept tiles, from shared memory, last first ----
    if (grp < n1) {
        int k = grp + (n1 - 1 - grp) / kCoopGroups * kCoopGroups;         // the group's last list entry
        if (k >= keep_from) {
            int s = coop_find_seg(segs, n_segs, tile_base + b + int64_t(k) * G);
#pragma unroll 1
            for (; k >= 0 && k >= keep_from; k -= kCoopGroups) {
                const int64_t gt = tile_base + b + int64_t(k) * G;
                while (segs[s].tile0 > gt) --s;
                coop_phase3<PARAM>(segs[s], gt, my_keep + ((k - keep_from) >> 2) * kTileElems, coef, gshard, master,
                                   exp_avg, exp_avg_sq, param, sc, t);
            }
        }
    }
    // ---- phase 3 (b): the other tiles, [0, nd), claimed one at a time from the top down ----
    // The group's thread 0 takes the next claim while the group updates the current tile;
    // the claim reaches the group through a two-slot shared word and one group barrier.
    const int nd = n_tiles > kKeepTotal * G ? int(n_tiles - kKeepTotal * G) : 0;
    if (nd > 0) {
        unsigned int nxt = 0;
        if (t == 0) nxt = atomicAdd(counter + 1, 1u);
        int s = n_segs - 1;                                 // claims come from the top down
#pragma unroll 1
        for (unsigned int par = 0;; par ^= 1u) {
            if (t == 0) claim_sh[grp][par] = nxt < unsigned(nd) ? nd - 1 - int(nxt) : -1;
            asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kThreads) : "memory");
            const int tt = claim_sh[grp][par];
            if (tt < 0) break;
            const int64_t gt = tile_base + tt;
            if (t == 0) nxt = atomicAdd(counter + 1, 1u);
            while (segs[s].tile0 > gt) --s;
            coop_phase3<PARAM>(segs[s], gt, nullptr, coef, gshard, master, exp_avg, exp_avg_sq, param, sc, t);
        }
    }
}

std::mutex g_coop_mu;
std::map<std::pair<const void*, int>, int> g_coop_grid;   // (kernel, device) -> co-resident CTAs

// CTAs of the kernel that fit on the current device at once (0 if none), cached.
template <typename K>
int coop_grid_of(K kernel) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    {
        std::lock_guard<std::mutex> lk(g_coop_mu);
        auto it = g_coop_grid.find(key);
        if (it != g_coop_grid.end()) return it->second;
    }
    int sms = 0, per_sm = 0, coop = 0;
    int blocks = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kCoopSmem)) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kCoopThreads, kCoopSmem) == cudaSuccess)
        blocks = sms * per_sm;
    cudaGetLastError();                   // a refused attribute leaves no error behind
    std::lock_guard<std::mutex> lk(g_coop_mu);
    g_coop_grid[key] = blocks;
    return blocks;
}

}  // namespace

cudaError_t launch_clip_coop(const Seg* segs, int n_segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                             const GradPtrs& gp, int N, float* gshard, float* master, float* m, float* v,
                             uint16_t* param, double* part, int max_part, unsigned int* counter, double* ws_norm,
                             float* ws_coef, float* norm_out, float max_norm, const AdamScal& sc, uint64_t wait_ns,
                             cudaStream_t st, bool* launched) {
    *launched = false;
    auto go = [&](auto kernel) -> cudaError_t {
        const int grid = coop_grid_of(kernel);
        // not here: the caller falls back (the kernel's tile indices are ints)
        if (grid <= 0 || grid > max_part || n_tiles >= (int64_t(1) << 31)) return cudaSuccess;
        cudaError_t e = cudaMemsetAsync(counter, 0, 2 * sizeof(unsigned int), st);
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kCoopThreads);
        cfg.dynamicSmemBytes = kCoopSmem;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, segs, n_segs, tile_base, n_tiles, gp, N, float(N), gshard, master, m, v,
                               param, part, counter, ws_norm, ws_coef, norm_out, max_norm, sc, wait_ns);
        if (e == cudaErrorCooperativeLaunchTooLarge) {                 // not all CTAs would fit: fall back
            cudaGetLastError();
            return cudaSuccess;
        }
        if (e == cudaSuccess) *launched = true;
        return e;
    };
    if (grad_bf16)
        return param ? go(k_clip_coop<uint16_t, true>) : go(k_clip_coop<uint16_t, false>);
    return param ? go(k_clip_coop<float, true>) : go(k_clip_coop<float, false>);
}

cudaError_t take_wait_error_coop(unsigned int* flag) { return take_local_wait_error(flag); }

}  // namespace fsdp
