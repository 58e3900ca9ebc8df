// kernels.cu -- the direct (register) kernels of libfsdpstate (sm_103a); the
// bulk-copy kernels are in staged.cu, allgather.cu and staged_rows.cu.
//
//   k_rs_adamw   fused reduce-scatter (fp32 mean over N gradient replicas, fixed
//                rank order) + AdamW on the fp32 master/exp_avg/exp_avg_sq shard +
//                bf16 recast of the updated shard: one HBM pass per shard element.
//   k_unshard_shift  all-gather (bitwise copy shard -> full) of the pieces whose
//                full-layout offset is not congruent to their shard offset mod 8
//                (the aligned ones go through bulk copies: k_unshard_bulk).
//   k_reshard    full layout -> rank shards (fp32 master and/or bf16 param), and
//   k_zero_pad   the zero-fill of shard padding.
//
// All kernels are persistent: the grid is a multiple of the SM count, each CTA
// walks tiles blockIdx.x, blockIdx.x + gridDim.x, ... of its segment range.  Each
// thread owns one 8-element vector per tile, aligned on the shard side; interior
// vectors use 16-byte loads and stores, the (at most two) partial vectors of a
// segment go element by element.  A segment whose full-layout offset is not
// congruent to its shard offset mod 8 (the "shifted" class) realigns its vectors
// across the warp: each lane takes its neighbour's vector with a shuffle.
// Memory-bound throughout: no tensor-core work (the path has no contraction).
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "device_ops.cuh"
#include "kernels.hpp"

namespace fsdp {
namespace {

// fp32 gradients on aligned segments, "split" thread mapping: within its warp's 256
// elements, lane l owns the two 4-element chunks [4l, 4l+4) and [128+4l, 128+4l+4),
// so every 16-byte load or store instruction of the warp covers 512 contiguous
// bytes (whole sectors).  Same arithmetic, same order as the other paths.
__device__ __forceinline__ void rs_tile_f32_split(const Seg& sg, int64_t gt, const GradPtrs& gp, int N,
                                                  float* __restrict__ master, float* __restrict__ exp_avg,
                                                  float* __restrict__ exp_avg_sq, uint16_t* __restrict__ param,
                                                  float* __restrict__ gout, const AdamScal& sc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t x0 = (seg_vec0(sg.shard) + (gt - sg.tile0) * kThreads) * kVec + warp * 256 + lane * 4;
    const int64_t lo = sg.shard, hi = sg.shard + sg.len;
    const int64_t delta = sg.full - sg.shard;
    if (x0 >= hi) return;
    const int64_t x1 = x0 + 128;
    const bool fast = x0 >= lo && x1 + 4 <= hi;
    if (fast) {
        const float4 pa = ld4(master + x0), pb = ld4(master + x1);
        const float4 ma = ld4(exp_avg + x0), mb = ld4(exp_avg + x1);
        const float4 va = ld4(exp_avg_sq + x0), vb = ld4(exp_avg_sq + x1);
        float acc[8];
        reduce_split_f32(gp, N, x0 + delta, x1 + delta, acc);
        // compute and store one 4-element chunk at a time (fewer live registers)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int64_t xc = c ? x1 : x0;
            const float4 pc = c ? pb : pa, mc = c ? mb : ma, vc = c ? vb : va;
            float p[4] = {pc.x, pc.y, pc.z, pc.w};
            float m[4] = {mc.x, mc.y, mc.z, mc.w};
            float v[4] = {vc.x, vc.y, vc.z, vc.w};
            float g[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                g[k] = mean_div(acc[4 * c + k], sc.nf);
                adamw1(sc, g[k], p[k], m[k], v[k]);
            }
            st4(master + xc, make_float4(p[0], p[1], p[2], p[3]));
            st4(exp_avg + xc, make_float4(m[0], m[1], m[2], m[3]));
            st4(exp_avg_sq + xc, make_float4(v[0], v[1], v[2], v[3]));
            if (param)
                *reinterpret_cast<uint2*>(param + xc) = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
            if (gout) st4(gout + xc, make_float4(g[0], g[1], g[2], g[3]));
        }
        return;
    }
    // a chunk at a segment edge: element by element
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
        const int64_t xc = c ? x1 : x0;
        const int64_t a = xc > lo ? xc : lo;
        const int64_t b = (xc + 4) < hi ? (xc + 4) : hi;
        for (int64_t e = a; e < b; ++e) {
            float acc = 0.0f;
            for (int q = 0; q < N; ++q) acc = __fadd_rn(acc, static_cast<const float*>(gp.p[q])[e + delta]);
            const float gg = mean_div(acc, sc.nf);
            float pp = master[e], mm = exp_avg[e], vv = exp_avg_sq[e];
            adamw1(sc, gg, pp, mm, vv);
            master[e] = pp; exp_avg[e] = mm; exp_avg_sq[e] = vv;
            if (param) param[e] = to_bf16(pp);
            if (gout) gout[e] = gg;
        }
    }
}

// SHIFT = false: every segment has its full-layout offset congruent to its shard
// offset mod 8 (plain 16-byte vectors on both sides).  SHIFT = true: none has, and
// the gradients go through the warp realignment.
// Occupancy: the aligned instances of the main configurations keep 3 CTAs (24
// warps) per SM -- at 2 the DRAM queue drains between tiles and a launch loses
// 5-20 % of bandwidth -- so they are held to 85 registers; the shifted ones, those
// that also write the gradient shard and bf16 gradients into fp32 parameters need
// more and keep 2 (no spills).
template <typename GT, bool PARAM, bool GOUT, bool SHIFT>
__global__ void __launch_bounds__(kThreads, (SHIFT || GOUT || (!PARAM && sizeof(GT) == 2)) ? 2 : 3)
k_rs_adamw(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles, GradPtrs gp, int N, int64_t F,
           float* __restrict__ master, float* __restrict__ exp_avg, float* __restrict__ exp_avg_sq,
           uint16_t* __restrict__ param, float* __restrict__ gout, AdamScal sc) {
    pdl_wait();
    const bool lane31 = (threadIdx.x & 31) == 31;
    int s = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t gt = tile_base + t;
        s = advance_seg(segs, s, gt);
        const Seg sg = segs[s];
        if (!SHIFT && sizeof(GT) == 4) {
            rs_tile_f32_split(sg, gt, gp, N, master, exp_avg, exp_avg_sq, param, gout, sc);
            continue;
        }
        const int64_t e0 = (seg_vec0(sg.shard) + (gt - sg.tile0) * kThreads + threadIdx.x) * kVec;
        const int64_t lo = sg.shard, hi = sg.shard + sg.len;
        const int64_t delta = sg.full - sg.shard;            // full index = shard index + delta
        const int64_t f0 = e0 + delta;
        const bool interior = e0 >= lo && e0 + kVec <= hi;
        const int d = int(delta & (kVec - 1));
        const int64_t fa = f0 - d;
        const bool have_a = fa >= 0 && fa + kVec <= F;
        const bool have_b = fa >= 0 && fa + 2 * kVec <= F;
        const bool fast = SHIFT ? (interior && have_a && have_b) : interior;
        // Issue the state loads before the gradient loads: both round trips overlap.
        float4 p0, p1, m0, m1, v0, v1;
        if (fast) {
            p0 = ld4(master + e0); p1 = ld4(master + e0 + 4);
            m0 = ld4(exp_avg + e0); m1 = ld4(exp_avg + e0 + 4);
            v0 = ld4(exp_avg_sq + e0); v1 = ld4(exp_avg_sq + e0 + 4);
        }
        float acc[8];
        if (!SHIFT) {
            // gradients 16-byte aligned where the state is: plain vector loads
            if (e0 >= hi) continue;
            if (fast) reduce8_vec<GT>(gp, N, f0, acc);
        } else {
            // misaligned segment (uniform over the tile): warp-collective realignment
            reduce8_shift<GT>(d, gp, N, fa, have_a, have_b, lane31, acc);
            if (e0 >= hi) continue;
        }

        if (fast) {
            // ---- interior vector: 16-byte state traffic ----
            float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            float g[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                g[k] = mean_div(acc[k], sc.nf);
                adamw1(sc, g[k], p[k], m[k], v[k]);
            }
            st4(master + e0, make_float4(p[0], p[1], p[2], p[3]));
            st4(master + e0 + 4, make_float4(p[4], p[5], p[6], p[7]));
            st4(exp_avg + e0, make_float4(m[0], m[1], m[2], m[3]));
            st4(exp_avg + e0 + 4, make_float4(m[4], m[5], m[6], m[7]));
            st4(exp_avg_sq + e0, make_float4(v[0], v[1], v[2], v[3]));
            st4(exp_avg_sq + e0 + 4, make_float4(v[4], v[5], v[6], v[7]));
            if (PARAM)
                stu4(param + e0, make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                                            pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7])));
            if (GOUT) {
                st4(gout + e0, make_float4(g[0], g[1], g[2], g[3]));
                st4(gout + e0 + 4, make_float4(g[4], g[5], g[6], g[7]));
            }
        } else {
            // ---- partial vector at a segment edge (or next to the buffer end): element by element ----
            const int64_t a = e0 > lo ? e0 : lo;
            const int64_t b = (e0 + kVec) < hi ? (e0 + kVec) : hi;
            for (int64_t e = a; e < b; ++e) {
                const float g = mean_div(reduce1<GT>(gp, N, e + delta), sc.nf);
                float p = master[e], m = exp_avg[e], v = exp_avg_sq[e];
                adamw1(sc, g, p, m, v);
                master[e] = p; exp_avg[e] = m; exp_avg_sq[e] = v;
                if (PARAM) param[e] = to_bf16(p);
                if (GOUT) gout[e] = g;
            }
        }
    }
}

// ----------------------------------------------------------------------------
// Unshard: bitwise copy shard -> full.  ET is the element's bit container.
// ----------------------------------------------------------------------------
template <typename ET> struct CopyVec {
    static constexpr int kWords = int(sizeof(ET)) * kVec / 4;   // 32-bit words per 8 elements: 4 or 8
    uint32_t w[kWords];
};

template <typename ET>
__device__ __forceinline__ CopyVec<ET> load_vec(const ET* p) {
    CopyVec<ET> v;
#pragma unroll
    for (int k = 0; k < CopyVec<ET>::kWords / 4; ++k) {
        const uint4 x = ld_once(p + k * (16 / sizeof(ET)));
        v.w[4 * k] = x.x; v.w[4 * k + 1] = x.y; v.w[4 * k + 2] = x.z; v.w[4 * k + 3] = x.w;
    }
    return v;
}

template <typename ET>
__device__ __forceinline__ void store_vec(ET* p, const CopyVec<ET>& v) {
#pragma unroll
    for (int k = 0; k < CopyVec<ET>::kWords / 4; ++k)
        stu4(p + k * (16 / sizeof(ET)), make_uint4(v.w[4 * k], v.w[4 * k + 1], v.w[4 * k + 2], v.w[4 * k + 3]));
}

// Elements O..O+7 of the window [S, X] as one vector (O compile-time).
template <typename ET, int O>
__device__ __forceinline__ CopyVec<ET> window(const CopyVec<ET>& S, const CopyVec<ET>& X) {
    constexpr int W = CopyVec<ET>::kWords;
    uint32_t w[2 * W];
#pragma unroll
    for (int k = 0; k < W; ++k) { w[k] = S.w[k]; w[W + k] = X.w[k]; }
    CopyVec<ET> r;
    if (sizeof(ET) == 4) {
#pragma unroll
        for (int k = 0; k < W; ++k) r.w[k] = w[O + k];
    } else if ((O & 1) == 0) {
#pragma unroll
        for (int k = 0; k < W; ++k) r.w[k] = w[(O >> 1) + k];
    } else {
#pragma unroll
        for (int k = 0; k < W; ++k) r.w[k] = __funnelshift_r(w[(O >> 1) + k], w[(O >> 1) + k + 1], 16);
    }
    return r;
}

template <typename ET>
__device__ __forceinline__ CopyVec<ET> window_any(int o, const CopyVec<ET>& S, const CopyVec<ET>& X) {
    switch (o) {
        case 1: return window<ET, 1>(S, X);
        case 2: return window<ET, 2>(S, X);
        case 3: return window<ET, 3>(S, X);
        case 4: return window<ET, 4>(S, X);
        case 5: return window<ET, 5>(S, X);
        case 6: return window<ET, 6>(S, X);
        default: return window<ET, 7>(S, X);
    }
}

// All-gather of the shifted class (pieces whose full-layout offset is not congruent
// to their shard offset mod 8); the aligned class goes through bulk copies
// (k_unshard_bulk).
template <typename ET>
__global__ void __launch_bounds__(kThreads)
k_unshard_shift(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles, const ET* __restrict__ src,
                ET* __restrict__ dst, int64_t src_limit) {
    pdl_wait();
    const bool lane31 = (threadIdx.x & 31) == 31;
    int s = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t gt = tile_base + t;
        s = advance_seg(segs, s, gt);
        const Seg sg = segs[s];
        const int64_t e0 = (seg_vec0(sg.shard) + (gt - sg.tile0) * kThreads + threadIdx.x) * kVec;
        const int64_t lo = sg.shard, hi = sg.shard + sg.len;
        const int64_t delta = sg.full - sg.shard;
        // Misaligned segment (uniform over the tile): every lane loads its aligned
        // source vector S and gets the next one X from its neighbour (lane 31 loads
        // it); lane t then stores the aligned destination vector [fa+8, fa+16),
        // made of S[8-d..7] and X[0..7-d].  Destination vectors that are not wholly
        // inside the segment are written element by element by the source owners.
        const int d = int(delta & (kVec - 1));
        CopyVec<ET> S{}, X{};
        if (e0 + kVec <= src_limit) S = load_vec(src + e0);
        if (lane31 && e0 + 2 * kVec <= src_limit) X = load_vec(src + e0 + kVec);
        {
            const CopyVec<ET> nb = shfl_down1(S);
            if (!lane31) X = nb;
        }
        if (e0 >= hi) continue;
        const int64_t fa = e0 + delta - d;                    // 8-aligned full index
        const int64_t rlo = sg.full, rhi = sg.full + sg.len;   // full range of the segment
        if (fa + kVec >= rlo && fa + 2 * kVec <= rhi) store_vec(dst + fa + kVec, window_any<ET>(kVec - d, S, X));
        if (fa >= rlo && fa + 2 * kVec <= rhi) continue;       // both my destination vectors are whole
        const int64_t a = e0 > lo ? e0 : lo;
        const int64_t b = (e0 + kVec) < hi ? (e0 + kVec) : hi;
        for (int64_t e = a; e < b; ++e) {
            const int64_t f = e + delta;
            const int64_t v0 = f - (f & (kVec - 1));
            if (!(v0 >= rlo && v0 + kVec <= rhi)) dst[f] = src[e];
        }
    }
}

// ----------------------------------------------------------------------------
// Reshard: full (fp32 or bf16) -> master fp32 and/or param bf16.
// ----------------------------------------------------------------------------
template <bool FULL_BF16>
__device__ __forceinline__ float load_full1(const void* full, int64_t i) {
    if (FULL_BF16) return bf16f(static_cast<const uint16_t*>(full)[i]);
    return static_cast<const float*>(full)[i];
}

template <bool FULL_BF16, bool MASTER, bool PARAM>
__global__ void __launch_bounds__(kThreads)
k_reshard(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles,
          const void* __restrict__ full, float* __restrict__ master, uint16_t* __restrict__ param) {
    pdl_wait();
    int s = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t gt = tile_base + t;
        s = advance_seg(segs, s, gt);
        const Seg sg = segs[s];
        const int64_t e0 = (seg_vec0(sg.shard) + (gt - sg.tile0) * kThreads + threadIdx.x) * kVec;
        const int64_t lo = sg.shard, hi = sg.shard + sg.len;
        if (e0 >= hi) continue;
        const int64_t delta = sg.full - sg.shard;
        if (e0 >= lo && e0 + kVec <= hi && (delta & (kVec - 1)) == 0) {
            float x[8];
            if (FULL_BF16) {
                const uint4 w = ldu4(static_cast<const uint16_t*>(full) + e0 + delta);
                x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
                x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
            } else {
                const float* f = static_cast<const float*>(full) + e0 + delta;
                const float4 a = ld4(f), b = ld4(f + 4);
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
            }
            if (MASTER) {
                st4(master + e0, make_float4(x[0], x[1], x[2], x[3]));
                st4(master + e0 + 4, make_float4(x[4], x[5], x[6], x[7]));
            }
            if (PARAM)
                stu4(param + e0, make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                            pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7])));
        } else {
            const int64_t a = e0 > lo ? e0 : lo;
            const int64_t b = (e0 + kVec) < hi ? (e0 + kVec) : hi;
            for (int64_t e = a; e < b; ++e) {
                const float x = load_full1<FULL_BF16>(full, e + delta);
                if (MASTER) master[e] = x;
                if (PARAM) param[e] = to_bf16(x);
            }
        }
    }
}

// Zero-fill of shard padding (pad segments): fp32 and/or bf16 arrays.
template <bool F32OUT, bool BF16OUT>
__global__ void __launch_bounds__(kThreads)
k_zero_pad(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles,
           float* __restrict__ a32, uint16_t* __restrict__ a16) {
    pdl_wait();
    int s = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t gt = tile_base + t;
        s = advance_seg(segs, s, gt);
        const Seg sg = segs[s];
        const int64_t e0 = (seg_vec0(sg.shard) + (gt - sg.tile0) * kThreads + threadIdx.x) * kVec;
        const int64_t lo = sg.shard, hi = sg.shard + sg.len;
        if (e0 >= hi) continue;
        if (e0 >= lo && e0 + kVec <= hi) {
            if (F32OUT) {
                st4(a32 + e0, make_float4(0.f, 0.f, 0.f, 0.f));
                st4(a32 + e0 + 4, make_float4(0.f, 0.f, 0.f, 0.f));
            }
            if (BF16OUT) stu4(a16 + e0, make_uint4(0u, 0u, 0u, 0u));
        } else {
            const int64_t a = e0 > lo ? e0 : lo;
            const int64_t b = (e0 + kVec) < hi ? (e0 + kVec) : hi;
            for (int64_t e = a; e < b; ++e) {
                if (F32OUT) a32[e] = 0.0f;
                if (BF16OUT) a16[e] = 0;
            }
        }
    }
}

// ----------------------------------------------------------------------------
// Grid sizing: persistent, (resident CTAs per SM) x (SM count), cached per device.
// ----------------------------------------------------------------------------
std::mutex g_grid_mu;
std::map<std::pair<const void*, int>, int> g_grid_cache;

template <typename K>
int grid_for(K kernel, int64_t n_tiles) {
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    int blocks = 0;
    {
        std::lock_guard<std::mutex> lk(g_grid_mu);
        auto it = g_grid_cache.find(key);
        if (it != g_grid_cache.end()) blocks = it->second;
    }
    if (blocks == 0) {
        int sms = 0, per_sm = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
        blocks = (sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
        std::lock_guard<std::mutex> lk(g_grid_mu);
        g_grid_cache[key] = blocks;
    }
    return int(n_tiles < blocks ? n_tiles : blocks);
}

}  // namespace

// ----------------------------------------------------------------------------
// Launchers (host).  They return the cudaError_t of the launch.
// ----------------------------------------------------------------------------
template <typename GT, bool SHIFT>
static cudaError_t launch_rs_t(const Seg* segs, int64_t tile_base, int64_t n_tiles, const GradPtrs& gp,
                               int N, int64_t F, float* master, float* m, float* v, uint16_t* param, float* gout,
                               const AdamScal& sc, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (param && gout) {
        auto k = k_rs_adamw<GT, true, true, SHIFT>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, gp, N, F, master,
                   m, v, param, gout, sc);
    } else if (param) {
        auto k = k_rs_adamw<GT, true, false, SHIFT>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, gp, N, F, master,
                   m, v, param, gout, sc);
    } else if (gout) {
        auto k = k_rs_adamw<GT, false, true, SHIFT>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, gp, N, F, master,
                   m, v, param, gout, sc);
    } else {
        auto k = k_rs_adamw<GT, false, false, SHIFT>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, gp, N, F, master,
                   m, v, param, gout, sc);
    }
    return e;
}

cudaError_t launch_rs_adamw(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool shifted, bool grad_bf16,
                            const GradPtrs& gp, int N, int64_t F, float* master, float* m, float* v,
                            uint16_t* param, float* gout, const AdamScal& sc, cudaStream_t st) {
    if (n_tiles <= 0) return cudaSuccess;
    if (grad_bf16)
        return shifted ? launch_rs_t<uint16_t, true>(segs, tile_base, n_tiles, gp, N, F, master, m, v, param, gout, sc, st)
                       : launch_rs_t<uint16_t, false>(segs, tile_base, n_tiles, gp, N, F, master, m, v, param, gout, sc, st);
    return shifted ? launch_rs_t<float, true>(segs, tile_base, n_tiles, gp, N, F, master, m, v, param, gout, sc, st)
                   : launch_rs_t<float, false>(segs, tile_base, n_tiles, gp, N, F, master, m, v, param, gout, sc, st);
}

template <typename ET>
static cudaError_t launch_unshard_t(const Seg* segs, int64_t tile_base, int64_t n_tiles, const void* src, void* dst,
                                    int64_t src_limit, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    auto k = k_unshard_shift<ET>;
    e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, static_cast<const ET*>(src),
                                                  static_cast<ET*>(dst), src_limit);
    return e;
}

cudaError_t launch_unshard_shifted(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool bf16, const void* src,
                                   void* dst, int64_t src_limit, cudaStream_t st) {
    if (n_tiles <= 0) return cudaSuccess;
    return bf16 ? launch_unshard_t<uint16_t>(segs, tile_base, n_tiles, src, dst, src_limit, st)
                : launch_unshard_t<uint32_t>(segs, tile_base, n_tiles, src, dst, src_limit, st);
}

template <bool FB>
static cudaError_t launch_reshard_t(const Seg* segs, int64_t tile_base, int64_t n_tiles, const void* full,
                                    float* master, uint16_t* param, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (master && param) {
        auto k = k_reshard<FB, true, true>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, full, master, param);
    } else if (master) {
        auto k = k_reshard<FB, true, false>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, full, master, param);
    } else {
        auto k = k_reshard<FB, false, true>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, full, master, param);
    }
    return e;
}

cudaError_t launch_reshard(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool full_bf16,
                           const void* full, float* master, uint16_t* param, cudaStream_t st) {
    if (n_tiles <= 0 || (!master && !param)) return cudaSuccess;
    return full_bf16 ? launch_reshard_t<true>(segs, tile_base, n_tiles, full, master, param, st)
                     : launch_reshard_t<false>(segs, tile_base, n_tiles, full, master, param, st);
}

cudaError_t launch_zero_pad(const Seg* segs, int64_t tile_base, int64_t n_tiles, float* a32, uint16_t* a16,
                            cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (n_tiles <= 0 || (!a32 && !a16)) return cudaSuccess;
    if (a32 && a16) {
        auto k = k_zero_pad<true, true>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, a32, a16);
    } else if (a32) {
        auto k = k_zero_pad<true, false>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, a32, a16);
    } else {
        auto k = k_zero_pad<false, true>;
        e = launch(k, dim3(grid_for(k, n_tiles)), dim3(kThreads), 0, st, segs, tile_base, n_tiles, a32, a16);
    }
    return e;
}

}  // namespace fsdp
