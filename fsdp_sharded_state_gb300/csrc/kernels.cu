// kernels.cu -- the device side of libfsdpstate (sm_103a).
//
//   k_rs_adamw   fused reduce-scatter (fp32 mean over N gradient replicas, fixed
//                rank order) + AdamW on the fp32 master/exp_avg/exp_avg_sq shard +
//                bf16 recast of the updated shard: one HBM pass per shard element.
//   k_unshard    all-gather of the rank shards into the full layout (bitwise copy).
//   k_reshard    full layout -> rank shards (fp32 master and/or bf16 param), and
//   k_zero_pad   the zero-fill of shard padding.
//
// All kernels are persistent: the grid is a multiple of the SM count, each CTA
// walks tiles blockIdx.x, blockIdx.x + gridDim.x, ... of its segment range.  Each
// thread owns one 8-element vector per tile, aligned on the shard side; interior
// vectors use 16-byte loads and stores, the (at most two) partial vectors of a
// segment go element by element.  A segment whose full-layout offset is not
// congruent to its shard offset mod 8 reads its gradients element by element.
// Memory-bound throughout: no tensor-core work (the path has no contraction).
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "kernels.hpp"

namespace fsdp {
namespace {

// ----------------------------------------------------------------------------
// AdamW on one element.  Every operation is one fp32 IEEE operation rounded to
// nearest even; the _rn intrinsics keep the compiler from contracting them.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void adamw1(const AdamScal& s, float g, float& p, float& m, float& v) {
    const float pp = __fmul_rn(p, s.decay);
    const float mm = __fmaf_rn(s.beta1, m, __fmul_rn(s.om1, g));
    const float gg = __fmul_rn(s.om2, g);
    const float vv = __fmaf_rn(s.beta2, v, __fmul_rn(gg, g));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(vv), s.bc2s), s.eps);
    const float upd = __fdiv_rn(mm, den);
    p = __fmaf_rn(-s.step_size, upd, pp);
    m = mm;
    v = vv;
}

template <typename GT> struct GradIO;

// bf16 gradients: one 16-byte load per replica covers the 8 elements.
template <> struct GradIO<uint16_t> {
    static constexpr int kBatch = 8;
    struct Vec { uint4 w; };
    static __device__ __forceinline__ Vec load(const void* base, int64_t i) {
        return Vec{ld_once(static_cast<const uint16_t*>(base) + i)};
    }
    static __device__ __forceinline__ void add(float (&a)[8], const Vec& x) {
        a[0] = __fadd_rn(a[0], bf16lo(x.w.x)); a[1] = __fadd_rn(a[1], bf16hi(x.w.x));
        a[2] = __fadd_rn(a[2], bf16lo(x.w.y)); a[3] = __fadd_rn(a[3], bf16hi(x.w.y));
        a[4] = __fadd_rn(a[4], bf16lo(x.w.z)); a[5] = __fadd_rn(a[5], bf16hi(x.w.z));
        a[6] = __fadd_rn(a[6], bf16lo(x.w.w)); a[7] = __fadd_rn(a[7], bf16hi(x.w.w));
    }
    static __device__ __forceinline__ float load1(const void* base, int64_t i) {
        return bf16f(static_cast<const uint16_t*>(base)[i]);
    }
};

// fp32 gradients: two 16-byte loads per replica.
template <> struct GradIO<float> {
    static constexpr int kBatch = 4;
    struct Vec { uint4 a, b; };
    static __device__ __forceinline__ Vec load(const void* base, int64_t i) {
        const float* p = static_cast<const float*>(base) + i;
        return Vec{ld_once(p), ld_once(p + 4)};
    }
    static __device__ __forceinline__ void add(float (&a)[8], const Vec& x) {
        a[0] = __fadd_rn(a[0], __uint_as_float(x.a.x)); a[1] = __fadd_rn(a[1], __uint_as_float(x.a.y));
        a[2] = __fadd_rn(a[2], __uint_as_float(x.a.z)); a[3] = __fadd_rn(a[3], __uint_as_float(x.a.w));
        a[4] = __fadd_rn(a[4], __uint_as_float(x.b.x)); a[5] = __fadd_rn(a[5], __uint_as_float(x.b.y));
        a[6] = __fadd_rn(a[6], __uint_as_float(x.b.z)); a[7] = __fadd_rn(a[7], __uint_as_float(x.b.w));
    }
    static __device__ __forceinline__ float load1(const void* base, int64_t i) {
        return static_cast<const float*>(base)[i];
    }
};

// Sum of the N replicas at 8 consecutive full-layout elements starting at f
// (16-byte aligned), in rank order.  Loads are issued in batches so that a batch
// is in flight together.
template <typename GT>
__device__ __forceinline__ void reduce8_vec(const GradPtrs& gp, int N, int64_t f, float (&acc)[8]) {
    using IO = GradIO<GT>;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
#pragma unroll 1
    for (int q0 = 0; q0 < N; q0 += IO::kBatch) {
        typename IO::Vec buf[IO::kBatch];
#pragma unroll
        for (int b = 0; b < IO::kBatch; ++b)
            if (q0 + b < N) buf[b] = IO::load(gp.p[q0 + b], f);
#pragma unroll
        for (int b = 0; b < IO::kBatch; ++b)
            if (q0 + b < N) IO::add(acc, buf[b]);
    }
}

template <typename GT>
__device__ __forceinline__ float reduce1(const GradPtrs& gp, int N, int64_t f) {
    float acc = 0.0f;
#pragma unroll 1
    for (int q = 0; q < N; ++q) acc = __fadd_rn(acc, GradIO<GT>::load1(gp.p[q], f));
    return acc;
}

template <typename GT, bool PARAM, bool GOUT>
__global__ void __launch_bounds__(kThreads)
k_rs_adamw(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles, GradPtrs gp, int N,
           float* __restrict__ master, float* __restrict__ exp_avg, float* __restrict__ exp_avg_sq,
           uint16_t* __restrict__ param, float* __restrict__ gout, AdamScal sc) {
    int s = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t gt = tile_base + t;
        s = advance_seg(segs, s, gt);
        const Seg sg = segs[s];
        const int64_t e0 = (sg.shard / kVec + (gt - sg.tile0) * kThreads + threadIdx.x) * kVec;
        const int64_t lo = sg.shard, hi = sg.shard + sg.len;
        if (e0 >= hi) continue;
        const int64_t delta = sg.full - sg.shard;            // full index = shard index + delta

        if (e0 >= lo && e0 + kVec <= hi) {
            // ---- interior vector: 16-byte state traffic ----
            float4 p0 = ld4(master + e0), p1 = ld4(master + e0 + 4);
            float4 m0 = ld4(exp_avg + e0), m1 = ld4(exp_avg + e0 + 4);
            float4 v0 = ld4(exp_avg_sq + e0), v1 = ld4(exp_avg_sq + e0 + 4);
            float acc[8];
            if ((delta & (kVec - 1)) == 0) {
                reduce8_vec<GT>(gp, N, e0 + delta, acc);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] = reduce1<GT>(gp, N, e0 + delta + k);
            }
            float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            float g[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                g[k] = __fdiv_rn(acc[k], sc.nf);
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
            // ---- partial vector at a segment edge: element by element ----
            const int64_t a = e0 > lo ? e0 : lo;
            const int64_t b = (e0 + kVec) < hi ? (e0 + kVec) : hi;
            for (int64_t e = a; e < b; ++e) {
                const float g = __fdiv_rn(reduce1<GT>(gp, N, e + delta), sc.nf);
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
template <typename ET>
__global__ void __launch_bounds__(kThreads)
k_unshard(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles,
          const ET* __restrict__ src, ET* __restrict__ dst) {
    constexpr int kU4 = int(sizeof(ET)) * kVec / 16;   // 16-byte words per vector: 1 or 2
    int s = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t gt = tile_base + t;
        s = advance_seg(segs, s, gt);
        const Seg sg = segs[s];
        const int64_t e0 = (sg.shard / kVec + (gt - sg.tile0) * kThreads + threadIdx.x) * kVec;
        const int64_t lo = sg.shard, hi = sg.shard + sg.len;
        if (e0 >= hi) continue;
        const int64_t delta = sg.full - sg.shard;
        if (e0 >= lo && e0 + kVec <= hi && (delta & (kVec - 1)) == 0) {
            uint4 w[kU4];
#pragma unroll
            for (int k = 0; k < kU4; ++k) w[k] = ld_once(src + e0 + k * (16 / sizeof(ET)));
#pragma unroll
            for (int k = 0; k < kU4; ++k) stu4(dst + e0 + delta + k * (16 / sizeof(ET)), w[k]);
        } else {
            const int64_t a = e0 > lo ? e0 : lo;
            const int64_t b = (e0 + kVec) < hi ? (e0 + kVec) : hi;
            for (int64_t e = a; e < b; ++e) dst[e + delta] = src[e];
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
    int s = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t gt = tile_base + t;
        s = advance_seg(segs, s, gt);
        const Seg sg = segs[s];
        const int64_t e0 = (sg.shard / kVec + (gt - sg.tile0) * kThreads + threadIdx.x) * kVec;
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
    int s = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t gt = tile_base + t;
        s = advance_seg(segs, s, gt);
        const Seg sg = segs[s];
        const int64_t e0 = (sg.shard / kVec + (gt - sg.tile0) * kThreads + threadIdx.x) * kVec;
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
template <typename GT>
static cudaError_t launch_rs_t(const Seg* segs, int64_t tile_base, int64_t n_tiles, const GradPtrs& gp,
                               int N, float* master, float* m, float* v, uint16_t* param, float* gout,
                               const AdamScal& sc, cudaStream_t st) {
    if (param && gout) {
        auto k = k_rs_adamw<GT, true, true>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc);
    } else if (param) {
        auto k = k_rs_adamw<GT, true, false>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc);
    } else if (gout) {
        auto k = k_rs_adamw<GT, false, true>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc);
    } else {
        auto k = k_rs_adamw<GT, false, false>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc);
    }
    return cudaGetLastError();
}

cudaError_t launch_rs_adamw(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                            const GradPtrs& gp, int N, float* master, float* m, float* v,
                            uint16_t* param, float* gout, const AdamScal& sc, cudaStream_t st) {
    if (n_tiles <= 0) return cudaSuccess;
    return grad_bf16 ? launch_rs_t<uint16_t>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc, st)
                     : launch_rs_t<float>(segs, tile_base, n_tiles, gp, N, master, m, v, param, gout, sc, st);
}

cudaError_t launch_unshard(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool bf16,
                           const void* src, void* dst, cudaStream_t st) {
    if (n_tiles <= 0) return cudaSuccess;
    if (bf16) {
        auto k = k_unshard<uint16_t>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles,
                                                      static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst));
    } else {
        auto k = k_unshard<uint32_t>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles,
                                                      static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst));
    }
    return cudaGetLastError();
}

template <bool FB>
static cudaError_t launch_reshard_t(const Seg* segs, int64_t tile_base, int64_t n_tiles, const void* full,
                                    float* master, uint16_t* param, cudaStream_t st) {
    if (master && param) {
        auto k = k_reshard<FB, true, true>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, full, master, param);
    } else if (master) {
        auto k = k_reshard<FB, true, false>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, full, master, param);
    } else {
        auto k = k_reshard<FB, false, true>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, full, master, param);
    }
    return cudaGetLastError();
}

cudaError_t launch_reshard(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool full_bf16,
                           const void* full, float* master, uint16_t* param, cudaStream_t st) {
    if (n_tiles <= 0 || (!master && !param)) return cudaSuccess;
    return full_bf16 ? launch_reshard_t<true>(segs, tile_base, n_tiles, full, master, param, st)
                     : launch_reshard_t<false>(segs, tile_base, n_tiles, full, master, param, st);
}

cudaError_t launch_zero_pad(const Seg* segs, int64_t tile_base, int64_t n_tiles, float* a32, uint16_t* a16,
                            cudaStream_t st) {
    if (n_tiles <= 0 || (!a32 && !a16)) return cudaSuccess;
    if (a32 && a16) {
        auto k = k_zero_pad<true, true>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, a32, a16);
    } else if (a32) {
        auto k = k_zero_pad<true, false>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, a32, a16);
    } else {
        auto k = k_zero_pad<false, true>;
        k<<<grid_for(k, n_tiles), kThreads, 0, st>>>(segs, tile_base, n_tiles, a32, a16);
    }
    return cudaGetLastError();
}

}  // namespace fsdp
