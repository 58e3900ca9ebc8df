// device_ops.cuh -- device building blocks shared by the libfsdpstate kernels:
// the AdamW element update, gradient vector I/O, and the reductions over the N
// gradient replicas (aligned vectors, warp-realigned vectors, single elements).
#pragma once

#include "common.cuh"

namespace fsdp {

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

// ----------------------------------------------------------------------------
// The mean's division x / n by the rank count n (a float holding an integer >= 1).
// When n is a power of two, 1/n is exact, so x * (1/n) is the same real number as
// x / n and rounds to the same float -- subnormal results, zeros and infinities
// included -- for far fewer instructions than an IEEE division.  Otherwise the
// division.  (n is the same for a whole launch: the test and the reciprocal are loop
// invariants.)
// ----------------------------------------------------------------------------
__device__ __forceinline__ float mean_div(float x, float n) {
    const bool pow2 = (__float_as_uint(n) & 0x807FFFFFu) == 0u && n >= 1.0f;
    return pow2 ? __fmul_rn(x, __frcp_rn(n)) : __fdiv_rn(x, n);
}

template <typename GT> struct GradIO;

// bf16 gradients: one 16-byte load per replica covers the 8 elements.
template <> struct GradIO<uint16_t> {
    static constexpr int kBatch = 8;
    static constexpr int kWords = 4;                 // 32-bit words per 8-element vector
    struct Vec { uint32_t w[4]; };
    static __device__ __forceinline__ Vec load(const void* base, int64_t i) {
        const uint4 x = ld_once(static_cast<const uint16_t*>(base) + i);
        return Vec{{x.x, x.y, x.z, x.w}};
    }
    // element e (0..15) of the window [A, B], as fp32 (bf16 widens exactly)
    static __device__ __forceinline__ float elem(const Vec& A, const Vec& B, int e) {
        const uint32_t w = e < 8 ? A.w[e >> 1] : B.w[(e - 8) >> 1];
        return (e & 1) ? bf16hi(w) : bf16lo(w);
    }
    static __device__ __forceinline__ float load1(const void* base, int64_t i) {
        return bf16f(static_cast<const uint16_t*>(base)[i]);
    }
};

// fp32 gradients: two 16-byte loads per replica.
template <> struct GradIO<float> {
    static constexpr int kBatch = 4;
    static constexpr int kWords = 8;
    struct Vec { uint32_t w[8]; };
    static __device__ __forceinline__ Vec load(const void* base, int64_t i) {
        const float* p = static_cast<const float*>(base) + i;
        const uint4 a = ld_once(p), b = ld_once(p + 4);
        return Vec{{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
    }
    static __device__ __forceinline__ float elem(const Vec& A, const Vec& B, int e) {
        return __uint_as_float(e < 8 ? A.w[e] : B.w[e - 8]);
    }
    static __device__ __forceinline__ float load1(const void* base, int64_t i) {
        return static_cast<const float*>(base)[i];
    }
};

template <typename V>
__device__ __forceinline__ V shfl_down1(const V& v) {
    V r;
#pragma unroll
    for (int k = 0; k < int(sizeof(v.w) / 4); ++k) r.w[k] = __shfl_down_sync(0xffffffffu, v.w[k], 1);
    return r;
}

// Sum of the N replicas at 8 consecutive full-layout elements starting at f
// (16-byte aligned), in rank order.  Loads are issued in batches so that a batch
// is in flight together.
// (Replicas gp.p[first .. first+N).)
template <typename GT>
__device__ __forceinline__ void reduce8_vec(const GradPtrs& gp, int N, int64_t f, float (&acc)[8], int first = 0) {
    using IO = GradIO<GT>;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
#pragma unroll 1
    for (int q0 = 0; q0 < N; q0 += IO::kBatch) {
        typename IO::Vec buf[IO::kBatch];
#pragma unroll
        for (int b = 0; b < IO::kBatch; ++b)
            if (q0 + b < N) buf[b] = IO::load(gp.p[first + q0 + b], f);
#pragma unroll
        for (int b = 0; b < IO::kBatch; ++b)
            if (q0 + b < N) {
                const typename IO::Vec& x = buf[b];
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] = __fadd_rn(acc[k], IO::elem(x, x, k));
            }
    }
}

// Elements d..d+7 (d in 1..7, warp-uniform) of the 16-element window [A, B] as fp32.
__device__ __forceinline__ void window8(const GradIO<uint16_t>::Vec& A, const GradIO<uint16_t>::Vec& B, int d,
                                        float (&out)[8]) {
    const uint32_t w[8] = {A.w[0], A.w[1], A.w[2], A.w[3], B.w[0], B.w[1], B.w[2], B.w[3]};
    uint32_t x[5];
    switch (d >> 1) {                       // whole 32-bit words first ...
        case 0: x[0] = w[0]; x[1] = w[1]; x[2] = w[2]; x[3] = w[3]; x[4] = w[4]; break;
        case 1: x[0] = w[1]; x[1] = w[2]; x[2] = w[3]; x[3] = w[4]; x[4] = w[5]; break;
        case 2: x[0] = w[2]; x[1] = w[3]; x[2] = w[4]; x[3] = w[5]; x[4] = w[6]; break;
        default: x[0] = w[3]; x[1] = w[4]; x[2] = w[5]; x[3] = w[6]; x[4] = w[7]; break;
    }
    const bool odd = d & 1;                 // ... then one bf16 if d is odd
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t y = odd ? __funnelshift_r(x[k], x[k + 1], 16) : x[k];
        out[2 * k] = bf16lo(y);
        out[2 * k + 1] = bf16hi(y);
    }
}

template <int D>
__device__ __forceinline__ void window8_f32(const GradIO<float>::Vec& A, const GradIO<float>::Vec& B,
                                            uint32_t (&x)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = (D + k) < 8 ? A.w[(D + k) & 7] : B.w[(D + k - 8) & 7];
}

__device__ __forceinline__ void window8(const GradIO<float>::Vec& A, const GradIO<float>::Vec& B, int d,
                                        float (&out)[8]) {
    uint32_t x[8];
    switch (d) {
        case 1: window8_f32<1>(A, B, x); break;
        case 2: window8_f32<2>(A, B, x); break;
        case 3: window8_f32<3>(A, B, x); break;
        case 4: window8_f32<4>(A, B, x); break;
        case 5: window8_f32<5>(A, B, x); break;
        case 6: window8_f32<6>(A, B, x); break;
        default: window8_f32<7>(A, B, x); break;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) out[k] = __uint_as_float(x[k]);
}

// The same sum when the 8 full-layout elements start d elements (warp-uniform,
// 1..7) past a 16-byte boundary fa.  Warp-collective: every lane loads its own
// aligned vector A at fa, takes its neighbour's (the next aligned vector) with a
// shuffle and reads elements d..d+7 of the pair; lane 31 loads the next vector
// itself.  have_a / have_b say whether A / the next vector lie inside the buffer.
template <typename GT>
__device__ __forceinline__ void reduce8_shift(int d, const GradPtrs& gp, int N, int64_t fa, bool have_a,
                                              bool have_b, bool lane31, float (&acc)[8]) {
    using IO = GradIO<GT>;
    constexpr int kB = IO::kWords == 4 ? 8 : 4;     // replicas in flight per batch
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
#pragma unroll 1
    for (int q0 = 0; q0 < N; q0 += kB) {
        typename IO::Vec A[kB], B[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            if (q0 + b < N) {
                A[b] = have_a ? IO::load(gp.p[q0 + b], fa) : typename IO::Vec{};
                B[b] = (lane31 && have_b) ? IO::load(gp.p[q0 + b], fa + kVec) : typename IO::Vec{};
            }
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            if (q0 + b < N) {                                   // uniform: all lanes shuffle
                const typename IO::Vec nb = shfl_down1(A[b]);
                float x[8];
                window8(A[b], lane31 ? B[b] : nb, d, x);
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] = __fadd_rn(acc[k], x[k]);
            }
        }
    }
}

// Sum, in rank order, of the N fp32 replicas at the two 4-element chunks a lane owns
// under the "split" mapping (full-layout offsets fa and fb, 16-byte aligned): acc[0..3]
// for fa, acc[4..7] for fb; 2 replicas x 2 chunks in flight.
__device__ __forceinline__ void reduce_split_f32(const GradPtrs& gp, int N, int64_t fa, int64_t fb,
                                                 float (&acc)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
#pragma unroll 1
    for (int q0 = 0; q0 < N; q0 += 2) {
        uint4 ga[2], gb[2];
#pragma unroll
        for (int b = 0; b < 2; ++b)
            if (q0 + b < N) {
                const float* g = static_cast<const float*>(gp.p[q0 + b]);
                ga[b] = ld_once(g + fa);
                gb[b] = ld_once(g + fb);
            }
#pragma unroll
        for (int b = 0; b < 2; ++b)
            if (q0 + b < N) {
                acc[0] = __fadd_rn(acc[0], __uint_as_float(ga[b].x));
                acc[1] = __fadd_rn(acc[1], __uint_as_float(ga[b].y));
                acc[2] = __fadd_rn(acc[2], __uint_as_float(ga[b].z));
                acc[3] = __fadd_rn(acc[3], __uint_as_float(ga[b].w));
                acc[4] = __fadd_rn(acc[4], __uint_as_float(gb[b].x));
                acc[5] = __fadd_rn(acc[5], __uint_as_float(gb[b].y));
                acc[6] = __fadd_rn(acc[6], __uint_as_float(gb[b].z));
                acc[7] = __fadd_rn(acc[7], __uint_as_float(gb[b].w));
            }
    }
}

template <typename GT>
__device__ __forceinline__ float reduce1(const GradPtrs& gp, int N, int64_t f) {
    float acc = 0.0f;
#pragma unroll 1
    for (int q = 0; q < N; ++q) acc = __fadd_rn(acc, GradIO<GT>::load1(gp.p[q], f));
    return acc;
}

}  // namespace fsdp
