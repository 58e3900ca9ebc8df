// common.cuh -- shared definitions of the libfsdpstate kernels (device side).
//
// Work decomposition used by every kernel: a launch covers a contiguous range of
// "segments".  A segment is one contiguous piece of one rank's shard row that maps
// to one contiguous piece of the full layout:
//     shard element  x in [shard, shard + len)   <->   full element  x - shard + full.
// Segments are cut into tiles of kThreads vectors of kVec elements; vectors are
// aligned on the SHARD side (vector v covers shard elements [8v, 8v+8)), so the
// first and last vector of a segment may be partial.  Tile prefix sums (tile0) let
// a persistent grid walk the tiles of any unit range in order.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace fsdp {

constexpr int kVec = 8;                       // elements per thread per tile
constexpr int kThreads = 256;                 // threads per CTA
constexpr int64_t kTileElems = int64_t(kVec) * kThreads;
constexpr int kMaxRanks = 64;

struct Seg {
    int64_t shard;   // absolute element index in the [N][stride] shard arrays
    int64_t full;    // absolute element index in the full layout (-1: none, padding)
    int64_t len;     // elements
    int64_t tile0;   // index of the segment's first tile in its list
};

// First vector of a segment's first tile: tiles sit on absolute multiples of
// kTileElems shard elements, so every warp's accesses are whole cache lines
// whatever the row stride.
__host__ __device__ inline int64_t seg_vec0(int64_t shard) { return (shard / kTileElems) * kThreads; }

// Tiles a segment occupies.
__host__ __device__ inline int64_t seg_tiles(int64_t shard, int64_t len) {
    if (len <= 0) return 0;
    const int64_t v0 = seg_vec0(shard);
    const int64_t v1 = (shard + len + kVec - 1) / kVec;
    return (v1 - v0 + kThreads - 1) / kThreads;
}

struct GradPtrs {
    const void* p[kMaxRanks];
};

// Per-step AdamW constants, each formed on the host in double and rounded once.
struct AdamScal {
    float decay;       // 1 - lr*wd
    float om1, om2;    // 1 - beta1, 1 - beta2
    float step_size;   // lr / (1 - beta1^t)
    float bc2s;        // sqrt(1 - beta2^t)
    float beta1, beta2, eps;
    float nf;          // (float)N, the divisor of the mean
};

#ifdef __CUDACC__
// ---- raw bf16 <-> fp32 (bf16 is the top half of a binary32) ---------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

// Two fp32 -> packed bf16x2, round to nearest even (CUDA's conversion).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}
__device__ __forceinline__ uint16_t to_bf16(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ---- 16-byte memory operations ---------------------------------------------------
// Gradient replicas are read exactly once per step: stream them past L1.  The asm
// is volatile with a memory clobber, so the compiler keeps it after pdl_wait() (and
// in order with every other memory access) whatever the address depends on: a
// replica written by the grid before this one is never read ahead of the wait.
__device__ __forceinline__ uint4 ld_once(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
    return r;
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ uint4 ldu4(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void stu4(void* p, uint4 x) { *reinterpret_cast<uint4*>(p) = x; }

// Finds, for tile gt, the segment that holds it, starting from the caller's cached
// index s (tiles are visited in increasing order by each CTA).
__device__ __forceinline__ int advance_seg(const Seg* __restrict__ segs, int s, int64_t gt) {
    while (segs[s + 1].tile0 <= gt) ++s;
    return s;
}

// ---- programmatic dependent launch ---------------------------------------------
// Every kernel of the library is launched with programmatic stream serialization
// (launch() below) and calls pdl_wait() before its first global-memory access: it
// waits there until the grid before it on the stream has completed with its memory
// visible (at once when there is none to wait for).  Nothing is read or written
// before the wait, so every ordering the stream gives is kept.  No kernel triggers
// its dependents early: the next grid launches as this one's CTAs exit (the
// implicit trigger), so its launch overlaps this grid's tail and memory flush
// instead of following them.  Measured on GB300 against plain launches: FULL_SHARD
// step on the 128 MiB fp32 layout 275.8 against 283.0 us, on 2^24+1 bf16 at N = 8
// 129.3 against 136.3 us, the 4-block Llama unchanged.  An early trigger (at kernel
// entry) made the staged reduce-scatter 2.4 % slower on bf16 layouts, its CTAs
// then waiting resident beside the all-gather's.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}
#endif  // __CUDACC__

}  // namespace fsdp
