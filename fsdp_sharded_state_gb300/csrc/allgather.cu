// allgather.cu -- the all-gather of the aligned class by bulk copies (sm_103a):
// global -> shared -> global with cp.async.bulk, no thread touching the data.
//
// "NCCL ZeRO/FSDP state sharding", "ZeRO-3 方向": all_gather_into_tensor of the N
// rank shards into the padded flat parameter; "第18章 FSDP" §18.8: FSDP2's copy-in /
// all-gather / copy-out.  The shifted class goes through k_unshard_shift (kernels.cu).
#include <type_traits>

#include "pipeline.cuh"
#include "staged.hpp"

namespace fsdp {
namespace {

// ----------------------------------------------------------------------------
// All-gather of the aligned class by bulk copies: global -> shared -> global.
// ----------------------------------------------------------------------------
// Pieces whose full-layout offset is congruent to their shard offset mod 8 start
// 16-byte aligned on both sides, so the bulk-copy engine can move them without a
// thread touching the data: per tile, one cp.async.bulk global->shared and one
// cp.async.bulk shared->global of its aligned interior.  Each CTA is one warp with
// a small ring of tile buffers (Ring below); 4 CTAs per SM.  Measured on GB300
// (bf16, 1-3 GB): as fast as a device copy of the same bytes; 1 or 3 loads ahead,
// 3, 5 or 8 CTAs per SM, or deeper rings were 2-8 % slower, and one CTA per SM
// with 8 loads ahead ran at 40 %.  Lane 0 issues the copies; the at most 7
// elements at each end of a segment that the copies leave out are copied by the
// warp's lanes with plain loads and stores.
constexpr int kUCtasPerSm = 4;
// Loads ahead and ring buffers per CTA: about 32 KB in flight per SM for both element
// sizes (bf16 tiles are 4 KB: 2 ahead; fp32 tiles 8 KB: 1 ahead).  Measured on GB300:
// fp32 128 MiB all-gather 44.2 us with 1 ahead against 46.5 us with 2.
template <int ES>
struct Ring {
    static constexpr int ahead = ES == 4 ? 1 : 2;
    static constexpr int size = ahead + 2;
};

template <int ES>
__global__ void __launch_bounds__(32)
k_unshard_bulk(const Seg* __restrict__ segs, int64_t tile_base, int64_t n_tiles, const unsigned char* src,
               unsigned char* dst, uint64_t wait_ns) {
    constexpr int64_t E = 16 / ES;              // elements per 16 bytes
    using W = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
    __shared__ __align__(128) unsigned char buf[Ring<ES>::size][kTileElems * ES];
    __shared__ __align__(8) uint64_t bars[Ring<ES>::size];
    const int lane = threadIdx.x;
    const int64_t G = gridDim.x;
    const int64_t n_mine = blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + G - 1) / G : 0;
    const uint32_t bar0 = smem_addr(&bars[0]);
    if (lane == 0) {
        for (int k = 0; k < Ring<ES>::size; ++k) mbar_init(bar0 + 8 * k, 1);
        mbar_fence_init();
    }
    __syncwarp();
    pdl_wait();

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
            const int k = int(j % Ring<ES>::size);
            const uint32_t bytes = p.b > p.a ? uint32_t(p.b - p.a) * ES : 0u;
            mbar_arrive_tx(bar0 + 8 * k, bytes);
            if (bytes) bulk_g2s(smem_addr(&buf[k][(p.a - p.t0) * ES]), src + p.a * ES, bytes, bar0 + 8 * k);
        }
    };
    for (int64_t j = 0; j < n_mine && j < Ring<ES>::ahead; ++j) load(j);
    int64_t j = 0;
    bool ok = true;
    for (; j < n_mine; ++j) {
        if (j + Ring<ES>::ahead < n_mine) {
            // buffer (j + ahead) mod ring was last stored from by tile j + ahead - ring
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(Ring<ES>::size - Ring<ES>::ahead - 1) : "memory");
            __syncwarp();
            load(j + Ring<ES>::ahead);
        }
        const int k = int(j % Ring<ES>::size);
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * k, uint32_t((j / Ring<ES>::size) & 1), wait_ns));
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
        for (int64_t q = j + 1; q < n_mine && q <= j + Ring<ES>::ahead; ++q)
            mbar_wait_bounded(bar0 + 8 * int(q % Ring<ES>::size), uint32_t((q / Ring<ES>::size) & 1), wait_ns);
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
}

}  // namespace

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
    if (bf16) return launch(k_unshard_bulk<2>, dim3(unsigned(blocks)), dim3(32), 0, st, segs, tile_base, n_tiles, s8, d8,
                            wait_ns);
    return launch(k_unshard_bulk<4>, dim3(unsigned(blocks)), dim3(32), 0, st, segs, tile_base, n_tiles, s8, d8, wait_ns);
}

cudaError_t take_wait_error_allgather(unsigned int* flag) { return take_local_wait_error(flag); }

}  // namespace fsdp
