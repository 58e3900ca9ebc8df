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
//
// A launch with enough tiles claims them from a counter pair (claims.cu), as the
// pipeline kernels do: lane 0 starts on the CTA's own first kUClaimTiles tiles, then
// takes kUClaimTiles consecutive tiles per claim when it needs the next tile to load,
// and records each loaded tile in a small ring that the store side reads.  Measured on
// GB300, FULL_SHARD steps with two all-gathers: bf16 layouts from 2^24 to 2^29
// parameters (13 tiles per CTA and more) 0.3-2 % faster with the claims; fp32 (8 KB
// tiles, one load ahead) 1.2 % faster at 2^26 parameters (54 tiles per CTA) and 1 % at
// 2^28, but 0.2-1 % slower at 2^25 (27 tiles per CTA: the 128 MiB layouts), so fp32
// claims from kUClaimMinTilesPerCtaF32 tiles per CTA.
constexpr int kUCtasPerSm = 4;
constexpr int kUClaimTiles = 2;                 // tiles per claim
constexpr int64_t kUClaimMinTilesPerCta = 8;    // shorter launches split their tiles statically
constexpr int64_t kUClaimMinTilesPerCtaF32 = 48;
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
               unsigned char* dst, uint64_t wait_ns, unsigned int* claim) {
    constexpr int64_t E = 16 / ES;              // elements per 16 bytes
    using W = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
    __shared__ __align__(128) unsigned char buf[Ring<ES>::size][kTileElems * ES];
    __shared__ __align__(8) uint64_t bars[Ring<ES>::size];
    __shared__ int64_t seq[Ring<ES>::size];     // the tile of item j, at j mod size
    const int lane = threadIdx.x;
    const int64_t G = gridDim.x;
    // items of this CTA: known with the static split, else found when the claims run out
    int64_t n_mine = claim ? INT64_MAX : (blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + G - 1) / G : 0);
    unsigned int next = 0;                      // lane 0: the claim in flight
    // lane 0: what is left of the current batch; the first is the CTA's own, [b B, b B + B),
    // so no claim is waited for at the start, and the claims hand out the tiles from G B on
    int64_t bat = int64_t(blockIdx.x) * kUClaimTiles;
    int64_t bat_end = bat + kUClaimTiles < n_tiles ? bat + kUClaimTiles : n_tiles;
    if (claim && lane == 0) next = atomicAdd(claim, unsigned(kUClaimTiles));
    const uint32_t bar0 = smem_addr(&bars[0]);
    if (lane == 0) {
        for (int k = 0; k < Ring<ES>::size; ++k) mbar_init(bar0 + 8 * k, 1);
        mbar_fence_init();
    }
    __syncwarp();
    pdl_wait();

    struct Piece { int64_t t0, s0, s1, delta, a, b; };     // tile range, aligned interior [a, b)
    auto piece = [&](int& cur, int64_t t) {
        const int64_t gt = tile_base + t;
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
    // Loads item j (lane 0; j one more each call): its tile -- the static split's, or the
    // next of the claimed batch, claiming again when it is used up -- into seq, or, when
    // there is none, n_mine = j.  Every lane then takes n_mine from lane 0.
    auto load = [&](int64_t j) {
        if (lane == 0) {
            int64_t t;
            if (claim) {
                if (bat >= bat_end) {
                    const int64_t c = G * kUClaimTiles + int64_t(next);
                    bat = c;
                    bat_end = c + kUClaimTiles < n_tiles ? c + kUClaimTiles : n_tiles;
                    if (c < n_tiles) next = atomicAdd(claim, unsigned(kUClaimTiles));
                }
                t = bat < bat_end ? bat++ : n_tiles;
            } else {
                t = blockIdx.x + j * G;
            }
            if (t >= n_tiles) {
                n_mine = j;
            } else {
                const int k = int(j % Ring<ES>::size);
                seq[k] = t;
                const Piece p = piece(load_cur, t);
                const uint32_t bytes = p.b > p.a ? uint32_t(p.b - p.a) * ES : 0u;
                mbar_arrive_tx(bar0 + 8 * k, bytes);
                if (bytes) bulk_g2s(smem_addr(&buf[k][(p.a - p.t0) * ES]), src + p.a * ES, bytes, bar0 + 8 * k);
            }
        }
        n_mine = __shfl_sync(0xffffffffu, n_mine, 0);
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
        __syncwarp();
        const Piece p = piece(store_cur, seq[k]);
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
    if (claim && lane == 0) {
        // done claiming (here on every path): the last CTA out leaves the pair at zero
        __threadfence();
        if (atomicAdd(claim + 1, 1u) == unsigned(G) - 1u) {
            atomicExch(claim, 0u);
            atomicExch(claim + 1, 0u);
        }
    }
    __syncwarp();
}

}  // namespace

cudaError_t launch_unshard_bulk(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool bf16, const void* src,
                                void* dst, uint64_t wait_ns, cudaStream_t st, bool claims) {
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
    unsigned int* claim = nullptr;
    int slot = -1, cdev = -1;
    if (claims && n_tiles >= (bf16 ? kUClaimMinTilesPerCta : kUClaimMinTilesPerCtaF32) * blocks &&
        n_tiles < (int64_t(1) << 31))
        claim = claim_acquire(st, &slot, &cdev);
    e = bf16 ? launch(k_unshard_bulk<2>, dim3(unsigned(blocks)), dim3(32), 0, st, segs, tile_base, n_tiles, s8, d8,
                      wait_ns, claim)
             : launch(k_unshard_bulk<4>, dim3(unsigned(blocks)), dim3(32), 0, st, segs, tile_base, n_tiles, s8, d8,
                      wait_ns, claim);
    claim_release(slot, cdev, st, e == cudaSuccess);
    return e;
}

cudaError_t take_wait_error_allgather(unsigned int* flag) { return take_local_wait_error(flag); }

}  // namespace fsdp
