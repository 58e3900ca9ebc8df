// noalloc.cu -- fsdp_reduce_scatter_adamw_noalloc: the fused reduce-scatter +
// AdamW + bf16 recast for callers that cannot allocate device memory.
//
// The regular entry point keeps each layout's segment table in device memory it
// allocates with cudaMalloc on first use.  Some callers cannot allow that: code
// running under a pre-sized memory pool or a custom allocator that owns all device
// memory, graph-building or real-time paths that must not hit the driver's
// allocator (cudaMalloc can synchronize the device and may fail under memory
// pressure mid-step), and embedders that forbid hidden allocations in a library.
// This variant instead stages the table in one fixed array that lives in the
// library image (it runs the same kernel as fsdp_reduce_scatter_adamw, staged or
// direct, neither of which allocates): `g_noalloc_segs` below, FSDP_NOALLOC_MAX_SEGMENTS entries of 32
// bytes (256 KiB), present on every GPU that loads the library until the process
// exits.  The entry point calls no cudaMalloc, cudaFree or other allocating
// routine.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fsdp_state.h"
#include "internal.hpp"
#include "kernels.hpp"
#include "layout.hpp"
#include "staged.hpp"

namespace {

using fsdp::Seg;

// The shared scratch.  Host code must not use this name as an address (on the
// host it is only a stand-in); it takes the device address from
// cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) Seg g_noalloc_segs[FSDP_NOALLOC_MAX_SEGMENTS];

constexpr int kMaxDevices = 64;
// Held by a call from its first table copy to its last launch, so that the copies and
// launches of two host threads on one stream are queued call by call, never
// interleaved (a kernel always reads the table its own call wrote).
std::mutex g_mu;
Seg* g_addr[kMaxDevices] = {};   // device address of g_noalloc_segs, per device (under g_mu)

// Set-up, once per device, with that device current: the device address of the
// scratch array.  (It loads the library's module on that device if needed.)  The
// cached address belongs to the device's current context: a cudaDeviceReset ends
// that context, so no call may follow one in this process.  Called under g_mu.
int scratch_address(Seg** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fsdp::detail::cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return FSDP_EINVAL;
    if (!g_addr[dev]) {
        Seg* p = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_segs);
        if (e != cudaSuccess) return fsdp::detail::cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
        if (!p) return FSDP_ECUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return FSDP_OK;
}

}  // namespace

extern "C" int fsdp_reduce_scatter_adamw_noalloc(const fsdp_layout* L, int32_t ub, int32_t ue,
                                                 const void* const* grads, int32_t grad_dtype, float* master,
                                                 float* exp_avg, float* exp_avg_sq, void* param_shards,
                                                 float* grad_shard_out, const fsdp_adamw_hparams* hp,
                                                 int64_t step, fsdp_stream_t stream) {
    fsdp::detail::NvtxRange nvtx_range("fsdp_reduce_scatter_adamw_noalloc");
    // ---- the same argument checks as fsdp_reduce_scatter_adamw ----
    int rc;
    if ((rc = fsdp::detail::check_units(L, ub, ue))) return rc;
    if (grad_dtype != FSDP_F32 && grad_dtype != FSDP_BF16) return FSDP_EDTYPE;
    if (!grads || !hp || step < 1) return FSDP_EINVAL;
    for (int32_t q = 0; q < L->N; ++q)
        if ((rc = fsdp::detail::check_ptr(grads[q]))) return rc;
    if ((rc = fsdp::detail::check_ptr(master)) || (rc = fsdp::detail::check_ptr(exp_avg)) ||
        (rc = fsdp::detail::check_ptr(exp_avg_sq)))
        return rc;
    if ((param_shards && !fsdp::detail::aligned16(param_shards)) ||
        (grad_shard_out && !fsdp::detail::aligned16(grad_shard_out)))
        return FSDP_EALIGN;
    if ((rc = fsdp::detail::check_hparams(hp))) return rc;
    if (L->mode == FSDP_ZERO1) return FSDP_EINVAL;

    // ---- the table entries this call reads: for each alignment class, the data
    //      segments of the unit range plus the entry after them (next unit's first
    //      segment or the sentinel); then, when grad_shard_out is given, the pad
    //      segments likewise ----
    const fsdp::SegList* cls[2] = {&L->data_al, &L->data_sh};
    int64_t n_cls[2];
    for (int c = 0; c < 2; ++c) n_cls[c] = int64_t(cls[c]->unit_begin[ue] - cls[c]->unit_begin[ub]) + 1;
    const int32_t pb = L->pad.unit_begin[ub], pe = L->pad.unit_begin[ue];
    const int64_t n_pad = grad_shard_out ? int64_t(pe - pb) + 1 : 0;
    if (n_cls[0] + n_cls[1] + n_pad > FSDP_NOALLOC_MAX_SEGMENTS) return FSDP_EINVAL;   // beyond the fixed scratch

    std::lock_guard<std::mutex> lk(g_mu);             // through the last launch of this call
    Seg* scratch = nullptr;
    if ((rc = scratch_address(&scratch))) return rc;

    const fsdp::AdamScal sc = fsdp::detail::adam_scalars(hp, step, L->N);
    fsdp::GradPtrs gp{};
    for (int32_t q = 0; q < L->N; ++q) gp.p[q] = grads[q];

    // The same kernel choice as fsdp_reduce_scatter_adamw (neither kernel allocates).
    const bool bf16 = grad_dtype == FSDP_BF16;
    bool staged = false;
    if ((rc = fsdp::detail::choose_staged(fsdp::staged_fits(L->N, bf16), true, &staged))) return rc;

    // Stream-ordered: the table is written before this call's kernels read it.
    // Nothing in the scratch needs to start at zero: every entry read is written first.
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    Seg* next = scratch;
    if (staged) {
        // one launch over the combined data list (fewer entries than the two classes)
        const int32_t sb = L->data.unit_begin[ub], se = L->data.unit_begin[ue];
        const int64_t n = int64_t(se - sb) + 1;
        e = cudaMemcpyAsync(next, L->data.segs.data() + sb, size_t(n) * sizeof(Seg), cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return fsdp::detail::cuda_fail(e, "cudaMemcpyAsync(no-allocation table)");
        const int64_t t0 = L->data.segs[sb].tile0, t1 = L->data.segs[se].tile0;
        // no claim counters: their ring is allocated on first use, and this call allocates nothing
        e = fsdp::launch_rs_adamw_staged(next, t0, t1 - t0, bf16, gp, L->N, master, exp_avg, exp_avg_sq,
                                         static_cast<uint16_t*>(param_shards), grad_shard_out, sc,
                                         fsdp::detail::kWaitNs, st, nullptr, false);
        if (e != cudaSuccess) return fsdp::detail::cuda_fail(e, "k_rs_adamw_staged launch");
        next += n;
    }
    for (int c = 0; c < 2 && !staged; ++c) {
        const int32_t sb = cls[c]->unit_begin[ub], se = cls[c]->unit_begin[ue];
        e = cudaMemcpyAsync(next, cls[c]->segs.data() + sb, size_t(n_cls[c]) * sizeof(Seg), cudaMemcpyHostToDevice,
                            st);
        if (e != cudaSuccess) return fsdp::detail::cuda_fail(e, "cudaMemcpyAsync(no-allocation table)");
        const int64_t t0 = cls[c]->segs[sb].tile0, t1 = cls[c]->segs[se].tile0;
        e = fsdp::launch_rs_adamw(next, t0, t1 - t0, c == 1, grad_dtype == FSDP_BF16, gp, L->N, L->F, master, exp_avg,
                                  exp_avg_sq, static_cast<uint16_t*>(param_shards), grad_shard_out, sc, st);
        if (e != cudaSuccess) return fsdp::detail::cuda_fail(e, "k_rs_adamw launch");
        next += n_cls[c];
    }
    if (grad_shard_out) {
        Seg* pad = next;
        e = cudaMemcpyAsync(pad, L->pad.segs.data() + pb, size_t(n_pad) * sizeof(Seg), cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return fsdp::detail::cuda_fail(e, "cudaMemcpyAsync(no-allocation pad table)");
        const int64_t q0 = L->pad.segs[pb].tile0, q1 = L->pad.segs[pe].tile0;
        e = fsdp::launch_zero_pad(pad, q0, q1 - q0, grad_shard_out, nullptr, st);
        if (e != cudaSuccess) return fsdp::detail::cuda_fail(e, "k_zero_pad launch");
    }
    return FSDP_OK;
}
