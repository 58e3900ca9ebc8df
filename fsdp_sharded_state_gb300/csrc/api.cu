// api.cu -- the extern "C" entry points of libfsdpstate (declared in
// include/fsdp_state.h): argument validation, per-device segment tables, the
// AdamW step constants and the kernel launches.  Every check runs before the
// first launch, so an error return leaves all outputs untouched.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/fsdp_state.h"
#include "internal.hpp"
#include "kernels.hpp"
#include "layout.hpp"
#include "staged.hpp"

using fsdp::Seg;
using fsdp::SegList;

namespace fsdp {
namespace detail {

thread_local char g_cuda_err[256] = "";

// Kernel choice of the reduce-scatter calls (fsdp_rs_kernel).
std::atomic<int> g_rs_kernel{FSDP_RS_AUTO};

int choose_staged(bool fits, bool preferred, bool* staged) {
    const int kind = g_rs_kernel.load();
    if (kind == FSDP_RS_STAGED && !fits) return FSDP_EINVAL;
    *staged = kind == FSDP_RS_STAGED || (kind == FSDP_RS_AUTO && fits && preferred);
    return FSDP_OK;
}

int rs_kernel_choice() { return g_rs_kernel.load(); }

int cuda_fail(cudaError_t e, const char* where) {
    std::snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s (%s)", where, cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return FSDP_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device copy of the layout's three segment lists for the current device.
int device_tables(const fsdp_layout* Lc, const Seg** base) {
    fsdp_layout* L = const_cast<fsdp_layout*>(Lc);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(L->mu);
    auto it = L->dev.find(dev);
    if (it != L->dev.end()) {
        *base = it->second.base;
        return FSDP_OK;
    }
    const SegList* lists[] = {&L->data, &L->gather, &L->pad, &L->data_al, &L->data_sh, &L->gather_al, &L->gather_sh,
                              &L->fullr};
    size_t n = 0;
    for (const SegList* l : lists) n += l->segs.size();
    Seg* d = nullptr;
    e = cudaMalloc(&d, n * sizeof(Seg));
    if (e != cudaSuccess) {
        cuda_fail(e, "cudaMalloc(segment tables)");
        return FSDP_ENOMEM;
    }
    std::vector<Seg> h;
    h.reserve(n);
    for (const SegList* l : lists) h.insert(h.end(), l->segs.begin(), l->segs.end());   // dev_off order
    e = cudaMemcpy(d, h.data(), n * sizeof(Seg), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(d);
        return cuda_fail(e, "cudaMemcpy(segment tables)");
    }
    L->dev[dev] = fsdp::DeviceTables{d};
    *base = d;
    return FSDP_OK;
}

Range range_of(const SegList& l, const Seg* dev_base, int32_t ub, int32_t ue) {
    const int32_t sb = l.unit_begin[ub], se = l.unit_begin[ue];
    const int64_t t0 = l.segs[sb].tile0, t1 = l.segs[se].tile0;
    return Range{dev_base + l.dev_off + sb, t0, t1 - t0, se - sb};
}

int check_units(const fsdp_layout* L, int32_t ub, int32_t ue) {
    if (!L) return FSDP_EINVAL;
    if (ub < 0 || ue > L->U || ub > ue) return FSDP_EINVAL;
    return FSDP_OK;
}

int check_ptr(const void* p) {
    if (!p) return FSDP_EINVAL;
    if (!aligned16(p)) return FSDP_EALIGN;
    return FSDP_OK;
}

int check_hparams(const fsdp_adamw_hparams* hp) {
    if (!hp) return FSDP_EINVAL;
    const float lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps, wd = hp->weight_decay;
    if (!std::isfinite(lr) || !std::isfinite(b1) || !std::isfinite(b2) || !std::isfinite(eps) ||
        !std::isfinite(wd))
        return FSDP_EINVAL;
    if (lr < 0.f || b1 < 0.f || b1 >= 1.f || b2 < 0.f || b2 >= 1.f || eps <= 0.f || wd < 0.f ||
        double(lr) * double(wd) > 1.0)
        return FSDP_EINVAL;
    return FSDP_OK;
}

AdamScal adam_scalars(const fsdp_adamw_hparams* hp, int64_t step, int32_t n_avg) {
    // formed in double from the fp32 hyper-parameters, rounded once
    AdamScal sc;
    const double b1 = hp->beta1, b2 = hp->beta2, lr = hp->lr, wd = hp->weight_decay;
    const double bc1 = 1.0 - std::pow(b1, double(step));
    const double bc2 = 1.0 - std::pow(b2, double(step));
    sc.decay = float(1.0 - lr * wd);
    sc.om1 = float(1.0 - b1);
    sc.om2 = float(1.0 - b2);
    sc.step_size = float(lr / bc1);
    sc.bc2s = float(std::sqrt(bc2));
    sc.beta1 = hp->beta1;
    sc.beta2 = hp->beta2;
    sc.eps = hp->eps;
    sc.nf = float(n_avg);
    return sc;
}

// The buffer and layout checks of the fused step (hyper-parameters aside), in the
// order the fused entry points apply them.
int check_rs_buffers(const fsdp_layout* L, int32_t ub, int32_t ue, const void* const* grads, int32_t grad_dtype,
                     const float* master, const float* exp_avg, const float* exp_avg_sq, const void* param_shards,
                     const float* grad_shard_out) {
    int rc = check_units(L, ub, ue);
    if (rc) return rc;
    if (grad_dtype != FSDP_F32 && grad_dtype != FSDP_BF16) return FSDP_EDTYPE;
    if (!grads) return FSDP_EINVAL;
    for (int32_t q = 0; q < L->N; ++q)
        if ((rc = check_ptr(grads[q]))) return rc;
    if ((rc = check_ptr(master)) || (rc = check_ptr(exp_avg)) || (rc = check_ptr(exp_avg_sq))) return rc;
    if (param_shards && !aligned16(param_shards)) return FSDP_EALIGN;
    if (grad_shard_out && !aligned16(grad_shard_out)) return FSDP_EALIGN;
    if (L->mode == FSDP_ZERO1) return FSDP_EINVAL;
    return FSDP_OK;
}

// The device block of the step constants is read by the kernels as an AdamScal.
static_assert(sizeof(fsdp_adamw_step_consts) == 48, "step constants block");
static_assert(offsetof(fsdp_adamw_step_consts, decay) == offsetof(AdamScal, decay) &&
                  offsetof(fsdp_adamw_step_consts, om1) == offsetof(AdamScal, om1) &&
                  offsetof(fsdp_adamw_step_consts, om2) == offsetof(AdamScal, om2) &&
                  offsetof(fsdp_adamw_step_consts, step_size) == offsetof(AdamScal, step_size) &&
                  offsetof(fsdp_adamw_step_consts, bc2s) == offsetof(AdamScal, bc2s) &&
                  offsetof(fsdp_adamw_step_consts, beta1) == offsetof(AdamScal, beta1) &&
                  offsetof(fsdp_adamw_step_consts, beta2) == offsetof(AdamScal, beta2) &&
                  offsetof(fsdp_adamw_step_consts, eps) == offsetof(AdamScal, eps) &&
                  offsetof(fsdp_adamw_step_consts, n_avg) == offsetof(AdamScal, nf),
              "step constants block matches AdamScal");

}  // namespace detail
}  // namespace fsdp

using namespace fsdp::detail;

extern "C" {

int fsdp_layout_create(int32_t n_tensors, const int32_t* ndim, const int64_t* dims, const int32_t* unit_id,
                       const int32_t* dtype, int32_t n_ranks, int32_t mode, fsdp_layout** out) {
    if (!out) return FSDP_EINVAL;
    if (n_tensors > (1 << 24)) return FSDP_EINVAL;
    fsdp_layout* L = new (std::nothrow) fsdp_layout();
    if (!L) return FSDP_ENOMEM;
    int rc;
    try {
        rc = fsdp::build_layout(L, n_tensors, ndim, dims, unit_id, dtype, n_ranks, mode);
    } catch (const std::bad_alloc&) {
        rc = FSDP_ENOMEM;
    }
    if (rc != FSDP_OK) {
        delete L;
        return rc;
    }
    *out = L;
    return FSDP_OK;
}

void fsdp_layout_destroy(fsdp_layout* L) {
    if (!L) return;
    int cur = -1;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    for (auto& kv : L->dev) {
        if (cudaSetDevice(kv.first) == cudaSuccess) cudaFree(kv.second.base);
    }
    if (have_cur && !L->dev.empty()) cudaSetDevice(cur);
    delete L;
}

int fsdp_layout_query(const fsdp_layout* L, fsdp_layout_info* o) {
    if (!L || !o) return FSDP_EINVAL;
    o->n_tensors = L->T;
    o->n_units = L->U;
    o->n_ranks = L->N;
    o->mode = L->mode;
    o->numel = L->P;
    o->shard_numel = L->S;
    o->shard_stride = L->stride;
    o->full_numel = L->F;
    o->pad_numel = int64_t(L->N) * L->S - L->P;
    o->n_segments = L->n_data_segments;
    return FSDP_OK;
}

int fsdp_layout_unit(const fsdp_layout* L, int32_t u, int64_t* shard_off, int64_t* shard_numel,
                     int64_t* full_off, int64_t* full_numel, int64_t* numel) {
    if (!L || u < 0 || u >= L->U) return FSDP_EINVAL;
    if (shard_off) *shard_off = L->u_shard_off[u];
    if (shard_numel) *shard_numel = L->u_S[u];
    if (full_off) *full_off = L->u_full_off[u];
    if (full_numel) *full_numel = L->mode == FSDP_FLAT ? int64_t(L->N) * L->u_S[u] : L->u_numel[u];
    if (numel) *numel = L->u_numel[u];
    return FSDP_OK;
}

int fsdp_layout_tensor(const fsdp_layout* L, int32_t t, int32_t* unit, int64_t* numel, int64_t* full_off,
                       int64_t* shard_off, int64_t* rows_per_rank) {
    if (!L || t < 0 || t >= L->T) return FSDP_EINVAL;
    if (unit) *unit = L->unit[t];
    if (numel) *numel = L->numel[t];
    if (full_off) *full_off = L->t_full_off[t];
    if (shard_off) *shard_off = L->mode != FSDP_FLAT ? L->t_shard_off[t] : -1;
    if (rows_per_rank) *rows_per_rank = L->mode == FSDP_DIM0 ? L->rows[t] : -1;
    return FSDP_OK;
}

int fsdp_layout_segment(const fsdp_layout* L, int32_t t, int32_t r, int64_t* shard_off, int64_t* full_off,
                        int64_t* len, int64_t* pad) {
    if (!L || t < 0 || t >= L->T || r < 0 || r >= L->N) return FSDP_EINVAL;
    int64_t so, fo, n, pd;
    if (L->mode == FSDP_ZERO1) {
        so = L->t_shard_off[t];
        fo = L->t_full_off[t];
        n = L->owner[t] == r ? L->numel[t] : 0;
        pd = 0;
    } else if (L->mode == FSDP_FLAT) {
        const int32_t u = L->unit[t];
        const int64_t Su = L->u_S[u];
        const int64_t a = L->t_unit_off[t], b = a + L->numel[t];   // tensor range in the unit's flat
        const int64_t ra = int64_t(r) * Su, rb = ra + Su;          // rank range
        int64_t lo = a < ra ? ra : a;
        if (lo > rb) lo = rb;
        const int64_t hi = b < rb ? b : rb;
        n = hi > lo ? hi - lo : 0;
        so = L->u_shard_off[u] + (lo - ra);
        fo = L->u_full_off[u] + lo;
        pd = 0;
    } else {
        const int64_t c = L->rows[t];
        const int64_t rb = std::min<int64_t>(int64_t(r) * c, L->d0[t]);
        const int64_t re = std::min<int64_t>(int64_t(r + 1) * c, L->d0[t]);
        n = (re - rb) * L->inner[t];
        so = L->t_shard_off[t];
        fo = L->t_full_off[t] + rb * L->inner[t];
        pd = c * L->inner[t] - n;
    }
    if (shard_off) *shard_off = so;
    if (full_off) *full_off = fo;
    if (len) *len = n;
    if (pad) *pad = pd;
    return FSDP_OK;
}

int fsdp_layout_owner(const fsdp_layout* L, int32_t t, int32_t* rank) {
    if (!L || t < 0 || t >= L->T || !rank) return FSDP_EINVAL;
    if (L->mode != FSDP_ZERO1) return FSDP_EINVAL;
    *rank = L->owner[t];
    return FSDP_OK;
}

int fsdp_state_bytes(const fsdp_layout* L, int32_t stage, int32_t rank, int32_t physical, int64_t pb,
                     int64_t gb, int64_t ob, int64_t step_bytes, int64_t out[3]) {
    if (!L || !out || stage < 0 || stage > 3 || rank < 0 || rank >= L->N) return FSDP_EINVAL;
    if (pb < 0 || gb < 0 || ob < 0 || step_bytes < 0) return FSDP_EINVAL;
    int64_t own = 0;
    if (physical) {
        own = L->S;
    } else {
        // Logical elements of this rank: the data segments in its row.
        const int64_t lo = int64_t(rank) * L->stride, hi = lo + L->stride;
        for (size_t i = 0; i + 1 < L->data.segs.size(); ++i) {   // the list's last entry is its sentinel
            const Seg& s = L->data.segs[i];
            if (s.shard >= lo && s.shard < hi) own += s.len;
        }
    }
    const int64_t sharded_or_full[2] = {L->P, own};
    out[0] = sharded_or_full[stage >= 3] * pb;
    out[1] = sharded_or_full[stage >= 2] * gb;
    out[2] = sharded_or_full[stage >= 1] * ob + int64_t(L->T) * step_bytes;
    return FSDP_OK;
}

int fsdp_collective_payload(const fsdp_layout* L, int32_t strategy, int32_t n_groups,
                            fsdp_collective_payload_info* out) {
    if (!L || !out || strategy < FSDP_NO_SHARD || strategy > FSDP_HYBRID_SHARD || n_groups < 1) return FSDP_EINVAL;
    if (strategy != FSDP_HYBRID_SHARD && n_groups != 1) return FSDP_EINVAL;
    // Collectives of one step per strategy, as multiples of the layout's P: all-reduce,
    // forward all-gather, backward all-gather, reduce-scatter, broadcast.
    static const int8_t kUses[5][5] = {
        {1, 0, 0, 0, 0},   // NO_SHARD: the gradient all-reduce
        {1, 0, 0, 0, 1},   // ZeRO-1: the same, then the updated parameters broadcast by their owners
        {0, 1, 0, 1, 0},   // SHARD_GRAD_OP
        {0, 1, 1, 1, 0},   // FULL_SHARD
        {0, 1, 1, 1, 0},   // HYBRID_SHARD inside a group; its all-reduce across groups is added below
    };
    const int8_t* u = kUses[strategy];
    out->allreduce_input = u[0] * L->P;
    out->forward_allgather = u[1] * L->P;
    out->backward_allgather = u[2] * L->P;
    out->reducescatter_input = u[3] * L->P;
    out->broadcast = u[4] * L->P;
    // Ring algorithms, elements one rank sends: all-gather, reduce-scatter and the
    // owners' broadcast pass on (N-1) of N chunks of the buffer; an all-reduce is a
    // reduce-scatter followed by an all-gather, twice that.
    const double N = double(L->N);
    const double gather_like = double(out->forward_allgather + out->backward_allgather + out->reducescatter_input +
                                      out->broadcast);
    double bus = gather_like * (N - 1.0) / N + 2.0 * double(out->allreduce_input) * (N - 1.0) / N;
    if (strategy == FSDP_HYBRID_SHARD) {
        // the reduced shard of each rank, all-reduced across the n_groups replica groups
        out->allreduce_input = L->S;
        bus += 2.0 * double(L->S) * double(n_groups - 1) / double(n_groups);
    }
    out->bus_elements = bus;
    return FSDP_OK;
}

int fsdp_layout_prepare(fsdp_layout* L) {
    fsdp::detail::NvtxRange nvtx_range("fsdp_layout_prepare");
    if (!L) return FSDP_EINVAL;
    const Seg* base = nullptr;
    return device_tables(L, &base);
}

int fsdp_unshard(const fsdp_layout* L, int32_t ub, int32_t ue, const void* shards, void* full,
                 int32_t elem_dtype, fsdp_stream_t stream) {
    fsdp::detail::NvtxRange nvtx_range("fsdp_unshard");
    int rc = check_units(L, ub, ue);
    if (rc) return rc;
    if (elem_dtype != FSDP_F32 && elem_dtype != FSDP_BF16) return FSDP_EDTYPE;
    if (L->mode == FSDP_ZERO1) return FSDP_EINVAL;          // parameters are replicated: nothing to gather
    if ((rc = check_ptr(shards)) || (rc = check_ptr(full))) return rc;
    const Seg* base = nullptr;
    if ((rc = device_tables(L, &base))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool bf16 = elem_dtype == FSDP_BF16;
    // aligned class: bulk copies through shared memory; shifted class: warp realignment
    const Range A = range_of(L->gather_al, base, ub, ue);
    cudaError_t e = fsdp::launch_unshard_bulk(A.segs, A.tile_base, A.n_tiles, bf16, shards, full, kWaitNs, st);
    if (e != cudaSuccess) return cuda_fail(e, "k_unshard_bulk launch");
    const Range R = range_of(L->gather_sh, base, ub, ue);
    e = fsdp::launch_unshard_shifted(R.segs, R.tile_base, R.n_tiles, bf16, shards, full, int64_t(L->N) * L->stride, st);
    if (e != cudaSuccess) return cuda_fail(e, "k_unshard_shift launch");
    return FSDP_OK;
}

int fsdp_reduce_scatter_adamw(const fsdp_layout* L, int32_t ub, int32_t ue, const void* const* grads,
                              int32_t grad_dtype, float* master, float* exp_avg, float* exp_avg_sq,
                              void* param_shards, float* grad_shard_out, const fsdp_adamw_hparams* hp,
                              int64_t step, fsdp_stream_t stream) {
    fsdp::detail::NvtxRange nvtx_range("fsdp_reduce_scatter_adamw");
    int rc = check_rs_buffers(L, ub, ue, grads, grad_dtype, master, exp_avg, exp_avg_sq, param_shards,
                              grad_shard_out);
    if (rc) return rc;
    if (!hp || step < 1) return FSDP_EINVAL;
    if ((rc = check_hparams(hp))) return rc;
    const fsdp::AdamScal sc = adam_scalars(hp, step, L->N);

    fsdp::GradPtrs gp{};
    for (int32_t q = 0; q < L->N; ++q) gp.p[q] = grads[q];

    const Seg* base = nullptr;
    if ((rc = device_tables(L, &base))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    const bool bf16 = grad_dtype == FSDP_BF16;
    bool staged = false;
    if ((rc = choose_staged(fsdp::staged_fits(L->N, bf16), true, &staged))) return rc;
    if (staged) {
        const Range R = range_of(L->data, base, ub, ue);
        e = fsdp::launch_rs_adamw_staged(R.segs, R.tile_base, R.n_tiles, bf16, gp, L->N, master, exp_avg, exp_avg_sq,
                                         static_cast<uint16_t*>(param_shards), grad_shard_out, sc, kWaitNs, st);
        if (e != cudaSuccess) return cuda_fail(e, "k_rs_adamw_staged launch");
    } else {
        for (int shifted = 0; shifted < 2; ++shifted) {
            const Range R = range_of(shifted ? L->data_sh : L->data_al, base, ub, ue);
            e = fsdp::launch_rs_adamw(R.segs, R.tile_base, R.n_tiles, shifted, bf16, gp, L->N, L->F, master, exp_avg,
                                      exp_avg_sq, static_cast<uint16_t*>(param_shards), grad_shard_out, sc, st);
            if (e != cudaSuccess) return cuda_fail(e, "k_rs_adamw launch");
        }
    }
    if (grad_shard_out) {
        const Range P = range_of(L->pad, base, ub, ue);
        e = fsdp::launch_zero_pad(P.segs, P.tile_base, P.n_tiles, grad_shard_out, nullptr, st);
        if (e != cudaSuccess) return cuda_fail(e, "k_zero_pad launch");
    }
    return FSDP_OK;
}

int fsdp_adamw_step_consts_make(const fsdp_layout* L, const fsdp_adamw_hparams* hp, int64_t step,
                                fsdp_adamw_step_consts* out) {
    if (!L || !hp || !out || step < 1) return FSDP_EINVAL;
    const int rc = check_hparams(hp);
    if (rc) return rc;
    const fsdp::AdamScal sc = adam_scalars(hp, step, L->N);
    fsdp_adamw_step_consts c{};
    c.decay = sc.decay;
    c.om1 = sc.om1;
    c.om2 = sc.om2;
    c.step_size = sc.step_size;
    c.bc2s = sc.bc2s;
    c.beta1 = sc.beta1;
    c.beta2 = sc.beta2;
    c.eps = sc.eps;
    c.n_avg = sc.nf;
    *out = c;
    return FSDP_OK;
}

int fsdp_adamw_step_consts_upload(fsdp_adamw_step_consts* dev_dst, const fsdp_adamw_step_consts* host_src,
                                  fsdp_stream_t stream) {
    int rc = check_ptr(dev_dst);
    if (rc) return rc;
    if (!host_src) return FSDP_EINVAL;
    const cudaError_t e = cudaMemcpyAsync(dev_dst, host_src, sizeof(fsdp_adamw_step_consts), cudaMemcpyHostToDevice,
                                          reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FSDP_OK : cuda_fail(e, "cudaMemcpyAsync(step constants)");
}

int fsdp_reduce_scatter_adamw_consts(const fsdp_layout* L, int32_t ub, int32_t ue, const void* const* grads,
                                     int32_t grad_dtype, float* master, float* exp_avg, float* exp_avg_sq,
                                     void* param_shards, float* grad_shard_out, const fsdp_adamw_step_consts* consts,
                                     fsdp_stream_t stream) {
    fsdp::detail::NvtxRange nvtx_range("fsdp_reduce_scatter_adamw_consts");
    int rc = check_rs_buffers(L, ub, ue, grads, grad_dtype, master, exp_avg, exp_avg_sq, param_shards,
                              grad_shard_out);
    if (rc) return rc;
    if ((rc = check_ptr(consts))) return rc;
    // the block may be device, managed or page-locked host memory: the kernel reads it
    // through the address the device sees; other host memory is refused
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, consts) != cudaSuccess) {
        (void)cudaGetLastError();   // not sticky: clear it
        return FSDP_EINVAL;
    }
    if ((pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeHost && pa.type != cudaMemoryTypeManaged) ||
        !pa.devicePointer)
        return FSDP_EINVAL;
    const fsdp::AdamScal* dconsts = static_cast<const fsdp::AdamScal*>(pa.devicePointer);
    if (!aligned16(dconsts)) return FSDP_EALIGN;
    const bool bf16 = grad_dtype == FSDP_BF16;
    if (!fsdp::staged_fits(L->N, bf16)) return FSDP_EINVAL;
    fsdp::GradPtrs gp{};
    for (int32_t q = 0; q < L->N; ++q) gp.p[q] = grads[q];
    const Seg* base = nullptr;
    if ((rc = device_tables(L, &base))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Range R = range_of(L->data, base, ub, ue);
    const fsdp::AdamScal unused{};   // the kernel reads the device block instead
    cudaError_t e = fsdp::launch_rs_adamw_staged(R.segs, R.tile_base, R.n_tiles, bf16, gp, L->N, master, exp_avg,
                                                 exp_avg_sq, static_cast<uint16_t*>(param_shards), grad_shard_out,
                                                 unused, kWaitNs, st, dconsts);
    if (e != cudaSuccess) return cuda_fail(e, "k_rs_adamw_staged launch");
    if (grad_shard_out) {
        const Range P = range_of(L->pad, base, ub, ue);
        e = fsdp::launch_zero_pad(P.segs, P.tile_base, P.n_tiles, grad_shard_out, nullptr, st);
        if (e != cudaSuccess) return cuda_fail(e, "k_zero_pad launch");
    }
    return FSDP_OK;
}

int fsdp_reshard(const fsdp_layout* L, int32_t ub, int32_t ue, const void* full, int32_t full_dtype,
                 float* master, void* param_shards, fsdp_stream_t stream) {
    fsdp::detail::NvtxRange nvtx_range("fsdp_reshard");
    int rc = check_units(L, ub, ue);
    if (rc) return rc;
    if (!full) return FSDP_OK;   // release only: the full buffer is the caller's
    if (full_dtype != FSDP_F32 && full_dtype != FSDP_BF16) return FSDP_EDTYPE;
    if ((rc = check_ptr(full))) return rc;
    if (!master && !param_shards) return FSDP_EINVAL;
    if ((master && !aligned16(master)) || (param_shards && !aligned16(param_shards))) return FSDP_EALIGN;
    const Seg* base = nullptr;
    if ((rc = device_tables(L, &base))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Range D = range_of(L->data, base, ub, ue);
    cudaError_t e = fsdp::launch_reshard(D.segs, D.tile_base, D.n_tiles, full_dtype == FSDP_BF16, full, master,
                                         static_cast<uint16_t*>(param_shards), st);
    if (e != cudaSuccess) return cuda_fail(e, "k_reshard launch");
    const Range P = range_of(L->pad, base, ub, ue);
    e = fsdp::launch_zero_pad(P.segs, P.tile_base, P.n_tiles, master, static_cast<uint16_t*>(param_shards), st);
    if (e != cudaSuccess) return cuda_fail(e, "k_zero_pad launch");
    return FSDP_OK;
}

int fsdp_check_status(fsdp_stream_t stream) {
    fsdp::detail::NvtxRange nvtx_range("fsdp_check_status");
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetLastError");
    unsigned int gave_up = 0;
    e = fsdp::take_wait_error(&gave_up);
    if (e != cudaSuccess) return cuda_fail(e, "wait status read");
    return gave_up ? FSDP_ETIMEOUT : FSDP_OK;
}

int fsdp_set_rs_kernel(int32_t kind) {
    if (kind != FSDP_RS_AUTO && kind != FSDP_RS_DIRECT && kind != FSDP_RS_STAGED) return FSDP_EINVAL;
    return g_rs_kernel.exchange(kind);
}

int fsdp_rs_kernel_for(const fsdp_layout* L, int32_t grad_dtype) {
    if (!L) return FSDP_EINVAL;
    if (grad_dtype != FSDP_F32 && grad_dtype != FSDP_BF16) return FSDP_EDTYPE;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const int kind = g_rs_kernel.load();
    if (kind == FSDP_RS_DIRECT) return FSDP_RS_DIRECT;
    if (kind == FSDP_RS_STAGED) return FSDP_RS_STAGED;
    return fsdp::staged_fits(L->N, grad_dtype == FSDP_BF16) ? FSDP_RS_STAGED : FSDP_RS_DIRECT;
}

int fsdp_wait_selftest(int64_t timeout_ns, fsdp_stream_t stream) {
    fsdp::detail::NvtxRange nvtx_range("fsdp_wait_selftest");
    if (timeout_ns <= 0 || timeout_ns > 10000000000LL) return FSDP_EINVAL;
    const cudaError_t e = fsdp::launch_wait_selftest(uint64_t(timeout_ns), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "k_wait_selftest launch");
    return FSDP_OK;
}

const char* fsdp_error_string(int status) {
    switch (status) {
        case FSDP_OK: return "FSDP_OK: success";
        case FSDP_EINVAL: return "FSDP_EINVAL: invalid argument";
        case FSDP_EDTYPE: return "FSDP_EDTYPE: dtype mismatch or unsupported dtype";
        case FSDP_ESHAPE: return "FSDP_ESHAPE: inconsistent shapes or unit ids";
        case FSDP_EALIGN: return "FSDP_EALIGN: buffer not 16-byte aligned";
        case FSDP_EOVERFLOW: return "FSDP_EOVERFLOW: element count overflows int64";
        case FSDP_ECUDA: return "FSDP_ECUDA: CUDA error";
        case FSDP_ETIMEOUT: return "FSDP_ETIMEOUT: bounded device wait gave up";
        case FSDP_ENOMEM: return "FSDP_ENOMEM: allocation failed";
        default: return "unknown fsdp_status";
    }
}

const char* fsdp_last_cuda_error(void) { return g_cuda_err; }

}  // extern "C"
