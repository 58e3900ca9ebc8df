// internal.hpp -- helpers shared by the libfsdpstate entry points (api.cu, rows.cu).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/fsdp_state.h"
#include "common.cuh"
#include "layout.hpp"

namespace fsdp {
namespace detail {

// Segment range and tile range of units [ub, ue) in one list.
struct Range {
    const Seg* segs;
    int64_t tile_base, n_tiles;
    int32_t n_segs;     // segments in the range (the sentinel after them not counted)
};

int cuda_fail(cudaError_t e, const char* where);        // records the error text, returns FSDP_ECUDA
bool aligned16(const void* p);
int device_tables(const fsdp_layout* L, const Seg** base);   // per-device copy of the segment lists
Range range_of(const SegList& l, const Seg* dev_base, int32_t ub, int32_t ue);
int check_units(const fsdp_layout* L, int32_t ub, int32_t ue);
int check_ptr(const void* p);                            // non-NULL and 16-byte aligned
int check_hparams(const fsdp_adamw_hparams* hp);
AdamScal adam_scalars(const fsdp_adamw_hparams* hp, int64_t step, int32_t n_avg);

// An NVTX range over one library call: the call's name on a profiler's timeline
// (Nsight Systems, ncu --nvtx); without a tool attached the push and pop do nothing.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Time limit of each mbarrier wait in the staged kernels.
constexpr uint64_t kWaitNs = 1000000000ull;

// Whether a call runs its staged kernel, under the process-wide choice
// (fsdp_set_rs_kernel), whether the staged kernel fits this call and whether the
// automatic choice prefers it (measured faster): FSDP_OK and *staged set, or
// FSDP_EINVAL when the staged kernel is forced but does not fit.
int choose_staged(bool fits, bool preferred, bool* staged);

// The process-wide kernel choice (fsdp_set_rs_kernel): FSDP_RS_AUTO, _DIRECT or _STAGED.
int rs_kernel_choice();

}  // namespace detail
}  // namespace fsdp
