// layout.hpp -- host-side layout engine of libfsdpstate.
//
// Computes, from a tensor list, the flatten/pad/shard layout of the FSDP pages
// (FLAT: FSDP1 FlatParameter per wrap unit; DIM0: FSDP2 per-tensor Shard(0)) and
// the three segment lists the kernels walk:
//   data    (rank, piece) -> logical elements:        reduce-scatter+AdamW, reshard
//   gather  (rank, piece) -> elements the all-gather copies:  unshard
//           (FLAT: the whole S_u slot, padding included; DIM0: the owned rows)
//   fullr   the logical ranges of the full layout, tiled on the full side:
//           per-replica work on the gradients (accumulation)
//   pad     (rank, piece) -> padding elements of the shard rows (and, attached to
//           the last unit, each row's physical tail [S, stride)): reshard zero-fill,
//           grad_shard_out zero-fill
// The data and gather lists are also kept split by alignment class: pieces whose
// full-layout offset is congruent to their shard offset mod 8 ("aligned": 16-byte
// vectors line up on both sides) and the rest ("shifted"), so that each class runs
// in a kernel compiled for it.
#pragma once

#include <cstdint>
#include <map>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace fsdp {

struct SegList {
    std::vector<Seg> segs;             // ordered by unit, then rank, then tensor; + sentinel
    std::vector<int32_t> unit_begin;   // U+1 entries: first segment of each unit
    int64_t dev_off = 0;               // element offset of this list in the device table
};

struct DeviceTables {
    Seg* base = nullptr;               // all three lists, back to back
};

}  // namespace fsdp

struct fsdp_layout {
    int32_t T = 0, U = 0, N = 0, mode = 0;
    int64_t P = 0, S = 0, stride = 0, F = 0;
    std::vector<int64_t> numel, d0, inner, rows, t_full_off, t_shard_off, t_unit_off;
    std::vector<int32_t> unit, dtype;
    std::vector<int64_t> u_numel, u_S, u_shard_off, u_full_off;
    fsdp::SegList data, gather, pad;
    fsdp::SegList data_al, data_sh, gather_al, gather_sh;   // split by alignment class
    fsdp::SegList fullr;        // logical full-layout ranges (shard field = full index)
    std::vector<int32_t> owner;  // ZeRO-1: owner rank of each tensor
    int64_t n_data_segments = 0;

    std::mutex mu;                                  // guards dev
    std::map<int, fsdp::DeviceTables> dev;          // per CUDA device
};

namespace fsdp {

// Builds the layout; returns an fsdp_status.
int build_layout(fsdp_layout* L, int32_t n_tensors, const int32_t* ndim, const int64_t* dims,
                 const int32_t* unit_id, const int32_t* dtype, int32_t n_ranks, int32_t mode);

}  // namespace fsdp
