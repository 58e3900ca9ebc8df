// staged.hpp -- host-side launchers of the bulk-copy staged kernels (staged.cu).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"

namespace fsdp {

// Whether at least two pipeline stages (3 fp32 state slices + N gradient slices
// of one 2048-element tile each) fit in one CTA's shared memory on this device.
bool staged_fits(int N, bool grad_bf16);

// Fused reduce-scatter + AdamW + cast over one segment range of either alignment
// class; wait_ns bounds every mbarrier wait.
cudaError_t launch_rs_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                   const GradPtrs& gp, int N, float* master, float* m, float* v, uint16_t* param,
                                   float* gout, const AdamScal& sc, uint64_t wait_ns, cudaStream_t st);

// All-gather (shard -> full, bitwise) of a segment range of the aligned class.
cudaError_t launch_unshard_bulk(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool bf16, const void* src,
                                void* dst, uint64_t wait_ns, cudaStream_t st);

// One kernel whose only wait cannot complete: exercises the bounded-wait exit.
cudaError_t launch_wait_selftest(uint64_t wait_ns, cudaStream_t st);

// Reads and clears the device's "a bounded wait gave up" word (synchronous).
cudaError_t take_wait_error(unsigned int* flag);

}  // namespace fsdp
