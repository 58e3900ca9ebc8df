// kernels.hpp -- host-side launchers of the libfsdpstate kernels (kernels.cu).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace fsdp {

// shifted: the segment range is the "shifted" alignment class (see layout.hpp).
cudaError_t launch_rs_adamw(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool shifted, bool grad_bf16,
                            const GradPtrs& gp, int N, int64_t F, float* master, float* m, float* v,
                            uint16_t* param, float* gout, const AdamScal& sc, cudaStream_t st);

// All-gather of a segment range of the shifted class (warp realignment).
cudaError_t launch_unshard_shifted(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool bf16, const void* src,
                                   void* dst, int64_t src_limit, cudaStream_t st);

cudaError_t launch_reshard(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool full_bf16,
                           const void* full, float* master, uint16_t* param, cudaStream_t st);

cudaError_t launch_zero_pad(const Seg* segs, int64_t tile_base, int64_t n_tiles, float* a32,
                            uint16_t* a16, cudaStream_t st);

}  // namespace fsdp
