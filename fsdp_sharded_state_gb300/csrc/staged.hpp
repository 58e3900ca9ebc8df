// staged.hpp -- host-side launchers of the bulk-copy kernels (staged.cu, allgather.cu,
// staged_rows.cu).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"

namespace fsdp {

// Whether at least two pipeline stages fit in one CTA's shared memory on this
// device.  Fused step: a stage holds 2048 elements of the 3 fp32 state arrays and of
// the N gradient replicas.  HSDP: of 3R state arrays and R*N replicas (and every
// state copy must start on a 16-byte boundary: copy % 4 == 0, R <= 3).  Clip pass 1:
// of the N replicas.
bool staged_fits(int N, bool grad_bf16);
bool hsdp_staged_fits(int N, int R, bool grad_bf16, int64_t copy);
bool norm_staged_fits(int N, bool grad_bf16);

// ZeRO-1: the owner state (3 slices) and the N replicas in one stage.
bool zero1_staged_fits(int N, bool grad_bf16);

// Partials k_rs_norm_staged writes for a launch over n_tiles tiles (one per
// consumer warp of each CTA).
int norm_staged_partials(int64_t n_tiles);

// A launch's claim counters (claims.cu): a zeroed pair of device words (units claimed,
// CTAs done) that no launch that may overlap this one uses, or nullptr (stream capture,
// no free slot, no ring): then the launch splits its units statically.  After queueing
// the launch (or failing to), claim_release(slot, dev, st, launched) records the slot's
// event on st.  Thread-safe.
unsigned int* claim_acquire(cudaStream_t st, int* slot, int* dev);
void claim_release(int slot, int dev, cudaStream_t st, bool launched);

// Each launcher covers one segment range of either alignment class; wait_ns
// bounds every mbarrier wait.
cudaError_t launch_rs_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                   const GradPtrs& gp, int N, float* master, float* m, float* v, uint16_t* param,
                                   float* gout, const AdamScal& sc, uint64_t wait_ns, cudaStream_t st,
                                   const AdamScal* dsc = nullptr,    // dsc: constants read on the device
                                   bool claims = true);              // false: no claim counters (no allocation)

// The last micro-batch of a no_sync accumulation fused with the step: replica q
// contributes acc.p[q] (fp32 accumulator) + micro.p[q] (micro_bf16 ? bf16 : fp32),
// full layout; the accumulators are read only.  Replicas come in groups where all N
// pairs and the state do not fit two stages.  acc_rs_staged_fits: one pair does.
cudaError_t launch_acc_rs_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool micro_bf16,
                                       const GradPtrs& acc, const GradPtrs& micro, int N, float* master, float* m,
                                       float* v, uint16_t* param, float* gout, const AdamScal& sc, uint64_t wait_ns,
                                       cudaStream_t st);
bool acc_rs_staged_fits(bool micro_bf16);

// HSDP: replicas gp.p[rho*N + q]; state copy rho at element offset rho * copy; rf = R.
cudaError_t launch_hsdp_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                     const GradPtrs& gp, int N, int R, int64_t copy, float* master, float* m,
                                     float* v, uint16_t* param, const AdamScal& sc, float rf, uint64_t wait_ns,
                                     cudaStream_t st);

// Clip pass 1: the fp32 mean into gout and the sums of squares into part[0 .. *n_part).
cudaError_t launch_rs_norm_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                  const GradPtrs& gp, int N, float* gout, double* part, int* n_part, uint64_t wait_ns,
                                  cudaStream_t st);

// Accumulation over the logical full-layout ranges (segs: the "fullr" list): for
// each replica q, acc[q] = micro[q] (first) or acc[q] + micro[q].  acc and micro are
// host arrays of N device pointers.
cudaError_t launch_accumulate_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, int N, float* const* acc,
                                     const void* const* micro, bool micro_bf16, bool first, uint64_t wait_ns,
                                     cudaStream_t st);

// Clip pass 3: g = gshard * (*coef), written back, then AdamW + cast (always fits).
cudaError_t launch_adamw_scaled_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, float* gshard,
                                       const float* coef, float* master, float* m, float* v, uint16_t* param,
                                       const AdamScal& sc, uint64_t wait_ns, cudaStream_t st);

// ZeRO-1 owner step + broadcast: master (bf16 replicas) or NULL (fp32 replicas: the
// owner's replica is its parameter); replicas is a host array of N device pointers.
cudaError_t launch_zero1_adamw_staged(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                                      const GradPtrs& gp, void* const* replicas, int N, int64_t stride,
                                      float* master, float* m, float* v, const AdamScal& sc, uint64_t wait_ns,
                                      cudaStream_t st);

// All-gather (shard -> full, bitwise) of a segment range of the aligned class; with
// claims, a launch with at least 8 (bf16) or 48 (fp32) tiles per CTA claims them from a
// counter pair.
cudaError_t launch_unshard_bulk(const Seg* segs, int64_t tile_base, int64_t n_tiles, bool bf16, const void* src,
                                void* dst, uint64_t wait_ns, cudaStream_t st, bool claims = true);

// One kernel whose only wait cannot complete: exercises the bounded-wait exit.
cudaError_t launch_wait_selftest(uint64_t wait_ns, cudaStream_t st);

// The sharded clip step in one cooperative launch (clip_coop.cu) over a segment range
// (tiles of the misaligned class take a per-element path: meant for ranges where they
// are rare): the reduce-scatter into gshard (its last tiles per CTA held in
// shared memory), the sums of squares into part[0 .. grid), a grid-wide barrier on
// *counter (cleared on the stream first; bounded by wait_ns), the norm and coefficient
// (CTA 0 stores them in ws_norm, ws_coef and norm_out), AdamW on the clipped shard.
// *launched is false, with nothing queued but the counter's clear, when the device
// cannot hold the whole grid at once or its grid would need more than max_part partials:
// the caller then runs the two-pass form.
cudaError_t launch_clip_coop(const Seg* segs, int n_segs, int64_t tile_base, int64_t n_tiles, bool grad_bf16,
                             const GradPtrs& gp, int N, float* gshard, float* master, float* m, float* v,
                             uint16_t* param, double* part, int max_part, unsigned int* counter, double* ws_norm,
                             float* ws_coef, float* norm_out, float max_norm, const AdamScal& sc, uint64_t wait_ns,
                             cudaStream_t st, bool* launched);

// Reads and clears the "a bounded wait gave up" words of every staged translation
// unit on the current device (synchronous).
cudaError_t take_wait_error(unsigned int* flag);
cudaError_t take_wait_error_allgather(unsigned int* flag);   // allgather.cu only
cudaError_t take_wait_error_rows(unsigned int* flag);        // staged_rows.cu only
cudaError_t take_wait_error_coop(unsigned int* flag);        // clip_coop.cu only

}  // namespace fsdp
