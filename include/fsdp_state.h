/*
 * fsdp_state.h -- C ABI of libfsdpstate, the FSDP / ZeRO-3 sharded-state step
 * on one GB300 (sm_103a), with N data-parallel ranks simulated as buffers in
 * one GPU's memory.
 *
 * The calls follow the way the FSDP pages state the problem:
 *   - flatten + pad + shard of a wrap unit (FSDP1 FlatParameter) or per-tensor
 *     dim-0 sharding (FSDP2 Shard(0)):  fsdp_layout_create / _query / _unit /
 *     _tensor / _segment;
 *   - the all-gather that rebuilds the full parameter before forward and again
 *     before backward:  fsdp_unshard;
 *   - the gradient reduce-scatter (fp32 reduce dtype, mean over ranks), the
 *     AdamW step of each rank's 1/N shard and the bf16 recast of the updated
 *     shard, fused into one pass:  fsdp_reduce_scatter_adamw;
 *   - initial sharding, summon_full_params(writeback) and the release of the
 *     full buffer after use:  fsdp_reshard;
 *   - per-rank model-state bytes of ZeRO stages 0-3:  fsdp_state_bytes; per-rank
 *     collective payload of a step under each sharding strategy:
 *     fsdp_collective_payload.
 *
 * Sources (titles and sections of the pages this restates):
 *   [FSDP-ch18]  "第18章 FSDP：ZeRO 风格的参数分片" (yangyitao.com PyTorch book)
 *   [ZeRO-state] "NCCL ZeRO/FSDP state sharding" (blog.cptz.space)
 *   [FSDP2-doc]  "PyTorch FSDP2 后端特性介绍" (MindSpeed-LLM docs)
 *   [titan]      torchtitan FSDP2 article (gsyq.cn)
 *
 * Conventions shared by every call
 *   - Return value: FSDP_OK (0) or a negative fsdp_status.  All arguments are
 *     validated before anything is launched; on error nothing is launched and
 *     no output is touched.
 *   - Memory: every data buffer is owned by the caller and must stay alive until
 *     the work queued on the given stream has finished.  Device buffers are
 *     plain device pointers (cudaMalloc, or any allocator), 16-byte aligned
 *     (else FSDP_EALIGN).  The library owns only the layout object, the
 *     small per-device copy of its segment tables, and per device a ring of 1024
 *     work-claim counter pairs (8 KB and 1024 events, set up by the first launch
 *     that uses one).
 *   - Streams: fsdp_stream_t is a cudaStream_t (NULL = legacy default stream).
 *     Launch calls are asynchronous and never synchronize; only
 *     fsdp_check_status and fsdp_layout_prepare block.  Kernels are launched as
 *     programmatic dependents of the work before them on the stream: each waits,
 *     before touching memory, for that work to complete, so stream order is kept
 *     exactly; only the launch latency between consecutive kernels is hidden.
 *   - Work claims: a bulk-copy (staged) launch with at least 8 tiles per CTA --
 *     the fused step, HSDP, accumulation, the fused last micro-batch, ZeRO-1, the
 *     staged clip update, the all-gather (fp32 from 48 tiles per CTA) -- hands its
 *     tiles to its CTAs through a counter pair from the device's ring, so that
 *     faster SMs take more of them; results do not depend on which CTA takes a
 *     tile.  A pair is reused only after the event recorded behind its last launch
 *     has completed (cudaEventQuery), and the kernel leaves it at zero.  Under
 *     stream capture, with no free pair, or from fsdp_reduce_scatter_adamw_noalloc,
 *     the tiles are split statically instead.  The ring is set up (cudaMalloc,
 *     cudaMemset, cudaEventCreate) by the first such launch on a device: make it
 *     before any stream capture, as the layout tables (fsdp_layout_prepare).
 *   - Shard arrays are [N][stride] row-major: rank r's shard starts at element
 *     r*stride; stride = fsdp_layout_info.shard_stride >= S.  The layout picks
 *     stride mod 8 so that as many rank views as possible sit at a shard index
 *     congruent to their full-layout index mod 8 (16-byte vectors line up on both
 *     sides); when that costs nothing, stride is a multiple of 64.
 *   - The full layout: FLAT -- per unit, the padded flat parameter of N*S_u
 *     elements (tensors are views into it, padding at the end), units
 *     concatenated; DIM0 -- the tensors concatenated, each in its own row-major
 *     shape, no padding.
 *   - Threads: a layout is immutable after creation; it may be used from any
 *     thread and stream.  fsdp_layout_destroy must not race with other calls.
 */
#ifndef FSDP_STATE_H
#define FSDP_STATE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FSDP_OK = 0,
    FSDP_EINVAL = -1,     /* bad argument: NULL, range, unknown enum, bad hyper-parameter  */
    FSDP_EDTYPE = -2,     /* mixed dtypes inside one FLAT unit, or unsupported dtype       */
    FSDP_ESHAPE = -3,     /* inconsistent shapes / unit ids                                */
    FSDP_EALIGN = -4,     /* a buffer is not 16-byte aligned                               */
    FSDP_EOVERFLOW = -5,  /* an element count does not fit the int64 / device index range  */
    FSDP_ECUDA = -6,      /* a CUDA call failed (fsdp_last_cuda_error names it)            */
    FSDP_ETIMEOUT = -7,   /* a bounded device-side wait gave up (fsdp_check_status)        */
    FSDP_ENOMEM = -8      /* host or device allocation of the layout tables failed         */
} fsdp_status;

/* FLAT = FSDP1 FlatParameter ([FSDP-ch18] §18.12; [ZeRO-state] "FlatParameter 与
 * Padding"): the tensors of a unit are flattened, concatenated and padded to
 * N*ceil(P_u/N); rank r owns flat elements [r*S_u, (r+1)*S_u), S_u = ceil(P_u/N).
 * DIM0 = FSDP2 per-parameter Shard(0) ([FSDP2-doc] "DTensor": [4096,4096] on 8
 * ranks -> [512,4096]; [titan] §2.3): each tensor of d0 rows gets a slot of
 * c = ceil(d0/N) rows on every rank; rank r owns rows [min(rc,d0), min((r+1)c,d0)),
 * the rest of its slot is zero padding (a rank may own no row).
 * ZERO1 = ZeRO-1 owner partition ([ZeRO-state] "ZeRO-1：Optimizer State
 * Sharding"): parameters stay whole and replicated; each tensor's optimizer state
 * lives on one owner rank.  Owners: tensors by size, largest first, each to the
 * rank with the fewest elements so far (lowest rank on ties) -- balanced by size,
 * not by count.  The owner's row holds its tensors in tensor order, each at an
 * offset congruent to its full-layout offset mod 8.  The full layout is the
 * tensors concatenated (P elements); fsdp_unshard does not apply. */
typedef enum { FSDP_FLAT = 0, FSDP_DIM0 = 1, FSDP_ZERO1 = 2 } fsdp_mode;

typedef enum { FSDP_F32 = 0, FSDP_BF16 = 1 } fsdp_dtype;

typedef struct fsdp_layout fsdp_layout;      /* opaque, host-owned, immutable */
typedef struct CUstream_st* fsdp_stream_t;    /* same type as cudaStream_t    */

/* AdamW hyper-parameters (decoupled weight decay; Adam with bias correction). */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} fsdp_adamw_hparams;

typedef struct {
    int32_t n_tensors, n_units, n_ranks, mode;
    int64_t numel;          /* P: logical elements, sum of tensor numels              */
    int64_t shard_numel;    /* S: elements of one rank's shard (sum over units)       */
    int64_t shard_stride;   /* physical row stride of [N][stride] shard arrays (>= S)  */
    int64_t full_numel;     /* elements of the full layout (FLAT: N*S, DIM0: P)       */
    int64_t pad_numel;      /* N*S - P: padding elements over all ranks               */
    int64_t n_segments;     /* (tensor or unit, rank) pieces holding logical elements */
} fsdp_layout_info;

/* Creates a layout of n_tensors tensors.
 *   ndim[t]      number of dimensions of tensor t (0 = scalar, counted as [1])
 *   dims         all dimensions, concatenated in tensor order (sum(ndim) entries)
 *   unit_id[t]   wrap unit (FSDP1) / param group (FSDP2) of tensor t: starts at 0,
 *                nondecreasing, steps of 0 or 1 (else FSDP_ESHAPE)
 *   dtype[t]     fsdp_dtype of tensor t's parameter; may be NULL (all the same).
 *                In FLAT mode all tensors of a unit must share a dtype, as a
 *                FlatParameter requires one dtype ([FSDP-ch18] §18.12) -> FSDP_EDTYPE.
 *   n_ranks      N >= 1 simulated data-parallel ranks (<= FSDP_MAX_RANKS)
 *   mode         FSDP_FLAT or FSDP_DIM0
 * Pure host computation: needs no GPU.  *out is set only on FSDP_OK. */
#define FSDP_MAX_RANKS 64
int fsdp_layout_create(int32_t n_tensors, const int32_t* ndim, const int64_t* dims,
                       const int32_t* unit_id, const int32_t* dtype, int32_t n_ranks,
                       int32_t mode, fsdp_layout** out);

/* Frees the layout and its device tables (on every device they were made on).
 * NULL is accepted.  No call may be using the layout or have queued work that
 * reads its tables. */
void fsdp_layout_destroy(fsdp_layout* layout);

/* The layout's sizes ([ZeRO-state] "FlatParameter 与 Padding": the padded physical
 * numel N*ceil(P/N) against the logical P, and the shard numel each rank holds;
 * "Canonical ZeRO 状态公式": the per-rank element counts the state formulas use):
 * P, S, the row stride of the shard arrays, the full-layout size, the padding over
 * all ranks and the number of (tensor or unit, rank) pieces.  Host only.
 * FSDP_EINVAL when an argument is NULL. */
int fsdp_layout_query(const fsdp_layout* layout, fsdp_layout_info* out);

/* Unit u: its shard offset and size S_u inside a rank row, its offset and size
 * in the full layout, and its logical element count P_u. */
int fsdp_layout_unit(const fsdp_layout* layout, int32_t unit, int64_t* shard_off,
                     int64_t* shard_numel, int64_t* full_off, int64_t* full_numel,
                     int64_t* numel);

/* Tensor t: its unit, numel, offset in the full layout; DIM0 only: its shard
 * offset inside a rank row and its rows per rank slot c (FLAT: both -1, since a
 * FLAT tensor's shard position depends on the rank -- use fsdp_layout_segment). */
int fsdp_layout_tensor(const fsdp_layout* layout, int32_t tensor, int32_t* unit,
                       int64_t* numel, int64_t* full_off, int64_t* shard_off,
                       int64_t* rows_per_rank);

/* Rank r's view of tensor t ([ZeRO-state] "FlatParameter 与 Padding": a rank's
 * view of an original parameter may be a 1-D piece, or empty):
 *   *shard_off  position of the view inside rank r's row (element index)
 *   *full_off   position of the same elements in the full layout
 *   *len        number of logical elements (0 when the rank holds none)
 *   *pad        DIM0: padding elements in rank r's slot of tensor t; FLAT: 0
 *               (FLAT padding belongs to the unit; see fsdp_layout_unit).
 * When *len == 0, *shard_off and *full_off are where the view would start. */
int fsdp_layout_segment(const fsdp_layout* layout, int32_t tensor, int32_t rank,
                        int64_t* shard_off, int64_t* full_off, int64_t* len, int64_t* pad);

/* Per-rank model-state bytes of ZeRO stage 0..3 ([ZeRO-state] "Canonical ZeRO
 * 状态公式": stage 0 keeps P, P, 2P per rank; stage 1 shards the optimizer state
 * (2P/N), stage 2 also the gradient (P/N), stage 3 also the parameter (P/N)).
 *   param_bytes, grad_bytes   bytes per parameter / gradient element
 *   optim_bytes               optimizer bytes per element (8: fp32 exp_avg +
 *                             exp_avg_sq; 12 with an fp32 master copy, [titan] §2.3)
 *   step_bytes                optimizer metadata per tensor (Adam's step scalar)
 *   physical                  1: a sharded state counts the rank's padded slot
 *                             (S elements); 0: only the logical elements it owns
 * out[0..2] = parameter, gradient, optimizer bytes held by `rank`. */
int fsdp_state_bytes(const fsdp_layout* layout, int32_t stage, int32_t rank, int32_t physical,
                     int64_t param_bytes, int64_t grad_bytes, int64_t optim_bytes,
                     int64_t step_bytes, int64_t out[3]);

/* Collective payload of one training step, per rank ([ZeRO-state] "Logical Payload
 * 模型": the logical total of each collective's input buffer, in elements, not the bytes
 * a ring algorithm moves; the ring all-reduce moves 2(N-1)/N of its input per rank.
 * [FSDP-ch18] §18.2: one all-reduce about 2 Psi for DDP, reduce-scatter plus
 * all-gather 2 Psi, FULL_SHARD 3 Psi).
 *   strategy   FSDP_NO_SHARD (DDP: the gradient all-reduce), FSDP_ZERO1_OPT (the same
 *              all-reduce, then each owner broadcasts its updated parameters, about P),
 *              FSDP_SHARD_GRAD_OP (forward all-gather, reduce-scatter), FSDP_FULL_SHARD
 *              (forward and backward all-gather, reduce-scatter), FSDP_HYBRID_SHARD
 *              (FULL_SHARD inside each of n_groups groups of N ranks, then an all-reduce
 *              of each rank's reduced shard, S elements, across the groups; [FSDP-ch18]
 *              §18.9)
 *   n_groups   replica groups: >= 1 for FSDP_HYBRID_SHARD, else 1 (else FSDP_EINVAL)
 * out: the logical inputs (P = the layout's logical elements) and bus_elements, the
 * elements one rank sends, and receives, under ring algorithms: (N-1)/N of the buffer
 * for an all-gather, a reduce-scatter or the owners' broadcast (equal shares), 2(N-1)/N
 * for an all-reduce (2(R-1)/R of S across R groups).  Multiply by the element size of
 * each collective's dtype for bytes.  Host only. */
typedef enum {
    FSDP_NO_SHARD = 0, FSDP_ZERO1_OPT = 1, FSDP_SHARD_GRAD_OP = 2, FSDP_FULL_SHARD = 3, FSDP_HYBRID_SHARD = 4
} fsdp_strategy;
typedef struct {
    int64_t allreduce_input, forward_allgather, backward_allgather, reducescatter_input, broadcast;
    double bus_elements;
} fsdp_collective_payload_info;
int fsdp_collective_payload(const fsdp_layout* layout, int32_t strategy, int32_t n_groups,
                            fsdp_collective_payload_info* out);

/* Allocates and uploads the layout's segment tables on the current CUDA device
 * and blocks until they are there.  Launch calls do this themselves on their
 * first use of a layout on a device; call it first to keep that allocation out
 * of a timed region or of a stream capture.  FSDP_ENOMEM / FSDP_ECUDA on failure. */
int fsdp_layout_prepare(fsdp_layout* layout);

/* Unshard = all-gather of units [unit_begin, unit_end) ([ZeRO-state] "ZeRO-3 方向：
 * Parameter Sharding": all_gather_into_tensor(padded_unsharded_flat_param,
 * sharded_flat_param); [FSDP-ch18] §18.3 and §18.8: FSDP2 copy-in, one all-gather,
 * copy-out).  Reads the N rank shards, writes the full layout of those units:
 *   FLAT: every shard element, padding included, to full[u_off + r*S_u + k]
 *         (the padded flat parameter; its padding comes out as the shards' zeros);
 *   DIM0: the owned rows of each tensor to their place in the full tensor.
 *   param_shards  device, [N][stride] of elem_dtype (bf16 param shards, or the
 *                 fp32 master when the parameter dtype is fp32)
 *   full          device, full-layout buffer of elem_dtype (full_numel elements;
 *                 only the units' ranges are written)
 * The copy is bitwise.  Async on `stream`. */
int fsdp_unshard(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                 const void* param_shards, void* full, int32_t elem_dtype, fsdp_stream_t stream);

/* The fused reduce-scatter + AdamW + bf16 recast of units [unit_begin, unit_end),
 * one pass over the rank shards:
 *   (1) reduce-scatter ([ZeRO-state] "ZeRO-2 方向：Gradient Sharding":
 *       reduce_scatter_tensor(new_sharded_grad, padded_grad)): for rank r and its
 *       shard element j, g = (sum over q = 0..N-1, in that order, of
 *       float(G_q[full index of (r, j)])) / N in fp32 (reduce_dtype = float32,
 *       [FSDP-ch18] §18.6); padding elements have g = 0;
 *   (2) AdamW on rank r's fp32 shard of master / exp_avg / exp_avg_sq
 *       ([ZeRO-state] "Optimizer Step 的所有权": each rank updates only its
 *       shard), in this order, every operation rounded to fp32:
 *         p *= 1 - lr*wd;  m = fma(b1, m, (1-b1)*g);  v = fma(b2, v, ((1-b2)*g)*g);
 *         p = fma(-lr/(1-b1^t), m / (sqrt(v)/sqrt(1-b2^t) + eps), p)
 *       (the four step constants formed in double, rounded to fp32 once);
 *   (3) param_shards = bf16(p), round to nearest even ([FSDP-ch18] §18.6:
 *       bf16 parameters for the all-gather, fp32 master for Adam).
 *   grad_replicas  host array of N device pointers; replica q is rank q's full
 *                  gradient in the full layout (full_numel elements of
 *                  grad_dtype).  FLAT padding positions are never read.
 *   master, exp_avg, exp_avg_sq   device, [N][stride] fp32, updated in place.
 *                  Padding elements are not touched: they stay +0 when they
 *                  start at +0 (fsdp_reshard writes them so), which is exactly
 *                  what AdamW does to them with g = 0 when 0 <= lr*wd <= 1.
 *   param_shards   device, [N][stride] bf16, or NULL when the parameter dtype is
 *                  fp32 (the master is then the parameter).
 *   grad_shard_out optional device [N][stride] fp32: the reduced gradient shard
 *                  (FSDP's _saved_grad_shard), padding written as +0; or NULL.
 *   hp             lr >= 0, 0 <= beta < 1, eps > 0, weight_decay >= 0,
 *                  lr*weight_decay <= 1, all finite (else FSDP_EINVAL).
 *   step           1-based step count t shared by all elements.
 * Async on `stream`. */
int fsdp_reduce_scatter_adamw(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                              const void* const* grad_replicas, int32_t grad_dtype,
                              float* master, float* exp_avg, float* exp_avg_sq,
                              void* param_shards, float* grad_shard_out,
                              const fsdp_adamw_hparams* hp, int64_t step, fsdp_stream_t stream);

/* Reshard of units [unit_begin, unit_end).
 *   full == NULL: release only -- the full buffer is the caller's to free or
 *     reuse ([FSDP-ch18] §18.3: after use the full copy is dropped and the rank is
 *     back to 1/N); nothing is launched.
 *   full != NULL: scatter the full layout into the rank shards, the initial
 *     sharding of a constructed model and the writeback of
 *     summon_full_params(writeback=True) ([FSDP-ch18] §18.17):
 *     master (fp32, or NULL) gets the values, param_shards (bf16, or NULL) gets
 *     their bf16 rounding (nearest even); padding elements get +0, and when the
 *     range ends at the last unit, so does each row's tail [S, stride).
 *   full_dtype     FSDP_F32 or FSDP_BF16 (bf16 values widen exactly).
 * Async on `stream`. */
int fsdp_reshard(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                 const void* full, int32_t full_dtype, float* master, void* param_shards,
                 fsdp_stream_t stream);

/* The pages have no counterpart of this call: their collectives report errors
 * through NCCL and the process group, which this library replaces with kernels.
 * Blocks until `stream` is idle and reports any CUDA error seen there
 * (FSDP_ECUDA), or, failing that, a bounded device-side wait that gave up on the
 * current device since the last check (FSDP_ETIMEOUT; the record is cleared). */
int fsdp_check_status(fsdp_stream_t stream);

/* Static text for a status code; never NULL. */
const char* fsdp_error_string(int status);

/* Text of the last CUDA error seen by this thread in a library call ("" if none). */
const char* fsdp_last_cuda_error(void);

/* ZeRO-1 layouts: the owner rank of tensor t (FSDP_EINVAL for other modes). */
int fsdp_layout_owner(const fsdp_layout* layout, int32_t tensor, int32_t* rank);

/* Sharded clip_grad_norm_ between the reduce-scatter and AdamW ([FSDP-ch18]
 * §18.18: every rank computes the sum of squares of its gradient shard, one
 * all-reduce adds them, the square root is the global norm, every rank scales its
 * own shard).  The clip coefficient follows torch's clip_grad_norm_ (L2 norm):
 * coef = min(1, max_norm / (norm + 1e-6)), formed in double and rounded to fp32
 * once; each reduced gradient is multiplied by it (one fp32 rounding) and then
 * goes through the AdamW and bf16 steps of fsdp_reduce_scatter_adamw.
 * Under the automatic kernel choice, when the rank views of the unit range sit at shard
 * indices congruent to their full-layout indices mod 8 but for at most one 2048-element
 * tile in 256 (fsdp_layout_segment tells each piece's class), one cooperative launch on
 * `stream` runs the whole step: each CTA reduce-scatters a fixed set of tiles into
 * the fp32 gradient shard -- holding the last of them in shared memory -- and writes
 * its partial sum of squares; after a grid-wide barrier (bounded: it gives up after
 * 1 s and records FSDP_ETIMEOUT for fsdp_check_status) every CTA adds the partials in
 * double in the same order, forms the coefficient, scales and updates the tiles it
 * holds, then takes the other tiles one at a time from a shared counter in the
 * workspace and scales and updates them (the tile sets of the sums are fixed, so the
 * norm is the same in every run).
 * Otherwise (or when the device cannot hold the whole grid at once), two passes: the
 * reduce-scatter writes the fp32 gradient shard and per-CTA partial sums of squares
 * (fixed order, so the norm is reproducible on a given GPU); the update pass adds the
 * partials in double (every CTA in the same order), forms the coefficient, scales the
 * shard and runs AdamW.  (With the staged kernels forced, one extra single-CTA kernel
 * forms the norm between them.)
 *   grad_shard  required device [N][stride] fp32: receives the CLIPPED reduced
 *               gradient (padding +0); it is also the working buffer.
 *   max_norm    > 0 and finite.
 *   workspace   device scratch of fsdp_clip_workspace_bytes() bytes, 16-byte
 *               aligned, owned by the caller; no initial contents needed.  It holds
 *               the call's partial sums (and the cooperative launch's barrier and tile counters)
 *               until the call's work has run: calls whose work may overlap on the GPU
 *               (other streams) need workspaces of their own.
 *   norm_out    optional device float[2] (8-byte aligned): total norm, coef.
 * Other arguments and errors as fsdp_reduce_scatter_adamw. */
size_t fsdp_clip_workspace_bytes(void);
int fsdp_reduce_scatter_clip_adamw(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                                   const void* const* grad_replicas, int32_t grad_dtype,
                                   float* master, float* exp_avg, float* exp_avg_sq,
                                   void* param_shards, float* grad_shard, float max_norm,
                                   void* workspace, float* norm_out,
                                   const fsdp_adamw_hparams* hp, int64_t step, fsdp_stream_t stream);

/* Gradient accumulation without synchronisation ([FSDP-ch18] §18.26: no_sync /
 * set_requires_gradient_sync(False) -- the unsharded gradients accumulate
 * locally and the reduce-scatter runs once, on the last micro-batch).  For every
 * rank q and every logical element of units [unit_begin, unit_end) in the full
 * layout: acc[q] = micro[q] (first != 0) or acc[q] + micro[q], in fp32.  Feed the
 * accumulators to fsdp_reduce_scatter_adamw (grad_dtype FSDP_F32) afterwards.
 *   acc    host array of N device pointers, fp32 full-layout buffers (FLAT
 *          padding positions are not touched)
 *   micro  host array of N device pointers, micro_dtype full-layout gradients */
int fsdp_accumulate_grads(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                          float* const* acc, const void* const* micro, int32_t micro_dtype,
                          int32_t first, fsdp_stream_t stream);

/* The last micro-batch of a gradient accumulation without synchronisation, fused with
 * the reduce-scatter + AdamW + cast ([FSDP-ch18] §18.26: the micro-batches before the
 * last accumulate their unsharded gradients locally; the last one runs with
 * synchronisation, its gradients added to the accumulated ones and reduce-scattered).
 * For rank r and shard element j with full-layout index f:
 *   g = (sum over q = 0..N-1, in that order, of (acc[q][f] + micro[q][f])) / N
 * in fp32 (each acc + micro one fp32 addition, as fsdp_accumulate_grads makes it), then
 * AdamW and the cast exactly as fsdp_reduce_scatter_adamw.  Bit for bit the results of
 * fsdp_accumulate_grads(first = 0) followed by fsdp_reduce_scatter_adamw(FSDP_F32) on
 * the accumulators, in one pass that reads each accumulator once and writes none: the
 * accumulators are read only (FSDP frees the unsharded gradients after the
 * reduce-scatter).
 *   acc    host array of N device pointers: fp32 full-layout accumulators
 *   micro  host array of N device pointers: the last micro-batch, micro_dtype
 * Other arguments, checks and results as fsdp_reduce_scatter_adamw (grad_shard_out
 * optional; the kernel choice of fsdp_set_rs_kernel applies: staged by default, with
 * the replicas in groups where all N pairs of slices do not fit). */
int fsdp_accumulate_reduce_scatter_adamw(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                                         const float* const* acc, const void* const* micro, int32_t micro_dtype,
                                         float* master, float* exp_avg, float* exp_avg_sq, void* param_shards,
                                         float* grad_shard_out, const fsdp_adamw_hparams* hp, int64_t step,
                                         fsdp_stream_t stream);

/* HSDP step ([FSDP-ch18] §18.9: shard inside a group, replicate across groups;
 * reduce-scatter in the shard dimension, then one all-reduce across the replica
 * groups; torchtitan article §3).  R = n_groups groups of N ranks (R*N <=
 * FSDP_MAX_RANKS); grad_replicas[rho*N + q] is rank q of group rho.  For every
 * shard element: g_rho = (sum over q, in order, of G[rho][q]) / N, then
 * g = (sum over rho, in order, of g_rho) / R -- the book's order (the torchtitan
 * article puts the all-reduce first) -- and every group's copy of the state gets
 * the same AdamW update.
 *   master, exp_avg, exp_avg_sq, param_shards: R copies of [N][stride], copy rho
 *   at element rho*N*stride (param_shards bf16 or NULL). */
int fsdp_hsdp_reduce_scatter_adamw(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                                   int32_t n_groups, const void* const* grad_replicas, int32_t grad_dtype,
                                   float* master, float* exp_avg, float* exp_avg_sq, void* param_shards,
                                   const fsdp_adamw_hparams* hp, int64_t step, fsdp_stream_t stream);

/* ZeRO-1 step on an FSDP_ZERO1 layout ([ZeRO-state] "ZeRO-1：Optimizer State
 * Sharding": gradients all-reduced, every rank updates only the parameters it
 * owns, then broadcasts them).  For every element: g = (sum over q of G_q) / N;
 * the owner's AdamW; the updated parameter is written into all N replicas.
 *   grad_replicas  N device pointers, full layout (P elements), grad_dtype
 *   master         [N][stride] fp32 owner rows, required with bf16 replicas;
 *                  NULL with fp32 replicas (the owner's replica is the parameter)
 *   exp_avg, exp_avg_sq  [N][stride] fp32 owner rows
 *   param_replicas host array of N device pointers, full layout, param_dtype
 * fsdp_reshard fills master from full parameters; fsdp_unshard does not apply. */
int fsdp_zero1_adamw_broadcast(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                               const void* const* grad_replicas, int32_t grad_dtype,
                               float* master, float* exp_avg, float* exp_avg_sq,
                               void* const* param_replicas, int32_t param_dtype,
                               const fsdp_adamw_hparams* hp, int64_t step, fsdp_stream_t stream);

/* Kernel choice of the calls that reduce over gradient replicas (process-wide;
 * the pages have no counterpart, the result is the same either way, bit for bit,
 * except the clip norm's last bits, see below): fsdp_reduce_scatter_adamw,
 * passes 1 and 3 of fsdp_reduce_scatter_clip_adamw,
 * fsdp_hsdp_reduce_scatter_adamw, fsdp_accumulate_grads and
 * fsdp_zero1_adamw_broadcast.
 *   FSDP_RS_AUTO    the staged kernel where at least two of its pipeline stages fit
 *                   in one CTA's shared memory, else the direct kernels; the clip
 *                   runs as one cooperative launch where at most one tile in 256 of
 *                   its unit range is misaligned, else as the direct passes.  A stage
 *                   holds 2048 elements of each array the call reads: for
 *                   fsdp_reduce_scatter_adamw the three fp32 state arrays and the N
 *                   gradient replicas, the replicas in groups where all of them do
 *                   not fit (bf16 N > 16, fp32 N > 8; always fits); for HSDP 3R
 *                   state arrays and R*N replicas (R <= 3,
 *                   and N*stride a multiple of 4); for the clip pass the N replicas;
 *                   for accumulation one micro-batch replica and its accumulator
 *                   (always fits); for ZeRO-1 the owner's state and the N replicas.
 *                   The default.
 *   FSDP_RS_DIRECT  the direct kernels: 16-byte loads straight into registers, one
 *                   launch per alignment class.
 *   FSDP_RS_STAGED  the staged kernels: the bulk-copy engine (cp.async.bulk) moves
 *                   each tile of every input array into shared memory, an mbarrier
 *                   per stage counts the bytes, one launch for both alignment
 *                   classes.  A call whose staged kernel does not fit returns
 *                   FSDP_EINVAL.
 * The clip norm is a double sum whose grouping differs between the forms (one
 * partial per CTA of the passes, per warp of the staged pass, per CTA of the
 * cooperative launch over other tiles); all are deterministic run to run.
 * Returns the previous choice, or FSDP_EINVAL for an unknown one.  Not ordered
 * with calls in flight on other threads. */
typedef enum { FSDP_RS_AUTO = 0, FSDP_RS_DIRECT = 1, FSDP_RS_STAGED = 2 } fsdp_rs_kernel;
int fsdp_set_rs_kernel(int32_t kind);

/* The kernel fsdp_reduce_scatter_adamw would run for this layout and gradient
 * dtype on the current device under the current choice: FSDP_RS_DIRECT or
 * FSDP_RS_STAGED (FSDP_EINVAL / FSDP_EDTYPE for a bad argument, FSDP_ECUDA if the
 * device cannot be queried).  Launches per call: staged 1, direct 1 per alignment
 * class present (fsdp_layout_segment tells the class of each piece). */
int fsdp_rs_kernel_for(const fsdp_layout* layout, int32_t grad_dtype);

/* Diagnostic of the bounded device waits: launches one kernel whose mbarrier
 * expects 16 bytes that nothing delivers.  Its wait gives up after timeout_ns
 * nanoseconds (0 < timeout_ns <= 10^10) and records the failure; the next
 * fsdp_check_status returns FSDP_ETIMEOUT and clears it.  The staged kernel
 * records a wait that gives up the same way (limit: 1 s per wait). */
int fsdp_wait_selftest(int64_t timeout_ns, fsdp_stream_t stream);

/* The step constants of the fused update in memory, for CUDA graphs.  The pages
 * have no counterpart of these three calls.  fsdp_reduce_scatter_adamw forms its
 * per-step AdamW constants on the host and passes them as kernel arguments, so a
 * CUDA graph that captured it would replay one step's bias corrections forever.
 * fsdp_reduce_scatter_adamw_consts runs the same step with those constants read
 * from a block in memory when the kernel runs; a captured graph is replayed after
 * the next step's block has been written there.  The block may be page-locked host
 * memory, which the host rewrites between replays with no copy in the graph, or
 * device memory filled on the stream (fsdp_adamw_step_consts_upload).
 *
 * fsdp_adamw_step_consts_make fills the 48-byte block for `step` exactly as
 * fsdp_reduce_scatter_adamw forms it (each constant in double from the fp32
 * hyper-parameters, rounded to fp32 once): decay = 1 - lr*wd, om1 = 1 - beta1,
 * om2 = 1 - beta2, step_size = lr / (1 - beta1^step), bc2s = sqrt(1 - beta2^step),
 * beta1, beta2, eps, n_avg = N.  Host only; hp and step are checked as in
 * fsdp_reduce_scatter_adamw (FSDP_EINVAL).
 *
 * fsdp_reduce_scatter_adamw_consts: arguments, checks and results as
 * fsdp_reduce_scatter_adamw (bit for bit, given the block of the same step), with
 *   consts   16-byte aligned (else FSDP_EALIGN) block in device, managed or
 *            page-locked host memory (pageable host memory: FSDP_EINVAL).  The
 *            kernel reads it when it runs, once per thread, with loads that use no
 *            cached copy; it must hold the step's constants then and must not be
 *            rewritten until the kernel has finished.
 * It always runs the staged kernel (the default of fsdp_reduce_scatter_adamw),
 * whatever fsdp_set_rs_kernel chose.  Launching it during stream capture needs
 * the layout's device tables to exist already (fsdp_layout_prepare, or any
 * earlier call on the device). */
typedef struct {
    float decay, om1, om2, step_size, bc2s, beta1, beta2, eps, n_avg;
    float reserved[3];
} fsdp_adamw_step_consts;
int fsdp_adamw_step_consts_make(const fsdp_layout* layout, const fsdp_adamw_hparams* hp, int64_t step,
                                fsdp_adamw_step_consts* out);
int fsdp_reduce_scatter_adamw_consts(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                                     const void* const* grad_replicas, int32_t grad_dtype,
                                     float* master, float* exp_avg, float* exp_avg_sq,
                                     void* param_shards, float* grad_shard_out,
                                     const fsdp_adamw_step_consts* consts, fsdp_stream_t stream);
/* Copies a block of step constants from host memory into the device block, on
 * `stream` (cudaMemcpyAsync, 48 bytes).  Captured in a CUDA graph it becomes a copy
 * that reads host_src when the graph runs, so host_src must be page-locked (pinned)
 * there and must not be rewritten before that replay has run.  dev_dst 16-byte
 * aligned (else FSDP_EALIGN); host_src non-NULL. */
int fsdp_adamw_step_consts_upload(fsdp_adamw_step_consts* dev_dst, const fsdp_adamw_step_consts* host_src,
                                  fsdp_stream_t stream);

/* fsdp_reduce_scatter_adamw_noalloc -- the pages have no counterpart of this call.
 * The same computation, arguments, checks, kernel choice and results as
 * fsdp_reduce_scatter_adamw,
 * for callers that cannot allocate device memory: a pre-sized pool or custom
 * allocator that owns all device memory, a step that must not enter the driver's
 * allocator (cudaMalloc may synchronize the device or fail under memory pressure),
 * or an embedder that forbids hidden allocations in a library.  It calls no
 * cudaMalloc, cudaFree or other allocating routine: the segment table its kernels
 * read is staged, on `stream`, in one fixed array inside the library image of
 * FSDP_NOALLOC_MAX_SEGMENTS 32-byte entries (256 KiB), which every GPU that loads
 * the library holds until the process exits.
 *   - The unit range may need at most FSDP_NOALLOC_MAX_SEGMENTS entries: the
 *     range's (tensor or unit, rank) pieces + 2, plus, when grad_shard_out is given,
 *     its padding pieces + 1.  A larger range returns FSDP_EINVAL with nothing
 *     launched; split it into smaller unit ranges.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.  The
 *     address is kept for the rest of the process: after a cudaDeviceReset of that
 *     device it is stale, so do not call this entry point after one.
 *   - All calls share the one array and each call rewrites the entries it reads
 *     before its kernels run, so no state carries over between calls.  Calls whose
 *     work overlaps on the GPU race on the array: issue them on one stream, or order
 *     them with events.  Host threads may call it at the same time: a lock held from
 *     a call's table copy to its last launch keeps each call's copy and kernels
 *     together on the stream.
 *   - A CUDA error is recorded for fsdp_last_cuda_error, as by the other calls. */
#define FSDP_NOALLOC_MAX_SEGMENTS 8192
int fsdp_reduce_scatter_adamw_noalloc(const fsdp_layout* layout, int32_t unit_begin, int32_t unit_end,
                                      const void* const* grad_replicas, int32_t grad_dtype,
                                      float* master, float* exp_avg, float* exp_avg_sq,
                                      void* param_shards, float* grad_shard_out,
                                      const fsdp_adamw_hparams* hp, int64_t step, fsdp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FSDP_STATE_H */
