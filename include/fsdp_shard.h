/*
 * fsdp_shard.h -- C ABI of the FSDP per-unit shard engine (GB300, sm_103a).
 *
 * One FSDP unit (a group of parameters gathered and reduced together, e.g.
 * one Transformer block) is sharded over R ranks. The R ranks are virtual:
 * each rank's buffers are separate device allocations on one GPU, and the
 * "collectives" are the kernels below, which read and write those buffers.
 *
 * The operations, and where the FSDP pages define them:
 *   fsdp_layout                dim-0 ceil-div sharding of every parameter
 *                              ("从源码理解 FSDP", §2.1 intra-tensor partition;
 *                              "FSDP Transformer Block Sharding Example",
 *                              4-GPU layout: FSDP2 per-parameter table and the
 *                              FSDP1 FlatParameter ranges).
 *   fsdp_pack_flat             shard from full: each rank keeps its slice
 *                              ("从源码理解 FSDP", §4.2 init_shard_from_full;
 *                              FlatParameter = concat(flatten(p_i)), padded).
 *   fsdp_all_gather_unflatten  every rank rebuilds the full unit from all
 *                              shards, as the original parameter shapes
 *                              ("从源码理解 FSDP", §2.2 gather_tensor;
 *                              "FSDP Transformer Block Sharding Example",
 *                              All-Gather mechanism and FSDP1 unflatten;
 *                              "FSDP Training Step Walkthrough", Step 1.1).
 *   fsdp_reduce_scatter_adamw  element-wise sum of the R ranks' full local
 *                              gradients in fp32, averaged, rank r keeping its
 *                              own slice ("从源码理解 FSDP", §2.3 scatter_tensor;
 *                              "FSDP Training Step Walkthrough", Step 4.4;
 *                              reduce dtype fp32 per the block page's mixed
 *                              precision policy), fused with the sharded AdamW
 *                              step on that slice ("从源码理解 FSDP", §2.4
 *                              FSDPAdamW; walkthrough Step 6).
 *
 * Conventions (all entry points):
 *  - Every call checks its arguments on the host before it launches
 *    anything: the layout and hyper-parameters, every pointer array and
 *    every pointer in it (non-NULL, 16-byte aligned), and that no output
 *    range [p, p + bytes) overlaps any other buffer's range, where bytes is
 *    what the layout says the buffer holds (e.g. P elements of grad_dtype
 *    for a full gradient), and that every buffer is device memory of one
 *    device (cudaPointerGetAttributes). A failed check returns a negative
 *    status, sets the thread's fsdp_last_error() message and launches
 *    nothing. A plain pointer carries no size or dtype, so the library
 *    cannot see that an allocation is too short or holds another dtype:
 *    that is the caller's part (the Python binding checks both on every
 *    tensor before the call). No kernel traps or asserts.
 *  - Kernel calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and never synchronise. They run on the device
 *    that owns the first output buffer, which every buffer of the call must
 *    be on; the calling thread's current device is the same after the call
 *    as before it.
 *  - Buffer arguments are host arrays of R device pointers, one per virtual
 *    rank, indexed by rank. The caller owns all device memory and the
 *    stream; the library owns only the opaque layout (host memory).
 *  - Every device pointer must be 16-byte aligned (else FSDP_EALIGN).
 *    Output buffers must not overlap each other or any input (else
 *    FSDP_EINVAL); read-only inputs may alias each other.
 *  - The full unit is the parameters concatenated row-major in unit order,
 *    with no gaps; parameter i starts at FSDP_Q_PARAM_FULL_OFFSET(i).
 *  - Per-rank shard buffers (FSDP_Q_SHARD_NUMEL elements each):
 *      FSDP_PER_PARAM: parameter i occupies a segment starting at
 *        FSDP_Q_PARAM_SHARD_OFFSET(i) of ceil(d0_i/R)*inner_i elements
 *        rounded up to a multiple of FSDP_SEG_ALIGN; the rank's own rows come
 *        first, zero padding after.
 *      FSDP_FLAT: S = ceil(P/R); rank r holds flat elements [r*S, (r+1)*S)
 *        of the unit, the part past P being zero padding.
 *      FSDP_ZERO3: parameters, whole and in unit order, fill rank 0 until
 *        it holds at least ceil(P/R) elements, then rank 1, and so on, the
 *        last rank taking the rest ("从源码理解 FSDP", §2.1: ZeRO-3 assigns
 *        whole tensors to owner ranks; the closing rule is this library's
 *        reading). Each rank's buffer holds its own parameters in unit
 *        order, each segment padded to FSDP_SEG_ALIGN; every buffer is as
 *        long as the longest. The all-gather is then the owner's broadcast
 *        and the reduce-scatter a reduce to the owner.
 *    Padding is never part of a result: the kernels do not read it and do
 *    not write it (fsdp_pack_flat writes it as zero).
 */
#ifndef FSDP_SHARD_H
#define FSDP_SHARD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FSDP_OK = 0,
    FSDP_EINVAL = -1,       /* bad argument: NULL, count, range, aliasing */
    FSDP_EALIGN = -2,       /* a device pointer is not 16-byte aligned */
    FSDP_ERANGE = -3,       /* a size overflows int64 element arithmetic */
    FSDP_ECUDA = -4,        /* a CUDA runtime call or kernel launch failed */
    FSDP_EUNSUPPORTED = -5  /* dtype or mode the library does not implement */
} fsdp_status;

typedef enum {
    FSDP_FLAT = 1,      /* FSDP1: one FlatParameter per unit */
    FSDP_PER_PARAM = 2, /* FSDP2: every parameter sharded on dim 0 */
    FSDP_ZERO3 = 3      /* ZeRO-3 inter-tensor: every parameter whole on one owner rank */
} fsdp_mode;

typedef enum { FSDP_F32 = 0, FSDP_BF16 = 1 } fsdp_dtype;

#define FSDP_MAX_RANKS 64
#define FSDP_SEG_ALIGN 8

typedef struct fsdp_layout_s fsdp_layout_t; /* opaque; host memory */

/* Build the layout of one unit of `n_params` parameters (n_params >= 0).
 * Parameter i has shape [dim0[i], ...] with inner[i] = product of the dims
 * after dim 0 (1 for a vector); dim0[i], inner[i] >= 0 (0 = empty
 * parameter). 1 <= R <= FSDP_MAX_RANKS. param_dtype is the dtype of the
 * shard buffers that the all-gather reads and of its full outputs (the fp32
 * master is always fp32); grad_dtype is the dtype of the full local
 * gradients. On success *out owns a new layout (free it with
 * fsdp_layout_destroy). Errors: FSDP_EINVAL (NULL, bad R/mode/dims),
 * FSDP_ERANGE (element counts past 2^60), FSDP_EUNSUPPORTED (dtype). */
fsdp_status fsdp_layout(fsdp_mode mode, int R, int n_params, const int64_t *dim0,
                        const int64_t *inner, fsdp_dtype param_dtype, fsdp_dtype grad_dtype,
                        fsdp_layout_t **out);

void fsdp_layout_destroy(fsdp_layout_t *layout);

typedef enum {
    FSDP_Q_FULL_NUMEL = 0,            /* P: elements of the full unit */
    FSDP_Q_SHARD_NUMEL = 1,           /* elements of one rank's shard buffer */
    FSDP_Q_PADDED_NUMEL = 2,          /* R * FSDP_Q_SHARD_NUMEL */
    FSDP_Q_N_PARAMS = 3,
    FSDP_Q_RANKS = 4,
    FSDP_Q_MODE = 5,
    FSDP_Q_PARAM_DTYPE = 6,
    FSDP_Q_GRAD_DTYPE = 7,
    FSDP_Q_PARAM_FULL_OFFSET = 8,     /* (i): offset of parameter i in the full unit */
    FSDP_Q_PARAM_SHARD_OFFSET = 9,    /* (i): segment offset (ZERO3: in the owner's buffer);
                                         FLAT: EINVAL */
    FSDP_Q_PARAM_SHARD_ROWS = 10,     /* (i): s_i = ceil(dim0_i / R) (ZERO3: dim0_i) */
    FSDP_Q_PARAM_RANK_ROW_START = 11, /* (i, r): first dim-0 row rank r holds */
    FSDP_Q_PARAM_RANK_ROWS = 12,      /* (i, r): rows rank r holds (0 = empty) */
    FSDP_Q_RANK_NUMEL = 13,           /* (r): real (non-padding) elements rank r holds */
    FSDP_Q_PARAM_OWNER = 14           /* (i): ZERO3 owner rank of parameter i; else EINVAL */
} fsdp_query;

/* Read one property of the layout into *out. `i` (parameter) and `r`
 * (rank) are used only by the queries that name them. Errors: FSDP_EINVAL. */
fsdp_status fsdp_layout_query(const fsdp_layout_t *layout, fsdp_query what, int i, int r,
                              int64_t *out);

/* Shard from full. `full`: device, P fp32 values of the unit. Writes, for
 * every rank r, master[r] (fp32 shard buffer) and, when param_dtype is
 * BF16, param_shard[r] = round-to-nearest-even bf16 of master[r]. For an
 * F32 layout param_shard must be NULL (the master is the parameter shard).
 * Padding is written as zero. Not on the per-step path. */
fsdp_status fsdp_pack_flat(const fsdp_layout_t *layout, const float *full,
                           void *const *param_shard, float *const *master, void *stream);

/* All-gather + unflatten. shard[r]: rank r's parameter shard buffer in
 * param_dtype (for F32 layouts, the fp32 master). full_out[d]: destination
 * rank d's full unit (P elements of param_dtype). Every destination receives
 * the same bytes: full_out[d][j] = the shard element that holds unit
 * element j. A bit copy: no rounding. */
fsdp_status fsdp_all_gather_unflatten(const fsdp_layout_t *layout, const void *const *shard,
                                      void *const *full_out, void *stream);

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
} fsdp_adamw_hp;

/* Reduce-scatter + sharded AdamW, in place on each rank's fp32 state.
 * grad_full[q]: rank q's full local gradient of the unit (P elements of
 * grad_dtype). For each element e that rank r owns, with j its unit index:
 *   acc = g_0[j]; acc = acc + g_1[j]; ...; acc = acc + g_{R-1}[j]   (fp32)
 *   g   = acc * fl(1/R)
 *   w = w*(1 - lr*wd); m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*(g*g);
 *   w = w - (lr/(1 - b1^step)) * (m / (sqrt(v)/sqrt(1 - b2^step) + eps))
 * every operation an fp32 operation rounded to nearest even; the scalars
 * are formed in double from `hp` and `step` and rounded once to fp32.
 * master/m/v[r]: fp32 shard buffers, read and written. param_shard_out[r]:
 * BF16 layouts only (else NULL): receives bf16 RNE of the new master.
 * grad_shard_out: NULL, or R fp32 shard buffers that receive g (for checks;
 * not needed for training). step >= 1; 0 <= beta1, beta2 < 1; eps > 0.
 * For R = 4 or 8 (bf16 gradients) and R = 2 or 4 (fp32 gradients), on
 * launches of at least ~10,000 tiles of 2,048 elements (units of ~20M
 * parameters and up; ~5,000 tiles when most rank pieces start off the
 * 8-element grid), the kernel stages the gradient slices in shared memory
 * with bulk copies and waits for them at most ~2 s; see
 * fsdp_stage_wait_timeouts. The results are the same either way. */
fsdp_status fsdp_reduce_scatter_adamw(const fsdp_layout_t *layout, const void *const *grad_full,
                                      float *const *master, float *const *m, float *const *v,
                                      void *const *param_shard_out, float *const *grad_shard_out,
                                      const fsdp_adamw_hp *hp, int64_t step, void *stream);

/* Prefetch step of two units: the reduce-scatter + AdamW of unit L (the
 * arguments and results of fsdp_reduce_scatter_adamw) followed on the same
 * stream by the all-gather + unflatten of unit G (those of
 * fsdp_all_gather_unflatten) -- the schedule of the pages, which gather the
 * next unit while the current one's gradients are reduced ("FSDP2 的参数全
 * 聚合、梯度归约分片与显存峰值", §07 forward prefetch; "从源码理解 FSDP", §5.2
 * layer-wise all-gather overlap). Both operations are validated together:
 * every buffer of one must be disjoint from every output of the other (so G
 * may not be the unit being updated), which leaves the library free to order
 * or overlap them. On GB300 the two launches back to back were faster than
 * any single launch interleaving them, so that is what is issued.
 * Errors as for the two calls. */
fsdp_status fsdp_reduce_scatter_adamw_gather(
    const fsdp_layout_t *L, const void *const *grad_full, float *const *master, float *const *m,
    float *const *v, void *const *param_shard_out, float *const *grad_shard_out,
    const fsdp_adamw_hp *hp, int64_t step, const fsdp_layout_t *G, const void *const *shard,
    void *const *full_out, void *stream);

/* ZeRO-1's optimizer step ("从源码理解 FSDP", §1.2, the ZeRO stages: the
 * gradients are all-reduced, so every rank holds the whole averaged
 * gradient, and each rank updates only the parameters and optimizer state of
 * its own partition, which an all-gather then shares). grad_avg_full[r]:
 * rank r's full averaged fp32 gradient, P elements, as fsdp_all_reduce with
 * an FSDP_F32 output leaves it. For each element that rank r owns, with j its
 * unit index: g = grad_avg_full[r][j], then the AdamW update of
 * fsdp_reduce_scatter_adamw on master/m/v[r] and param_shard_out[r] (BF16
 * layouts only, else NULL). With fsdp_all_reduce's output the results equal
 * fsdp_reduce_scatter_adamw's on the same gradients bit for bit. Errors: as
 * fsdp_reduce_scatter_adamw. */
fsdp_status fsdp_adamw_from_reduced(const fsdp_layout_t *layout, const float *const *grad_avg_full,
                                    float *const *master, float *const *m, float *const *v,
                                    void *const *param_shard_out, const fsdp_adamw_hp *hp,
                                    int64_t step, void *stream);

/* All-reduce, the DDP collective that FSDP is compared against ("FSDP
 * Training Step Walkthrough", per-step communication summary; "FSDP2 的参数
 * 全聚合、梯度归约分片与显存峰值", §01 and §09). Every rank d receives, for
 * every unit element j, the same fixed-order average as the reduce-scatter:
 *   acc = g_0[j] + g_1[j] + ... + g_{R-1}[j] (fp32, left to right);
 *   out[d][j] = acc * fl(1/R), stored as fp32 or as its bf16 rounding.
 * So gathering the fp32 reduce-scatter shards reproduces out[d] bit for bit.
 * grad_full[q]: rank q's P elements of the layout's grad_dtype; out[d]: P
 * elements of out_dtype. Only R, P and the grad dtype of the layout are
 * used. Errors: FSDP_EINVAL, FSDP_EALIGN, FSDP_EUNSUPPORTED (out_dtype). */
fsdp_status fsdp_all_reduce(const fsdp_layout_t *layout, const void *const *grad_full,
                            void *const *out, fsdp_dtype out_dtype, void *stream);

/* Gradient accumulation over micro-batches ("FSDP2 的参数全聚合、梯度归约分片
 * 与显存峰值", §08: every micro-batch runs forward and backward, the update
 * happens once per K micro-batches). For every rank q and unit element j:
 *   first != 0:  acc_full[q][j] = g_q[j]                 (exact widening)
 *   first == 0:  acc_full[q][j] = acc_full[q][j] + g_q[j]   (one fp32 add)
 * acc_full[q]: rank q's P fp32 accumulators (read and written); grad_full[q]:
 * P elements of the layout's grad_dtype. The accumulated gradient is the
 * plain sum over micro-batches; scale the loss for any 1/K normalisation.
 * Errors: FSDP_EINVAL, FSDP_EALIGN. */
fsdp_status fsdp_accumulate_grad(const fsdp_layout_t *layout, float *const *acc_full,
                                 const void *const *grad_full, int first, void *stream);

/* The last micro-batch fused into the optimizer step: exactly
 * fsdp_reduce_scatter_adamw, except that rank q's gradient is
 * acc_full[q][j] + grad_full[q][j] (one fp32 add per rank, then the same
 * rank-ordered fold). Bit-identical to fsdp_accumulate_grad of the last
 * micro-batch followed by fsdp_reduce_scatter_adamw on the accumulators, and
 * saves one write and one read of the accumulators. acc_full is read only.
 * Errors as fsdp_reduce_scatter_adamw. */
fsdp_status fsdp_reduce_scatter_adamw_accum(const fsdp_layout_t *layout,
                                            const float *const *acc_full,
                                            const void *const *grad_full, float *const *master,
                                            float *const *m, float *const *v,
                                            void *const *param_shard_out,
                                            float *const *grad_shard_out, const fsdp_adamw_hp *hp,
                                            int64_t step, void *stream);

/* Several units in one call: the all-gather + unflatten of n_units units,
 * each exactly as fsdp_all_gather_unflatten would do it, issued as one
 * kernel launch (or a few, past 256 parameters or 64 per-rank pointers per
 * launch). This is the pages' bucketing taken one level up: many small
 * collectives fused into one ("从源码理解 FSDP", §5.3 bucketing small tensors
 * into one communication; "FSDP2 的参数全聚合、梯度归约分片与显存峰值", §05
 * how grouping sets the size of each all-gather). It exists for small units,
 * whose per-call host work and per-launch ramp dominate their streaming time.
 * layouts[u]: unit u's layout; all share R and the dtypes (else FSDP_EINVAL);
 * one layout may serve several units. shard and full_out hold n_units*R
 * device pointers, unit-major: entry u*R + r is unit u's rank r. Every buffer
 * is validated as in the one-unit call, and outputs must not overlap any
 * buffer of any unit. Units with no elements are skipped (their pointers may
 * be NULL). Errors: as fsdp_all_gather_unflatten, plus FSDP_EINVAL for
 * n_units < 1 or a NULL layout. */
fsdp_status fsdp_all_gather_unflatten_units(int n_units, const fsdp_layout_t *const *layouts,
                                            const void *const *shard, void *const *full_out,
                                            void *stream);

/* The reduce-scatter + AdamW step of n_units units in one call (see
 * fsdp_all_gather_unflatten_units for the grouping and the pointer arrays,
 * which here are grad_full, master, m, v, param_shard_out and, if not NULL,
 * grad_shard_out, each n_units*R entries, unit-major). Every unit takes the
 * same hyper-parameters and step, and gets exactly the result of
 * fsdp_reduce_scatter_adamw. param_shard_out is required for BF16 layouts and
 * must be NULL for F32 layouts. Errors: as fsdp_reduce_scatter_adamw, plus
 * FSDP_EINVAL for n_units < 1 or a NULL layout. */
fsdp_status fsdp_reduce_scatter_adamw_units(int n_units, const fsdp_layout_t *const *layouts,
                                            const void *const *grad_full, float *const *master,
                                            float *const *m, float *const *v,
                                            void *const *param_shard_out,
                                            float *const *grad_shard_out, const fsdp_adamw_hp *hp,
                                            int64_t step, void *stream);

/* Measurement helper; the pages have no counterpart. Writes the 32-bit
 * `pattern` over the first `bytes` bytes of each of the n device buffers
 * dst[0..n) (1 <= n <= FSDP_MAX_RANKS; bytes a multiple of 32; buffers
 * 32-byte aligned, disjoint, on one device), with the all-gather's store
 * pattern and grid. Timing it gives the write-only stream ceiling that
 * bounds the all-gather (which writes R bytes per byte read) and the
 * all-reduce. Errors: FSDP_EINVAL, FSDP_EALIGN, FSDP_ECUDA. */
fsdp_status fsdp_write_stream(void *const *dst, int n, int64_t bytes, uint32_t pattern,
                              void *stream);

/* Implementation status; the pages have no counterpart. The number of
 * thread blocks of the staged reduce-scatter kernel on CUDA device `device`
 * that gave up waiting for their gradient bulk copies (after ~2 s each),
 * since the library was loaded. A block that gives up leaves the rest of its
 * tiles unwritten, so any nonzero count means the results of the calls
 * since the last read of 0 are invalid. Waits for all work on the device
 * (cudaDeviceSynchronize) before it reads; restores the caller's current
 * device. Errors: FSDP_EINVAL (count NULL, device < 0), FSDP_ECUDA. */
fsdp_status fsdp_stage_wait_timeouts(int device, uint64_t *count);

/* Self-test of that bounded wait; the pages have no counterpart. Launches
 * one thread block on `device` that waits on an mbarrier whose phase cannot
 * complete (bytes announced that no copy delivers), gives up after 20 ms and
 * counts itself in a counter of its own (fsdp_stage_wait_timeouts is not
 * touched). *gave_up receives the number of blocks that gave up: 1. The
 * device stays usable. Synchronises the device; restores the caller's
 * current device. Errors: FSDP_EINVAL (gave_up NULL, device < 0),
 * FSDP_ECUDA. */
fsdp_status fsdp_stage_wait_selftest(int device, uint64_t *gave_up);

/* Message for the last non-OK status returned on the calling thread. */
const char *fsdp_last_error(void);

/* Library version string. */
const char *fsdp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FSDP_SHARD_H */
