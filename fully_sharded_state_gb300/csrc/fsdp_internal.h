// fsdp_internal.h -- types shared by the library's host code (fsdp_capi.cpp)
// and its kernels (fsdp_kernels.cu). Not part of the public ABI.
#pragma once

#include <cstdint>
#include <vector>

#include "fsdp_shard.h"

namespace fsdp {

// Work decomposition. A tile is kTile consecutive elements of one rank's
// piece of one segment; each thread of a CTA owns kElemsPerThread of them
// (one 16-byte vector of bf16, two of fp32).
constexpr int kThreads = 256;
constexpr int kElemsPerThread = 8;
constexpr int64_t kTile = (int64_t)kThreads * kElemsPerThread;
// The all-gather's threads own 16 elements each (one 32-byte vector of bf16),
// so its tiles are twice as long.
constexpr int kGatherEPT = 16;
constexpr int64_t kGatherTile = (int64_t)kThreads * kGatherEPT;
// Segment descriptors travel in the kernel parameter block; larger units are
// split into several launches.
constexpr int kMaxSegsPerLaunch = 256;

// One FSDP2 parameter, or the whole FSDP1 FlatParameter, as the kernels see
// it. Rank r holds full elements [full_off + r*rank_stride, + n_r) with
// n_r = clamp(numel - r*rank_stride, 0, rank_stride), stored at shard_off in
// its shard buffer, followed by padding up to pad_len.
struct Seg {
    int64_t full_off;
    int64_t numel;
    int64_t rank_stride;
    int64_t shard_off;
    int64_t pad_len;
    int64_t tile_begin;      // first tile of this segment within its launch
    int64_t tiles_per_rank;  // tiles of a rank that holds rank_stride (or pad_len) elements
    int32_t owner;           // -1: dim-0 slices as above; >= 0: the whole segment
                             // (numel elements) belongs to this rank
    int32_t base;            // where this segment's unit starts in the launch's per-rank
                             // pointer arrays: rank r's buffer is entry base + r
    int64_t unit_numel;      // P of the segment's unit: the length of its full and
                             // gradient buffers
};

// The segments of one launch and its tile count. elems: the elements its
// tiles cover; aligned_elems: those in rank pieces whose full and shard
// starts are both 32-byte aligned (the all-gather's vector paths need it).
struct LaunchPlan {
    std::vector<Seg> segs;
    int64_t total_tiles = 0;
    int64_t elems = 0;
    int64_t aligned_elems = 0;
    int64_t aligned8_elems = 0;  // those whose full and shard starts are multiples
                                 // of 8 elements (the reduce-scatter's vectors)
};

// AdamW scalars, formed on the host in double and rounded once to fp32.
struct AdamScalars {
    float decay;      // 1 - lr*wd
    float b1, omb1;   // beta1, 1 - beta1
    float b2, omb2;   // beta2, 1 - beta2
    float step_size;  // lr / (1 - beta1^t)
    float bc2_sqrt;   // sqrt(1 - beta2^t)
    float eps;
    float inv_R;      // fl(1/R)
};

fsdp_status set_error(fsdp_status st, const char *fmt, ...);

// Kernel launchers (fsdp_kernels.cu). Arguments are validated by the caller.
fsdp_status launch_pack(const fsdp_layout_t *L, const float *full, void *const *param_shard,
                        float *const *master, void *stream);
// The gather and the reduce-scatter take n >= 1 layouts with the same R and
// dtypes; every per-rank pointer array then holds n*R entries, unit-major
// (entry u*R + r is unit u's rank r).
fsdp_status launch_all_gather(int n, const fsdp_layout_t *const *Ls, const void *const *shard,
                              void *const *full_out, void *stream);
// acc: NULL, or fp32 gradient accumulators added to grad (rank by rank)
// before the fold.
fsdp_status launch_rs_adamw(int n, const fsdp_layout_t *const *Ls, const void *const *grad,
                            float *const *master, float *const *m, float *const *v,
                            void *const *param_shard_out, float *const *grad_shard_out,
                            const AdamScalars &c, void *stream, const float *const *acc);
fsdp_status launch_accumulate(const fsdp_layout_t *L, float *const *acc, const void *const *grad,
                              int first, void *stream);
fsdp_status launch_adamw_reduced(const fsdp_layout_t *L, const float *const *grad_avg,
                                 float *const *master, float *const *m, float *const *v,
                                 void *const *param_shard_out, const AdamScalars &c, void *stream);
fsdp_status launch_all_reduce(const fsdp_layout_t *L, const void *const *grad, void *const *out,
                              fsdp_dtype out_dtype, void *stream);
fsdp_status launch_write_stream(void *const *dst, int n, int64_t bytes, uint32_t pattern,
                                void *stream);
fsdp_status read_stage_wait_timeouts(int device, uint64_t *count);
fsdp_status run_stage_wait_selftest(int device, uint64_t *gave_up);
fsdp_status launch_rs_adamw_gather(const fsdp_layout_t *A, const void *const *grad,
                                   float *const *master, float *const *m, float *const *v,
                                   void *const *param_shard_out, float *const *grad_shard_out,
                                   const AdamScalars &c, const fsdp_layout_t *B,
                                   const void *const *shard, void *const *full_out, void *stream);

}  // namespace fsdp

struct fsdp_layout_s {
    fsdp_mode mode;
    int R;
    int n;
    fsdp_dtype param_dtype;
    fsdp_dtype grad_dtype;
    std::vector<int64_t> dim0, inner, full_off, shard_off, shard_rows;
    std::vector<int64_t> owner;  // ZERO3: owner rank of each parameter
    int64_t P;            // full numel
    int64_t shard_numel;  // per-rank shard buffer numel
    std::vector<fsdp::LaunchPlan> valid_plans;   // kTile tiles over owned elements (reduce)
    std::vector<fsdp::LaunchPlan> gather_plans;  // kGatherTile tiles over owned elements
    std::vector<fsdp::LaunchPlan> padded_plans;  // kTile tiles over whole shard buffers (pack)
};
