// fsdp_kernels.cu -- the shard engine's kernels for sm_103a (GB300).
//
// Every kernel here streams HBM: nothing is a dense contraction, so there is
// no tensor-core work. The layout-driven kernels (pack, all-gather, fused
// reduce-scatter + AdamW) share one work decomposition: a launch covers up to
// kMaxSegsPerLaunch segments (parameters, one FlatParameter, or ZeRO-3 tensors
// with their owner ranks, from one unit or several); each segment's rank
// pieces are cut into tiles (kTile elements; kGatherTile for the gather); a
// persistent grid (a few CTAs per SM) walks the tiles in order, so at any
// moment the grid touches one contiguous window of every buffer. A thread
// owns 8 consecutive elements of a tile (16 in the gather): one 16-byte
// vector per bf16 stream, two per fp32 stream. Shard offsets are always
// multiples of 8 elements; a tile whose full-buffer start is not (ragged
// FSDP1 boundaries, odd row widths) is realigned: the gather stages its
// shard elements in shared memory, the staged reduce-scatter stages the
// 16-byte span around it and the register one (bf16, R = 8) loads aligned
// chunks, each shifting the words into place in registers; the other
// register reduce-scatters take a scalar path with the same per-element
// arithmetic. The all-reduce and gradient-accumulation kernels tile the flat
// unit index the same way.
//
// Segment descriptors and the per-rank pointers travel in the kernel
// parameter block (__grid_constant__), so the kernels need no device memory
// beyond the caller's buffers (and two counters of abandoned waits, below).
//
// The fused reduce-scatter + AdamW brings each tile's R gradient slices into
// shared memory with cp.async.bulk, a few tiles ahead, on per-stage
// mbarriers (rs_adamw_staged_kernel) on large launches where R is a
// compile-time 4 or 8 (bf16 gradients) or 2 or 4 (fp32 gradients); otherwise
// every load is a register load.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "fsdp_internal.h"

namespace fsdp {
namespace {

constexpr int kMaxR = FSDP_MAX_RANKS;

// Resident CTAs per SM of each kernel's persistent grid. Measured on GB300
// with 218M-parameter Llama units, R = 8 (one launch per point):
//   reduce-scatter + AdamW: 2/SM 1.520 ms, 3/SM 1.389 ms, 4/SM (the register
//   limit) 1.498 ms.
// Fewer CTAs, each streaming its tiles in order, keep a narrower window of
// every buffer open at once; past these points HBM does not go faster.
constexpr int kRsCtasPerSm = 3;
// ... but 4 on launches of at most kRsSmallLaunchTiles tiles, whose data
// mostly sits in L2 (flat units, reduce-scatter alone, 4/SM vs 3/SM: 512
// tiles bf16 R = 4 0.92, 1,536 tiles bf16 R = 4 0.97 and fp32 R = 4 0.95,
// bf16 R = 8 1.00, fp32 R = 2 1.02; 3,626 tiles bf16 R = 4 1.06).
constexpr int kRsCtasPerSmSmall = 4;
constexpr int64_t kRsSmallLaunchTiles = 2048;
// The staged form (gradient slices by cp.async.bulk, 3 stages of 32 KB for
// bf16 R = 8): 1/SM 2.08 ms, 2/SM 1.327 ms on the same unit, and 1.331 ms
// right after a gather-shaped write stream, where the register form takes
// 1.398 ms (a replica of both kernels, one process).
constexpr int kRsStagedCtasPerSm = 2;
// Stage sizing: a stage (R slices of one tile) of at most kRsStageMaxBytes
// of gradients, and as many stages (2 to 8) as fit, with their barriers and
// tile descriptors, in kRsStagedSmemBudget: two CTAs and their 1 KB
// reservations then fit the 196 KB shared-memory carveout. Past it the SM
// takes the 228 KB carveout, L1 drops from 60 KB to 28 KB, and a Llama unit's
// reduce-scatter took 1.351 ms instead of 1.305.
constexpr int kRsStageMaxBytes = 32 * 1024;
constexpr int kRsStagedSmemBudget = 97 * 1024;
// When staging pays (staged / register time, flat units, alone):
//   R x gradient bytes = 8 or 16 (bf16 R = 4, 8; fp32 R = 2, 4): 0.92-0.97
//   from 16K tiles (54 per staged CTA), about even at 6K-8K, 1.05-1.3
//   below 4K tiles, where the ring of stages never fills;
//   R x gradient bytes = 4 (bf16 R = 2): 1.08-1.3 at every size.
constexpr int kRsStageMinGradBytes = 8;
constexpr int kRsStagedMinTilesPerCta = 32;
// A launch whose elements mostly sit in rank pieces that start off the
// 8-element grid stages from 16 tiles per CTA: the staged kernel realigns
// them at full speed, while the register kernel's scalar path is slow
// (misaligned flat units, 5,859 tiles, staged / register: bf16 R = 4 0.87,
// bf16 R = 8 0.93, fp32 R = 4 0.86; 2,929 tiles: bf16 R = 4 1.06).
constexpr int kRsStagedMinTilesPerCtaMisaligned = 16;
// all-gather (256 threads, 16 elements per thread): 1/SM 0.613 ms,
// 2/SM 0.668 ms, 3/SM 0.667 ms on a Llama unit, whose tiles are full and
// aligned. A launch whose elements mostly sit in misaligned or partial tiles
// (the ragged fp32 workload: 2 % aligned, tiles 86 % full) runs faster with
// more CTAs to overlap their latencies: 1/SM 0.067 ms, 2/SM 0.053, 4/SM
// 0.051, 8/SM 0.052.
constexpr int kGatherCtasPerSm = 1;
constexpr int kGatherCtasPerSmIrregular = 4;
// pack (set-up): 1/SM 0.810, 2/SM 0.482, 3/SM 0.404, 4/SM 0.356, 6/SM
// 0.421, 8/SM 0.418 ms.
constexpr int kPackCtasPerSm = 4;
// all-reduce (bf16 grads -> fp32 outputs), pipelined with 32-byte stores:
// 1/SM 1.575 ms, 2/SM 1.676 ms, 3/SM 1.665 ms (a replica of the kernel).
constexpr int kAllReduceCtasPerSm = 1;
constexpr int kAccumulateCtasPerSm = 3;

struct PackParams {
    const float *full;
    float *master[kMaxR];
    uint16_t *pshard[kMaxR];
    int R;
    int nseg;
    int64_t total_tiles;
    Seg seg[kMaxSegsPerLaunch];
};

struct GatherParams {
    const unsigned char *shard[kMaxR];
    unsigned char *full[kMaxR];
    int R;
    int wide;  // every shard and full pointer is 32-byte aligned
    int nseg;
    int64_t total_tiles;
    Seg seg[kMaxSegsPerLaunch];
};

struct RsParams {
    const void *grad[kMaxR];
    const float *acc[kMaxR];  // gradient accumulators (NULL unless accumulating)
    float *master[kMaxR];
    float *m[kMaxR];
    float *v[kMaxR];
    uint16_t *pshard[kMaxR];
    float *gshard[kMaxR];
    AdamScalars c;
    int R;
    int nseg;
    int64_t total_tiles;
    Seg seg[kMaxSegsPerLaunch];
};

// ---------------------------------------------------------------- tiles ----

struct Tile {
    int rank;        // the tile's rank within its unit
    int base;        // the unit's first entry in the per-rank pointer arrays
    int64_t fbase;   // full-buffer index of the tile's first element
    int64_t sbase;   // shard-buffer index of the tile's first element
    int64_t len;     // elements in the tile
    int64_t nvalid;  // padded traversal: elements of the tile that the rank owns
    int64_t unit_numel;  // P of the tile's unit (the full and gradient buffers' length)
};

// kT: the kernel's tile length.
template <int64_t kT>
__device__ __forceinline__ Tile locate(const Seg *seg, int nseg, int64_t t, bool padded)
{
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (seg[mid].tile_begin <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    const Seg &s = seg[lo];
    int64_t tl = t - s.tile_begin;
    int r, first_of_rank;
    int64_t off, owned;
    if (s.owner >= 0) {  // a whole parameter on its owner rank
        r = (int)s.owner;
        first_of_rank = 0;
        off = tl * kT;
        owned = s.numel;
    } else {
        r = (int)(tl / s.tiles_per_rank);
        first_of_rank = r;
        off = (tl - (int64_t)r * s.tiles_per_rank) * kT;
        owned = s.numel - (int64_t)r * s.rank_stride;
        owned = owned < 0 ? 0 : (owned > s.rank_stride ? s.rank_stride : owned);
    }
    int64_t piece = padded ? s.pad_len : owned;
    Tile T;
    T.rank = r;
    T.base = s.base;
    T.fbase = s.full_off + (int64_t)first_of_rank * s.rank_stride + off;
    T.sbase = s.shard_off + off;
    T.len = piece - off < kT ? piece - off : kT;
    int64_t nv = owned - off;
    T.nvalid = nv < 0 ? 0 : (nv > T.len ? T.len : nv);
    T.unit_numel = s.unit_numel;
    return T;
}

// ------------------------------------------------------ memory helpers ----

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(void *p, uint4 v)
{
    __stcs(reinterpret_cast<uint4 *>(p), v);
}
__device__ __forceinline__ float4 ld_f4(const float *p)
{
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_f4(float *p, float4 v)
{
    __stcs(reinterpret_cast<float4 *>(p), v);
}

// ---------------------------------------- bulk copies and mbarriers ----

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival that also announces `bytes` of bulk copies to come.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for phase `parity` of `bar` for at most `limit_ns` of the global
// timer, and at most 2^27 polls should the timer not advance; false if it
// gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t round = 0; round < (1u << 22); round++) {
        for (int k = 0; k < 32; k++)
            if (mbar_try_wait(bar, parity))
                return true;
        if (global_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}
constexpr uint64_t kStageWaitNs = 2000000000ull;  // a stage's copies: 2 s

// CTAs that gave up waiting for their bulk copies (read by the host through
// fsdp_stage_wait_timeouts). Zero unless a copy failed to arrive.
__device__ unsigned long long g_stage_wait_timeouts;
// The same count for the self-test below, kept apart so that it never
// touches the real one.
__device__ unsigned long long g_selftest_wait_timeouts;

// Self-test of the bounded wait: one CTA waits on an mbarrier whose phase
// cannot complete (one arrival announcing 16 bytes that no copy delivers),
// gives up after limit_ns and counts itself. No copy is in flight, so the
// CTA may leave with the phase open.
__global__ void stage_wait_selftest_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
        mbar_arrive_expect_tx(&bar, 16);
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
    if (__syncthreads_or(!ok) && threadIdx.x == 0)
        atomicAdd(&g_selftest_wait_timeouts, 1ull);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h)
{
    return __uint_as_float((uint32_t)h << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ---------------------------------------------------------------- pack ----

template <bool kBf16>
__global__ void __launch_bounds__(kThreads) pack_kernel(const __grid_constant__ PackParams p)
{
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const Tile T = locate<kTile>(p.seg, p.nseg, t, true);  // one unit: base 0
        float *dst = p.master[T.rank] + T.sbase;
        uint16_t *dst16 = kBf16 ? p.pshard[T.rank] + T.sbase : nullptr;
        const float *src = p.full + T.fbase;
        const int64_t e = (int64_t)threadIdx.x * kElemsPerThread;
        const bool aligned = ((T.fbase | T.sbase) & (kElemsPerThread - 1)) == 0;
        if (aligned && e + kElemsPerThread > T.len) {
            // the tile's last, partial group of this thread's 8 elements
            for (int64_t q = e; q < T.len; q++) {
                float x = q < T.nvalid ? src[q] : 0.0f;
                dst[q] = x;
                if (kBf16)
                    dst16[q] = f32_to_bf16_bits(x);
            }
            continue;
        }
        if (aligned) {
            // 8 elements: owned ones from the full unit, the rest zero padding
            float x[8];
            if (e + kElemsPerThread <= T.nvalid) {
                const float4 a = __ldcs(reinterpret_cast<const float4 *>(src + e));
                const float4 b = __ldcs(reinterpret_cast<const float4 *>(src + e + 4));
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
            } else {
#pragma unroll
                for (int k = 0; k < 8; k++)
                    x[k] = e + k < T.nvalid ? src[e + k] : 0.0f;
            }
            st_f4(dst + e, make_float4(x[0], x[1], x[2], x[3]));
            st_f4(dst + e + 4, make_float4(x[4], x[5], x[6], x[7]));
            if (kBf16) {
                uint4 v;
                v.x = (uint32_t)f32_to_bf16_bits(x[0]) | ((uint32_t)f32_to_bf16_bits(x[1]) << 16);
                v.y = (uint32_t)f32_to_bf16_bits(x[2]) | ((uint32_t)f32_to_bf16_bits(x[3]) << 16);
                v.z = (uint32_t)f32_to_bf16_bits(x[4]) | ((uint32_t)f32_to_bf16_bits(x[5]) << 16);
                v.w = (uint32_t)f32_to_bf16_bits(x[6]) | ((uint32_t)f32_to_bf16_bits(x[7]) << 16);
                st_stream(dst16 + e, v);
            }
            continue;
        }
#pragma unroll
        for (int k = 0; k < kElemsPerThread; k++) {
            int64_t q = threadIdx.x + (int64_t)k * kThreads;
            if (q < T.len) {
                float x = q < T.nvalid ? src[q] : 0.0f;
                dst[q] = x;
                if (kBf16)
                    dst16[q] = f32_to_bf16_bits(x);
            }
        }
    }
}

// ----------------------------------------------------- all-gather ----------
//
// The gather writes R bytes for every byte it reads, so its store pattern
// sets its speed. Each thread owns 16 consecutive elements of a
// kGatherTile-element tile: with 32-byte aligned buffers every store
// instruction writes whole 32-byte sectors (one 32-byte vector per
// destination for bf16, two for fp32). Two 16-byte halves of one sector
// written by separate instructions cost about 1.8x the DRAM time of
// whole-sector writes on GB300 (a write-only stream of 8 fp32 buffers: 3.7
// TB/s with 16-byte halves, 6.5 TB/s with 32-byte stores). Tiles that are
// only 16-byte aligned use 16-byte vectors laid out so that a warp's
// instruction still covers 512 contiguous bytes; other tiles copy element
// by element.
//
// Measured interplay on GB300 (Llama unit, R = 8, gather then reduce-scatter
// as in a step): after this gather the reduce-scatter takes 1.376 ms, after
// a gather whose threads store 16 bytes each (512 bytes per warp
// instruction) 1.327 ms, with identical reduce-scatter code and identical
// placement of its CTAs on the SMs; the 16-byte gather itself takes
// 0.627-0.666 ms against 0.613 ms here. The sum is about 1 % in favour of
// the 16-byte gather; this one is kept because it alone holds the gather
// above 80 % of the nominal HBM bandwidth.

constexpr int kGatherThreads = kThreads;
static_assert(kGatherThreads * kGatherEPT == kGatherTile, "a gather CTA covers one tile");

template <int kEB> struct ElemOf;
template <> struct ElemOf<2> { using T = unsigned short; };
template <> struct ElemOf<4> { using T = unsigned int; };

__device__ __forceinline__ void ld32(const void *p, uint4 &a, uint4 &b)
{
    asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                   "=r"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ void st32(void *p, const uint4 &a, const uint4 &b)
{
    asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x),
                 "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

// One all-gather tile: the tile's shard elements go to the same place of
// every destination's full buffer. kEB = element bytes (2 bf16, 4 fp32); the
// copy is bitwise. PP is any parameter block with `shard`, `full` and `wide`
// (1 when every shard and full pointer of the launch is 32-byte aligned);
// `stage` is the CTA's shared buffer of kGatherTile elements. Every thread of
// the CTA calls this with the same tile.
template <int RC, int kEB, class PP>
__device__ __forceinline__ void gather_tile(const PP &p, int R, const Tile &T,
                                            unsigned char *stage)
{
    using E = typename ElemOf<kEB>::T;
    constexpr int kV = 16 / kEB;                     // elements per 16-byte vector
    constexpr int kW = 32 / kEB;                     // elements per 32-byte vector
    constexpr int kWide = kGatherEPT / kW;           // 32-byte vectors per thread
    constexpr int kNarrow = kGatherTile / (kGatherThreads * kV);  // 16-byte vectors per thread
    const int n = RC > 0 ? RC : R;
    const E *src = reinterpret_cast<const E *>(p.shard[T.base + T.rank]) + T.sbase;
    // destination pointers in registers when R is known at compile time
    constexpr int kN = RC > 0 ? RC : 1;
    unsigned char *fl[kN];
    unsigned char *const *full = p.full + T.base;
    if (RC > 0) {
#pragma unroll
        for (int d = 0; d < kN; d++)
            fl[d] = p.full[T.base + d];
        full = fl;
    }
    const int64_t off = T.fbase | T.sbase;
    const int tid = threadIdx.x;
    if (p.wide && (off & (kW - 1)) == 0) {
        const int64_t e = (int64_t)tid * kGatherEPT;
        if (e + kGatherEPT <= T.len) {
            uint4 x[kWide][2];
#pragma unroll
            for (int k = 0; k < kWide; k++)
                ld32(src + e + k * kW, x[k][0], x[k][1]);
#pragma unroll 8
            for (int d = 0; d < n; d++) {
                E *dst = reinterpret_cast<E *>(full[d]) + T.fbase + e;
#pragma unroll
                for (int k = 0; k < kWide; k++)
                    st32(dst + k * kW, x[k][0], x[k][1]);
            }
            return;
        }
        for (int64_t q = e; q < T.len && q < e + kGatherEPT; q++) {
            const E x = src[q];
            for (int d = 0; d < n; d++)
                reinterpret_cast<E *>(full[d])[T.fbase + q] = x;
        }
        return;
    }
    if ((off & (kV - 1)) == 0) {
        uint4 x[kNarrow];  // every load of this thread before its stores
#pragma unroll
        for (int k = 0; k < kNarrow; k++) {
            const int64_t e = (int64_t)(tid + k * kGatherThreads) * kV;
            if (e + kV <= T.len)
                x[k] = ld_stream(src + e);
        }
#pragma unroll
        for (int k = 0; k < kNarrow; k++) {
            const int64_t e = (int64_t)(tid + k * kGatherThreads) * kV;
            if (e + kV <= T.len) {
#pragma unroll 8
                for (int d = 0; d < n; d++)
                    st_stream(reinterpret_cast<E *>(full[d]) + T.fbase + e, x[k]);
            } else {
                for (int64_t q = e; q < T.len; q++) {
                    const E x = src[q];
                    for (int d = 0; d < n; d++)
                        reinterpret_cast<E *>(full[d])[T.fbase + q] = x;
                }
            }
        }
        return;
    }
    if ((T.sbase & (kV - 1)) == 0) {
        // Only the full side is misaligned (odd row widths, ragged FlatParameter
        // boundaries; shard segments start aligned): stage the tile's shard
        // elements in shared memory with aligned 16-byte loads, then write
        // every destination in aligned 16-byte vectors read from the stage at
        // the shifted offset; the few elements before the first and after the
        // last aligned destination vector go one by one.
        E *sE = reinterpret_cast<E *>(stage);
        const int64_t nvec = T.len / kV;
        for (int64_t v = tid; v < nvec; v += kGatherThreads)
            reinterpret_cast<uint4 *>(stage)[v] = ld_stream(src + v * kV);
        for (int64_t q = nvec * kV + tid; q < T.len; q += kGatherThreads)
            sE[q] = src[q];
        __syncthreads();
        const int64_t head = (kV - (T.fbase & (kV - 1))) & (kV - 1);
        const int64_t body = T.len > head ? (T.len - head) / kV : 0;
        for (int64_t v = tid; v < body; v += kGatherThreads) {
            const int64_t q0 = head + v * kV;
            uint4 x;
            E *xe = reinterpret_cast<E *>(&x);
#pragma unroll
            for (int i = 0; i < kV; i++)
                xe[i] = sE[q0 + i];
#pragma unroll 8
            for (int d = 0; d < n; d++)
                st_stream(reinterpret_cast<E *>(full[d]) + T.fbase + q0, x);
        }
        for (int64_t q = tid; q < T.len; q += kGatherThreads) {
            if (q >= head && q < head + body * kV)
                continue;
            const E x = sE[q];
            for (int d = 0; d < n; d++)
                reinterpret_cast<E *>(full[d])[T.fbase + q] = x;
        }
        __syncthreads();  // the stage is free for the next tile
        return;
    }
    // element by element, four loads of a thread before their stores
#pragma unroll 1
    for (int k0 = 0; k0 < kGatherEPT; k0 += 4) {
        E x[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int64_t q = tid + (int64_t)(k0 + k) * kGatherThreads;
            x[k] = q < T.len ? src[q] : E(0);
        }
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int64_t q = tid + (int64_t)(k0 + k) * kGatherThreads;
            if (q < T.len)
                for (int d = 0; d < n; d++)
                    reinterpret_cast<E *>(full[d])[T.fbase + q] = x[k];
        }
    }
}

// kUnits: the launch holds several units (segments carry their unit's
// pointer base); otherwise the base is a compile-time 0 and the per-rank
// pointers are read from the parameter block at fixed offsets.
template <int RC, int kEB, bool kUnits>
__global__ void __launch_bounds__(kGatherThreads)
    all_gather_kernel(const __grid_constant__ GatherParams p)
{
    // one tile's shard elements, for tiles whose full side is misaligned
    __shared__ __align__(16) unsigned char stage[kGatherTile * kEB];
    const int R = RC > 0 ? RC : p.R;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        Tile T = locate<kGatherTile>(p.seg, p.nseg, t, false);
        if (!kUnits)
            T.base = 0;
        gather_tile<RC, kEB>(p, R, T, stage);
    }
}

// ------------------------------------------- reduce-scatter + AdamW --------

struct AdamOut {
    float w, m, v;
};

// One element's AdamW step; each operation is a single fp32 operation
// rounded to nearest even (no FMA contraction), in the documented order.
__device__ __forceinline__ AdamOut adamw_elem(const AdamScalars &c, float g, float w, float m,
                                              float v)
{
    AdamOut o;
    float wd = __fmul_rn(w, c.decay);
    o.m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
    o.v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.omb2, __fmul_rn(g, g)));
    float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(o.v), c.bc2_sqrt), c.eps);
    o.w = __fsub_rn(wd, __fmul_rn(c.step_size, __fdiv_rn(o.m, denom)));
    return o;
}

template <bool kGradBf16>
__device__ __forceinline__ float load_grad(const void *g, int64_t j)
{
    if (kGradBf16)
        return bf16_bits_to_f32(__ldcs(reinterpret_cast<const unsigned short *>(g) + j));
    return __ldcs(reinterpret_cast<const float *>(g) + j);
}

// The R gradient (and accumulator) pointers of one unit, and the state
// buffers of the rank that owns a tile.
struct RankPtrs {
    const void *const *grad;  // [R]: each rank's full local gradient
    const float *const *acc;  // [R]: accumulators (only read when accumulating)
    float *master, *m, *v;
    uint16_t *pshard;
    float *gshard;
};

template <class PP>
__device__ __forceinline__ RankPtrs rank_ptrs(const PP &p, const Tile &T)
{
    const int i = T.base + T.rank;
    return {p.grad + T.base, p.acc + T.base, p.master[i], p.m[i], p.v[i], p.pshard[i],
            p.gshard[i]};
}

// Rank q's gradient at unit index j; with accumulators, the accumulated
// earlier micro-batches plus this one (one fp32 add).
template <bool kGradBf16, bool kAccum>
__device__ __forceinline__ float rank_grad(const RankPtrs &b, int q, int64_t j)
{
    float g = load_grad<kGradBf16>(b.grad[q], j);
    if (kAccum)
        g = __fadd_rn(__ldcs(b.acc[q] + j), g);
    return g;
}

// Scalar path: rank-ordered fp32 fold of element j, averaged, then AdamW on
// shard element s.
template <bool kGradBf16, bool kParamBf16, bool kAccum>
__device__ __forceinline__ void rs_adamw_scalar(const RankPtrs &b, const AdamScalars &c, int R,
                                                int64_t j, int64_t s)
{
    float acc = rank_grad<kGradBf16, kAccum>(b, 0, j);
    for (int q = 1; q < R; q++)
        acc = __fadd_rn(acc, rank_grad<kGradBf16, kAccum>(b, q, j));
    const float g = __fmul_rn(acc, c.inv_R);
    AdamOut o = adamw_elem(c, g, b.master[s], b.m[s], b.v[s]);
    b.master[s] = o.w;
    b.m[s] = o.m;
    b.v[s] = o.v;
    if (kParamBf16)
        b.pshard[s] = f32_to_bf16_bits(o.w);
    if (b.gshard)
        b.gshard[s] = g;
}

// Two elements of a misaligned tile at once, with R known at compile time:
// every load of both comes before any store, so their latencies overlap
// (the compiler cannot move loads above the stores, which it must assume
// may alias). Element 1 is skipped when has1 is false.
template <int RC, bool kGradBf16, bool kParamBf16, bool kAccum>
__device__ __forceinline__ void rs_adamw_scalar_pair(const RankPtrs &b, const AdamScalars &c,
                                                     int64_t j0, int64_t s0, int64_t j1,
                                                     int64_t s1, bool has1)
{
    float g0[RC], g1[RC];
#pragma unroll
    for (int q = 0; q < RC; q++) {
        g0[q] = rank_grad<kGradBf16, kAccum>(b, q, j0);
        g1[q] = has1 ? rank_grad<kGradBf16, kAccum>(b, q, j1) : 0.0f;
    }
    const float w0 = b.master[s0], m0 = b.m[s0], v0 = b.v[s0];
    const float w1 = has1 ? b.master[s1] : 0.0f, m1 = has1 ? b.m[s1] : 0.0f,
                v1 = has1 ? b.v[s1] : 0.0f;
    float a0 = g0[0], a1 = g1[0];
#pragma unroll
    for (int q = 1; q < RC; q++) {
        a0 = __fadd_rn(a0, g0[q]);
        a1 = __fadd_rn(a1, g1[q]);
    }
    a0 = __fmul_rn(a0, c.inv_R);
    a1 = __fmul_rn(a1, c.inv_R);
    const AdamOut o0 = adamw_elem(c, a0, w0, m0, v0);
    b.master[s0] = o0.w;
    b.m[s0] = o0.m;
    b.v[s0] = o0.v;
    if (kParamBf16)
        b.pshard[s0] = f32_to_bf16_bits(o0.w);
    if (b.gshard)
        b.gshard[s0] = a0;
    if (has1) {
        const AdamOut o1 = adamw_elem(c, a1, w1, m1, v1);
        b.master[s1] = o1.w;
        b.m[s1] = o1.m;
        b.v[s1] = o1.v;
        if (kParamBf16)
            b.pshard[s1] = f32_to_bf16_bits(o1.w);
        if (b.gshard)
            b.gshard[s1] = a1;
    }
}

__device__ __forceinline__ void unpack_bf16x8(uint4 x, float out[8])
{
    out[0] = bf16_lo(x.x); out[1] = bf16_hi(x.x);
    out[2] = bf16_lo(x.y); out[3] = bf16_hi(x.y);
    out[4] = bf16_lo(x.z); out[5] = bf16_hi(x.z);
    out[6] = bf16_lo(x.w); out[7] = bf16_hi(x.w);
}

// Loads the 8 gradient values of one rank at element j (8-aligned) as fp32.
template <bool kGradBf16>
__device__ __forceinline__ void load_grad8(const void *g, int64_t j, float out[8])
{
    if (kGradBf16) {
        unpack_bf16x8(ld_stream(reinterpret_cast<const uint16_t *>(g) + j), out);
    } else {
        float4 a = ld_f4(reinterpret_cast<const float *>(g) + j);
        float4 b = ld_f4(reinterpret_cast<const float *>(g) + j + 4);
        out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
        out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    }
}

// Rank-ordered fp32 fold of the 8 gradient elements starting at unit index j
// (8-aligned): acc[k] = g_0[j+k] + g_1[j+k] + ... + g_{R-1}[j+k], one rounding
// per add. grad[q] is rank q's full gradient.
template <int RC, bool kGradBf16>
__device__ __forceinline__ void fold8(const void *const *grad, int R, int64_t j, float acc[8])
{
    if (RC > 0 && kGradBf16) {
        constexpr int kR = RC > 0 ? RC : 1;
        uint4 raw[kR];  // all R loads in flight before the first add
#pragma unroll
        for (int q = 0; q < kR; q++)
            raw[q] = ld_stream(reinterpret_cast<const uint16_t *>(grad[q]) + j);
        unpack_bf16x8(raw[0], acc);
#pragma unroll
        for (int q = 1; q < kR; q++) {
            float g[8];
            unpack_bf16x8(raw[q], g);
#pragma unroll
            for (int k = 0; k < 8; k++)
                acc[k] = __fadd_rn(acc[k], g[k]);
        }
    } else if (RC > 0) {
        constexpr int kR = RC > 0 ? RC : 1;
        float g[kR][8];
#pragma unroll
        for (int q = 0; q < kR; q++)
            load_grad8<kGradBf16>(grad[q], j, g[q]);
#pragma unroll
        for (int k = 0; k < 8; k++) {
            float a = g[0][k];
#pragma unroll
            for (int q = 1; q < kR; q++)
                a = __fadd_rn(a, g[q][k]);
            acc[k] = a;
        }
    } else {
        load_grad8<kGradBf16>(grad[0], j, acc);
        for (int q = 1; q < R; q++) {
            float g[8];
            load_grad8<kGradBf16>(grad[q], j, g);
#pragma unroll
            for (int k = 0; k < 8; k++)
                acc[k] = __fadd_rn(acc[k], g[k]);
        }
    }
}

// The fold when rank q's gradient is accumulator q plus this micro-batch's
// g_q: a = acc_q[j+k] + g_q[j+k], then the same left fold over ranks.
template <int RC, bool kGradBf16>
__device__ __forceinline__ void fold8_accum(const RankPtrs &b, int R, int64_t j, float out[8])
{
    const int n = RC > 0 ? RC : R;
#pragma unroll 2
    for (int q = 0; q < n; q++) {
        float g[8];
        load_grad8<kGradBf16>(b.grad[q], j, g);
        const float4 a0 = ld_f4(b.acc[q] + j), a1 = ld_f4(b.acc[q] + j + 4);
        const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const float x = __fadd_rn(a[k], g[k]);
            out[k] = q == 0 ? x : __fadd_rn(out[k], x);
        }
    }
}

// The 8 shard elements at s of one rank: acc holds their rank-ordered
// gradient sums (scaled by 1/R here), w/m/v their loaded state. AdamW, then
// the stores of master, m, v, the bf16 shard and the gradient shard.
template <bool kParamBf16>
__device__ __forceinline__ void adamw8_store(const AdamScalars &c, const RankPtrs &b, int64_t s,
                                             float acc[8], float4 w0, float4 w1, float4 m0,
                                             float4 m1, float4 v0, float4 v1)
{
    float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int k = 0; k < 8; k++) {
        acc[k] = __fmul_rn(acc[k], c.inv_R);
        AdamOut o = adamw_elem(c, acc[k], wv[k], mv[k], vv[k]);
        wv[k] = o.w;
        mv[k] = o.m;
        vv[k] = o.v;
    }
    st_f4(b.master + s, make_float4(wv[0], wv[1], wv[2], wv[3]));
    st_f4(b.master + s + 4, make_float4(wv[4], wv[5], wv[6], wv[7]));
    st_f4(b.m + s, make_float4(mv[0], mv[1], mv[2], mv[3]));
    st_f4(b.m + s + 4, make_float4(mv[4], mv[5], mv[6], mv[7]));
    st_f4(b.v + s, make_float4(vv[0], vv[1], vv[2], vv[3]));
    st_f4(b.v + s + 4, make_float4(vv[4], vv[5], vv[6], vv[7]));
    if (kParamBf16) {
        uint4 o;
        o.x = (uint32_t)f32_to_bf16_bits(wv[0]) | ((uint32_t)f32_to_bf16_bits(wv[1]) << 16);
        o.y = (uint32_t)f32_to_bf16_bits(wv[2]) | ((uint32_t)f32_to_bf16_bits(wv[3]) << 16);
        o.z = (uint32_t)f32_to_bf16_bits(wv[4]) | ((uint32_t)f32_to_bf16_bits(wv[5]) << 16);
        o.w = (uint32_t)f32_to_bf16_bits(wv[6]) | ((uint32_t)f32_to_bf16_bits(wv[7]) << 16);
        st_stream(b.pshard + s, o);
    }
    if (b.gshard) {
        st_f4(b.gshard + s, make_float4(acc[0], acc[1], acc[2], acc[3]));
        st_f4(b.gshard + s + 4, make_float4(acc[4], acc[5], acc[6], acc[7]));
    }
}

// Eight elements of kEB bytes that start A words plus bshift / 8 bytes into
// the 16-byte chunks held in w[], widened to fp32: each output word is a
// funnel shift of two neighbouring input words.
template <int kEB, int A>
struct Realign {
    static constexpr int kOut = 2 * kEB;                    // words of 8 elements
    static constexpr int kChunks = (kOut + A + 1 + 3) / 4;  // 16-byte chunks covering them
    static __device__ __forceinline__ void to_f32(const uint32_t *w, uint32_t bshift, float g[8])
    {
        uint32_t o[kOut];
#pragma unroll
        for (int m = 0; m < kOut; m++)
            o[m] = __funnelshift_r(w[m + A], w[m + A + 1 < 4 * kChunks ? m + A + 1 : m + A],
                                   bshift);
        if (kEB == 2) {
            unpack_bf16x8(make_uint4(o[0], o[1], o[2], o[3]), g);
        } else {
#pragma unroll
            for (int k = 0; k < 8; k++)
                g[k] = __uint_as_float(o[k]);
        }
    }
};

// The rank-ordered fold of the 8 gradient elements that start A words plus
// bshift / 8 bytes past unit index cb (a 16-byte boundary), read from the
// gradient buffers with aligned 16-byte loads. The caller checks that the
// chunks lie inside the buffers.
template <int RC, bool kGradBf16, int A>
__device__ __forceinline__ void fold8_realigned_global(const void *const *grad, int64_t cb,
                                                       uint32_t bshift, float acc[8])
{
    constexpr int kEB = kGradBf16 ? 2 : 4;
    using RA = Realign<kEB, A>;
#pragma unroll
    for (int q = 0; q < RC; q++) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const unsigned char *>(grad[q]) + cb * kEB);
        uint32_t w[4 * RA::kChunks];
#pragma unroll
        for (int c = 0; c < RA::kChunks; c++) {
            const uint4 v = ld_stream(src + c);
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
        }
        float g[8];
        RA::to_f32(w, bshift, g);
#pragma unroll
        for (int k = 0; k < 8; k++)
            acc[k] = q == 0 ? g[k] : __fadd_rn(acc[k], g[k]);
    }
}

// A tile whose full-buffer start is off a 16-byte boundary (its shard start
// is aligned): each thread takes its 8 consecutive elements as on the
// vector path, reading the gradients with aligned 16-byte loads that it
// realigns in registers. The threads' chunks overlap, so DRAM sees each
// byte once. A thread whose chunks would pass the buffers' last whole vector
// (only at the unit's end), and the tile's last partial vector, go element
// by element.
template <int RC, bool kGradBf16, bool kParamBf16>
__device__ __forceinline__ void rs_adamw_tile_realigned(const AdamScalars &c, const RankPtrs &b,
                                                        const Tile &T)
{
    constexpr int kEB = kGradBf16 ? 2 : 4;
    constexpr int kVE = 16 / kEB;
    constexpr int kMaxChunkElems = Realign<kEB, 3>::kChunks * kVE;
    const int64_t e = (int64_t)threadIdx.x * kElemsPerThread;
    if (e >= T.len)
        return;
    const int64_t j = T.fbase + e;
    const int64_t cb = j & ~(int64_t)(kVE - 1);
    const int64_t cap = T.unit_numel & ~(int64_t)(kVE - 1);
    if (e + kElemsPerThread > T.len || cb + kMaxChunkElems > cap) {
        const int64_t stop = e + kElemsPerThread < T.len ? e + kElemsPerThread : T.len;
        for (int64_t q = e; q < stop; q++)
            rs_adamw_scalar<kGradBf16, kParamBf16, false>(b, c, RC, T.fbase + q, T.sbase + q);
        return;
    }
    const int64_t s = T.sbase + e;
    float4 w0 = ld_f4(b.master + s), w1 = ld_f4(b.master + s + 4);
    float4 m0 = ld_f4(b.m + s), m1 = ld_f4(b.m + s + 4);
    float4 v0 = ld_f4(b.v + s), v1 = ld_f4(b.v + s + 4);
    const int sh = (int)(j - cb) * kEB;  // the same for every thread of the tile
    const uint32_t bshift = 8u * (uint32_t)(sh & 3);
    float acc[8];
    switch (sh >> 2) {
    case 0: fold8_realigned_global<RC, kGradBf16, 0>(b.grad, cb, bshift, acc); break;
    case 1: fold8_realigned_global<RC, kGradBf16, 1>(b.grad, cb, bshift, acc); break;
    case 2: fold8_realigned_global<RC, kGradBf16, 2>(b.grad, cb, bshift, acc); break;
    default: fold8_realigned_global<RC, kGradBf16, 3>(b.grad, cb, bshift, acc); break;
    }
    adamw8_store<kParamBf16>(c, b, s, acc, w0, w1, m0, m1, v0, v1);
}

// One reduce-scatter + AdamW tile.
template <int RC, bool kGradBf16, bool kParamBf16, bool kAccum, class PP>
__device__ __forceinline__ void rs_adamw_tile(const PP &p, int R, const Tile &T)
{
    RankPtrs b = rank_ptrs(p, T);
    // With R known at compile time the unit's R gradient pointers are read
    // from the parameter block into registers once per tile; the loads below
    // then index registers, not the parameter block through a generic
    // pointer (which cost ~4 % of a Llama unit's time). The accumulating
    // form keeps the generic pointers: its rank loop is not fully unrolled.
    constexpr int kN = RC > 0 ? RC : 1;
    const void *gl[kN];
    if (RC > 0 && !kAccum) {
#pragma unroll
        for (int q = 0; q < kN; q++)
            gl[q] = p.grad[T.base + q];
        b.grad = gl;
    }
    if (((T.fbase | T.sbase) & (kElemsPerThread - 1)) != 0) {
        // bf16 gradients at R = 8 only (misaligned 7.4M-parameter unit: 0.0668
        // -> 0.0597 ms). With fp32 gradients the scalar pairs below were as
        // fast (the realigning loads fetch 48 bytes per 32 used); at R = 4 the
        // extra code cost the L2-resident 3.1M-parameter block 2-4 %.
        if constexpr (RC == 8 && !kAccum && kGradBf16) {
            if ((T.sbase & (kElemsPerThread - 1)) == 0) {
                rs_adamw_tile_realigned<RC, kGradBf16, kParamBf16>(p.c, b, T);
                return;
            }
        }
        if constexpr (RC > 0) {
#pragma unroll 1
            for (int k = 0; k < kElemsPerThread; k += 2) {
                const int64_t e0 = threadIdx.x + (int64_t)k * kThreads, e1 = e0 + kThreads;
                if (e0 < T.len)
                    rs_adamw_scalar_pair<RC, kGradBf16, kParamBf16, kAccum>(
                        b, p.c, T.fbase + e0, T.sbase + e0, T.fbase + e1, T.sbase + e1,
                        e1 < T.len);
            }
        } else {
#pragma unroll 1
            for (int k = 0; k < kElemsPerThread; k++) {
                const int64_t e = threadIdx.x + (int64_t)k * kThreads;
                if (e < T.len)
                    rs_adamw_scalar<kGradBf16, kParamBf16, kAccum>(b, p.c, R, T.fbase + e,
                                                                   T.sbase + e);
            }
        }
        return;
    }
    const int64_t e = (int64_t)threadIdx.x * kElemsPerThread;
    if (e + kElemsPerThread > T.len) {
        for (int64_t q = e; q < T.len; q++)
            rs_adamw_scalar<kGradBf16, kParamBf16, kAccum>(b, p.c, R, T.fbase + q, T.sbase + q);
        return;
    }
    const int64_t j = T.fbase + e;
    const int64_t s = T.sbase + e;
    // issue every load of this thread before any arithmetic
    float acc[8];
    float4 w0 = ld_f4(b.master + s), w1 = ld_f4(b.master + s + 4);
    float4 m0 = ld_f4(b.m + s), m1 = ld_f4(b.m + s + 4);
    float4 v0 = ld_f4(b.v + s), v1 = ld_f4(b.v + s + 4);
    if (kAccum)
        fold8_accum<RC, kGradBf16>(b, R, j, acc);
    else
        fold8<RC, kGradBf16>(b.grad, R, j, acc);
    adamw8_store<kParamBf16>(p.c, b, s, acc, w0, w1, m0, m1, v0, v1);
}

// kUnits as for the all-gather.
template <int RC, bool kGradBf16, bool kParamBf16, bool kAccum, bool kUnits>
__global__ void __launch_bounds__(kThreads) rs_adamw_kernel(const __grid_constant__ RsParams p)
{
    const int R = RC > 0 ? RC : p.R;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        Tile T = locate<kTile>(p.seg, p.nseg, t, false);
        if (!kUnits)
            T.base = 0;
        rs_adamw_tile<RC, kGradBf16, kParamBf16, kAccum>(p, R, T);
    }
}

// ------------------------------ reduce-scatter + AdamW, staged gradients ----
//
// The same tiles and arithmetic as rs_adamw_kernel, with each tile's R
// gradient slices brought into shared memory by cp.async.bulk: thread 0
// issues R 1-D copies of the tile onto its stage's mbarrier, stages() tiles
// ahead of the threads that consume them, and re-fills a stage once every
// thread has read it. The threads load the fp32 state (master, m, v) of
// their 8 elements themselves, before they wait. A tile whose start is off a
// 16-byte boundary in the full buffer is staged from the boundary below it
// and realigned in registers (fold8_staged_at); shard offsets are always
// multiples of 8. The last partial vector of a tile goes element by element.
//
// Every wait gives up after kStageWaitNs: the CTA then counts itself in
// g_stage_wait_timeouts, lets the copies it issued land (again bounded) and
// returns, leaving its remaining tiles unwritten.

// per_stage: a stage's slices, barrier and tile descriptor, in bytes
constexpr int stages_for(int per_stage)
{
    return per_stage <= 0 ? 1
           : kRsStagedSmemBudget / per_stage < 2 ? 2
           : kRsStagedSmemBudget / per_stage > 8 ? 8
                                                 : kRsStagedSmemBudget / per_stage;
}

// What the consumers of a stage need of its tile, written by thread 0 when
// it issues the tile's copies: the consumers read it from shared memory
// instead of searching the segment table and indexing the parameter block.
struct StageTile {
    int64_t fbase, sbase, len, unit_numel;
    float *master, *m, *v;
    uint16_t *pshard;
    int32_t rank, base;
};
static_assert(sizeof(StageTile) == 72, "a compact stage descriptor");

template <int RC, bool kGradBf16>
struct RsStage {
    static constexpr int kEB = kGradBf16 ? 2 : 4;
    static constexpr int kVE = 16 / kEB;             // elements per 16-byte vector
    static constexpr int kData = (int)kTile * kEB;   // one rank's elements of a tile
    // A slice holds a tile's elements from the 16-byte boundary at or below
    // its start to the one at or above its end (up to kVE - 1 elements more
    // on each side); the realigning reads (below) stay inside it too.
    static constexpr int kSlice = kData + 2 * kVE * kEB;
    static constexpr int kBytes = RC * kSlice;       // one stage
    static constexpr bool kOn = RC > 0 && RC * kEB >= kRsStageMinGradBytes &&
                                kBytes - 2 * RC * kVE * kEB <= kRsStageMaxBytes;
    static constexpr int stages()
    {
        return stages_for(kBytes + (int)sizeof(uint64_t) + (int)sizeof(StageTile));
    }
    static constexpr size_t smem()
    {
        return (size_t)stages() * (kBytes + sizeof(uint64_t) + sizeof(StageTile));
    }
};

// What a stage holds of tile T's gradient slices: the elements from
// `first`, the 16-byte boundary at or below T.fbase (`lead` = T.fbase -
// first), to the 16-byte boundary at or above the tile's end, but not past
// the last whole vector of the gradient buffers (P = T.unit_numel elements,
// 16-byte aligned bases); `nst` elements, `bytes` per rank. So the copies
// stay inside the buffers, and only the unit's very last tile can leave a
// few elements (those past the buffers' last whole vector) unstaged.
struct StagedSpan {
    int64_t first;
    int lead;
    int nst;
    uint32_t bytes;
};

template <class S>
__device__ __forceinline__ StagedSpan staged_span(const Tile &T)
{
    StagedSpan z;
    z.first = T.fbase & ~(int64_t)(S::kVE - 1);
    z.lead = (int)(T.fbase - z.first);
    int64_t last = (T.fbase + T.len + S::kVE - 1) & ~(int64_t)(S::kVE - 1);
    const int64_t cap = T.unit_numel & ~(int64_t)(S::kVE - 1);
    if (last > cap)
        last = cap;
    z.nst = last > z.first ? (int)(last - z.first) : 0;
    z.bytes = (uint32_t)z.nst * S::kEB;
    return z;
}

template <bool kUnits, class PP>
__device__ __forceinline__ Tile rs_tile(const PP &p, int64_t t)
{
    Tile T = locate<kTile>(p.seg, p.nseg, t, false);
    if (!kUnits)
        T.base = 0;
    return T;
}

// The rank-ordered fold of the 8 staged gradient elements at tile offset e.
template <int RC, bool kGradBf16>
__device__ __forceinline__ void fold8_staged(const unsigned char *st, int64_t e, float acc[8])
{
    using S = RsStage<RC, kGradBf16>;
    if (kGradBf16) {
        uint4 raw[RC];
#pragma unroll
        for (int q = 0; q < RC; q++)
            raw[q] = *reinterpret_cast<const uint4 *>(st + q * S::kSlice + e * 2);
        unpack_bf16x8(raw[0], acc);
#pragma unroll
        for (int q = 1; q < RC; q++) {
            float g[8];
            unpack_bf16x8(raw[q], g);
#pragma unroll
            for (int k = 0; k < 8; k++)
                acc[k] = __fadd_rn(acc[k], g[k]);
        }
    } else {
#pragma unroll
        for (int q = 0; q < RC; q++) {
            const float4 a = *reinterpret_cast<const float4 *>(st + q * S::kSlice + e * 4);
            const float4 c = *reinterpret_cast<const float4 *>(st + q * S::kSlice + e * 4 + 16);
            const float g[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
            for (int k = 0; k < 8; k++)
                acc[k] = q == 0 ? g[k] : __fadd_rn(acc[k], g[k]);
        }
    }
}

// The same fold for a tile that starts off a 16-byte boundary: the thread's
// 8 elements begin at stage element i0 = lead + e, i0 * kEB bytes into each
// slice, sh = that mod 16 being the same for every thread of the tile (A =
// sh / 4 whole words, B = sh mod 4 bytes). Each slice is read with aligned
// 16-byte loads covering the elements, and the words are shifted into place.
// Elements at stage index nst and beyond (at the end of the unit, past the
// buffers' last whole vector) were not copied; they are read from the
// gradient buffers.
template <int RC, bool kGradBf16, int A>
__device__ __forceinline__ void fold8_realigned(const unsigned char *st, int64_t i0, int nst,
                                                const void *const *grad, int64_t j, float acc[8])
{
    using S = RsStage<RC, kGradBf16>;
    constexpr int kChunks = Realign<S::kEB, A>::kChunks;
    const int ob = (int)((i0 * S::kEB) & ~(int64_t)15);
    const uint32_t bshift = 8u * (uint32_t)((i0 * S::kEB) & 3);
#pragma unroll
    for (int q = 0; q < RC; q++) {
        const unsigned char *sl = st + q * S::kSlice + ob;
        uint32_t w[4 * kChunks];
#pragma unroll
        for (int c = 0; c < kChunks; c++) {
            const uint4 v = *reinterpret_cast<const uint4 *>(sl + 16 * c);
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
        }
        float g[8];
        Realign<S::kEB, A>::to_f32(w, bshift, g);
        if (i0 + 8 > nst) {
#pragma unroll
            for (int k = 0; k < 8; k++)
                if (i0 + k >= nst)
                    g[k] = load_grad<kGradBf16>(grad[q], j + k);
        }
#pragma unroll
        for (int k = 0; k < 8; k++)
            acc[k] = q == 0 ? g[k] : __fadd_rn(acc[k], g[k]);
    }
}

template <int RC, bool kGradBf16>
__device__ __forceinline__ void fold8_staged_at(const unsigned char *st, int64_t i0, int nst,
                                                const void *const *grad, int64_t j, float acc[8])
{
    switch ((int)((i0 * RsStage<RC, kGradBf16>::kEB) & 15) >> 2) {
    case 0: fold8_realigned<RC, kGradBf16, 0>(st, i0, nst, grad, j, acc); break;
    case 1: fold8_realigned<RC, kGradBf16, 1>(st, i0, nst, grad, j, acc); break;
    case 2: fold8_realigned<RC, kGradBf16, 2>(st, i0, nst, grad, j, acc); break;
    default: fold8_realigned<RC, kGradBf16, 3>(st, i0, nst, grad, j, acc); break;
    }
}

template <int RC, bool kGradBf16, bool kParamBf16, bool kUnits>
__global__ void __launch_bounds__(kThreads, kRsStagedCtasPerSm)
    rs_adamw_staged_kernel(const __grid_constant__ RsParams p)
{
    using S = RsStage<RC, kGradBf16>;
    static_assert(S::kOn, "staging needs a compile-time R whose stage fits");
    constexpr int NS = S::stages();
    extern __shared__ __align__(128) unsigned char stage[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(stage + (size_t)NS * S::kBytes);
    StageTile *desc = reinterpret_cast<StageTile *>(bar + NS);
    const int tid = threadIdx.x;
    // thread 0: tile t's descriptor and gradient copies onto stage k (a
    // phase with no bytes completes at once)
    auto issue = [&](const Tile &T, int k) {
        const RankPtrs b = rank_ptrs(p, T);
        desc[k] = {T.fbase, T.sbase, T.len, T.unit_numel, b.master, b.m, b.v, b.pshard,
                   T.rank, T.base};
        const StagedSpan z = staged_span<S>(T);
        mbar_arrive_expect_tx(&bar[k], z.bytes * RC);
        if (z.bytes != 0) {
            unsigned char *dst = stage + (size_t)k * S::kBytes;
#pragma unroll
            for (int q = 0; q < RC; q++)
                bulk_load(dst + q * S::kSlice,
                          static_cast<const unsigned char *>(p.grad[T.base + q]) +
                              z.first * S::kEB,
                          z.bytes, &bar[k]);
        }
    };
    if (tid == 0) {
        for (int k = 0; k < NS; k++)
            mbar_init(&bar[k], 1);
        mbar_init_fence();
        for (int k = 0; k < NS; k++) {
            const int64_t t = blockIdx.x + (int64_t)k * gridDim.x;
            if (t < p.total_tiles)
                issue(rs_tile<kUnits>(p, t), k);
        }
    }
    __syncthreads();
    const int64_t e = (int64_t)tid * kElemsPerThread;
    int64_t i = 0;  // this CTA's tile count: stage i % NS, phase i / NS
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x, i++) {
        const int k = (int)(i % NS);
        // written by thread 0 at least one barrier ago
        const StageTile &d = desc[k];
        Tile T;
        T.fbase = d.fbase;
        T.sbase = d.sbase;
        T.len = d.len;
        T.unit_numel = d.unit_numel;
        T.rank = d.rank;
        T.base = d.base;
        T.nvalid = d.len;
        const RankPtrs b = {p.grad + d.base, p.acc + d.base, d.master, d.m, d.v, d.pshard,
                            p.gshard[d.base + d.rank]};
        // shard offsets are multiples of 8 (segment starts are padded), so
        // every full vector of a tile takes the vector path
        const bool vec =
            e + kElemsPerThread <= T.len && (T.sbase & (kElemsPerThread - 1)) == 0;
        const int64_t s = T.sbase + e;
        float4 w0, w1, m0, m1, v0, v1;
        if (vec) {
            w0 = ld_f4(b.master + s);
            w1 = ld_f4(b.master + s + 4);
            m0 = ld_f4(b.m + s);
            m1 = ld_f4(b.m + s + 4);
            v0 = ld_f4(b.v + s);
            v1 = ld_f4(b.v + s + 4);
        }
        // thread 0 finds the tile that will refill stage k while its loads fly
        const int64_t tn = t + (int64_t)NS * gridDim.x;
        Tile Tn;
        if (tid == 0 && tn < p.total_tiles)
            Tn = rs_tile<kUnits>(p, tn);
        const bool ok = mbar_wait_bounded(&bar[k], (uint32_t)((i / NS) & 1), kStageWaitNs);
        if (ok) {
            if (vec) {
                const StagedSpan z = staged_span<S>(T);
                const unsigned char *st = stage + (size_t)k * S::kBytes;
                float acc[8];
                if (z.lead == 0 && e + kElemsPerThread <= z.nst)
                    fold8_staged<RC, kGradBf16>(st, e, acc);
                else
                    fold8_staged_at<RC, kGradBf16>(st, z.lead + e, z.nst, b.grad, T.fbase + e,
                                                   acc);
                adamw8_store<kParamBf16>(p.c, b, s, acc, w0, w1, m0, m1, v0, v1);
            } else {
                // the tile's last partial vector, element by element
                const int64_t stop = e + kElemsPerThread < T.len ? e + kElemsPerThread : T.len;
                for (int64_t q = e; q < stop; q++)
                    rs_adamw_scalar<kGradBf16, kParamBf16, false>(b, p.c, RC, T.fbase + q,
                                                                  T.sbase + q);
            }
        }
        // every thread is done with stage k; all learn whether a wait gave up
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicAdd(&g_stage_wait_timeouts, 1ull);
                // the copies of this tile and the next NS - 1 were issued
                for (int j = 0; j < NS; j++) {
                    if (t + (int64_t)j * gridDim.x >= p.total_tiles)
                        break;
                    const int64_t ij = i + j;
                    mbar_wait_bounded(&bar[ij % NS], (uint32_t)((ij / NS) & 1), kStageWaitNs);
                }
            }
            return;
        }
        if (tid == 0 && tn < p.total_tiles)
            issue(Tn, k);
    }
}

// ------------------------------------------ AdamW from a reduced gradient ----
//
// ZeRO-1's update: the gradients were all-reduced already, so every rank's
// full buffer holds the averaged fp32 gradient, and rank r updates the
// elements it owns from its own buffer: no sum, and the scalars' inv_R is 1
// (an exact multiply). The same tiles and AdamW epilogue as the fused
// reduce-scatter, so with the all-reduce's output the results are the fused
// kernel's bit for bit.
template <bool kParamBf16>
__global__ void __launch_bounds__(kThreads) adamw_reduced_kernel(const __grid_constant__ RsParams p)
{
    const int64_t e = (int64_t)threadIdx.x * kElemsPerThread;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const Tile T = locate<kTile>(p.seg, p.nseg, t, false);  // one unit: base 0
        if (e >= T.len)
            continue;
        const RankPtrs b = rank_ptrs(p, T);
        const float *g = static_cast<const float *>(p.grad[T.rank]);
        const int64_t s = T.sbase + e;
        if (((T.fbase & 3) | (T.sbase & 3)) == 0 && e + kElemsPerThread <= T.len) {
            const int64_t j = T.fbase + e;
            const float4 g0 = ld_f4(g + j), g1 = ld_f4(g + j + 4);
            float4 w0 = ld_f4(b.master + s), w1 = ld_f4(b.master + s + 4);
            float4 m0 = ld_f4(b.m + s), m1 = ld_f4(b.m + s + 4);
            float4 v0 = ld_f4(b.v + s), v1 = ld_f4(b.v + s + 4);
            float acc[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            adamw8_store<kParamBf16>(p.c, b, s, acc, w0, w1, m0, m1, v0, v1);
        } else {
            const int64_t stop = e + kElemsPerThread < T.len ? e + kElemsPerThread : T.len;
            for (int64_t q = e; q < stop; q++) {
                const int64_t sq = T.sbase + q;
                const float gq = __fmul_rn(__ldcs(g + T.fbase + q), p.c.inv_R);
                const AdamOut o = adamw_elem(p.c, gq, b.master[sq], b.m[sq], b.v[sq]);
                b.master[sq] = o.w;
                b.m[sq] = o.m;
                b.v[sq] = o.v;
                if (kParamBf16)
                    b.pshard[sq] = f32_to_bf16_bits(o.w);
            }
        }
    }
}

// ------------------------------------------------- gradient accumulation ----
//
// acc[q] = g[q] (first micro-batch) or acc[q] + g[q], fp32, for every rank
// q. Tiles run over (rank, flat unit index); tile starts are multiples of
// kTile, so only each rank's last partial vector takes the scalar path.

struct AccumParams {
    float *acc[kMaxR];
    const void *grad[kMaxR];
    int R;
    int first;
    int64_t P;
    int64_t tiles_per_rank;
    int64_t total_tiles;
};

template <bool kGradBf16>
__global__ void __launch_bounds__(kThreads) accumulate_kernel(const __grid_constant__ AccumParams p)
{
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const int q = (int)(t / p.tiles_per_rank);
        const int64_t base = (t - (int64_t)q * p.tiles_per_rank) * kTile;
        const int64_t len = p.P - base < kTile ? p.P - base : kTile;
        const int64_t e = (int64_t)threadIdx.x * kElemsPerThread;
        float *a = p.acc[q];
        if (e + kElemsPerThread <= len) {
            const int64_t j = base + e;
            float g[8];
            load_grad8<kGradBf16>(p.grad[q], j, g);
            if (!p.first) {
                const float4 a0 = ld_f4(a + j), a1 = ld_f4(a + j + 4);
                const float x[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int k = 0; k < 8; k++)
                    g[k] = __fadd_rn(x[k], g[k]);
            }
            st_f4(a + j, make_float4(g[0], g[1], g[2], g[3]));
            st_f4(a + j + 4, make_float4(g[4], g[5], g[6], g[7]));
        } else {
            for (int64_t j = base + e; j < base + len; j++) {
                const float g = load_grad<kGradBf16>(p.grad[q], j);
                a[j] = p.first ? g : __fadd_rn(a[j], g);
            }
        }
    }
}

// --------------------------------------------------------- all-reduce ----
//
// DDP's collective on virtual ranks: every rank's output receives the
// rank-ordered fp32 average of the R full gradients (or its bf16 rounding).
// Tiles run over the flat unit index; every tile start is a multiple of
// kTile, so only the unit's last partial vector takes the scalar path.
//
// With R known at compile time the kernel is software-pipelined: a thread
// issues the R gradient loads of its next tile before the 2R (or R) stores
// of the current one, so loads stay in flight while the stores drain; one
// CTA per SM then keeps HBM busy. fp32 outputs are stored as one 32-byte
// vector per rank when every output is 32-byte aligned (whole sectors; see
// the all-gather). Measured on a Llama unit (R = 8, bf16 in, fp32 out):
// 1.73 ms unpipelined with 16-byte stores at 2 CTAs/SM, 1.58 ms pipelined
// with 32-byte stores at 1 CTA/SM.

struct ReduceParams {
    const void *grad[kMaxR];
    void *out[kMaxR];
    float inv_R;
    int R;
    int wide;  // every output pointer is 32-byte aligned
    int64_t P;
    int64_t total_tiles;
};

// R ranks' 8 gradient values at one index, held in registers: bf16 as one
// 16-byte vector per rank, fp32 as two.
template <int kR, bool kGradBf16> struct Grad8 {
    uint4 v[kR][kGradBf16 ? 1 : 2];
};

template <int kR, bool kGradBf16, class PP>
__device__ __forceinline__ void load_ranks8(const PP &p, int64_t j, Grad8<kR, kGradBf16> &g)
{
#pragma unroll
    for (int q = 0; q < kR; q++) {
        if (kGradBf16) {
            g.v[q][0] = ld_stream(reinterpret_cast<const uint16_t *>(p.grad[q]) + j);
        } else {
            const float *f = reinterpret_cast<const float *>(p.grad[q]) + j;
            g.v[q][0] = ld_stream(f);
            g.v[q][kGradBf16 ? 0 : 1] = ld_stream(f + 4);
        }
    }
}

template <int kR, bool kGradBf16>
__device__ __forceinline__ void fold_ranks8(const Grad8<kR, kGradBf16> &g, float acc[8])
{
#pragma unroll
    for (int q = 0; q < kR; q++) {
        float x[8];
        if (kGradBf16) {
            unpack_bf16x8(g.v[q][0], x);
        } else {
            const uint4 a = g.v[q][0], b = g.v[q][kGradBf16 ? 0 : 1];
            x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
            x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
            x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
            x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
        }
#pragma unroll
        for (int k = 0; k < 8; k++)
            acc[k] = q == 0 ? x[k] : __fadd_rn(acc[k], x[k]);
    }
}

// Stores one thread's 8 averaged values at unit index j to every output.
template <bool kOutBf16>
__device__ __forceinline__ void store_ranks8(const ReduceParams &p, int R, int64_t j,
                                             const float acc[8])
{
    if (kOutBf16) {
        uint4 b;
        b.x = (uint32_t)f32_to_bf16_bits(acc[0]) | ((uint32_t)f32_to_bf16_bits(acc[1]) << 16);
        b.y = (uint32_t)f32_to_bf16_bits(acc[2]) | ((uint32_t)f32_to_bf16_bits(acc[3]) << 16);
        b.z = (uint32_t)f32_to_bf16_bits(acc[4]) | ((uint32_t)f32_to_bf16_bits(acc[5]) << 16);
        b.w = (uint32_t)f32_to_bf16_bits(acc[6]) | ((uint32_t)f32_to_bf16_bits(acc[7]) << 16);
#pragma unroll 8
        for (int d = 0; d < R; d++)
            st_stream(static_cast<uint16_t *>(p.out[d]) + j, b);
        return;
    }
    const uint4 lo = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                                __float_as_uint(acc[2]), __float_as_uint(acc[3]));
    const uint4 hi = make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                __float_as_uint(acc[6]), __float_as_uint(acc[7]));
    if (p.wide) {
#pragma unroll 8
        for (int d = 0; d < R; d++)
            st32(static_cast<float *>(p.out[d]) + j, lo, hi);
    } else {
#pragma unroll 8
        for (int d = 0; d < R; d++) {
            st_stream(static_cast<float *>(p.out[d]) + j, lo);
            st_stream(static_cast<float *>(p.out[d]) + j + 4, hi);
        }
    }
}

// Elements [base + e, base + len) one by one (the unit's last partial vector).
template <bool kGradBf16, bool kOutBf16>
__device__ __forceinline__ void all_reduce_scalar(const ReduceParams &p, int R, int64_t from,
                                                  int64_t to)
{
    for (int64_t q = from; q < to; q++) {
        float acc = load_grad<kGradBf16>(p.grad[0], q);
        for (int r = 1; r < R; r++)
            acc = __fadd_rn(acc, load_grad<kGradBf16>(p.grad[r], q));
        acc = __fmul_rn(acc, p.inv_R);
        for (int d = 0; d < R; d++) {
            if (kOutBf16)
                static_cast<uint16_t *>(p.out[d])[q] = f32_to_bf16_bits(acc);
            else
                static_cast<float *>(p.out[d])[q] = acc;
        }
    }
}

template <int RC, bool kGradBf16, bool kOutBf16>
__global__ void __launch_bounds__(kThreads) all_reduce_kernel(const __grid_constant__ ReduceParams p)
{
    const int64_t e = (int64_t)threadIdx.x * kElemsPerThread;
    if constexpr (RC > 0) {
        // a tile is "full" for this thread when its 8 elements exist
        auto full = [&](int64_t t) { return t < p.total_tiles && t * kTile + e + 8 <= p.P; };
        Grad8<RC, kGradBf16> g;
        int64_t t = blockIdx.x;
        if (full(t))
            load_ranks8<RC, kGradBf16>(p, t * kTile + e, g);
        for (; t < p.total_tiles; t += gridDim.x) {
            const int64_t j = t * kTile + e;
            if (!full(t)) {  // the unit's last, partial tile
                all_reduce_scalar<kGradBf16, kOutBf16>(p, RC, j, p.P);
                continue;
            }
            float acc[8];
            fold_ranks8<RC, kGradBf16>(g, acc);
            const int64_t tn = t + gridDim.x;
            if (full(tn))
                load_ranks8<RC, kGradBf16>(p, tn * kTile + e, g);
#pragma unroll
            for (int k = 0; k < 8; k++)
                acc[k] = __fmul_rn(acc[k], p.inv_R);
            store_ranks8<kOutBf16>(p, RC, j, acc);
        }
    } else {
        const int R = p.R;
        for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
            const int64_t j = t * kTile + e;
            if (j + 8 > p.P) {
                all_reduce_scalar<kGradBf16, kOutBf16>(p, R, j, p.P);
                continue;
            }
            float acc[8];
            fold8<0, kGradBf16>(p.grad, R, j, acc);
#pragma unroll
            for (int k = 0; k < 8; k++)
                acc[k] = __fmul_rn(acc[k], p.inv_R);
            store_ranks8<kOutBf16>(p, R, j, acc);
        }
    }
}

// ------------------------------------------------------- write stream ----
//
// Measurement helper, not a step of the method: writes a 32-bit pattern to n
// buffers with the all-gather's store pattern (one 32-byte vector per buffer
// per thread, 128-thread CTAs, the gather's grid), so that the write-only
// stream ceiling that bounds the gather and the all-reduce can be measured
// in the same run as they are.

struct WriteParams {
    unsigned char *dst[kMaxR];
    int n;
    uint32_t pattern;
    int64_t chunks;  // 32-byte chunks per buffer
};

__global__ void __launch_bounds__(kGatherThreads) write_stream_kernel(const __grid_constant__ WriteParams p)
{
    const uint4 v = make_uint4(p.pattern, p.pattern, p.pattern, p.pattern);
    for (int64_t c = blockIdx.x * (int64_t)kGatherThreads + threadIdx.x; c < p.chunks;
         c += (int64_t)gridDim.x * kGatherThreads)
        for (int d = 0; d < p.n; d++)
            st32(p.dst[d] + c * 32, v, v);
}

// ------------------------------------------------------------ launching ----

struct DeviceInfo {
    int sms = 0;
    std::unordered_map<const void *, int> blocks_per_sm;
};

std::mutex g_dev_mu;
std::unordered_map<int, DeviceInfo> g_dev;

// Makes the device that owns a buffer current for the life of the scope and
// gives the caller's current device back when it ends.
class DeviceScope {
  public:
    DeviceScope() = default;
    DeviceScope(const DeviceScope &) = delete;
    DeviceScope &operator=(const DeviceScope &) = delete;
    ~DeviceScope()
    {
        if (changed_)
            cudaSetDevice(prev_);
    }

    fsdp_status enter(const void *p)
    {
        cudaPointerAttributes a;
        cudaError_t err = cudaPointerGetAttributes(&a, p);
        if (err != cudaSuccess)
            return set_error(FSDP_ECUDA, "cudaPointerGetAttributes: %s", cudaGetErrorString(err));
        if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
            return set_error(FSDP_EINVAL, "output buffer %p is not device memory", p);
        if ((err = cudaGetDevice(&prev_)) != cudaSuccess)
            return set_error(FSDP_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
        if (prev_ != a.device) {
            if ((err = cudaSetDevice(a.device)) != cudaSuccess)
                return set_error(FSDP_ECUDA, "cudaSetDevice: %s", cudaGetErrorString(err));
            changed_ = true;
        }
        dev_ = a.device;
        return FSDP_OK;
    }
    int device() const { return dev_; }

  private:
    int prev_ = -1, dev_ = -1;
    bool changed_ = false;
};

// Persistent grid size for `kernel` on `dev`: resident CTAs per SM (at most
// `max_per_sm`) x SMs.
fsdp_status grid_for(int dev, const void *kernel, int threads, int64_t tiles, int max_per_sm,
                     int *grid, size_t smem = 0)
{
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    cudaError_t err;
    if (d.sms == 0 &&
        (err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return set_error(FSDP_ECUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(err));
    auto it = d.blocks_per_sm.find(kernel);
    if (it == d.blocks_per_sm.end()) {
        if (smem > 48 * 1024 &&
            (err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem)) != cudaSuccess)
            return set_error(FSDP_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(err));
        int nb = 0;
        if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem)) !=
            cudaSuccess)
            return set_error(FSDP_ECUDA, "cudaOccupancyMaxActiveBlocksPerMultiprocessor: %s",
                             cudaGetErrorString(err));
        it = d.blocks_per_sm.emplace(kernel, nb < 1 ? 1 : nb).first;
    }
    int per = it->second < max_per_sm ? it->second : max_per_sm;
    int64_t g = (int64_t)per * d.sms;
    *grid = (int)(tiles < g ? tiles : g);
    return FSDP_OK;
}

fsdp_status check_launch(const char *what)
{
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return set_error(FSDP_ECUDA, "%s launch failed: %s", what, cudaGetErrorString(err));
    return FSDP_OK;
}

template <typename Params>
void fill_segs(Params &p, const LaunchPlan &plan)
{
    p.nseg = (int)plan.segs.size();
    p.total_tiles = plan.total_tiles;
    memcpy(p.seg, plan.segs.data(), plan.segs.size() * sizeof(Seg));
}

template <typename Params, typename Kernel>
fsdp_status run(int dev, Kernel kernel, Params &p, cudaStream_t stream, const char *what,
                int max_per_sm, int threads = kThreads, size_t smem = 0)
{
    int grid = 0;
    fsdp_status st = grid_for(dev, reinterpret_cast<const void *>(kernel), threads,
                              p.total_tiles, max_per_sm, &grid, smem);
    if (st != FSDP_OK)
        return st;
    kernel<<<grid, threads, smem, stream>>>(p);
    return check_launch(what);
}

bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// One kernel launch of a call over n units: its segments, and for each unit
// slot k of the launch the caller's unit index units[k]. Slot k's rank r
// buffer is entry k*R + r of the launch's pointer arrays (Seg::base = k*R).
struct Launch {
    const LaunchPlan *plan = nullptr;  // a layout's own plan (one unit), or
    LaunchPlan merged;                 // segments merged from several units
    std::vector<int> units;
    const LaunchPlan &get() const { return plan ? *plan : merged; }
};

// Which of a layout's plans a kernel walks.
using Plans = std::vector<LaunchPlan> fsdp_layout_s::*;

// The launches of a call over n layouts sharing R: consecutive units share
// a launch while the launch holds at most kMaxSegsPerLaunch segments and
// kMaxR pointers per array. One unit takes its layout's own plans.
std::vector<Launch> plan_launches(int n, const fsdp_layout_t *const *Ls, Plans plans)
{
    std::vector<Launch> out;
    if (n == 1) {
        for (const LaunchPlan &pl : Ls[0]->*plans) {
            out.emplace_back();
            out.back().plan = &pl;
            out.back().units.push_back(0);
        }
        return out;
    }
    const int R = Ls[0]->R;
    const int max_units = kMaxR / R;
    Launch cur;
    for (int u = 0; u < n; u++) {
        for (const LaunchPlan &pl : Ls[u]->*plans) {
            const bool has_slot = !cur.units.empty() && cur.units.back() == u;
            if ((!has_slot && (int)cur.units.size() == max_units) ||
                cur.merged.segs.size() + pl.segs.size() > (size_t)kMaxSegsPerLaunch) {
                out.push_back(std::move(cur));
                cur = Launch();
            }
            if (cur.units.empty() || cur.units.back() != u)
                cur.units.push_back(u);
            const int32_t base = (int32_t)(cur.units.size() - 1) * R;
            for (Seg s : pl.segs) {
                s.tile_begin += cur.merged.total_tiles;
                s.base = base;
                cur.merged.segs.push_back(s);
            }
            cur.merged.total_tiles += pl.total_tiles;
            cur.merged.elems += pl.elems;
            cur.merged.aligned_elems += pl.aligned_elems;
            cur.merged.aligned8_elems += pl.aligned8_elems;
        }
    }
    if (!cur.units.empty())
        out.push_back(std::move(cur));
    return out;
}

// Entry k*R + r of a launch's pointer array = the caller's entry u*R + r of
// unit slot k's unit u (NULL when the caller passed no array).
template <typename T, typename A>
void bind(T *dst, A src, const Launch &l, int R)
{
    for (size_t k = 0; k < l.units.size(); k++)
        for (int r = 0; r < R; r++)
            dst[k * R + r] = src ? (T)src[(size_t)l.units[k] * R + r] : nullptr;
}

}  // namespace

fsdp_status launch_pack(const fsdp_layout_t *L, const float *full, void *const *param_shard,
                        float *const *master, void *stream)
{
    DeviceScope ds;
    fsdp_status st = ds.enter(master[0]);
    if (st != FSDP_OK)
        return st;
    if (L->mode == FSDP_ZERO3) {
        // a rank's buffer past its own parameters is covered by no segment
        for (int r = 0; r < L->R; r++) {
            cudaError_t err = cudaMemsetAsync(master[r], 0, L->shard_numel * 4,
                                              (cudaStream_t)stream);
            if (err == cudaSuccess && param_shard)
                err = cudaMemsetAsync(param_shard[r], 0, L->shard_numel * 2,
                                      (cudaStream_t)stream);
            if (err != cudaSuccess)
                return set_error(FSDP_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(err));
        }
    }
    PackParams p;
    memset(&p, 0, sizeof p);
    p.full = full;
    p.R = L->R;
    for (const Launch &l : plan_launches(1, &L, &fsdp_layout_s::padded_plans)) {
        bind(p.master, master, l, L->R);
        bind(p.pshard, param_shard, l, L->R);
        fill_segs(p, l.get());
        st = L->param_dtype == FSDP_BF16
                 ? run(ds.device(), pack_kernel<true>, p, (cudaStream_t)stream, "pack",
                       kPackCtasPerSm)
                 : run(ds.device(), pack_kernel<false>, p, (cudaStream_t)stream, "pack",
                       kPackCtasPerSm);
        if (st != FSDP_OK)
            return st;
    }
    return FSDP_OK;
}

template <bool kUnits>
static fsdp_status gather_dispatch(int dev, int R, bool bf16, GatherParams &p, cudaStream_t s,
                                   int per)
{
    const char *w = "all_gather";
    const int th = kGatherThreads;
    switch (bf16 ? R : -R) {
    case 2: return run(dev, all_gather_kernel<2, 2, kUnits>, p, s, w, per, th);
    case 4: return run(dev, all_gather_kernel<4, 2, kUnits>, p, s, w, per, th);
    case 8: return run(dev, all_gather_kernel<8, 2, kUnits>, p, s, w, per, th);
    case -2: return run(dev, all_gather_kernel<2, 4, kUnits>, p, s, w, per, th);
    case -4: return run(dev, all_gather_kernel<4, 4, kUnits>, p, s, w, per, th);
    case -8: return run(dev, all_gather_kernel<8, 4, kUnits>, p, s, w, per, th);
    default:
        return bf16 ? run(dev, all_gather_kernel<0, 2, kUnits>, p, s, w, per, th)
                    : run(dev, all_gather_kernel<0, 4, kUnits>, p, s, w, per, th);
    }
}

fsdp_status launch_all_gather(int n, const fsdp_layout_t *const *Ls, const void *const *shard,
                              void *const *full_out, void *stream)
{
    DeviceScope ds;
    fsdp_status st = ds.enter(full_out[0]);
    if (st != FSDP_OK)
        return st;
    const fsdp_layout_t *L = Ls[0];
    const int dev = ds.device();
    GatherParams p;
    memset(&p, 0, sizeof p);
    p.R = L->R;
    cudaStream_t s = (cudaStream_t)stream;
    const bool bf16 = L->param_dtype == FSDP_BF16;
    for (const Launch &l : plan_launches(n, Ls, &fsdp_layout_s::gather_plans)) {
        bind(p.shard, shard, l, L->R);
        bind(p.full, full_out, l, L->R);
        fill_segs(p, l.get());
        p.wide = 1;
        for (size_t k = 0; k < l.units.size() * L->R; k++)
            p.wide &= aligned32(p.shard[k]) && aligned32(p.full[k]);
        // irregular: under half the elements in aligned rank pieces, or the
        // tiles under three quarters full on average
        const LaunchPlan &pl = l.get();
        const bool irregular = 2 * pl.aligned_elems < pl.elems ||
                               4 * pl.elems < 3 * pl.total_tiles * kGatherTile;
        const int per = irregular ? kGatherCtasPerSmIrregular : kGatherCtasPerSm;
        st = l.units.size() > 1 ? gather_dispatch<true>(dev, L->R, bf16, p, s, per)
                                : gather_dispatch<false>(dev, L->R, bf16, p, s, per);
        if (st != FSDP_OK)
            return st;
    }
    return FSDP_OK;
}

// The staged kernel where R is a compile-time constant whose stage fits, no
// accumulators are read and the launch gives every staged CTA at least
// kRsStagedMinTilesPerCta tiles; the register kernel otherwise.
template <int RC, bool kGradBf16, bool kParamBf16, bool kAccum, bool kUnits>
static fsdp_status rs_run(int dev, RsParams &p, cudaStream_t s, int min_tiles_per_cta)
{
    using S = RsStage<RC, kGradBf16>;
    if constexpr (!kAccum && S::kOn) {
        auto kernel = rs_adamw_staged_kernel<RC, kGradBf16, kParamBf16, kUnits>;
        int grid = 0;
        fsdp_status st = grid_for(dev, reinterpret_cast<const void *>(kernel), kThreads,
                                  p.total_tiles, kRsStagedCtasPerSm, &grid, S::smem());
        if (st != FSDP_OK)
            return st;
        if (p.total_tiles >= (int64_t)min_tiles_per_cta * grid) {
            kernel<<<grid, kThreads, S::smem(), s>>>(p);
            return check_launch("rs_adamw_staged");
        }
    }
    return run(dev, rs_adamw_kernel<RC, kGradBf16, kParamBf16, kAccum, kUnits>, p, s,
               "rs_adamw",
               p.total_tiles <= kRsSmallLaunchTiles ? kRsCtasPerSmSmall : kRsCtasPerSm);
}

template <bool kGradBf16, bool kParamBf16, bool kAccum, bool kUnits>
static fsdp_status rs_dispatch(int dev, int R, RsParams &p, cudaStream_t s, int mt)
{
    switch (R) {
    case 2: return rs_run<2, kGradBf16, kParamBf16, kAccum, kUnits>(dev, p, s, mt);
    case 4: return rs_run<4, kGradBf16, kParamBf16, kAccum, kUnits>(dev, p, s, mt);
    case 8: return rs_run<8, kGradBf16, kParamBf16, kAccum, kUnits>(dev, p, s, mt);
    default: return rs_run<0, kGradBf16, kParamBf16, kAccum, kUnits>(dev, p, s, mt);
    }
}

// Accumulating launches always hold one unit.
template <bool kAccum, bool kUnits>
static fsdp_status rs_dispatch_dtypes(int dev, const fsdp_layout_t *L, RsParams &p, cudaStream_t s,
                                      const LaunchPlan &pl)
{
    const int mt = 2 * pl.aligned8_elems < pl.elems ? kRsStagedMinTilesPerCtaMisaligned
                                                    : kRsStagedMinTilesPerCta;
    const bool gb = L->grad_dtype == FSDP_BF16, pb = L->param_dtype == FSDP_BF16;
    if (gb && pb)
        return rs_dispatch<true, true, kAccum, kUnits>(dev, L->R, p, s, mt);
    if (gb)
        return rs_dispatch<true, false, kAccum, kUnits>(dev, L->R, p, s, mt);
    if (pb)
        return rs_dispatch<false, true, kAccum, kUnits>(dev, L->R, p, s, mt);
    return rs_dispatch<false, false, kAccum, kUnits>(dev, L->R, p, s, mt);
}

fsdp_status launch_rs_adamw(int n, const fsdp_layout_t *const *Ls, const void *const *grad,
                            float *const *master, float *const *m, float *const *v,
                            void *const *param_shard_out, float *const *grad_shard_out,
                            const AdamScalars &c, void *stream, const float *const *acc)
{
    DeviceScope ds;
    fsdp_status st = ds.enter(master[0]);
    if (st != FSDP_OK)
        return st;
    const fsdp_layout_t *L = Ls[0];
    const int R = L->R;
    RsParams p;
    memset(&p, 0, sizeof p);
    p.R = R;
    p.c = c;
    cudaStream_t s = (cudaStream_t)stream;
    for (const Launch &l : plan_launches(n, Ls, &fsdp_layout_s::valid_plans)) {
        bind(p.grad, grad, l, R);
        bind(p.acc, acc, l, R);
        bind(p.master, master, l, R);
        bind(p.m, m, l, R);
        bind(p.v, v, l, R);
        bind(p.pshard, param_shard_out, l, R);
        bind(p.gshard, grad_shard_out, l, R);
        fill_segs(p, l.get());
        if (acc)
            st = rs_dispatch_dtypes<true, false>(ds.device(), L, p, s, l.get());
        else if (l.units.size() > 1)
            st = rs_dispatch_dtypes<false, true>(ds.device(), L, p, s, l.get());
        else
            st = rs_dispatch_dtypes<false, false>(ds.device(), L, p, s, l.get());
        if (st != FSDP_OK)
            return st;
    }
    return FSDP_OK;
}

fsdp_status launch_adamw_reduced(const fsdp_layout_t *L, const float *const *grad_avg,
                                 float *const *master, float *const *m, float *const *v,
                                 void *const *param_shard_out, const AdamScalars &c, void *stream)
{
    DeviceScope ds;
    fsdp_status st = ds.enter(master[0]);
    if (st != FSDP_OK)
        return st;
    RsParams p;
    memset(&p, 0, sizeof p);
    p.R = L->R;
    p.c = c;
    p.c.inv_R = 1.0f;  // the gradient is averaged already
    for (int r = 0; r < L->R; r++) {
        p.grad[r] = grad_avg[r];
        p.master[r] = master[r];
        p.m[r] = m[r];
        p.v[r] = v[r];
        p.pshard[r] = param_shard_out ? static_cast<uint16_t *>(param_shard_out[r]) : nullptr;
    }
    cudaStream_t s = (cudaStream_t)stream;
    for (const LaunchPlan &pl : L->valid_plans) {
        fill_segs(p, pl);
        st = L->param_dtype == FSDP_BF16
                 ? run(ds.device(), adamw_reduced_kernel<true>, p, s, "adamw_reduced", kRsCtasPerSm)
                 : run(ds.device(), adamw_reduced_kernel<false>, p, s, "adamw_reduced",
                       kRsCtasPerSm);
        if (st != FSDP_OK)
            return st;
    }
    return FSDP_OK;
}

fsdp_status launch_accumulate(const fsdp_layout_t *L, float *const *acc, const void *const *grad,
                              int first, void *stream)
{
    DeviceScope ds;
    fsdp_status st = ds.enter(acc[0]);
    if (st != FSDP_OK)
        return st;
    AccumParams p;
    memset(&p, 0, sizeof p);
    p.R = L->R;
    p.first = first ? 1 : 0;
    p.P = L->P;
    p.tiles_per_rank = (L->P + kTile - 1) / kTile;
    p.total_tiles = p.tiles_per_rank * L->R;
    for (int r = 0; r < L->R; r++) {
        p.acc[r] = acc[r];
        p.grad[r] = grad[r];
    }
    cudaStream_t s = (cudaStream_t)stream;
    if (L->grad_dtype == FSDP_BF16)
        return run(ds.device(), accumulate_kernel<true>, p, s, "accumulate", kAccumulateCtasPerSm);
    return run(ds.device(), accumulate_kernel<false>, p, s, "accumulate", kAccumulateCtasPerSm);
}

// The reduce-scatter + AdamW of unit A, then the gather of unit B, on one
// stream. Single launches that interleave the two tile streams (tile by
// tile, in chunks of 2-32 tiles, or by splitting the CTAs) and two concurrent
// launches on two streams were all measured on GB300: none beat these two
// launches back to back (the interleaved forms were 9-17 % slower), so the
// prefetch is issued in order.
fsdp_status launch_rs_adamw_gather(const fsdp_layout_t *A, const void *const *grad,
                                   float *const *master, float *const *m, float *const *v,
                                   void *const *param_shard_out, float *const *grad_shard_out,
                                   const AdamScalars &c, const fsdp_layout_t *B,
                                   const void *const *shard, void *const *full_out, void *stream)
{
    fsdp_status st = launch_rs_adamw(1, &A, grad, master, m, v, param_shard_out, grad_shard_out,
                                     c, stream, nullptr);
    if (st != FSDP_OK)
        return st;
    return launch_all_gather(1, &B, shard, full_out, stream);
}

template <bool kGradBf16, bool kOutBf16>
static fsdp_status ar_dispatch(int dev, int R, ReduceParams &p, cudaStream_t s)
{
    const char *w = "all_reduce";
    switch (R) {
    case 2: return run(dev, all_reduce_kernel<2, kGradBf16, kOutBf16>, p, s, w, kAllReduceCtasPerSm);
    case 4: return run(dev, all_reduce_kernel<4, kGradBf16, kOutBf16>, p, s, w, kAllReduceCtasPerSm);
    case 8: return run(dev, all_reduce_kernel<8, kGradBf16, kOutBf16>, p, s, w, kAllReduceCtasPerSm);
    default: return run(dev, all_reduce_kernel<0, kGradBf16, kOutBf16>, p, s, w, kAllReduceCtasPerSm);
    }
}

fsdp_status launch_all_reduce(const fsdp_layout_t *L, const void *const *grad, void *const *out,
                              fsdp_dtype out_dtype, void *stream)
{
    DeviceScope ds;
    fsdp_status st = ds.enter(out[0]);
    if (st != FSDP_OK)
        return st;
    ReduceParams p;
    memset(&p, 0, sizeof p);
    p.R = L->R;
    p.P = L->P;
    p.inv_R = 1.0f / (float)L->R;
    p.total_tiles = (L->P + kTile - 1) / kTile;
    p.wide = 1;
    for (int r = 0; r < L->R; r++) {
        p.grad[r] = grad[r];
        p.out[r] = out[r];
        p.wide &= aligned32(out[r]);
    }
    cudaStream_t s = (cudaStream_t)stream;
    const bool gb = L->grad_dtype == FSDP_BF16, ob = out_dtype == FSDP_BF16;
    const int dev = ds.device();
    if (gb && ob)
        return ar_dispatch<true, true>(dev, L->R, p, s);
    if (gb)
        return ar_dispatch<true, false>(dev, L->R, p, s);
    if (ob)
        return ar_dispatch<false, true>(dev, L->R, p, s);
    return ar_dispatch<false, false>(dev, L->R, p, s);
}

fsdp_status launch_write_stream(void *const *dst, int n, int64_t bytes, uint32_t pattern,
                                void *stream)
{
    DeviceScope ds;
    fsdp_status st = ds.enter(dst[0]);
    if (st != FSDP_OK)
        return st;
    WriteParams p;
    memset(&p, 0, sizeof p);
    p.n = n;
    p.pattern = pattern;
    p.chunks = bytes / 32;
    for (int d = 0; d < n; d++)
        p.dst[d] = static_cast<unsigned char *>(dst[d]);
    int grid = 0;
    const int64_t blocks = (p.chunks + kGatherThreads - 1) / kGatherThreads;
    if ((st = grid_for(ds.device(), reinterpret_cast<const void *>(write_stream_kernel),
                       kGatherThreads, blocks, kGatherCtasPerSm, &grid)) != FSDP_OK)
        return st;
    write_stream_kernel<<<grid, kGatherThreads, 0, (cudaStream_t)stream>>>(p);
    return check_launch("write_stream");
}

fsdp_status run_stage_wait_selftest(int device, uint64_t *gave_up)
{
    int prev = -1;
    cudaError_t err = cudaGetDevice(&prev);
    if (err != cudaSuccess)
        return set_error(FSDP_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
    if (prev != device && (err = cudaSetDevice(device)) != cudaSuccess)
        return set_error(FSDP_ECUDA, "cudaSetDevice(%d): %s", device, cudaGetErrorString(err));
    unsigned long long before = 0, after = 0;
    err = cudaMemcpyFromSymbol(&before, g_selftest_wait_timeouts, sizeof before);
    if (err == cudaSuccess) {
        stage_wait_selftest_kernel<<<1, 32>>>(20000000ull);  // gives up after 20 ms
        err = cudaGetLastError();
    }
    if (err == cudaSuccess)
        err = cudaDeviceSynchronize();
    if (err == cudaSuccess)
        err = cudaMemcpyFromSymbol(&after, g_selftest_wait_timeouts, sizeof after);
    if (prev != device)
        cudaSetDevice(prev);
    if (err != cudaSuccess)
        return set_error(FSDP_ECUDA, "wait self-test: %s", cudaGetErrorString(err));
    *gave_up = after - before;
    return FSDP_OK;
}

fsdp_status read_stage_wait_timeouts(int device, uint64_t *count)
{
    int prev = -1;
    cudaError_t err = cudaGetDevice(&prev);
    if (err != cudaSuccess)
        return set_error(FSDP_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
    if (prev != device && (err = cudaSetDevice(device)) != cudaSuccess)
        return set_error(FSDP_ECUDA, "cudaSetDevice(%d): %s", device, cudaGetErrorString(err));
    unsigned long long n = 0;
    err = cudaDeviceSynchronize();
    if (err == cudaSuccess)
        err = cudaMemcpyFromSymbol(&n, g_stage_wait_timeouts, sizeof n);
    if (prev != device)
        cudaSetDevice(prev);
    if (err != cudaSuccess)
        return set_error(FSDP_ECUDA, "reading the wait-timeout count: %s", cudaGetErrorString(err));
    *count = n;
    return FSDP_OK;
}

}  // namespace fsdp
