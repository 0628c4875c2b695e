// fsdp_capi.cpp -- layout planner, argument validation and the extern "C"
// entry points of the shard engine. Host code only; the kernels live in
// fsdp_kernels.cu. Compiled with -ffp-contract=off so the AdamW scalars are
// formed exactly as documented in fsdp_shard.h.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <limits>
#include <new>
#include <string>

#include <cuda_runtime.h>

#include "fsdp_internal.h"

namespace fsdp {

static thread_local std::string g_last_error;

fsdp_status set_error(fsdp_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

namespace {

constexpr int64_t kMaxElems = int64_t(1) << 60;  // byte counts (x4) stay in int64

bool mul_ok(int64_t a, int64_t b, int64_t *out)
{
    if (a != 0 && b > kMaxElems / a)
        return false;
    *out = a * b;
    return true;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tiles of `tile` elements in one rank piece of `len` elements.
int64_t tiles_for(int64_t len, int64_t tile) { return ceil_div(len, tile); }

// Split segments into launches of at most kMaxSegsPerLaunch segments, with
// the tile numbering of each launch starting at 0. `padded` selects the
// traversal: owned elements only (gather, reduce) or whole shard buffers
// (pack); `tile` is the kernel's tile length. Segments without tiles are
// dropped.
std::vector<LaunchPlan> make_plans(const std::vector<Seg> &segs, int R, bool padded,
                                   int64_t tile, int64_t align)
{
    std::vector<LaunchPlan> plans;
    LaunchPlan cur;
    for (Seg s : segs) {
        // owned elements and those in aligned rank pieces (see LaunchPlan)
        int64_t elems = 0, aligned = 0, aligned8 = 0;
        const int pieces = s.owner >= 0 ? 1 : R;
        for (int r = 0; r < pieces; r++) {
            int64_t n = s.owner >= 0 ? s.numel : s.numel - (int64_t)r * s.rank_stride;
            n = n < 0 ? 0 : (s.owner < 0 && n > s.rank_stride ? s.rank_stride : n);
            const int64_t start = s.full_off + (s.owner >= 0 ? 0 : (int64_t)r * s.rank_stride);
            elems += n;
            if (start % align == 0 && s.shard_off % align == 0)
                aligned += n;
            if (start % 8 == 0 && s.shard_off % 8 == 0)
                aligned8 += n;
        }
        int64_t tiles;
        if (s.owner >= 0) {
            // a whole parameter on one rank: tiles over its (padded) length
            tiles = tiles_for(padded ? s.pad_len : s.numel, tile);
            s.tiles_per_rank = tiles;
        } else if (padded) {
            s.tiles_per_rank = tiles_for(s.pad_len, tile);
            tiles = s.tiles_per_rank * R;
        } else {
            if (s.numel == 0 || s.rank_stride == 0)
                continue;
            s.tiles_per_rank = tiles_for(s.rank_stride, tile);
            int64_t full_ranks = s.numel / s.rank_stride;
            int64_t rest = s.numel - full_ranks * s.rank_stride;
            tiles = full_ranks * s.tiles_per_rank + tiles_for(rest, tile);
        }
        if (tiles == 0)
            continue;
        if ((int)cur.segs.size() == kMaxSegsPerLaunch) {
            plans.push_back(cur);
            cur = LaunchPlan();
        }
        s.tile_begin = cur.total_tiles;
        cur.total_tiles += tiles;
        cur.elems += elems;
        cur.aligned_elems += aligned;
        cur.aligned8_elems += aligned8;
        cur.segs.push_back(s);
    }
    if (!cur.segs.empty())
        plans.push_back(cur);
    return plans;
}

// ZeRO-3 owners: parameters in unit order fill rank 0 until it holds at
// least ceil(P/R) elements, then rank 1, ...; the last rank takes the rest.
std::vector<int64_t> zero3_owners(const std::vector<int64_t> &numel, int R)
{
    int64_t total = 0;
    for (int64_t x : numel)
        total += x;
    const int64_t quota = ceil_div(total, R);
    std::vector<int64_t> owner(numel.size());
    int64_t rank = 0, held = 0;
    for (size_t i = 0; i < numel.size(); i++) {
        owner[i] = rank;
        held += numel[i];
        if (held >= quota && rank + 1 < R) {
            ++rank;
            held = 0;
        }
    }
    return owner;
}

// Rows [start, start+count) of a dim-0 extent d0 held by rank r.
void rank_rows(int64_t d0, int R, int r, int64_t *start, int64_t *count)
{
    int64_t s = ceil_div(d0, R);
    int64_t a = s * r;
    *start = a;
    *count = std::max<int64_t>(0, std::min<int64_t>(s, d0 - a));
}

int64_t rank_numel(const fsdp_layout_t *L, int r)
{
    if (L->mode == FSDP_ZERO3) {
        int64_t tot = 0;
        for (int i = 0; i < L->n; i++)
            if (L->owner[i] == r)
                tot += L->dim0[i] * L->inner[i];
        return tot;
    }
    if (L->mode == FSDP_FLAT)
        return std::max<int64_t>(0, std::min<int64_t>(L->shard_numel, L->P - r * L->shard_numel));
    int64_t tot = 0;
    for (int i = 0; i < L->n; i++) {
        int64_t a, c;
        rank_rows(L->dim0[i], L->R, r, &a, &c);
        tot += c * L->inner[i];
    }
    return tot;
}

int64_t esize(fsdp_dtype d) { return d == FSDP_BF16 ? 2 : 4; }

struct Span {
    uintptr_t lo, hi;
    bool out;
    const char *what;
    int rank;
};

// Checks a host array of R device pointers. Each entry must be non-NULL
// (when bytes > 0) and 16-byte aligned. `first` is the array index of
// entry 0 in error messages (multi-unit calls pass slices of longer arrays).
fsdp_status check_ptrs(const void *const *arr, int R, int64_t bytes, bool out, const char *what,
                       std::vector<Span> *spans, int first = 0)
{
    if (arr == nullptr)
        return set_error(FSDP_EINVAL, "%s: pointer array is NULL", what);
    for (int r = 0; r < R; r++) {
        const void *p = arr[r];
        if (bytes == 0)
            continue;
        if (p == nullptr)
            return set_error(FSDP_EINVAL, "%s[%d] is NULL", what, first + r);
        if (reinterpret_cast<uintptr_t>(p) & 15u)
            return set_error(FSDP_EALIGN, "%s[%d] = %p is not 16-byte aligned", what, first + r,
                             p);
        uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        spans->push_back({lo, lo + (uintptr_t)bytes, out, what, first + r});
    }
    return FSDP_OK;
}

// Any output overlapping another buffer is an error; inputs may alias.
fsdp_status check_overlap(std::vector<Span> &spans)
{
    std::sort(spans.begin(), spans.end(), [](const Span &a, const Span &b) { return a.lo < b.lo; });
    const Span *far_any = nullptr;
    const Span *far_out = nullptr;
    for (const Span &s : spans) {
        const Span *hit = nullptr;
        if (s.out && far_any && s.lo < far_any->hi)
            hit = far_any;
        else if (!s.out && far_out && s.lo < far_out->hi)
            hit = far_out;
        if (hit)
            return set_error(FSDP_EINVAL, "%s[%d] overlaps %s[%d]", s.what, s.rank, hit->what,
                             hit->rank);
        if (!far_any || s.hi > far_any->hi)
            far_any = &s;
        if (s.out && (!far_out || s.hi > far_out->hi))
            far_out = &s;
    }
    return FSDP_OK;
}

// Every buffer must be device memory of one device (the one the call runs
// on). A host or peer pointer would otherwise reach a kernel.
fsdp_status check_devices(const std::vector<Span> &spans)
{
    int dev = -1;
    for (const Span &s : spans) {
        cudaPointerAttributes a;
        cudaError_t err = cudaPointerGetAttributes(&a, reinterpret_cast<const void *>(s.lo));
        if (err != cudaSuccess)
            return set_error(FSDP_ECUDA, "cudaPointerGetAttributes(%s[%d]): %s", s.what, s.rank,
                             cudaGetErrorString(err));
        if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
            return set_error(FSDP_EINVAL, "%s[%d] = %p is not device memory", s.what, s.rank,
                             reinterpret_cast<const void *>(s.lo));
        if (dev < 0)
            dev = a.device;
        else if (a.device != dev)
            return set_error(FSDP_EINVAL, "%s[%d] is on device %d, other buffers on device %d",
                             s.what, s.rank, a.device, dev);
    }
    return FSDP_OK;
}

// The checks every call makes once its spans are collected: no output
// overlaps another buffer, and all buffers are on one device.
fsdp_status check_spans(std::vector<Span> &spans)
{
    fsdp_status st = check_overlap(spans);
    return st != FSDP_OK ? st : check_devices(spans);
}

fsdp_status check_gather_args(const fsdp_layout_t *L, const void *const *shard,
                              void *const *full_out, std::vector<Span> *spans, int first = 0)
{
    int64_t es = esize(L->param_dtype);
    fsdp_status st = check_ptrs(shard, L->R, L->shard_numel * es, false, "shard", spans, first);
    if (st != FSDP_OK)
        return st;
    return check_ptrs((const void *const *)full_out, L->R, L->P * es, true, "full_out", spans,
                      first);
}

fsdp_status check_hp(const fsdp_adamw_hp *hp, int64_t step)
{
    if (hp == nullptr)
        return set_error(FSDP_EINVAL, "AdamW hyper-parameters are NULL");
    if (step < 1)
        return set_error(FSDP_EINVAL, "step = %lld, must be >= 1", (long long)step);
    if (!(std::isfinite(hp->lr) && hp->lr >= 0) || !(hp->beta1 >= 0 && hp->beta1 < 1) ||
        !(hp->beta2 >= 0 && hp->beta2 < 1) || !(std::isfinite(hp->eps) && hp->eps > 0) ||
        !std::isfinite(hp->weight_decay))
        return set_error(FSDP_EINVAL, "bad AdamW hyper-parameters");
    return FSDP_OK;
}

fsdp_status check_rs_args(const fsdp_layout_t *L, const void *const *grad_full,
                          float *const *master, float *const *m, float *const *v,
                          void *const *param_shard_out, float *const *grad_shard_out,
                          std::vector<Span> *spans, int first = 0)
{
    fsdp_status st;
    int64_t sb = L->shard_numel * 4;
    if ((st = check_ptrs(grad_full, L->R, L->P * esize(L->grad_dtype), false, "grad_full",
                         spans, first)) != FSDP_OK)
        return st;
    if ((st = check_ptrs((const void *const *)master, L->R, sb, true, "master", spans, first)) !=
        FSDP_OK)
        return st;
    if ((st = check_ptrs((const void *const *)m, L->R, sb, true, "m", spans, first)) != FSDP_OK)
        return st;
    if ((st = check_ptrs((const void *const *)v, L->R, sb, true, "v", spans, first)) != FSDP_OK)
        return st;
    if (L->param_dtype == FSDP_BF16) {
        if ((st = check_ptrs((const void *const *)param_shard_out, L->R, L->shard_numel * 2, true,
                             "param_shard_out", spans, first)) != FSDP_OK)
            return st;
    } else if (param_shard_out != nullptr) {
        return set_error(FSDP_EINVAL, "param_shard_out must be NULL for an F32 layout");
    }
    if (grad_shard_out != nullptr &&
        (st = check_ptrs((const void *const *)grad_shard_out, L->R, sb, true, "grad_shard_out",
                         spans, first)) != FSDP_OK)
        return st;
    return FSDP_OK;
}

// A multi-unit call's layouts: n >= 1, none NULL, all with the first one's
// R and dtypes.
fsdp_status check_units(int n, const fsdp_layout_t *const *Ls, const char *fn)
{
    if (n < 1 || Ls == nullptr)
        return set_error(FSDP_EINVAL, "%s: need n_units >= 1 layouts (n_units = %d)", fn, n);
    for (int u = 0; u < n; u++) {
        if (Ls[u] == nullptr)
            return set_error(FSDP_EINVAL, "%s: layouts[%d] is NULL", fn, u);
        if (Ls[u]->R != Ls[0]->R || Ls[u]->param_dtype != Ls[0]->param_dtype ||
            Ls[u]->grad_dtype != Ls[0]->grad_dtype)
            return set_error(FSDP_EINVAL, "%s: layouts[%d] differs from layouts[0] in R or dtypes",
                             fn, u);
        if ((int64_t)n * Ls[0]->R > (int64_t)1 << 30)
            return set_error(FSDP_ERANGE, "%s: too many units", fn);
    }
    return FSDP_OK;
}

// Appends entries [u*R, (u+1)*R) of a per-rank pointer array (or nothing for
// a NULL array).
template <typename T>
void take(std::vector<T> &dst, T const *src, int u, int R)
{
    if (src)
        dst.insert(dst.end(), src + (size_t)u * R, src + (size_t)(u + 1) * R);
}

template <typename T>
T const *data_or_null(const std::vector<T> &v, const void *given)
{
    return given ? v.data() : nullptr;
}

// AdamW scalars formed in double from hp and step, rounded once to fp32.
AdamScalars adam_scalars(const fsdp_adamw_hp *hp, int64_t step, int R)
{
    AdamScalars c;
    c.decay = (float)(1.0 - hp->lr * hp->weight_decay);
    c.b1 = (float)hp->beta1;
    c.omb1 = (float)(1.0 - hp->beta1);
    c.b2 = (float)hp->beta2;
    c.omb2 = (float)(1.0 - hp->beta2);
    c.step_size = (float)(hp->lr / (1.0 - std::pow(hp->beta1, (double)step)));
    c.bc2_sqrt = (float)std::sqrt(1.0 - std::pow(hp->beta2, (double)step));
    c.eps = (float)hp->eps;
    c.inv_R = 1.0f / (float)R;
    return c;
}

}  // namespace
}  // namespace fsdp

using namespace fsdp;

extern "C" {

const char *fsdp_last_error(void) { return g_last_error.c_str(); }

const char *fsdp_version(void) { return "fsdp_shard 0.1 (sm_103a)"; }

fsdp_status fsdp_layout(fsdp_mode mode, int R, int n_params, const int64_t *dim0,
                        const int64_t *inner, fsdp_dtype param_dtype, fsdp_dtype grad_dtype,
                        fsdp_layout_t **out)
{
    if (out == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_layout: out is NULL");
    *out = nullptr;
    if (mode != FSDP_FLAT && mode != FSDP_PER_PARAM && mode != FSDP_ZERO3)
        return set_error(FSDP_EINVAL, "fsdp_layout: unknown mode %d", (int)mode);
    if (R < 1 || R > FSDP_MAX_RANKS)
        return set_error(FSDP_EINVAL, "fsdp_layout: R = %d outside [1, %d]", R, FSDP_MAX_RANKS);
    if (n_params < 0 || (n_params > 0 && (dim0 == nullptr || inner == nullptr)))
        return set_error(FSDP_EINVAL, "fsdp_layout: bad parameter list (n_params = %d)", n_params);
    if ((param_dtype != FSDP_F32 && param_dtype != FSDP_BF16) ||
        (grad_dtype != FSDP_F32 && grad_dtype != FSDP_BF16))
        return set_error(FSDP_EUNSUPPORTED, "fsdp_layout: unsupported dtype");

    fsdp_layout_t *L = new (std::nothrow) fsdp_layout_t();
    if (!L)
        return set_error(FSDP_EINVAL, "fsdp_layout: out of host memory");
    L->mode = mode;
    L->R = R;
    L->n = n_params;
    L->param_dtype = param_dtype;
    L->grad_dtype = grad_dtype;
    L->dim0.assign(dim0, dim0 + n_params);
    L->inner.assign(inner, inner + n_params);

    int64_t P = 0, seg_total = 0;
    std::vector<Seg> segs;
    for (int i = 0; i < n_params; i++) {
        int64_t d = dim0[i], w = inner[i], numel;
        if (d < 0 || w < 0) {
            delete L;
            return set_error(FSDP_EINVAL, "fsdp_layout: parameter %d has a negative dim", i);
        }
        if (!mul_ok(d, w, &numel) || P > kMaxElems - numel) {
            delete L;
            return set_error(FSDP_ERANGE, "fsdp_layout: unit too large at parameter %d", i);
        }
        int64_t rows = ceil_div(d, R);
        int64_t stride = rows * w;  // <= numel + R*w, no overflow past the check above
        int64_t pad = ceil_div(stride, FSDP_SEG_ALIGN) * FSDP_SEG_ALIGN;
        L->full_off.push_back(P);
        L->shard_rows.push_back(rows);
        L->shard_off.push_back(seg_total);
        if (mode == FSDP_PER_PARAM)
            segs.push_back({P, numel, stride, seg_total, pad, 0, 0, -1, 0, 0});
        P += numel;
        seg_total += pad;
    }
    L->P = P;
    if (mode == FSDP_PER_PARAM) {
        L->shard_numel = seg_total;
    } else if (mode == FSDP_FLAT) {
        int64_t S = ceil_div(P, R);
        L->shard_numel = S;
        segs.push_back({0, P, S, 0, S, 0, 0, -1, 0, 0});
    } else {
        std::vector<int64_t> numel(n_params);
        for (int i = 0; i < n_params; i++)
            numel[i] = dim0[i] * inner[i];
        L->owner = zero3_owners(numel, R);
        std::vector<int64_t> used(R, 0);
        int64_t longest = 0;
        for (int i = 0; i < n_params; i++) {
            const int64_t o = L->owner[i];
            const int64_t pad = ceil_div(numel[i], FSDP_SEG_ALIGN) * FSDP_SEG_ALIGN;
            L->shard_rows[i] = dim0[i];
            L->shard_off[i] = used[o];
            segs.push_back({L->full_off[i], numel[i], numel[i], used[o], pad, 0, 0, (int32_t)o, 0, 0});
            used[o] += pad;
            longest = std::max(longest, used[o]);
        }
        L->shard_numel = longest;
    }
    for (Seg &sg : segs)
        sg.unit_numel = P;
    int64_t padded;
    if (!mul_ok(L->shard_numel, R, &padded)) {
        delete L;
        return set_error(FSDP_ERANGE, "fsdp_layout: shard buffers too large");
    }
    const int64_t align = 32 / esize(param_dtype);
    L->valid_plans = make_plans(segs, R, false, kTile, align);
    L->gather_plans = make_plans(segs, R, false, kGatherTile, align);
    L->padded_plans = make_plans(segs, R, true, kTile, align);
    *out = L;
    return FSDP_OK;
}

void fsdp_layout_destroy(fsdp_layout_t *layout) { delete layout; }

fsdp_status fsdp_layout_query(const fsdp_layout_t *L, fsdp_query what, int i, int r, int64_t *out)
{
    if (L == nullptr || out == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_layout_query: NULL argument");
    bool need_i = (what >= FSDP_Q_PARAM_FULL_OFFSET && what <= FSDP_Q_PARAM_RANK_ROWS) ||
                  what == FSDP_Q_PARAM_OWNER;
    bool need_r = what == FSDP_Q_PARAM_RANK_ROW_START || what == FSDP_Q_PARAM_RANK_ROWS ||
                  what == FSDP_Q_RANK_NUMEL;
    if (need_i && (i < 0 || i >= L->n))
        return set_error(FSDP_EINVAL, "fsdp_layout_query: parameter index %d out of range", i);
    if (need_r && (r < 0 || r >= L->R))
        return set_error(FSDP_EINVAL, "fsdp_layout_query: rank %d out of range", r);
    int64_t a = 0, c = 0;
    switch (what) {
    case FSDP_Q_FULL_NUMEL: *out = L->P; break;
    case FSDP_Q_SHARD_NUMEL: *out = L->shard_numel; break;
    case FSDP_Q_PADDED_NUMEL: *out = L->shard_numel * L->R; break;
    case FSDP_Q_N_PARAMS: *out = L->n; break;
    case FSDP_Q_RANKS: *out = L->R; break;
    case FSDP_Q_MODE: *out = L->mode; break;
    case FSDP_Q_PARAM_DTYPE: *out = L->param_dtype; break;
    case FSDP_Q_GRAD_DTYPE: *out = L->grad_dtype; break;
    case FSDP_Q_PARAM_FULL_OFFSET: *out = L->full_off[i]; break;
    case FSDP_Q_PARAM_SHARD_OFFSET:
        if (L->mode == FSDP_FLAT)
            return set_error(FSDP_EINVAL, "fsdp_layout_query: FLAT layouts have no per-parameter "
                                          "shard offset");
        *out = L->shard_off[i];
        break;
    case FSDP_Q_PARAM_SHARD_ROWS: *out = L->shard_rows[i]; break;
    case FSDP_Q_PARAM_RANK_ROW_START:
        if (L->mode == FSDP_ZERO3)
            a = 0;
        else
            rank_rows(L->dim0[i], L->R, r, &a, &c);
        *out = a;
        break;
    case FSDP_Q_PARAM_RANK_ROWS:
        if (L->mode == FSDP_ZERO3)
            c = L->owner[i] == r ? L->dim0[i] : 0;
        else
            rank_rows(L->dim0[i], L->R, r, &a, &c);
        *out = c;
        break;
    case FSDP_Q_PARAM_OWNER:
        if (L->mode != FSDP_ZERO3)
            return set_error(FSDP_EINVAL, "fsdp_layout_query: only ZERO3 layouts have owners");
        *out = L->owner[i];
        break;
    case FSDP_Q_RANK_NUMEL: *out = rank_numel(L, r); break;
    default: return set_error(FSDP_EINVAL, "fsdp_layout_query: unknown query %d", (int)what);
    }
    return FSDP_OK;
}

fsdp_status fsdp_pack_flat(const fsdp_layout_t *L, const float *full, void *const *param_shard,
                           float *const *master, void *stream)
{
    if (L == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_pack_flat: layout is NULL");
    if (L->P == 0 && L->shard_numel == 0)
        return FSDP_OK;
    std::vector<Span> spans;
    fsdp_status st;
    if (L->P > 0) {
        if (full == nullptr)
            return set_error(FSDP_EINVAL, "fsdp_pack_flat: full is NULL");
        const void *f[1] = {full};
        if ((st = check_ptrs(f, 1, L->P * 4, false, "full", &spans)) != FSDP_OK)
            return st;
    }
    if ((st = check_ptrs((const void *const *)master, L->R, L->shard_numel * 4, true, "master",
                         &spans)) != FSDP_OK)
        return st;
    if (L->param_dtype == FSDP_BF16) {
        if ((st = check_ptrs((const void *const *)param_shard, L->R, L->shard_numel * 2, true,
                             "param_shard", &spans)) != FSDP_OK)
            return st;
    } else if (param_shard != nullptr) {
        return set_error(FSDP_EINVAL, "fsdp_pack_flat: param_shard must be NULL for an F32 "
                                      "layout (the master is the parameter shard)");
    }
    if ((st = check_spans(spans)) != FSDP_OK)
        return st;
    return launch_pack(L, full, param_shard, master, stream);
}

fsdp_status fsdp_all_gather_unflatten(const fsdp_layout_t *L, const void *const *shard,
                                      void *const *full_out, void *stream)
{
    if (L == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_all_gather_unflatten: layout is NULL");
    if (L->P == 0)
        return FSDP_OK;
    std::vector<Span> spans;
    fsdp_status st = check_gather_args(L, shard, full_out, &spans);
    if (st == FSDP_OK)
        st = check_spans(spans);
    if (st != FSDP_OK)
        return st;
    return launch_all_gather(1, &L, shard, full_out, stream);
}

fsdp_status fsdp_reduce_scatter_adamw(const fsdp_layout_t *L, const void *const *grad_full,
                                      float *const *master, float *const *m, float *const *v,
                                      void *const *param_shard_out, float *const *grad_shard_out,
                                      const fsdp_adamw_hp *hp, int64_t step, void *stream)
{
    if (L == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_reduce_scatter_adamw: layout is NULL");
    fsdp_status st = check_hp(hp, step);
    if (st != FSDP_OK || L->P == 0)
        return st;
    std::vector<Span> spans;
    st = check_rs_args(L, grad_full, master, m, v, param_shard_out, grad_shard_out, &spans);
    if (st == FSDP_OK)
        st = check_spans(spans);
    if (st != FSDP_OK)
        return st;
    return launch_rs_adamw(1, &L, grad_full, master, m, v, param_shard_out, grad_shard_out,
                           adam_scalars(hp, step, L->R), stream, nullptr);
}

fsdp_status fsdp_reduce_scatter_adamw_gather(
    const fsdp_layout_t *L, const void *const *grad_full, float *const *master, float *const *m,
    float *const *v, void *const *param_shard_out, float *const *grad_shard_out,
    const fsdp_adamw_hp *hp, int64_t step, const fsdp_layout_t *G, const void *const *shard,
    void *const *full_out, void *stream)
{
    if (L == nullptr || G == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_reduce_scatter_adamw_gather: layout is NULL");
    fsdp_status st = check_hp(hp, step);
    if (st != FSDP_OK)
        return st;
    std::vector<Span> spans;
    if (L->P > 0)
        st = check_rs_args(L, grad_full, master, m, v, param_shard_out, grad_shard_out, &spans);
    if (st == FSDP_OK && G->P > 0)
        st = check_gather_args(G, shard, full_out, &spans);
    if (st == FSDP_OK)
        st = check_spans(spans);
    if (st != FSDP_OK)
        return st;
    if (L->P == 0)
        return G->P == 0 ? FSDP_OK : launch_all_gather(1, &G, shard, full_out, stream);
    if (G->P == 0)
        return launch_rs_adamw(1, &L, grad_full, master, m, v, param_shard_out, grad_shard_out,
                               adam_scalars(hp, step, L->R), stream, nullptr);
    return launch_rs_adamw_gather(L, grad_full, master, m, v, param_shard_out, grad_shard_out,
                                  adam_scalars(hp, step, L->R), G, shard, full_out, stream);
}

fsdp_status fsdp_adamw_from_reduced(const fsdp_layout_t *L, const float *const *grad_avg_full,
                                    float *const *master, float *const *m, float *const *v,
                                    void *const *param_shard_out, const fsdp_adamw_hp *hp,
                                    int64_t step, void *stream)
{
    if (L == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_adamw_from_reduced: layout is NULL");
    fsdp_status st = check_hp(hp, step);
    if (st != FSDP_OK || L->P == 0)
        return st;
    std::vector<Span> spans;
    const int64_t sb = L->shard_numel * 4;
    if ((st = check_ptrs((const void *const *)grad_avg_full, L->R, L->P * 4, false,
                         "grad_avg_full", &spans)) != FSDP_OK ||
        (st = check_ptrs((const void *const *)master, L->R, sb, true, "master", &spans)) !=
            FSDP_OK ||
        (st = check_ptrs((const void *const *)m, L->R, sb, true, "m", &spans)) != FSDP_OK ||
        (st = check_ptrs((const void *const *)v, L->R, sb, true, "v", &spans)) != FSDP_OK)
        return st;
    if (L->param_dtype == FSDP_BF16) {
        if ((st = check_ptrs((const void *const *)param_shard_out, L->R, L->shard_numel * 2, true,
                             "param_shard_out", &spans)) != FSDP_OK)
            return st;
    } else if (param_shard_out != nullptr) {
        return set_error(FSDP_EINVAL, "param_shard_out must be NULL for an F32 layout");
    }
    if ((st = check_spans(spans)) != FSDP_OK)
        return st;
    return launch_adamw_reduced(L, grad_avg_full, master, m, v, param_shard_out,
                                adam_scalars(hp, step, L->R), stream);
}

fsdp_status fsdp_all_reduce(const fsdp_layout_t *L, const void *const *grad_full,
                            void *const *out, fsdp_dtype out_dtype, void *stream)
{
    if (L == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_all_reduce: layout is NULL");
    if (out_dtype != FSDP_F32 && out_dtype != FSDP_BF16)
        return set_error(FSDP_EUNSUPPORTED, "fsdp_all_reduce: unsupported output dtype");
    if (L->P == 0)
        return FSDP_OK;
    std::vector<Span> spans;
    fsdp_status st = check_ptrs(grad_full, L->R, L->P * esize(L->grad_dtype), false, "grad_full",
                                &spans);
    if (st == FSDP_OK)
        st = check_ptrs((const void *const *)out, L->R, L->P * esize(out_dtype), true, "out",
                        &spans);
    if (st == FSDP_OK)
        st = check_spans(spans);
    if (st != FSDP_OK)
        return st;
    return launch_all_reduce(L, grad_full, out, out_dtype, stream);
}

fsdp_status fsdp_accumulate_grad(const fsdp_layout_t *L, float *const *acc_full,
                                 const void *const *grad_full, int first, void *stream)
{
    if (L == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_accumulate_grad: layout is NULL");
    if (L->P == 0)
        return FSDP_OK;
    std::vector<Span> spans;
    fsdp_status st = check_ptrs(grad_full, L->R, L->P * esize(L->grad_dtype), false, "grad_full",
                                &spans);
    if (st == FSDP_OK)
        st = check_ptrs((const void *const *)acc_full, L->R, L->P * 4, true, "acc_full", &spans);
    if (st == FSDP_OK)
        st = check_spans(spans);
    if (st != FSDP_OK)
        return st;
    return launch_accumulate(L, acc_full, grad_full, first, stream);
}

fsdp_status fsdp_reduce_scatter_adamw_accum(const fsdp_layout_t *L, const float *const *acc_full,
                                            const void *const *grad_full, float *const *master,
                                            float *const *m, float *const *v,
                                            void *const *param_shard_out,
                                            float *const *grad_shard_out, const fsdp_adamw_hp *hp,
                                            int64_t step, void *stream)
{
    if (L == nullptr)
        return set_error(FSDP_EINVAL, "fsdp_reduce_scatter_adamw_accum: layout is NULL");
    fsdp_status st = check_hp(hp, step);
    if (st != FSDP_OK || L->P == 0)
        return st;
    std::vector<Span> spans;
    st = check_ptrs((const void *const *)acc_full, L->R, L->P * 4, false, "acc_full", &spans);
    if (st == FSDP_OK)
        st = check_rs_args(L, grad_full, master, m, v, param_shard_out, grad_shard_out, &spans);
    if (st == FSDP_OK)
        st = check_spans(spans);
    if (st != FSDP_OK)
        return st;
    return launch_rs_adamw(1, &L, grad_full, master, m, v, param_shard_out, grad_shard_out,
                           adam_scalars(hp, step, L->R), stream, acc_full);
}


fsdp_status fsdp_all_gather_unflatten_units(int n_units, const fsdp_layout_t *const *layouts,
                                            const void *const *shard, void *const *full_out,
                                            void *stream)
{
    const char *fn = "fsdp_all_gather_unflatten_units";
    fsdp_status st = check_units(n_units, layouts, fn);
    if (st != FSDP_OK)
        return st;
    if (shard == nullptr || full_out == nullptr)
        return set_error(FSDP_EINVAL, "%s: pointer array is NULL", fn);
    const int R = layouts[0]->R;
    std::vector<Span> spans;
    std::vector<const fsdp_layout_t *> Ls;
    std::vector<const void *> sh;
    std::vector<void *> fo;
    for (int u = 0; u < n_units; u++) {
        const fsdp_layout_t *L = layouts[u];
        if (L->P == 0)
            continue;  // an empty unit's pointers are not used
        st = check_gather_args(L, shard + (size_t)u * R, full_out + (size_t)u * R, &spans, u * R);
        if (st != FSDP_OK)
            return st;
        Ls.push_back(L);
        take(sh, shard, u, R);
        take(fo, full_out, u, R);
    }
    if (Ls.empty())
        return FSDP_OK;
    if ((st = check_spans(spans)) != FSDP_OK)
        return st;
    return launch_all_gather((int)Ls.size(), Ls.data(), sh.data(), fo.data(), stream);
}

fsdp_status fsdp_reduce_scatter_adamw_units(int n_units, const fsdp_layout_t *const *layouts,
                                            const void *const *grad_full, float *const *master,
                                            float *const *m, float *const *v,
                                            void *const *param_shard_out,
                                            float *const *grad_shard_out, const fsdp_adamw_hp *hp,
                                            int64_t step, void *stream)
{
    const char *fn = "fsdp_reduce_scatter_adamw_units";
    fsdp_status st = check_units(n_units, layouts, fn);
    if (st == FSDP_OK)
        st = check_hp(hp, step);
    if (st != FSDP_OK)
        return st;
    if (grad_full == nullptr || master == nullptr || m == nullptr || v == nullptr)
        return set_error(FSDP_EINVAL, "%s: pointer array is NULL", fn);
    const bool bf16 = layouts[0]->param_dtype == FSDP_BF16;
    if (bf16 != (param_shard_out != nullptr))
        return set_error(FSDP_EINVAL, "%s: param_shard_out must be given for BF16 layouts and "
                                      "NULL for F32 layouts", fn);
    const int R = layouts[0]->R;
    std::vector<Span> spans;
    std::vector<const fsdp_layout_t *> Ls;
    std::vector<const void *> g;
    std::vector<float *> ma, mm, vv, gs;
    std::vector<void *> ps;
    for (int u = 0; u < n_units; u++) {
        const fsdp_layout_t *L = layouts[u];
        if (L->P == 0)
            continue;
        const size_t o = (size_t)u * R;
        st = check_rs_args(L, grad_full + o, master + o, m + o, v + o,
                           param_shard_out ? param_shard_out + o : nullptr,
                           grad_shard_out ? grad_shard_out + o : nullptr, &spans, u * R);
        if (st != FSDP_OK)
            return st;
        Ls.push_back(L);
        take(g, grad_full, u, R);
        take(ma, master, u, R);
        take(mm, m, u, R);
        take(vv, v, u, R);
        take(ps, param_shard_out, u, R);
        take(gs, grad_shard_out, u, R);
    }
    if (Ls.empty())
        return FSDP_OK;
    if ((st = check_spans(spans)) != FSDP_OK)
        return st;
    return launch_rs_adamw((int)Ls.size(), Ls.data(), g.data(), ma.data(), mm.data(), vv.data(),
                           data_or_null(ps, param_shard_out), data_or_null(gs, grad_shard_out),
                           adam_scalars(hp, step, R), stream, nullptr);
}

fsdp_status fsdp_write_stream(void *const *dst, int n, int64_t bytes, uint32_t pattern,
                              void *stream)
{
    if (dst == nullptr || n < 1 || n > FSDP_MAX_RANKS || bytes < 0)
        return set_error(FSDP_EINVAL, "fsdp_write_stream: bad arguments");
    if (bytes % 32 != 0)
        return set_error(FSDP_EINVAL, "fsdp_write_stream: bytes must be a multiple of 32");
    if (bytes == 0)
        return FSDP_OK;
    std::vector<Span> spans;
    for (int d = 0; d < n; d++)
        if (dst[d] != nullptr && (reinterpret_cast<uintptr_t>(dst[d]) & 31u))
            return set_error(FSDP_EALIGN, "fsdp_write_stream: dst[%d] is not 32-byte aligned", d);
    fsdp_status st = check_ptrs((const void *const *)dst, n, bytes, true, "dst", &spans);
    if (st == FSDP_OK)
        st = check_spans(spans);
    if (st != FSDP_OK)
        return st;
    return launch_write_stream(dst, n, bytes, pattern, stream);
}

fsdp_status fsdp_stage_wait_timeouts(int device, uint64_t *count)
{
    if (count == nullptr || device < 0)
        return set_error(FSDP_EINVAL, "fsdp_stage_wait_timeouts: bad arguments");
    return read_stage_wait_timeouts(device, count);
}

fsdp_status fsdp_stage_wait_selftest(int device, uint64_t *gave_up)
{
    if (gave_up == nullptr || device < 0)
        return set_error(FSDP_EINVAL, "fsdp_stage_wait_selftest: bad arguments");
    return run_stage_wait_selftest(device, gave_up);
}

}  // extern "C"
