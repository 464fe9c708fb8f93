// Host-side View checks and the iteration space shared by the elementwise and
// row-reduction launches.
//
// A View is (shape, strides, offset, mask) and lowers to index arithmetic
// inside the kernels (limn, "Three rules hold it together").  Before any
// launch the host proves every reachable element lies inside the allocation
// (the in-bounds half of Litmus's "GPUSafetyCheck") and that a written View is
// injective (the race-free half: no two cells of the output share an address).
#include <algorithm>
#include <cstring>

#include "common.h"

namespace psg {

int64_t view_numel(const psg_view* v)
{
    int64_t n = 1;
    for (int d = 0; d < v->ndim; ++d) n *= v->shape[d];
    return n;
}

static bool dim_masked(const psg_view* v, int d)
{
    return v->mask_lo[d] > 0 || v->mask_hi[d] < v->shape[d];
}

bool view_has_mask(const psg_view* v)
{
    for (int d = 0; d < v->ndim; ++d)
        if (dim_masked(v, d)) return true;
    return false;
}

bool view_contiguous(const psg_view* v)
{
    if (view_has_mask(v)) return false;
    int64_t s = 1;
    for (int d = v->ndim - 1; d >= 0; --d) {
        if (v->shape[d] != 1 && v->strides[d] != s) return false;
        s *= v->shape[d];
    }
    return true;
}

psg_status check_view(const psg_view* v, bool for_write)
{
    if (!v) return PSG_E_INVALID_ARG;
    if (v->ndim < 0 || v->ndim > PSG_MAX_DIMS) return PSG_E_INVALID_ARG;
    if (!dtype_valid(v->dtype)) return PSG_E_UNSUPPORTED_DTYPE;
    if (v->extent < 0) return PSG_E_INVALID_ARG;
    bool empty = false;
    for (int d = 0; d < v->ndim; ++d) {
        if (v->shape[d] < 0 || v->strides[d] < 0) return PSG_E_INVALID_ARG;
        if (v->shape[d] > (int64_t(1) << 40)) return PSG_E_INVALID_ARG;
        if (v->strides[d] > (int64_t(1) << 44)) return PSG_E_INVALID_ARG;
        if (v->shape[d] == 0) empty = true;
    }
    if (empty) return PSG_OK;
    // the reachable box: per dim [max(lo,0), min(hi,shape))
    __int128 lo_off = v->offset, hi_off = v->offset;
    bool reads_nothing = false;
    for (int d = 0; d < v->ndim; ++d) {
        int64_t lo = std::max<int64_t>(v->mask_lo[d], 0);
        int64_t hi = std::min<int64_t>(v->mask_hi[d], v->shape[d]);
        if (hi <= lo) { reads_nothing = true; break; }
        lo_off += (__int128)lo * v->strides[d];
        hi_off += (__int128)(hi - 1) * v->strides[d];
    }
    if (for_write) {
        if (view_has_mask(v)) return PSG_E_UNSUPPORTED_LAYOUT;
        // injective: sort the dims of size > 1 by stride; each must step past
        // the whole span of the dims below it (mixed-radix, no aliasing)
        int idx[PSG_MAX_DIMS], k = 0;
        for (int d = 0; d < v->ndim; ++d)
            if (v->shape[d] > 1) idx[k++] = d;
        std::sort(idx, idx + k, [&](int a, int b) { return v->strides[a] < v->strides[b]; });
        __int128 span = 1;
        for (int i = 0; i < k; ++i) {
            int d = idx[i];
            if ((__int128)v->strides[d] < span) return PSG_E_UNSUPPORTED_LAYOUT;
            span = (__int128)v->strides[d] * v->shape[d];
        }
    }
    if (reads_nothing) return PSG_OK;
    if (lo_off < 0 || hi_off >= (__int128)v->extent) return PSG_E_OUT_OF_BOUNDS_VIEW;
    return PSG_OK;
}

psg_status build_space(const psg_view* const* views, int nviews, bool keep_last, Space* sp,
                       int64_t (*strides)[MAXD], int64_t (*mlo)[MAXD], int64_t (*mhi)[MAXD],
                       bool* masked)
{
    const psg_view* o = views[0];
    const int nd0 = o->ndim;
    // 1. dims kept: drop size-1 dims nobody masks (they never move an index)
    int keep[MAXD], nk = 0;
    for (int d = 0; d < nd0; ++d) {
        bool m = false;
        for (int v = 0; v < nviews; ++v) m = m || dim_masked(views[v], d);
        bool last = keep_last && d == nd0 - 1;
        if (o->shape[d] != 1 || m || last) keep[nk++] = d;
    }
    // 2. order: the first view's strides descending, so its stride-1 dim is
    //    innermost (limn, "Reading the schedule": loop order is chosen so the
    //    innermost loop walks stride-1 memory); a reduce axis stays last
    int nsort = keep_last && nk > 0 ? nk - 1 : nk;
    std::stable_sort(keep, keep + nsort, [&](int a, int b) { return o->strides[a] > o->strides[b]; });
    // 3. merge neighbours that are contiguous and unmasked in every view
    int64_t shp[MAXD];
    int64_t st[16][MAXD];
    int64_t lo[16][MAXD], hi[16][MAXD];
    int n = 0;
    for (int i = 0; i < nk; ++i) {
        int d = keep[i];
        bool can_merge = n > 0 && !(keep_last && i == nk - 1);
        if (can_merge) {
            for (int v = 0; v < nviews && can_merge; ++v) {
                const psg_view* w = views[v];
                if (dim_masked(w, d)) can_merge = false;
                if (lo[v][n - 1] != 0 || hi[v][n - 1] != shp[n - 1]) can_merge = false;
                if (st[v][n - 1] != w->strides[d] * w->shape[d]) can_merge = false;
            }
        }
        if (can_merge) {
            shp[n - 1] *= o->shape[d];
            for (int v = 0; v < nviews; ++v) {
                st[v][n - 1] = views[v]->strides[d];
                lo[v][n - 1] = 0;
                hi[v][n - 1] = shp[n - 1];
            }
        } else {
            shp[n] = o->shape[d];
            for (int v = 0; v < nviews; ++v) {
                st[v][n] = views[v]->strides[d];
                lo[v][n] = std::max<int64_t>(views[v]->mask_lo[d], 0);
                hi[v][n] = std::min<int64_t>(views[v]->mask_hi[d], views[v]->shape[d]);
            }
            ++n;
        }
    }
    if (n == 0) {  // scalar
        shp[0] = 1;
        for (int v = 0; v < nviews; ++v) { st[v][0] = 0; lo[v][0] = 0; hi[v][0] = 1; }
        n = 1;
    }
    sp->nd = n;
    sp->rows = 1;
    for (int d = 0; d < n; ++d) {
        sp->shape[d] = shp[d];
        if (d < n - 1) sp->rows *= shp[d];
    }
    sp->inner = shp[n - 1];
    sp->chunks = (sp->inner + VEC - 1) / VEC;
    for (int v = 0; v < nviews; ++v) {
        masked[v] = false;
        for (int d = 0; d < n; ++d) {
            strides[v][d] = st[v][d];
            mlo[v][d] = lo[v][d];
            mhi[v][d] = hi[v][d];
            if (lo[v][d] != 0 || hi[v][d] != shp[d]) masked[v] = true;
        }
    }
    return PSG_OK;
}

}  // namespace psg
