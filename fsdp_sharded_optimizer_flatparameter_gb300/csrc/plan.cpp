// FlatParameter planner and accounting (host only, no CUDA calls).
//
// Layout: "Infra: Data Parallel" (F. Pu), FSDP section, FSDP1 layout figure
// and subsection "FSDP1" - flatten and concatenate the parameters of each
// unit in order, pad with the fewest zeros that make the unit's length a
// multiple of N_d, cut into N_d equal contiguous shards.  Buckets (section
// "Naive Data Parallelism") are runs of floor(bucket_bytes / 2) consecutive
// bf16 gradient elements of one unit.
//
// Accounting: section "Zero Redundancy Optimizer (ZeRO)", memory figure
// (bytes of model states one GPU holds, k = 12) and communication paragraphs
// (bytes one rank sends per step, 16-bit elements).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "plan.h"

namespace zs {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }
void clear_error() { g_last_error.clear(); }

}  // namespace zs

using zs::set_error;

extern "C" const char* zs_last_error(void) { return zs::g_last_error.c_str(); }

static int plan_create(int32_t n_params, const int32_t* ndims, const int64_t* dims, const int32_t* unit_of_param,
                       int32_t n_d, int32_t stage, int64_t bucket_bytes, int32_t layout, zs_plan_t* out) {
    zs::clear_error();
    if (!out) { set_error("zs_plan_create: out is NULL"); return ZS_ERR_INVALID; }
    *out = nullptr;
    if (n_params < 1) { set_error("zs_plan_create: n_params must be >= 1"); return ZS_ERR_INVALID; }
    if (!ndims || !dims) { set_error("zs_plan_create: ndims/dims is NULL"); return ZS_ERR_INVALID; }
    if (n_d < 1 || n_d > ZS_MAX_RANKS) { set_error("zs_plan_create: n_d out of range"); return ZS_ERR_INVALID; }
    if (stage < ZS_STAGE_DP || stage > ZS_STAGE_ZERO3) { set_error("zs_plan_create: bad stage"); return ZS_ERR_INVALID; }

    zs_plan_s* p = new (std::nothrow) zs_plan_s();
    if (!p) { set_error("zs_plan_create: out of host memory"); return ZS_ERR_OOM_HOST; }
    try {
        p->n_d = n_d;
        p->stage = stage;
        p->layout = layout;
        p->param_numel.resize(n_params);
        p->param_d0.assign(n_params, 1);
        p->param_row.assign(n_params, 1);
        p->param_chunk.assign(n_params, 1);
        p->param_piece_off.assign(n_params, 0);
        p->param_offset.resize(n_params);
        p->param_unit.resize(n_params);

        // element counts
        int64_t d = 0;
        for (int32_t k = 0; k < n_params; ++k) {
            if (ndims[k] < 0 || ndims[k] > 8) { set_error("zs_plan_create: ndims out of range"); delete p; return ZS_ERR_INVALID; }
            int64_t n = 1;
            for (int32_t j = 0; j < ndims[k]; ++j, ++d) {
                if (dims[d] < 1) { set_error("zs_plan_create: every dimension must be >= 1"); delete p; return ZS_ERR_INVALID; }
                if (n > (int64_t(1) << 50) / dims[d]) { set_error("zs_plan_create: parameter too large"); delete p; return ZS_ERR_INVALID; }
                n *= dims[d];
                if (j == 0) p->param_d0[k] = dims[d];
            }
            p->param_numel[k] = n;
            p->param_row[k] = n / p->param_d0[k];       // a 0-d parameter is one row of one element
            p->param_chunk[k] = (p->param_d0[k] + n_d - 1) / n_d;
        }

        // units
        int32_t n_units = 1;
        if (unit_of_param) {
            int32_t mx = -1;
            for (int32_t k = 0; k < n_params; ++k) {
                if (unit_of_param[k] < 0 || unit_of_param[k] >= n_params) {
                    set_error("zs_plan_create: unit id out of range"); delete p; return ZS_ERR_INVALID;
                }
                mx = unit_of_param[k] > mx ? unit_of_param[k] : mx;
            }
            n_units = mx + 1;
            std::vector<char> used(n_units, 0);
            for (int32_t k = 0; k < n_params; ++k) used[unit_of_param[k]] = 1;
            for (int32_t u = 0; u < n_units; ++u)
                if (!used[u]) { set_error("zs_plan_create: unit ids must be 0..U-1 with none unused"); delete p; return ZS_ERR_INVALID; }
        }
        int64_t base = 0;
        for (int32_t u = 0; u < n_units; ++u) {
            int64_t off = base, piece = 0;
            for (int32_t k = 0; k < n_params; ++k) {
                int32_t ku = unit_of_param ? unit_of_param[k] : 0;
                if (ku != u) continue;
                p->param_unit[k] = u;
                if (layout == ZS_LAYOUT_FSDP2) {
                    // each parameter cut along dim 0: its rank-r piece sits at base + r*S + piece
                    p->param_piece_off[k] = piece;
                    p->param_offset[k] = base + piece;
                    piece += p->param_chunk[k] * p->param_row[k];
                } else {
                    p->param_offset[k] = off;
                }
                off += p->param_numel[k];
            }
            zs::Unit un;
            un.base = base;
            un.numel = off - base;
            if (layout == ZS_LAYOUT_FSDP2) {
                un.shard = piece;
                un.padded = piece * n_d;
            } else {
                un.padded = ((un.numel + n_d - 1) / n_d) * n_d;
                un.shard = un.padded / n_d;
            }
            p->units.push_back(un);
            p->numel += un.numel;
            p->shard_per_rank += un.shard;
            base += un.padded;
        }
        p->padded = base;

        // buckets
        int64_t max_unit = 1;
        for (const auto& un : p->units) max_unit = un.padded > max_unit ? un.padded : max_unit;
        p->bucket_elems = bucket_bytes <= 0 ? max_unit : bucket_bytes / 2;
        if (p->bucket_elems < 1) { set_error("zs_plan_create: bucket smaller than one bf16 element"); delete p; return ZS_ERR_INVALID; }
        for (int32_t u = 0; u < n_units; ++u) {
            const auto& un = p->units[u];
            for (int64_t s = 0; s < un.padded; s += p->bucket_elems) {
                int64_t e = s + p->bucket_elems < un.padded ? s + p->bucket_elems : un.padded;
                p->buckets.push_back({u, un.base + s, un.base + e});
            }
            if (p->buckets.size() > (size_t)INT32_MAX) { set_error("zs_plan_create: too many buckets"); delete p; return ZS_ERR_INVALID; }
        }
    } catch (const std::bad_alloc&) {
        delete p;
        set_error("zs_plan_create: out of host memory");
        return ZS_ERR_OOM_HOST;
    }
    *out = p;
    return ZS_OK;
}

extern "C" int zs_plan_create(int32_t n_params, const int32_t* ndims, const int64_t* dims,
                              const int32_t* unit_of_param, int32_t n_d, int32_t stage,
                              int64_t bucket_bytes, zs_plan_t* out) {
    return plan_create(n_params, ndims, dims, unit_of_param, n_d, stage, bucket_bytes, ZS_LAYOUT_FSDP1, out);
}

extern "C" int zs_plan_create_fsdp2(int32_t n_params, const int32_t* ndims, const int64_t* dims,
                                    const int32_t* unit_of_param, int32_t n_d, int32_t stage,
                                    int64_t bucket_bytes, zs_plan_t* out) {
    return plan_create(n_params, ndims, dims, unit_of_param, n_d, stage, bucket_bytes, ZS_LAYOUT_FSDP2, out);
}

extern "C" int zs_plan_layout(zs_plan_t p, int32_t* layout) {
    zs::clear_error();
    if (!p || !layout) { set_error("zs_plan_layout: NULL argument"); return ZS_ERR_INVALID; }
    *layout = p->layout;
    return ZS_OK;
}

extern "C" int zs_plan_param_rows(zs_plan_t p, int32_t k, int32_t rank, int64_t* row_begin, int64_t* nrows,
                                  int64_t* rows_per_rank, int64_t* row_elems) {
    zs::clear_error();
    if (!p || k < 0 || k >= (int32_t)p->param_numel.size() || rank < 0 || rank >= p->n_d) {
        set_error("zs_plan_param_rows: bad plan, parameter or rank");
        return ZS_ERR_INVALID;
    }
    const int64_t c = p->param_chunk[k], d0 = p->param_d0[k];
    const int64_t b = std::min<int64_t>((int64_t)rank * c, d0), e = std::min<int64_t>(((int64_t)rank + 1) * c, d0);
    if (row_begin) *row_begin = b;
    if (nrows) *nrows = e - b;
    if (rows_per_rank) *rows_per_rank = c;
    if (row_elems) *row_elems = p->param_row[k];
    return ZS_OK;
}

extern "C" void zs_plan_destroy(zs_plan_t plan) { delete plan; }

extern "C" int zs_plan_info(zs_plan_t p, int64_t* numel, int64_t* padded_numel, int64_t* shard_numel_per_rank,
                            int32_t* n_units, int32_t* n_buckets, int32_t* n_d, int32_t* stage) {
    zs::clear_error();
    if (!p) { set_error("zs_plan_info: plan is NULL"); return ZS_ERR_INVALID; }
    if (numel) *numel = p->numel;
    if (padded_numel) *padded_numel = p->padded;
    if (shard_numel_per_rank) *shard_numel_per_rank = p->shard_per_rank;
    if (n_units) *n_units = (int32_t)p->units.size();
    if (n_buckets) *n_buckets = (int32_t)p->buckets.size();
    if (n_d) *n_d = p->n_d;
    if (stage) *stage = p->stage;
    return ZS_OK;
}

extern "C" int zs_plan_unit(zs_plan_t p, int32_t u, int64_t* base, int64_t* numel, int64_t* padded_numel,
                            int64_t* shard_numel) {
    zs::clear_error();
    if (!p || u < 0 || u >= (int32_t)p->units.size()) { set_error("zs_plan_unit: bad plan or unit"); return ZS_ERR_INVALID; }
    const auto& un = p->units[u];
    if (base) *base = un.base;
    if (numel) *numel = un.numel;
    if (padded_numel) *padded_numel = un.padded;
    if (shard_numel) *shard_numel = un.shard;
    return ZS_OK;
}

extern "C" int zs_plan_bucket(zs_plan_t p, int32_t b, int32_t* unit, int64_t* begin, int64_t* end) {
    zs::clear_error();
    if (!p || b < 0 || b >= (int32_t)p->buckets.size()) { set_error("zs_plan_bucket: bad plan or bucket"); return ZS_ERR_INVALID; }
    const auto& bk = p->buckets[b];
    if (unit) *unit = bk.unit;
    if (begin) *begin = bk.begin;
    if (end) *end = bk.end;
    return ZS_OK;
}

extern "C" int zs_plan_bucket_rank_slice(zs_plan_t p, int32_t b, int32_t rank, int64_t* begin, int64_t* end) {
    zs::clear_error();
    if (!p || b < 0 || b >= (int32_t)p->buckets.size() || rank < 0 || rank >= p->n_d) {
        set_error("zs_plan_bucket_rank_slice: bad plan, bucket or rank");
        return ZS_ERR_INVALID;
    }
    const auto& bk = p->buckets[b];
    const auto& un = p->units[bk.unit];
    int64_t s_lo = un.base + (int64_t)rank * un.shard, s_hi = s_lo + un.shard;
    int64_t lo = bk.begin > s_lo ? bk.begin : s_lo;
    int64_t hi = bk.end < s_hi ? bk.end : s_hi;
    if (hi < lo) hi = lo;
    if (begin) *begin = lo;
    if (end) *end = hi;
    return ZS_OK;
}

extern "C" int zs_plan_param(zs_plan_t p, int32_t k, int32_t* unit, int64_t* flat_offset, int64_t* numel) {
    zs::clear_error();
    if (!p || k < 0 || k >= (int32_t)p->param_numel.size()) { set_error("zs_plan_param: bad plan or parameter"); return ZS_ERR_INVALID; }
    if (unit) *unit = p->param_unit[k];
    if (flat_offset) *flat_offset = p->param_offset[k];
    if (numel) *numel = p->param_numel[k];
    return ZS_OK;
}

extern "C" int zs_plan_param_segment(zs_plan_t p, int32_t k, int32_t rank, int64_t* flat_begin,
                                     int64_t* shard_offset, int64_t* len) {
    zs::clear_error();
    if (!p || k < 0 || k >= (int32_t)p->param_numel.size() || rank < 0 || rank >= p->n_d) {
        set_error("zs_plan_param_segment: bad plan, parameter or rank");
        return ZS_ERR_INVALID;
    }
    const auto& un = p->units[p->param_unit[k]];
    if (p->layout == ZS_LAYOUT_FSDP2) {
        // rank r's piece: rows [r*c, min((r+1)*c, d0)) at base + r*S + piece offset
        const int64_t c = p->param_chunk[k], d0 = p->param_d0[k];
        const int64_t b = std::min<int64_t>((int64_t)rank * c, d0), e = std::min<int64_t>(((int64_t)rank + 1) * c, d0);
        const int64_t n = (e - b) * p->param_row[k];
        if (flat_begin) *flat_begin = n ? un.base + (int64_t)rank * un.shard + p->param_piece_off[k] : 0;
        if (shard_offset) *shard_offset = n ? p->param_piece_off[k] : 0;
        if (len) *len = n;
        return ZS_OK;
    }
    int64_t lo = p->param_offset[k], hi = lo + p->param_numel[k];
    int64_t s_lo = un.base + (int64_t)rank * un.shard, s_hi = s_lo + un.shard;
    int64_t a = lo > s_lo ? lo : s_lo;
    int64_t b = hi < s_hi ? hi : s_hi;
    int64_t fb = 0, so = 0, n = 0;
    if (a < b) { fb = a; so = a - s_lo; n = b - a; }
    if (flat_begin) *flat_begin = fb;
    if (shard_offset) *shard_offset = so;
    if (len) *len = n;
    return ZS_OK;
}

extern "C" int zs_plan_memory_bytes(zs_plan_t p, int32_t stage, int64_t* bytes_per_rank) {
    zs::clear_error();
    if (!p || !bytes_per_rank || stage < 0 || stage > 3) { set_error("zs_plan_memory_bytes: bad argument"); return ZS_ERR_INVALID; }
    const int64_t S = p->shard_per_rank;
    int64_t b = 0;
    switch (stage) {
        case ZS_STAGE_DP:    b = 2 * p->numel + 2 * p->numel + 12 * p->numel; break;   // everything replicated
        case ZS_STAGE_ZERO1: b = 2 * p->padded + 2 * p->padded + 12 * S; break;        // state sharded
        case ZS_STAGE_ZERO2: b = 2 * p->padded + 2 * S + 12 * S; break;                // + gradients sharded
        case ZS_STAGE_ZERO3: b = 2 * S + 2 * S + 12 * S; break;                        // + parameters sharded
    }
    *bytes_per_rank = b;
    return ZS_OK;
}

extern "C" int zs_plan_comm_bytes(zs_plan_t p, int32_t stage, int32_t reshard_after_forward,
                                  int64_t* bytes_sent_per_rank) {
    zs::clear_error();
    if (!p || !bytes_sent_per_rank || stage < 0 || stage > 3) { set_error("zs_plan_comm_bytes: bad argument"); return ZS_ERR_INVALID; }
    // One reduce-scatter or all-gather of unit u: each rank sends the (N_d - 1) * S_u
    // elements it does not own (RS) or its shard to the N_d - 1 others (AG).
    int64_t one_pass = 0;
    for (const auto& un : p->units) one_pass += (int64_t)(p->n_d - 1) * un.shard;
    int64_t passes = 0;
    switch (stage) {
        case ZS_STAGE_DP:    passes = 2; break;                                  // ring all-reduce = RS + AG
        case ZS_STAGE_ZERO1:
        case ZS_STAGE_ZERO2: passes = 2; break;                                  // RS grads + AG params
        case ZS_STAGE_ZERO3: passes = reshard_after_forward ? 3 : 2; break;      // AG fwd (+ AG bwd) + RS
    }
    *bytes_sent_per_rank = 2 * passes * one_pass;
    return ZS_OK;
}

extern "C" int zs_adamw_scalars(const zs_adamw_hparams* hp, int64_t step, float* out8) {
    zs::clear_error();
    if (!hp || !out8) { set_error("zs_adamw_scalars: NULL argument"); return ZS_ERR_INVALID; }
    if (step < 1) { set_error("zs_adamw_scalars: step must be >= 1"); return ZS_ERR_INVALID; }
    const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, wd = hp->weight_decay;
    out8[0] = hp->beta1;
    out8[1] = hp->beta2;
    out8[2] = hp->eps;
    out8[3] = (float)(1.0 - lr * wd);
    out8[4] = (float)(1.0 - b1);
    out8[5] = (float)(1.0 - b2);
    out8[6] = (float)(lr / (1.0 - std::pow(b1, (double)step)));
    out8[7] = (float)std::sqrt(1.0 - std::pow(b2, (double)step));
    return ZS_OK;
}

extern "C" int zs_plan_pad_ranges(zs_plan_t p, int64_t* begins, int64_t* ends, int64_t capacity, int64_t* count) {
    zs::clear_error();
    if (!p || !count || capacity < 0 || (capacity > 0 && (!begins || !ends))) {
        set_error("zs_plan_pad_ranges: bad argument");
        return ZS_ERR_INVALID;
    }
    int64_t n = 0;
    auto emit = [&](int64_t b, int64_t e) {
        if (e <= b) return;
        if (n < capacity) {
            begins[n] = b;
            ends[n] = e;
        }
        ++n;
    };
    for (size_t u = 0; u < p->units.size(); ++u) {
        const auto& un = p->units[u];
        if (p->layout != ZS_LAYOUT_FSDP2) {
            emit(un.base + un.numel, un.base + un.padded);
            continue;
        }
        for (int32_t r = 0; r < p->n_d; ++r) {
            for (size_t k = 0; k < p->param_numel.size(); ++k) {
                if (p->param_unit[k] != (int32_t)u) continue;
                const int64_t c = p->param_chunk[k], d0 = p->param_d0[k], row = p->param_row[k];
                const int64_t b = std::min<int64_t>((int64_t)r * c, d0), e = std::min<int64_t>(((int64_t)r + 1) * c, d0);
                const int64_t start = un.base + (int64_t)r * un.shard + p->param_piece_off[k];
                emit(start + (e - b) * row, start + c * row);
            }
        }
    }
    *count = n;
    return ZS_OK;
}
