// Internal definition of the FlatParameter plan (host only).
//
// "Infra: Data Parallel" (F. Pu), FSDP section, subsection "FSDP1": the
// parameters of a unit are flattened and concatenated into one FlatParameter
// that is cut into N_d equal contiguous shards.  Each unit is padded on its
// own to a multiple of N_d; the units are laid out one after another in one
// global flat index space.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "zs.h"

namespace zs {

struct Unit {
    int64_t base;      // global flat index of the unit's first element
    int64_t numel;     // real elements
    int64_t padded;    // multiple of n_d
    int64_t shard;     // padded / n_d
};

struct Bucket {
    int32_t unit;
    int64_t begin;     // global flat range [begin, end)
    int64_t end;
};

}  // namespace zs

struct zs_plan_s {
    int32_t n_d = 0;
    int32_t stage = 0;
    int32_t layout = 0;                         // ZS_LAYOUT_FSDP1 or ZS_LAYOUT_FSDP2
    int64_t bucket_elems = 0;
    int64_t numel = 0;
    int64_t padded = 0;
    int64_t shard_per_rank = 0;                 // sum over units of S_u
    std::vector<int64_t> param_numel;
    std::vector<int64_t> param_offset;          // global flat index of the first element
    std::vector<int32_t> param_unit;
    // FSDP2 only: dim-0 rows, elements per row, rows per rank, offset of the piece in a rank's shard
    std::vector<int64_t> param_d0, param_row, param_chunk, param_piece_off;
    std::vector<zs::Unit> units;
    std::vector<zs::Bucket> buckets;
};

namespace zs {

// Thread-local message behind zs_last_error().
void set_error(const std::string& msg);
void clear_error();

// Rank owning global index i of unit u.
inline int32_t owner_in_unit(const Unit& u, int64_t i) { return (int32_t)((i - u.base) / u.shard); }

}  // namespace zs
