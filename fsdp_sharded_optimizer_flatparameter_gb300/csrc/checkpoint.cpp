// Sharded checkpoint: every simulated rank writes its own shards, loading re-cuts
// them for any rank count.
//
// "Infra: Data Parallel" (F. Pu), section "Fully Sharded Data Parallel (FSDP)",
// subsection "Checkpoint": ranks write the shards they own plus the metadata
// needed to restore them; loading follows the target run's sharding layout,
// so save and load may use different numbers of ranks; optimizer state is
// saved with the weights.  An element is identified across layouts by its
// position among its unit's real elements (padding is dropped and re-made).
//
// Files in `dir` (which must exist):
//   meta.txt          text: format tag, N_d, step, parameter shapes and units,
//                     per-unit (numel, padded, shard), the arrays and their types
//   rank-NNNNN.bin    rank r's shard of each array in the order params (bf16),
//                     master, m, v (fp32); each array is the rank's piece of every
//                     unit, units in order
// Both calls copy through a bounded host buffer with cudaMemcpyAsync on the
// given stream and synchronise that stream.
#include <algorithm>
#include <cerrno>
#include <cstdio>
#include <cstring>
#include <fstream>
#include <sstream>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "plan.h"

namespace {

constexpr size_t kChunk = size_t(64) << 20;            // host staging per copy
const int kElemBytes[4] = {2, 4, 4, 4};

int fail(const char* fn, const std::string& what, int code = ZS_ERR_INVALID) {
    zs::set_error(std::string(fn) + ": " + what);
    return code;
}

std::string rank_file(const std::string& dir, int r) {
    char name[32];
    std::snprintf(name, sizeof(name), "rank-%05d.bin", r);
    return dir + "/" + name;
}

struct SavedUnit {
    int64_t numel, padded, shard;
};

}  // namespace

extern "C" int zs_checkpoint_save(zs_plan_t plan, const char* dir, const void* shards, const float* master,
                                  const float* m, const float* v, int64_t step, void* stream) {
    static const char* fn = "zs_checkpoint_save";
    zs::clear_error();
    if (!plan || !dir || !shards || !master || !m || !v) return fail(fn, "NULL argument");
    if (plan->layout != ZS_LAYOUT_FSDP1) return fail(fn, "only FSDP1-layout plans are supported", ZS_ERR_UNSUPPORTED);
    cudaStream_t st = (cudaStream_t)stream;
    const std::string d(dir);
    {
        std::ofstream meta(d + "/meta.txt");
        if (!meta) return fail(fn, "cannot write " + d + "/meta.txt: " + std::strerror(errno));
        meta << "zs-checkpoint 1\n";
        meta << "n_d " << plan->n_d << "\n";
        meta << "step " << step << "\n";
        meta << "params " << plan->param_numel.size() << "\n";
        for (size_t k = 0; k < plan->param_numel.size(); ++k)
            meta << "p " << plan->param_numel[k] << " unit " << plan->param_unit[k] << "\n";
        meta << "units " << plan->units.size() << "\n";
        for (const auto& u : plan->units) meta << "u " << u.numel << " " << u.padded << " " << u.shard << "\n";
        meta << "arrays params:bf16 master:f32 m:f32 v:f32\n";
        if (!meta) return fail(fn, "writing meta.txt failed");
    }
    const void* src[4] = {shards, master, m, v};
    std::vector<char> buf(kChunk);
    for (int r = 0; r < plan->n_d; ++r) {
        FILE* f = std::fopen(rank_file(d, r).c_str(), "wb");
        if (!f) return fail(fn, "cannot write " + rank_file(d, r) + ": " + std::strerror(errno));
        for (int a = 0; a < 4; ++a) {
            const int eb = kElemBytes[a];
            for (const auto& u : plan->units) {
                const char* from = (const char*)src[a] + (size_t)(u.base + (int64_t)r * u.shard) * eb;
                size_t left = (size_t)u.shard * eb;
                while (left) {
                    const size_t n = left < kChunk ? left : kChunk;
                    cudaError_t e = cudaMemcpyAsync(buf.data(), from, n, cudaMemcpyDeviceToHost, st);
                    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
                    if (e != cudaSuccess) {
                        std::fclose(f);
                        return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
                    }
                    if (std::fwrite(buf.data(), 1, n, f) != n) {
                        std::fclose(f);
                        return fail(fn, "short write to " + rank_file(d, r));
                    }
                    from += n;
                    left -= n;
                }
            }
        }
        if (std::fclose(f) != 0) return fail(fn, "closing " + rank_file(d, r) + " failed");
    }
    return ZS_OK;
}

extern "C" int zs_checkpoint_load(zs_plan_t plan, const char* dir, void* shards, float* master, float* m, float* v,
                                  int64_t* step, void* stream) {
    static const char* fn = "zs_checkpoint_load";
    zs::clear_error();
    if (!plan || !dir || !shards || !master || !m || !v) return fail(fn, "NULL argument");
    if (plan->layout != ZS_LAYOUT_FSDP1) return fail(fn, "only FSDP1-layout plans are supported", ZS_ERR_UNSUPPORTED);
    cudaStream_t st = (cudaStream_t)stream;
    const std::string d(dir);

    // ---- metadata
    std::ifstream meta(d + "/meta.txt");
    if (!meta) return fail(fn, "cannot read " + d + "/meta.txt");
    std::string tag;
    int version = 0, saved_nd = 0;
    int64_t saved_step = 0;
    size_t n_params = 0, n_units = 0;
    std::string key;
    meta >> tag >> version;
    if (tag != "zs-checkpoint" || version != 1) return fail(fn, "not a zs checkpoint (meta.txt)");
    meta >> key >> saved_nd;
    if (key != "n_d" || saved_nd < 1 || saved_nd > ZS_MAX_RANKS) return fail(fn, "bad n_d in meta.txt");
    meta >> key >> saved_step;
    if (key != "step") return fail(fn, "bad step in meta.txt");
    meta >> key >> n_params;
    if (key != "params" || n_params != plan->param_numel.size())
        return fail(fn, "the checkpoint holds another model (parameter count differs)");
    for (size_t k = 0; k < n_params; ++k) {
        std::string p, unit_kw;
        int64_t numel = -1;
        int unit = -1;
        meta >> p >> numel >> unit_kw >> unit;
        if (p != "p" || unit_kw != "unit") return fail(fn, "bad parameter line in meta.txt");
        if (numel != plan->param_numel[k] || unit != plan->param_unit[k])
            return fail(fn, "the checkpoint holds another model (parameter " + std::to_string(k) + " differs)");
    }
    meta >> key >> n_units;
    if (key != "units" || n_units != plan->units.size()) return fail(fn, "the checkpoint holds another unit layout");
    std::vector<SavedUnit> su(n_units);
    for (size_t u = 0; u < n_units; ++u) {
        std::string tagu;
        meta >> tagu >> su[u].numel >> su[u].padded >> su[u].shard;
        if (tagu != "u" || su[u].numel != plan->units[u].numel || su[u].shard * saved_nd != su[u].padded)
            return fail(fn, "bad unit line in meta.txt");
    }
    if (!meta) return fail(fn, "truncated meta.txt");
    int64_t saved_shard_total = 0;
    std::vector<int64_t> unit_off(n_units);
    for (size_t u = 0; u < n_units; ++u) {
        unit_off[u] = saved_shard_total;
        saved_shard_total += su[u].shard;
    }

    // ---- data
    void* dst[4] = {shards, master, m, v};
    std::vector<FILE*> files(saved_nd, nullptr);
    auto close_all = [&]() {
        for (auto f : files)
            if (f) std::fclose(f);
    };
    for (int r = 0; r < saved_nd; ++r) {
        files[r] = std::fopen(rank_file(d, r).c_str(), "rb");
        if (!files[r]) {
            close_all();
            return fail(fn, "cannot read " + rank_file(d, r));
        }
        int64_t want = 0;
        for (int a = 0; a < 4; ++a) want += saved_shard_total * kElemBytes[a];
        std::fseek(files[r], 0, SEEK_END);
        if ((int64_t)std::ftell(files[r]) != want) {
            close_all();
            return fail(fn, rank_file(d, r) + " has the wrong size");
        }
    }
    std::vector<char> buf(kChunk);
    int64_t section = 0;                                   // byte offset of array a inside a rank file
    for (int a = 0; a < 4; ++a) {
        const int eb = kElemBytes[a];
        for (size_t u = 0; u < n_units; ++u) {
            const zs::Unit& du = plan->units[u];
            char* base = (char*)dst[a] + (size_t)du.base * eb;
            // the target's padding is zero
            if (du.padded > du.numel) {
                cudaError_t e = cudaMemsetAsync(base + (size_t)du.numel * eb, 0, (size_t)(du.padded - du.numel) * eb, st);
                if (e != cudaSuccess) {
                    close_all();
                    return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
                }
            }
            // unit-local real element j sits in saved rank j / S_u at position j % S_u of its piece
            for (int r = 0; r < saved_nd; ++r) {
                const int64_t lo = (int64_t)r * su[u].shard;
                const int64_t hi = std::min(lo + su[u].shard, su[u].numel);
                if (hi <= lo) continue;
                if (std::fseek(files[r], (long)(section + unit_off[u] * eb), SEEK_SET) != 0) {
                    close_all();
                    return fail(fn, "seek failed in " + rank_file(d, r));
                }
                size_t left = (size_t)(hi - lo) * eb;
                char* to = base + (size_t)lo * eb;
                while (left) {
                    const size_t n = left < kChunk ? left : kChunk;
                    if (std::fread(buf.data(), 1, n, files[r]) != n) {
                        close_all();
                        return fail(fn, "short read from " + rank_file(d, r));
                    }
                    cudaError_t e = cudaMemcpyAsync(to, buf.data(), n, cudaMemcpyHostToDevice, st);
                    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
                    if (e != cudaSuccess) {
                        close_all();
                        return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
                    }
                    to += n;
                    left -= n;
                }
            }
        }
        section += saved_shard_total * eb;
    }
    close_all();
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
    if (step) *step = saved_step;
    return ZS_OK;
}
