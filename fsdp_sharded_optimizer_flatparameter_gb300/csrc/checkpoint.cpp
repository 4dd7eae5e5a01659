// Sharded checkpoint: every simulated rank writes its own shards; loading lays
// them out for any target plan - another rank count, unit grouping or layout.
//
// "Infra: Data Parallel" (F. Pu), section "Fully Sharded Data Parallel (FSDP)",
// subsection "Checkpoint": ranks write the shards they own plus the metadata
// needed to restore them; loading follows the target run's sharding layout, so
// save and load may use different numbers of ranks; optimizer state is saved
// with the weights; FSDP1 and FSDP2 layouts both support this.
//
// An element is identified by (parameter k, position e in the parameter's own
// row-major order); no layout, rank count or unit grouping changes that.  Each
// parameter's elements lie in a few runs that are contiguous both in one saved
// rank file and in the target's flat space (a run ends where either side moves
// to another rank); loading copies run by run and zeroes the target's padding.
//
// Files in `dir` (which must exist):
//   meta.txt          text: format tag and version, N_d, step, layout, per parameter
//                     (numel, rows of dim 0, unit), per unit (numel, padded, shard),
//                     the arrays and their element types
//   rank-NNNNN.bin    rank r's shard of params (bf16), master, m, v (fp32), one after
//                     another; each is the rank's piece of every unit, units in order
// Transfers: both calls first wait for the caller's stream, then cut the data
// into chunks of at most 16 MiB, each a contiguous byte range of one rank file
// and of one device array, and share them out among worker threads (up to 16,
// contiguous runs of chunks of equal total size, so each worker reads or writes
// its files mostly sequentially).  A worker owns a non-blocking stream and two
// pinned staging buffers: while it writes one chunk to its file with pwrite, the
// device-to-host copy of its next chunk runs (save); while the host-to-device
// copy of one chunk runs, it reads the next with pread (load).  The calls return
// once every worker's copies have completed.
#include <algorithm>
#include <atomic>
#include <cerrno>
#include <cstdio>
#include <cstring>
#include <fstream>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cuda_runtime.h>

#include "plan.h"

namespace {

constexpr size_t kChunk = size_t(16) << 20;            // bytes per transfer chunk (and per staging buffer)
constexpr int kMaxWorkers = 16;
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

// Where element e of parameter k lives in a layout: the rank, the position inside that rank's
// shard (all units concatenated), and how many following elements stay contiguous there.
struct Layout {
    int32_t n_d = 0, layout = 0;
    std::vector<int64_t> numel, d0, row, chunk, unit, off_in_unit;   // per parameter
    std::vector<int64_t> u_shard, u_local, u_base;                   // per unit
    void finish() {
        const size_t K = numel.size(), U = u_shard.size();
        row.resize(K);
        chunk.resize(K);
        off_in_unit.assign(K, 0);
        std::vector<int64_t> acc(U, 0);
        for (size_t k = 0; k < K; ++k) {
            row[k] = numel[k] / d0[k];
            chunk[k] = (d0[k] + n_d - 1) / n_d;
            off_in_unit[k] = acc[unit[k]];
            acc[unit[k]] += layout == ZS_LAYOUT_FSDP2 ? chunk[k] * row[k] : numel[k];
        }
        u_local.assign(U, 0);
        u_base.assign(U, 0);
        for (size_t u = 1; u < U; ++u) {
            u_local[u] = u_local[u - 1] + u_shard[u - 1];
            u_base[u] = u_base[u - 1] + u_shard[u - 1] * n_d;
        }
    }
    // (rank, position in the rank's shard, contiguous run length)
    void locate(size_t k, int64_t e, int32_t* rank, int64_t* pos, int64_t* run) const {
        const int64_t u = unit[k], S = u_shard[u];
        if (layout == ZS_LAYOUT_FSDP2) {
            const int64_t i = e / row[k], j = e % row[k];
            const int64_t r = i / chunk[k];
            *rank = (int32_t)r;
            *pos = u_local[u] + off_in_unit[k] + (i - r * chunk[k]) * row[k] + j;
            const int64_t rows_end = std::min((r + 1) * chunk[k], d0[k]);
            *run = rows_end * row[k] - e;
        } else {
            const int64_t x = off_in_unit[k] + e;           // index inside the unit's flat range
            const int64_t r = x / S;
            *rank = (int32_t)r;
            *pos = u_local[u] + (x - r * S);
            *run = std::min((r + 1) * S - x, numel[k] - e);
        }
    }
    // global flat index of (rank, position in the rank's shard)
    int64_t global(size_t k, int32_t rank, int64_t pos) const {
        const int64_t u = unit[k];
        return u_base[u] + (int64_t)rank * u_shard[u] + (pos - u_local[u]);
    }
};

// One chunk: `bytes` bytes between file descriptor `fd` at `off` and device address `dev`.
struct Xfer {
    int fd;
    int64_t off;
    char* dev;
    size_t bytes;
};

// Appends [off, off + bytes) <-> [dev, dev + bytes) as chunks of at most kChunk bytes, first
// growing the last chunk when the range continues it on both sides.
void add_chunks(std::vector<Xfer>& out, int fd, int64_t off, char* dev, size_t bytes) {
    if (bytes && !out.empty()) {
        Xfer& t = out.back();
        if (t.fd == fd && t.off + (int64_t)t.bytes == off && t.dev + t.bytes == dev && t.bytes < kChunk) {
            const size_t n = std::min(bytes, kChunk - t.bytes);
            t.bytes += n;
            off += (int64_t)n;
            dev += n;
            bytes -= n;
        }
    }
    while (bytes) {
        const size_t n = bytes < kChunk ? bytes : kChunk;
        out.push_back({fd, off, dev, n});
        off += (int64_t)n;
        dev += n;
        bytes -= n;
    }
}

bool full_pwrite(int fd, const char* p, size_t n, int64_t off) {
    while (n) {
        const ssize_t w = ::pwrite(fd, p, n, (off_t)off);
        if (w < 0 && errno == EINTR) continue;
        if (w <= 0) return false;
        p += w;
        n -= (size_t)w;
        off += w;
    }
    return true;
}

bool full_pread(int fd, char* p, size_t n, int64_t off) {
    while (n) {
        const ssize_t r = ::pread(fd, p, n, (off_t)off);
        if (r < 0 && errno == EINTR) continue;
        if (r <= 0) return false;
        p += r;
        n -= (size_t)r;
        off += r;
    }
    return true;
}

struct Failure {
    std::mutex mu;
    std::atomic<bool> any{false};
    std::string what;
    int code = ZS_OK;
    void set(const std::string& w, int c) {
        std::lock_guard<std::mutex> lock(mu);
        if (!any.load()) {
            what = w;
            code = c;
            any.store(true);
        }
    }
};

// One worker: chunks [lo, hi) of `xs`, device <-> file through two pinned buffers on its own stream.
void worker(const std::vector<Xfer>& xs, size_t lo, size_t hi, bool save, int device, Failure* fail) {
    if (lo >= hi) return;
    cudaStream_t st = nullptr;
    cudaEvent_t ev[2] = {nullptr, nullptr};
    char* buf[2] = {nullptr, nullptr};
    auto cuda_fail = [&](cudaError_t e) { fail->set(cudaGetErrorString(e), ZS_ERR_CUDA); };
    cudaError_t e = cudaSetDevice(device);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) e = cudaEventCreateWithFlags(&ev[b], cudaEventDisableTiming);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) e = cudaHostAlloc((void**)&buf[b], kChunk, cudaHostAllocDefault);
    if (e != cudaSuccess) cuda_fail(e);
    if (save) {
        // D2H of chunk i + 1 runs while chunk i is written out
        if (e == cudaSuccess) e = cudaMemcpyAsync(buf[0], xs[lo].dev, xs[lo].bytes, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaEventRecord(ev[0], st);
        if (e != cudaSuccess && !fail->any.load()) cuda_fail(e);
        for (size_t i = lo; i < hi && !fail->any.load(); ++i) {
            const int b = (int)((i - lo) & 1);
            if (i + 1 < hi) {
                const int nb = b ^ 1;          // its last chunk was written out in the previous iteration
                e = cudaMemcpyAsync(buf[nb], xs[i + 1].dev, xs[i + 1].bytes, cudaMemcpyDeviceToHost, st);
                if (e == cudaSuccess) e = cudaEventRecord(ev[nb], st);
                if (e != cudaSuccess) {
                    cuda_fail(e);
                    break;
                }
            }
            e = cudaEventSynchronize(ev[b]);
            if (e != cudaSuccess) {
                cuda_fail(e);
                break;
            }
            if (!full_pwrite(xs[i].fd, buf[b], xs[i].bytes, xs[i].off)) {
                fail->set(std::string("write failed: ") + std::strerror(errno), ZS_ERR_INVALID);
                break;
            }
        }
    } else {
        // pread of chunk i runs while the H2D copy of chunk i - 1 is in flight
        for (size_t i = lo; i < hi && e == cudaSuccess && !fail->any.load(); ++i) {
            const int b = (int)((i - lo) & 1);
            if (i - lo >= 2) {                 // the copy out of this buffer two chunks ago must be done
                e = cudaEventSynchronize(ev[b]);
                if (e != cudaSuccess) {
                    cuda_fail(e);
                    break;
                }
            }
            if (!full_pread(xs[i].fd, buf[b], xs[i].bytes, xs[i].off)) {
                fail->set("short read from a rank file", ZS_ERR_INVALID);
                break;
            }
            e = cudaMemcpyAsync(xs[i].dev, buf[b], xs[i].bytes, cudaMemcpyHostToDevice, st);
            if (e == cudaSuccess) e = cudaEventRecord(ev[b], st);
            if (e != cudaSuccess) cuda_fail(e);
        }
    }
    // every copy of this worker has completed before its buffers go
    if (st) {
        cudaError_t se = cudaStreamSynchronize(st);
        if (se != cudaSuccess) cuda_fail(se);
    }
    for (int b = 0; b < 2; ++b) {
        if (buf[b]) cudaFreeHost(buf[b]);
        if (ev[b]) cudaEventDestroy(ev[b]);
    }
    if (st) cudaStreamDestroy(st);
}

// Runs every chunk on up to kMaxWorkers threads; returns ZS_OK or the first failure (message set).
int transfer(const char* fn, const std::vector<Xfer>& xs, bool save) {
    if (xs.empty()) return ZS_OK;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
    unsigned hw = std::thread::hardware_concurrency();
    size_t W = std::min<size_t>({(size_t)kMaxWorkers, hw ? (size_t)hw : 1, xs.size()});
    uint64_t total = 0;
    for (const auto& x : xs) total += x.bytes;
    // contiguous runs of chunks with about total / W bytes each
    std::vector<size_t> cut(1, 0);
    uint64_t acc = 0;
    for (size_t i = 0; i < xs.size() && cut.size() < W; ++i) {
        acc += xs[i].bytes;
        if (acc * W >= total * cut.size()) cut.push_back(i + 1);
    }
    cut.push_back(xs.size());
    Failure f;
    std::vector<std::thread> threads;
    for (size_t w = 0; w + 1 < cut.size(); ++w)
        threads.emplace_back(worker, std::cref(xs), cut[w], cut[w + 1], save, device, &f);
    for (auto& t : threads) t.join();
    if (f.any.load()) return fail(fn, f.what, f.code);
    return ZS_OK;
}

Layout layout_of(zs_plan_t p) {
    Layout L;
    L.n_d = p->n_d;
    L.layout = p->layout;
    L.numel = p->param_numel;
    L.d0 = p->param_d0;
    L.unit.assign(p->param_unit.begin(), p->param_unit.end());
    for (const auto& u : p->units) L.u_shard.push_back(u.shard);
    L.finish();
    return L;
}

}  // namespace

extern "C" int zs_checkpoint_save(zs_plan_t plan, const char* dir, const void* shards, const float* master,
                                  const float* m, const float* v, int64_t step, void* stream) {
    static const char* fn = "zs_checkpoint_save";
    zs::clear_error();
    if (!plan || !dir || !shards || !master || !m || !v) return fail(fn, "NULL argument");
    if (step < 0) return fail(fn, "step must be >= 0 (the number of optimizer steps taken)");
    cudaStream_t st = (cudaStream_t)stream;
    const std::string d(dir);
    {
        cudaError_t e = cudaStreamSynchronize(st);   // the arrays as the caller's stream leaves them
        if (e != cudaSuccess) return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
    }
    {
        std::ofstream meta(d + "/meta.txt");
        if (!meta) return fail(fn, "cannot write " + d + "/meta.txt: " + std::strerror(errno));
        meta << "zs-checkpoint 2\n";
        meta << "n_d " << plan->n_d << "\n";
        meta << "step " << step << "\n";
        meta << "layout " << plan->layout << "\n";
        meta << "params " << plan->param_numel.size() << "\n";
        for (size_t k = 0; k < plan->param_numel.size(); ++k)
            meta << "p " << plan->param_numel[k] << " d0 " << plan->param_d0[k] << " unit " << plan->param_unit[k] << "\n";
        meta << "units " << plan->units.size() << "\n";
        for (const auto& u : plan->units) meta << "u " << u.numel << " " << u.padded << " " << u.shard << "\n";
        meta << "arrays params:bf16 master:f32 m:f32 v:f32\n";
        if (!meta) return fail(fn, "writing meta.txt failed");
    }
    const void* src[4] = {shards, master, m, v};
    std::vector<int> fds(plan->n_d, -1);
    auto close_all = [&]() {
        bool ok = true;
        for (int& fd : fds)
            if (fd >= 0) {
                ok = ::close(fd) == 0 && ok;
                fd = -1;
            }
        return ok;
    };
    std::vector<Xfer> xs;
    for (int r = 0; r < plan->n_d; ++r) {
        fds[r] = ::open(rank_file(d, r).c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
        if (fds[r] < 0) {
            const std::string why = std::strerror(errno);
            close_all();
            return fail(fn, "cannot write " + rank_file(d, r) + ": " + why);
        }
        int64_t off = 0;
        for (int a = 0; a < 4; ++a) {
            const int eb = kElemBytes[a];
            for (const auto& u : plan->units) {
                char* from = (char*)src[a] + (size_t)(u.base + (int64_t)r * u.shard) * eb;
                add_chunks(xs, fds[r], off, from, (size_t)u.shard * eb);
                off += u.shard * eb;
            }
        }
    }
    const int rc = transfer(fn, xs, true);
    if (!close_all() && rc == ZS_OK) return fail(fn, "closing a rank file failed");
    if (rc != ZS_OK) return rc;
    return ZS_OK;
}

extern "C" int zs_checkpoint_load(zs_plan_t plan, const char* dir, void* shards, float* master, float* m, float* v,
                                  int64_t* step, void* stream) {
    static const char* fn = "zs_checkpoint_load";
    zs::clear_error();
    if (!plan || !dir || !shards || !master || !m || !v) return fail(fn, "NULL argument");
    cudaStream_t st = (cudaStream_t)stream;
    const std::string d(dir);

    // ---- metadata of the save
    std::ifstream meta(d + "/meta.txt");
    if (!meta) return fail(fn, "cannot read " + d + "/meta.txt");
    std::string tag, key;
    int version = 0;
    int64_t saved_step = 0;
    size_t n_params = 0, n_units = 0;
    Layout S;
    meta >> tag >> version;
    if (tag != "zs-checkpoint" || version != 2) return fail(fn, "not a zs checkpoint of format 2 (meta.txt)");
    meta >> key >> S.n_d;
    if (key != "n_d" || S.n_d < 1 || S.n_d > ZS_MAX_RANKS) return fail(fn, "bad n_d in meta.txt");
    meta >> key >> saved_step;
    if (key != "step" || !meta || saved_step < 0) return fail(fn, "bad step in meta.txt");
    meta >> key >> S.layout;
    if (key != "layout" || (S.layout != ZS_LAYOUT_FSDP1 && S.layout != ZS_LAYOUT_FSDP2)) return fail(fn, "bad layout in meta.txt");
    meta >> key >> n_params;
    if (key != "params" || n_params != plan->param_numel.size())
        return fail(fn, "the checkpoint holds another model (parameter count differs)");
    S.numel.resize(n_params);
    S.d0.resize(n_params);
    S.unit.resize(n_params);
    for (size_t k = 0; k < n_params; ++k) {
        std::string p, d0_kw, unit_kw;
        meta >> p >> S.numel[k] >> d0_kw >> S.d0[k] >> unit_kw >> S.unit[k];
        if (p != "p" || d0_kw != "d0" || unit_kw != "unit") return fail(fn, "bad parameter line in meta.txt");
        if (S.numel[k] != plan->param_numel[k] || S.d0[k] != plan->param_d0[k])
            return fail(fn, "the checkpoint holds another model (parameter " + std::to_string(k) + " differs)");
    }
    meta >> key >> n_units;
    if (key != "units" || n_units < 1 || n_units > n_params) return fail(fn, "bad unit count in meta.txt");
    for (size_t k = 0; k < n_params; ++k)
        if (S.unit[k] < 0 || S.unit[k] >= (int64_t)n_units) return fail(fn, "bad unit id in meta.txt");
    S.u_shard.resize(n_units);
    for (size_t u = 0; u < n_units; ++u) {
        std::string tagu;
        int64_t numel = 0, padded = 0;
        meta >> tagu >> numel >> padded >> S.u_shard[u];
        if (tagu != "u" || S.u_shard[u] * S.n_d != padded) return fail(fn, "bad unit line in meta.txt");
    }
    if (!meta) return fail(fn, "truncated meta.txt");
    S.finish();
    // the saved layout must place every element inside its rank's unit piece
    for (size_t k = 0; k < n_params; ++k) {
        int64_t need = S.layout == ZS_LAYOUT_FSDP2 ? S.off_in_unit[k] + S.chunk[k] * S.row[k]
                                                   : (S.off_in_unit[k] + S.numel[k] + S.n_d - 1) / S.n_d;
        int64_t have = S.layout == ZS_LAYOUT_FSDP2 ? S.u_shard[S.unit[k]] : S.u_shard[S.unit[k]];
        if (need > have) return fail(fn, "meta.txt shard sizes do not fit its parameters");
    }
    int64_t saved_shard_total = 0;
    for (auto x : S.u_shard) saved_shard_total += x;
    const Layout D = layout_of(plan);

    // ---- files
    std::vector<int> fds(S.n_d, -1);
    auto close_all = [&]() {
        for (int& fd : fds)
            if (fd >= 0) {
                ::close(fd);
                fd = -1;
            }
    };
    for (int r = 0; r < S.n_d; ++r) {
        fds[r] = ::open(rank_file(d, r).c_str(), O_RDONLY);
        if (fds[r] < 0) {
            close_all();
            return fail(fn, "cannot read " + rank_file(d, r));
        }
        int64_t want = 0;
        for (int a = 0; a < 4; ++a) want += saved_shard_total * kElemBytes[a];
        struct stat sb;
        if (::fstat(fds[r], &sb) != 0 || (int64_t)sb.st_size != want) {
            close_all();
            return fail(fn, rank_file(d, r) + " has the wrong size");
        }
    }

    // ---- data: padding of the target first, then every parameter run by run
    void* dst[4] = {shards, master, m, v};
    std::vector<int64_t> pad_b, pad_e;
    {
        int64_t count = 0;
        zs_plan_pad_ranges(plan, nullptr, nullptr, 0, &count);
        pad_b.resize(count + 1);
        pad_e.resize(count + 1);
        zs_plan_pad_ranges(plan, pad_b.data(), pad_e.data(), count, &count);
        pad_b.resize(count);
        pad_e.resize(count);
    }
    {
        cudaError_t e = cudaStreamSynchronize(st);   // the caller's work on the arrays is done
        if (e != cudaSuccess) {
            close_all();
            return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
        }
    }
    std::vector<Xfer> xs;
    int64_t section = 0;                                   // byte offset of array a inside a rank file
    for (int a = 0; a < 4; ++a) {
        const int eb = kElemBytes[a];
        for (size_t i = 0; i < pad_b.size(); ++i) {
            cudaError_t e = cudaMemsetAsync((char*)dst[a] + (size_t)pad_b[i] * eb, 0, (size_t)(pad_e[i] - pad_b[i]) * eb, st);
            if (e != cudaSuccess) {
                close_all();
                return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
            }
        }
        for (size_t k = 0; k < n_params; ++k) {
            for (int64_t e0 = 0; e0 < S.numel[k];) {
                int32_t rs, rd;
                int64_t ps, pd, ls, ld;
                S.locate(k, e0, &rs, &ps, &ls);
                D.locate(k, e0, &rd, &pd, &ld);
                const int64_t len = std::min(ls, ld);
                add_chunks(xs, fds[rs], section + ps * eb, (char*)dst[a] + (size_t)D.global(k, rd, pd) * eb,
                           (size_t)len * eb);
                e0 += len;
            }
        }
        section += saved_shard_total * eb;
    }
    const int rc = transfer(fn, xs, false);
    close_all();
    cudaError_t e = cudaStreamSynchronize(st);             // the padding memsets
    if (rc != ZS_OK) return rc;
    if (e != cudaSuccess) return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
    if (step) *step = saved_step;
    return ZS_OK;
}
