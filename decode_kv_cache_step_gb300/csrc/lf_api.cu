// C-ABI entry points of the LongFlow decode-step library: argument checks,
// split planning, scratch management, TMA descriptors and launches.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>  // header-only; ranges are free unless a profiler is attached

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "../../include/lf_decode.h"
#include "lf_kernels.h"

namespace {

constexpr int kVersion = 100;  // 0.1.0

// The header's step flags are the kernel's flag bits.
static_assert(LF_STEP_FILL_EMPTY_FIRST == lf::kFlagFillEmptyFirst &&
                  LF_STEP_MASK_EVICTED == lf::kFlagMaskEvicted &&
                  LF_STEP_LOG2_SCORES == lf::kFlagLog2Scores,
              "step flag bits");
constexpr int kMaxNChunk = 1024;
constexpr int kMaxS = 1 << 20;

thread_local char g_last_error[512] = "";

lf_status fail(lf_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

lf_status cuda_fail(cudaError_t e, const char* what) {
    return fail(LF_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ----------------------------------------------------------------- scratch --

struct Scratch {
    void* base = nullptr;
    size_t bytes = 0;
    uint32_t* dev_err = nullptr;   // never moves once created
    // Per unit, zero between steps: the decode-step kernel's chunk arrival
    // counters [units], the scoring kernel's [units], its 64-bit argmin
    // words [units], the ready flags [units] (lf::kCounterWordsPerUnit
    // words per unit in all).
    uint32_t* arrivals = nullptr;
    size_t arrivals_len = 0;
};

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, Scratch> g_scratch;

lf_status get_scratch(int dev, cudaStream_t stream, size_t need, size_t units, Scratch** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    Scratch& s = g_scratch[{dev, stream}];
    if (s.arrivals_len < units) {
        if (s.arrivals) {
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
            cudaFree(s.arrivals);
            s.arrivals = nullptr;
            s.arrivals_len = 0;
        }
        const size_t words = lf::kCounterWordsPerUnit * units;
        cudaError_t e = cudaMalloc(&s.arrivals, words * sizeof(uint32_t));
        if (e != cudaSuccess) return fail(LF_ERR_NO_MEMORY, "cudaMalloc(arrival counters): %s", cudaGetErrorString(e));
        e = cudaMemset(s.arrivals, 0, words * sizeof(uint32_t));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
        s.arrivals_len = units;
    }
    if (!s.dev_err) {
        cudaError_t e = cudaMalloc(&s.dev_err, 256);
        if (e != cudaSuccess) return fail(LF_ERR_NO_MEMORY, "cudaMalloc(error word): %s", cudaGetErrorString(e));
        e = cudaMemset(s.dev_err, 0, 256);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
    }
    if (s.bytes < need) {
        if (s.base) {
            // Work already queued on this stream may still use the old buffer.
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
            cudaFree(s.base);
            s.base = nullptr;
            s.bytes = 0;
        }
        const size_t grow = align_up(need + need / 8, size_t(1) << 21);
        cudaError_t e = cudaMalloc(&s.base, grow);
        if (e != cudaSuccess) {
            s.base = nullptr;
            return fail(LF_ERR_NO_MEMORY, "cudaMalloc(%zu bytes of scratch): %s", grow, cudaGetErrorString(e));
        }
        s.bytes = grow;
    }
    *out = &s;
    return LF_OK;
}

// ----------------------------------------------------------------- profile --

struct ProfRec {
    int kernel;
    cudaEvent_t start, stop;
};

std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

struct ProfScope {
    int kernel;
    cudaStream_t stream;
    cudaEvent_t start = nullptr, stop = nullptr;
    ProfScope(int k, cudaStream_t s) : kernel(k), stream(s) {
        std::lock_guard<std::mutex> lock(g_prof_mu);
        if (!g_prof_on) return;
        start = take_event();
        stop = take_event();
        if (start) cudaEventRecord(start, stream);
    }
    ~ProfScope() {
        if (!start || !stop) return;
        cudaEventRecord(stop, stream);
        std::lock_guard<std::mutex> lock(g_prof_mu);
        g_prof.push_back({kernel, start, stop});
    }
};

// Counts a launch under `kernel` without events of its own (its time is
// inside an enclosing ProfScope).
void prof_count(int kernel) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (g_prof_on) g_prof.push_back({kernel, nullptr, nullptr});
}

// ------------------------------------------------------------- device info --

int sm_count(int dev) {
    static std::mutex mu;
    static std::map<int, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cache[dev] = n;
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [units][S][D] bf16 as a 3-D tensor map, 64 x 64 x 1 boxes, 128-byte swizzle.
lf_status encode_cache_map_uncached(CUtensorMap* m, void* base, int D, int S, int units) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(LF_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                          static_cast<cuuint64_t>(units)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(S) * static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(lf::kBoxCols), static_cast<cuuint32_t>(lf::kTile), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LF_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
    return LF_OK;
}

// A tensor map is a pure function of (base, D, S, units), so the maps of the
// caches a caller steps over are kept (a small round-robin table) instead of
// being encoded again at every call.
struct MapKey {
    void* base;
    int D, S, units;
    bool operator==(const MapKey& o) const {
        return base == o.base && D == o.D && S == o.S && units == o.units;
    }
};
constexpr int kMapCacheSize = 64;
std::mutex g_map_mu;
MapKey g_map_keys[kMapCacheSize] = {};
CUtensorMap g_maps[kMapCacheSize];
int g_map_next = 0;

lf_status encode_cache_map(CUtensorMap* m, void* base, int D, int S, int units) {
    const MapKey k{base, D, S, units};
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        for (int i = 0; i < kMapCacheSize; ++i)
            if (g_map_keys[i].base && g_map_keys[i] == k) {
                *m = g_maps[i];
                return LF_OK;
            }
    }
    lf_status st = encode_cache_map_uncached(m, base, D, S, units);
    if (st != LF_OK) return st;
    std::lock_guard<std::mutex> lock(g_map_mu);
    g_map_keys[g_map_next] = k;
    g_maps[g_map_next] = *m;
    g_map_next = (g_map_next + 1) % kMapCacheSize;
    return LF_OK;
}

// Limit of the kernel's pipeline waits: 1 s, or LF_WAIT_LIMIT_NS (a
// diagnostic that makes the waits give up early, to exercise the timeout path).
uint64_t wait_limit_ns() {
    if (const char* env = std::getenv("LF_WAIT_LIMIT_NS")) {
        const long long v = std::atoll(env);
        if (v > 0) return static_cast<uint64_t>(v);
    }
    return 1000000000ull;
}

// ---------------------------------------------------------------- planning --

struct Plan {
    int tiles, chunk_tiles, nchunk, stages;
    bool cluster;  // the unit's chunks run as one thread-block cluster
    bool split;    // a top-1 step scores in a second kernel (split finish)
    int split_from = 0;  // with split: units below this still scan in their last CTA
    int fit = 0;   // clusters that can be resident at once: of the plan's size with a
                   // cluster merge, else of the largest size tried (-1: not considered)
};

// Units of at least this many slots take the split finish.
constexpr int kSplitMinSlots = 8192;

// Largest cluster the plan tries by default: 16 CTAs, a non-portable size
// (smaller ones are tried where it cannot be placed).
constexpr int kDefaultClusterChunks = 16;

// Split the slot axis of every unit into nchunk chunks of chunk_tiles tiles.
// Each CTA costs a fixed start-up and merge, so chunks stay long (13 to 32
// tiles) while the grid still has about 27 CTAs per SM (about 4100), the
// chunk count rounded down, to balance the tail (measured: 4 chunks of 13
// tiles beat 3 of 17 on the Fig. 1 shape by 1 us per step, 2 chunks of 19
// beat 3 of 13 on the 2400-slot ragged batch); units long enough for the
// split finish, which has no last-CTA scan on the tail, aim at 16 tiles
// (measured on 8 sequences of 16K slots: 16 chunks of 16 tiles 75.6 us per
// step against 80.5 for 20 of 13). A batch too small to fill the GPU that
// way uses short chunks of about 5 tiles instead. At most kMaxChunkTiles
// tiles and kMaxNChunk chunks.
Plan plan_split(int S, int units, int sms, bool want_cluster, int D, int G, bool score) {
    Plan pl;
    pl.tiles = (S + lf::kTile - 1) / lf::kTile;
    int nchunk = 0;
    if (const char* env = std::getenv("LF_CHUNK_TILES")) {
        const int ct = std::atoi(env);
        if (ct >= 1 && ct <= lf::kMaxChunkTiles) nchunk = (pl.tiles + ct - 1) / ct;
    }
    const bool forced_chunks = nchunk > 0;
    if (nchunk == 0) {
        const int longest = (pl.tiles + lf::kMaxChunkTiles - 1) / lf::kMaxChunkTiles;
        const int fill = static_cast<int>((27L * sms) / units);
        const int target = S >= kSplitMinSlots ? 16 : 13;
        if (static_cast<long>(units) * longest >= sms)
            nchunk = std::max(longest, std::min(fill, (pl.tiles + target - 1) / target));
        else
            nchunk = (pl.tiles + 4) / 5;
    }
    nchunk = std::max(nchunk, (pl.tiles + lf::kMaxChunkTiles - 1) / lf::kMaxChunkTiles);
    nchunk = std::min(std::max(nchunk, 1), std::min(pl.tiles, kMaxNChunk));
    pl.chunk_tiles = (pl.tiles + nchunk - 1) / nchunk;
    pl.nchunk = (pl.tiles + pl.chunk_tiles - 1) / pl.chunk_tiles;
    pl.stages = 2;
    if (const char* env = std::getenv("LF_STAGES")) pl.stages = (std::atoi(env) == 3) ? 3 : 2;
    // A grid whose clusters (one per unit, of at most cmax chunks) are all
    // resident at once merges inside thread-block clusters: the
    // latency-bound small batches gain the shorter merge. Larger grids keep
    // the last-CTA merge, where a finished CTA frees its slot at once instead
    // of waiting for its cluster (measured with clusters forced on the full
    // batches, same chunks, per step: the Fig. 1 shape 264.8 us against
    // 240.4, the ragged 2400-slot batch 269.0 against 234.7, the 16K-slot
    // workload 284.9 against 193.4). A cluster must sit within one GPC, so how
    // many fit at once comes from the occupancy query, not the SM count
    // (measured: 16 clusters of 8 one-per-SM CTAs, 128 of 152 SMs, took two
    // waves: 21.6 us per step against 10.4 for one cluster).
    // A step of such a grid is a chain of round trips that shortens with the
    // chunk, so among the splits whose clusters all fit the plan takes, for
    // each TMA ring, the one with the most chunks: the 2-stage ring at three
    // CTAs per SM, and the kDeepStages ring at one CTA per SM, which keeps
    // every tile of a short chunk in flight. Of the two it takes the shorter
    // modelled chain, about 0.55 us per tile of chunk on the deep ring and
    // 0.9 us per tile plus 0.9 on the 2-stage ring. Measured per step: one
    // 2400-slot Qwen3 sequence 7.7 us in 10 chunks of 4 tiles on the deep
    // ring, 9.1 in 13 of 3 on the 2-stage ring, 8.4 in 8 of 5 on the deep
    // ring; two ragged 2400-slot sequences 9.6 us in 13 of 3 on the 2-stage
    // ring against 10.3 in 5 of 8 on the deep ring; the 3200-slot Qwen3 shape
    // at batch 8, 6 chunks of 9 tiles in clusters 20.2 us against 30.8 for
    // the last-CTA merge over 10 of 5.
    // LF_CLUSTER=0 turns clusters off, =1 forces them whenever one cluster of
    // the split can be placed; LF_DEEP=0 keeps the 2-stage ring, =1 takes the
    // deep ring whenever its clusters all fit.
    pl.cluster = false;
    const char* cenv = std::getenv("LF_CLUSTER");
    const int cmode = cenv ? std::atoi(cenv) : -1;
    int cmax = kDefaultClusterChunks;
    if (const char* env = std::getenv("LF_CLUSTER_MAX"))
        cmax = std::min(std::max(std::atoi(env), 2), lf::kMaxClusterChunks);
    const char* denv = std::getenv("LF_DEEP");
    const int dmode = denv ? std::atoi(denv) : -1;
    pl.fit = -1;
    if (want_cluster && pl.stages == 2 && cmode != 0 && pl.tiles <= cmax * lf::kMaxChunkTiles) {
        struct Split {
            int ct = 0, nc = 0, fit = 0;
        };
        Split two, deep, first;
        // Splits by decreasing chunk count; a forced split (LF_CHUNK_TILES)
        // is the only one tried.
        const int n_hi = forced_chunks ? pl.nchunk : std::min(cmax, pl.tiles);
        for (int n0 = n_hi; n0 >= 1; --n0) {
            const int ct = (pl.tiles + n0 - 1) / n0;
            if (ct > lf::kMaxChunkTiles) break;
            const int nc = (pl.tiles + ct - 1) / ct;
            if (nc != n0) continue;  // the same split as a larger n0
            if (nc <= cmax) {
                const int f2 = lf::max_active_clusters(D, G, 2, score, nc);
                if (first.nc == 0) first = {ct, nc, f2};
                if (two.nc == 0 && units <= f2) two = {ct, nc, f2};
                // (The deep ring keeps a chunk's score terms in shared memory,
                // which bounds its chunk.)
                if (dmode != 0 && deep.nc == 0 &&
                    (!score || ct * lf::kTile <= lf::deep_term_slots(D, G))) {
                    const int fd = lf::max_active_clusters(D, G, lf::kDeepStages, score, nc);
                    if (units <= fd) deep = {ct, nc, fd};
                }
            }
            if (forced_chunks || (two.nc != 0 && (deep.nc != 0 || dmode == 0))) break;
        }
        Split pick;
        bool take_deep = false;
        if (deep.nc != 0 && (dmode == 1 || two.nc == 0 || 55 * deep.ct <= 90 * two.ct + 90)) {
            pick = deep;
            take_deep = true;
        } else if (two.nc != 0) {
            pick = two;
        } else if (cmode == 1 && first.fit > 0) {
            pick = first;  // forced: clusters in more than one wave
        }
        pl.fit = first.fit;
        if (pick.nc != 0) {
            pl.chunk_tiles = pick.ct;
            pl.nchunk = pick.nc;
            pl.cluster = true;
            pl.fit = pick.fit;
            if (take_deep) pl.stages = lf::kDeepStages;
        }
    }
    // Top-1 steps over long units without clusters score in a second kernel:
    // the last CTA's scan of every slot would otherwise run on the step's
    // tail at one SM's share of the memory system. LF_SPLIT=0 / 1 forces it
    // off / on (on: for every top-1 step without clusters).
    const char* senv = std::getenv("LF_SPLIT");
    const int smode = senv ? std::atoi(senv) : -1;
    pl.split = want_cluster && !pl.cluster && smode != 0 && (smode == 1 || S >= kSplitMinSlots);
    // A split grid of many waves merges its first units long before the
    // scoring kernel can start (it starts with the decode grid's last wave),
    // and by then their score terms have left L2. So the first 3/8 of the
    // units still scan in their last CTA while their terms are in L2, and
    // the scoring kernel takes the rest (measured on the 16K-slot workload,
    // 256 units of 16 chunks, about 9 waves; us per step, per event pair:
    // every unit split 199.6, the last 224 / 192 / 160 / 128 / 96 units
    // split 199.4 / 198.6 / 198.3 / 198.4 / 198.9). LF_SPLIT_TAIL sets how
    // many of the last units the scoring kernel takes.
    pl.split_from = 0;
    if (pl.split) {
        const long long ctas = static_cast<long long>(units) * pl.nchunk;
        if (ctas >= 4LL * 3 * sms) pl.split_from = units * 3 / 8;
        if (const char* env = std::getenv("LF_SPLIT_TAIL"))
            pl.split_from = std::max(0, units - std::max(1, std::atoi(env)));
    }
    return pl;
}

// ---------------------------------------------------------------- checking --

struct Shape {
    int B, Hq, Hkv, d, S, W;
    float scale;
};

lf_status check_shape(const Shape& s) {
    if (s.B < 1 || s.Hq < 1 || s.Hkv < 1 || s.d < 1 || s.S < 1)
        return fail(LF_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d Hq=%d Hkv=%d d=%d S=%d)", s.B, s.Hq, s.Hkv, s.d, s.S);
    if (s.Hq % s.Hkv != 0) return fail(LF_ERR_INVALID_ARG, "Hq (%d) is not a multiple of Hkv (%d)", s.Hq, s.Hkv);
    if (s.W < 0) return fail(LF_ERR_INVALID_ARG, "W must be >= 0 (got %d)", s.W);
    if (!std::isfinite(s.scale)) return fail(LF_ERR_INVALID_ARG, "scale must be finite");
    if (s.d != 64 && s.d != 128) return fail(LF_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", s.d);
    const int g = s.Hq / s.Hkv;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return fail(LF_ERR_UNSUPPORTED, "group size Hq/Hkv = %d (supported: 1, 2, 4, 8)", g);
    if (s.S > kMaxS) return fail(LF_ERR_UNSUPPORTED, "S = %d exceeds %d", s.S, kMaxS);
    if (static_cast<long>(s.B) * s.Hkv > 65535)
        return fail(LF_ERR_UNSUPPORTED, "B * Hkv = %ld exceeds 65535", static_cast<long>(s.B) * s.Hkv);
    return LF_OK;
}

lf_status check_ptr(const void* p, size_t align, const char* name) {
    if (!p) return fail(LF_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, align)) return fail(LF_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
    return LF_OK;
}

struct StepArgs {
    const void* q;
    void* k_cache;
    void* v_cache;
    int32_t* mask;
    const void* new_k;
    const void* new_v;
    const int32_t* write_slot;
    void* out;
    int32_t* next_slot;
    float* scores;
    int topk = 1;        // slots returned per unit into next_slot[B][Hkv][topk]
    int flags = 0;       // LF_STEP_* bits
    bool score = true;   // false: attention only (no score, no eviction, no ageing)
};

lf_status check_args(const StepArgs& a, const Shape& s) {
    lf_status st;
    if ((st = check_ptr(a.q, 16, "q")) != LF_OK) return st;
    if ((st = check_ptr(a.k_cache, 16, "k_cache")) != LF_OK) return st;
    if ((st = check_ptr(a.v_cache, 16, "v_cache")) != LF_OK) return st;
    if ((st = check_ptr(a.mask, 4, "mask")) != LF_OK) return st;
    if ((st = check_ptr(a.new_k, 16, "new_k")) != LF_OK) return st;
    if ((st = check_ptr(a.new_v, 16, "new_v")) != LF_OK) return st;
    if ((st = check_ptr(a.write_slot, 4, "write_slot")) != LF_OK) return st;
    if ((st = check_ptr(a.out, 16, "out")) != LF_OK) return st;
    if (a.score && (st = check_ptr(a.next_slot, 4, "next_slot")) != LF_OK) return st;
    if (a.scores && !aligned(a.scores, 4)) return fail(LF_ERR_INVALID_ARG, "scores is not 4-byte aligned");
    if (a.topk < 1 || a.topk > LF_MAX_TOPK)
        return fail(LF_ERR_INVALID_ARG, "k = %d is outside [1, %d]", a.topk, LF_MAX_TOPK);
    if (a.flags & ~(LF_STEP_FILL_EMPTY_FIRST | LF_STEP_MASK_EVICTED | LF_STEP_LOG2_SCORES))
        return fail(LF_ERR_INVALID_ARG, "unknown flag bits 0x%x", a.flags);
    return check_shape(s);
}

struct Layout {
    size_t ml, o, stash, cfold, tiles, total;
};

Layout scratch_layout(const Shape& s, const Plan& pl, size_t extra) {
    const size_t units = static_cast<size_t>(s.B) * s.Hkv;
    const size_t g = static_cast<size_t>(s.Hq / s.Hkv);
    Layout L;
    L.ml = 0;
    L.o = align_up(L.ml + units * pl.nchunk * g * sizeof(float2), 256);
    L.stash = align_up(L.o + units * pl.nchunk * g * s.d * sizeof(float), 256);
    L.cfold = align_up(L.stash + units * static_cast<size_t>(s.S) * g * sizeof(float), 256);
    L.tiles = align_up(L.cfold + units * g * sizeof(float), 256);
    L.total = align_up(L.tiles + units * pl.nchunk * sizeof(uint32_t), 256) + extra;
    return L;
}

// Enqueue one step. Arguments are already checked.
// Everything one step's launches need, resolved from the arguments, the
// scratch and the plan.
struct Launch {
    lf::StepParams sp;
    CUtensorMap tmK, tmV;
    Plan pl;
    int d, g, units;
    bool score;
};

lf_status build_launch(const StepArgs& a, const Shape& s, char* base, uint32_t* arrivals,
                       uint32_t* dev_err, const Layout& L, const Plan& pl, Launch* out) {
    const int units = s.B * s.Hkv;
    const int g = s.Hq / s.Hkv;
    Launch& r = *out;
    lf_status st = encode_cache_map(&r.tmK, a.k_cache, s.d, s.S, units);
    if (st != LF_OK) return st;
    if ((st = encode_cache_map(&r.tmV, a.v_cache, s.d, s.S, units)) != LF_OK) return st;
    lf::StepParams& sp = r.sp;
    sp = lf::StepParams{};
    sp.q = static_cast<const __nv_bfloat16*>(a.q);
    sp.k_cache = static_cast<__nv_bfloat16*>(a.k_cache);
    sp.v_cache = static_cast<__nv_bfloat16*>(a.v_cache);
    sp.mask = a.mask;
    sp.new_k = static_cast<const __nv_bfloat16*>(a.new_k);
    sp.new_v = static_cast<const __nv_bfloat16*>(a.new_v);
    sp.write_slot = a.write_slot;
    sp.out = static_cast<__nv_bfloat16*>(a.out);
    sp.next_slot = a.next_slot;
    sp.scores = a.scores;
    sp.part_o = reinterpret_cast<float*>(base + L.o);
    sp.part_ml = reinterpret_cast<float2*>(base + L.ml);
    sp.stash = reinterpret_cast<float*>(base + L.stash);
    sp.arrivals = arrivals;
    sp.dev_err = dev_err;
    sp.cfold = reinterpret_cast<float*>(base + L.cfold);
    sp.part_tiles = reinterpret_cast<uint32_t*>(base + L.tiles);
    sp.score_arrivals = arrivals + units;
    sp.best = reinterpret_cast<unsigned long long*>(arrivals + 2 * static_cast<size_t>(units));
    sp.ready = arrivals + 4 * static_cast<size_t>(units);
    sp.Hq = s.Hq;
    sp.Hkv = s.Hkv;
    sp.S = s.S;
    sp.W = s.W;
    sp.nchunk = pl.nchunk;
    sp.chunk_tiles = pl.chunk_tiles;
    sp.scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
    sp.wait_limit_ns = wait_limit_ns();
    sp.topk = a.score ? a.topk : 1;
    sp.flags = a.score ? a.flags : 0;
    sp.split = (a.score && pl.split && sp.topk == 1) ? 1 : 0;
    sp.split_from = sp.split ? pl.split_from : 0;
    if (!lf::step_fits(s.d, g, pl.stages, a.score, pl.nchunk, sp.topk))
        return fail(LF_ERR_UNSUPPORTED,
                    "k = %d with %d chunks of the slot axis does not fit in shared memory",
                    sp.topk, pl.nchunk);
    r.pl = pl;
    r.d = s.d;
    r.g = g;
    r.units = units;
    r.score = a.score;
    return LF_OK;
}

lf_status launch(const Launch& r, cudaStream_t stream) {
    // A named range around each launch for timeline profilers (nsys).
    struct NvtxRange {
        explicit NvtxRange(const char* n) { nvtxRangePushA(n); }
        ~NvtxRange() { nvtxRangePop(); }
    };
    cudaError_t e;
    // A split finish's two launches are one event pair (LF_KERNEL_DECODE_STEP):
    // an event recorded between them would end the programmatic dependency
    // that lets the scoring kernel start during the decode-step kernel's
    // tail. The scoring launch is counted under LF_KERNEL_SCORE.
    NvtxRange range(r.score ? "lf_decode_step" : "lf_decode_attention");
    ProfScope prof(r.score ? LF_KERNEL_DECODE_STEP : LF_KERNEL_ATTENTION, stream);
    const bool cluster = r.pl.cluster && r.sp.topk == 1;
    e = lf::launch_decode_step(r.d, r.g, r.pl.stages, r.score, cluster, r.tmK, r.tmV, r.sp,
                               r.units, stream);
    if (e != cudaSuccess && cluster) {
        // A cluster that cannot be scheduled: the last-CTA merge, scoring
        // in the same kernel.
        (void)cudaGetLastError();
        e = lf::launch_decode_step(r.d, r.g, 2, r.score, false, r.tmK, r.tmV, r.sp, r.units,
                                   stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode-step launch");
    if (r.sp.split) {
        prof_count(LF_KERNEL_SCORE);
        e = lf::launch_score(r.g, r.sp, r.units, stream);
        if (e != cudaSuccess) return cuda_fail(e, "scoring-kernel launch");
    }
    return LF_OK;
}

lf_status enqueue_step(const StepArgs& a, const Shape& s, cudaStream_t stream, Scratch* scr,
                       const Layout& L, const Plan& pl) {
    Launch r;
    lf_status st = build_launch(a, s, static_cast<char*>(scr->base), scr->arrivals, scr->dev_err,
                                L, pl, &r);
    if (st != LF_OK) return st;
    return launch(r, stream);
}

lf_status run_step(const StepArgs& a, const Shape& s, void* stream_v) {
    lf_status st = check_args(a, s);
    if (st != LF_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const Plan pl = plan_split(s.S, s.B * s.Hkv, sm_count(dev), a.topk == 1, s.d, s.Hq / s.Hkv,
                               a.score);
    const Layout L = scratch_layout(s, pl, 0);
    Scratch* scr = nullptr;
    if ((st = get_scratch(dev, stream, L.total, static_cast<size_t>(s.B) * s.Hkv, &scr)) != LF_OK) return st;
    g_last_error[0] = '\0';
    return enqueue_step(a, s, stream, scr, L, pl);
}

// ------------------------------------------------- static scratch variant --
//
// lf_decode_step_noalloc runs the same decode-step kernel with its scratch
// (softmax partials, per-slot score terms, arrival counters, error word) in
// this fixed device array instead of memory from cudaMalloc. Every device that
// loads this library holds the array until the process exits. In host code
// the name is only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, once per device, with that device current.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
// The array's last 256 bytes hold the entry point's device error word. It
// starts at zero with the module, every call ORs into it and none clears it;
// lf_device_errors reads (and may clear) it.
constexpr size_t kStaticErrOff = kStaticScratchBytes - 256;

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_base[kMaxDevices] = {};

lf_status static_scratch_base(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(LF_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_base[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_static_base[dev] = p;
    }
    *out = g_static_base[dev];
    return LF_OK;
}

}  // namespace

// ------------------------------------------------------- prepared steps --
//
// A prepared step fixes the buffers, shape and launch plan once: each run is
// the staging copies it needs, one or two kernel launches and the copies
// back, with no argument checks, plan, tensor-map lookup or pointer query.
// The handle owns its scratch, counters and error word, so runs of different
// handles never share state.

struct lf_step_handle {
    int dev = 0;
    cudaStream_t stream = nullptr;
    Launch r;
    void* mem = nullptr;        // scratch, then staging for I/O buffers not addressable in place
    uint32_t* words = nullptr;  // counter words (lf::kCounterWordsPerUnit per unit), then the error word
    uint32_t* dev_err = nullptr;
    struct Copy {
        void* dst;
        const void* src;
        size_t bytes;
    };
    Copy h2d[4];
    int n_h2d = 0;
    Copy d2h[2];
    int n_d2h = 0;
};

namespace {

void free_handle(lf_step_handle* h) {
    if (h->mem) cudaFree(h->mem);
    if (h->words) cudaFree(h->words);
    delete h;
}

}  // namespace

extern "C" {

lf_status lf_decode_step(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                         const void* new_k, const void* new_v, const int32_t* write_slot,
                         void* out, int32_t* next_slot, int B, int Hq, int Hkv, int d, int S,
                         int W, float scale, void* stream) {
    StepArgs a{q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot, nullptr};
    return run_step(a, Shape{B, Hq, Hkv, d, S, W, scale}, stream);
}

lf_status lf_decode_step_scores(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                                const void* new_k, const void* new_v,
                                const int32_t* write_slot, void* out, int32_t* next_slot,
                                float* scores, int B, int Hq, int Hkv, int d, int S, int W,
                                float scale, void* stream) {
    if (!scores) return fail(LF_ERR_INVALID_ARG, "scores is NULL");
    StepArgs a{q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot, scores};
    return run_step(a, Shape{B, Hq, Hkv, d, S, W, scale}, stream);
}

lf_status lf_decode_step_ex(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                            const void* new_k, const void* new_v, const int32_t* write_slot,
                            void* out, int32_t* next_slots, int k, int flags, float* scores,
                            int B, int Hq, int Hkv, int d, int S, int W, float scale,
                            void* stream) {
    StepArgs a{q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slots, scores};
    a.topk = k;
    a.flags = flags;
    return run_step(a, Shape{B, Hq, Hkv, d, S, W, scale}, stream);
}

lf_status lf_decode_attention(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                              const void* new_k, const void* new_v, const int32_t* write_slot,
                              void* out, int B, int Hq, int Hkv, int d, int S, float scale,
                              void* stream) {
    StepArgs a{q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, nullptr, nullptr};
    a.score = false;
    return run_step(a, Shape{B, Hq, Hkv, d, S, 0, scale}, stream);
}

lf_status lf_decode_step_host(const void* q_host, void* k_cache, void* v_cache, int32_t* mask,
                              const void* new_k_host, const void* new_v_host,
                              const int32_t* write_slot_host, void* out_host,
                              int32_t* next_slot_host, int B, int Hq, int Hkv, int d, int S,
                              int W, float scale, void* stream_v) {
    const Shape s{B, Hq, Hkv, d, S, W, scale};
    // Host buffers need no device alignment; the device staging copies are aligned.
    lf_status st;
    if (!q_host || !new_k_host || !new_v_host || !write_slot_host || !out_host || !next_slot_host)
        return fail(LF_ERR_INVALID_ARG, "a host buffer is NULL");
    if ((st = check_ptr(k_cache, 16, "k_cache")) != LF_OK) return st;
    if ((st = check_ptr(v_cache, 16, "v_cache")) != LF_OK) return st;
    if ((st = check_ptr(mask, 4, "mask")) != LF_OK) return st;
    if ((st = check_shape(s)) != LF_OK) return st;

    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const size_t units = static_cast<size_t>(B) * Hkv;
    const size_t q_bytes = static_cast<size_t>(B) * Hq * d * 2;
    const size_t kv_bytes = units * d * 2;
    const size_t i_bytes = units * 4;
    size_t off_q = 0, off_k = align_up(off_q + q_bytes, 256), off_v = align_up(off_k + kv_bytes, 256),
           off_w = align_up(off_v + kv_bytes, 256), off_o = align_up(off_w + i_bytes, 256),
           off_n = align_up(off_o + q_bytes, 256), staging = align_up(off_n + i_bytes, 256);
    const Plan pl = plan_split(S, static_cast<int>(units), sm_count(dev), true, d, Hq / Hkv, true);
    const Layout L = scratch_layout(s, pl, staging);
    Scratch* scr = nullptr;
    if ((st = get_scratch(dev, stream, L.total, static_cast<size_t>(s.B) * s.Hkv, &scr)) != LF_OK) return st;
    char* stg = static_cast<char*>(scr->base) + (L.total - staging);
    // Page-locked host buffers that this device can address (cudaHostAlloc /
    // cudaHostRegister memory; on GB300 over NVLink-C2C) are read and written
    // by the kernel in place; any other buffer goes through device staging
    // with one copy each way. LF_HOST_ZEROCOPY=0 stages every buffer.
    const char* zenv = std::getenv("LF_HOST_ZEROCOPY");
    const bool zero_copy = !(zenv && std::atoi(zenv) == 0);
    auto mapped = [&](const void* p, size_t align) -> void* {
        if (!zero_copy) return nullptr;
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        if (at.type != cudaMemoryTypeHost || !at.devicePointer ||
            reinterpret_cast<uintptr_t>(at.devicePointer) % align != 0)
            return nullptr;
        return at.devicePointer;
    };
    void* dq = mapped(q_host, 16);
    void* dk = mapped(new_k_host, 16);
    void* dv = mapped(new_v_host, 16);
    void* dw = mapped(write_slot_host, 4);
    void* dout = mapped(out_host, 16);
    void* dn = mapped(next_slot_host, 4);
    StepArgs a{dq ? dq : stg + off_q, k_cache, v_cache, mask, dk ? dk : stg + off_k,
               dv ? dv : stg + off_v,
               reinterpret_cast<int32_t*>(dw ? dw : stg + off_w), dout ? dout : stg + off_o,
               reinterpret_cast<int32_t*>(dn ? dn : stg + off_n), nullptr};
    g_last_error[0] = '\0';
    if ((!dq && (e = cudaMemcpyAsync(stg + off_q, q_host, q_bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess) ||
        (!dk && (e = cudaMemcpyAsync(stg + off_k, new_k_host, kv_bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess) ||
        (!dv && (e = cudaMemcpyAsync(stg + off_v, new_v_host, kv_bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess) ||
        (!dw && (e = cudaMemcpyAsync(stg + off_w, write_slot_host, i_bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess))
        return cuda_fail(e, "host-to-device copy");
    if ((st = enqueue_step(a, s, stream, scr, L, pl)) != LF_OK) return st;
    if ((!dout && (e = cudaMemcpyAsync(out_host, stg + off_o, q_bytes, cudaMemcpyDeviceToHost, stream)) != cudaSuccess) ||
        (!dn && (e = cudaMemcpyAsync(next_slot_host, stg + off_n, i_bytes, cudaMemcpyDeviceToHost, stream)) != cudaSuccess))
        return cuda_fail(e, "device-to-host copy");
    return LF_OK;
}

lf_status lf_decode_step_noalloc(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                                 const void* new_k, const void* new_v, const int32_t* write_slot,
                                 void* out, int32_t* next_slot, int B, int Hq, int Hkv, int d,
                                 int S, int W, float scale, void* stream_v) {
    const StepArgs a{q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot, nullptr};
    const Shape s{B, Hq, Hkv, d, S, W, scale};
    lf_status st = check_args(a, s);
    if (st != LF_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    const size_t units = static_cast<size_t>(B) * Hkv;
    const Plan pl = plan_split(S, static_cast<int>(units), sms > 0 ? sms : 1, true, d, Hq / Hkv, true);
    const Layout L = scratch_layout(s, pl, 0);
    // Per unit, the chunk and scoring-kernel arrival counters, the 64-bit
    // argmin word and the ready flag of a split finish.
    const size_t arrivals_off = align_up(L.total, 256);
    const size_t need = arrivals_off + lf::kCounterWordsPerUnit * units * sizeof(uint32_t);
    if (need + (kStaticScratchBytes - kStaticErrOff) > kStaticScratchBytes)
        return fail(LF_ERR_UNSUPPORTED,
                    "lf_decode_step_noalloc: this shape needs %zu bytes of scratch but the static "
                    "scratch holds %zu; use lf_decode_step or fewer B * Hkv * S slots",
                    need + (kStaticScratchBytes - kStaticErrOff), kStaticScratchBytes);
    void* base_v = nullptr;
    if ((st = static_scratch_base(dev, &base_v)) != LF_OK) return st;
    char* base = static_cast<char*>(base_v);
    // The arrival counters must start at zero (the kernels leave them so, but
    // a call that timed out may not have).
    if ((e = cudaMemsetAsync(base + arrivals_off, 0, need - arrivals_off, stream)) != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(static scratch)");
    Launch r;
    if ((st = build_launch(a, s, base, reinterpret_cast<uint32_t*>(base + arrivals_off),
                           reinterpret_cast<uint32_t*>(base + kStaticErrOff), L, pl, &r)) != LF_OK)
        return st;
    g_last_error[0] = '\0';
    return launch(r, stream);
}

lf_status lf_step_plan(int B, int Hq, int Hkv, int d, int S, int topk, int32_t* plan) {
    if (!plan) return fail(LF_ERR_INVALID_ARG, "plan is null");
    if (topk < 1 || topk > LF_MAX_TOPK)
        return fail(LF_ERR_INVALID_ARG, "k = %d is outside [1, %d]", topk, LF_MAX_TOPK);
    const Shape s{B, Hq, Hkv, d, S, 0, 1.f};
    lf_status st = check_shape(s);
    if (st != LF_OK) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const Plan pl = plan_split(S, B * Hkv, sm_count(dev), topk == 1, d, Hq / Hkv, true);
    plan[0] = pl.nchunk;
    plan[1] = pl.chunk_tiles;
    plan[2] = pl.stages;
    plan[3] = pl.cluster ? 1 : 0;
    plan[4] = pl.split ? 1 : 0;
    plan[5] = pl.fit;
    return LF_OK;
}

lf_status lf_step_prepare(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                          const void* new_k, const void* new_v, const int32_t* write_slot,
                          void* out, int32_t* next_slot, int B, int Hq, int Hkv, int d, int S,
                          int W, float scale, void* stream_v, lf_step_handle** handle) {
    if (!handle) return fail(LF_ERR_INVALID_ARG, "handle is NULL");
    *handle = nullptr;
    const Shape s{B, Hq, Hkv, d, S, W, scale};
    lf_status st;
    if (!q || !new_k || !new_v || !write_slot || !out || !next_slot)
        return fail(LF_ERR_INVALID_ARG, "an input or output buffer is NULL");
    if ((st = check_ptr(k_cache, 16, "k_cache")) != LF_OK) return st;
    if ((st = check_ptr(v_cache, 16, "v_cache")) != LF_OK) return st;
    if ((st = check_ptr(mask, 4, "mask")) != LF_OK) return st;
    if ((st = check_shape(s)) != LF_OK) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");

    const size_t units = static_cast<size_t>(B) * Hkv;
    const size_t q_bytes = static_cast<size_t>(B) * Hq * d * 2;
    const size_t kv_bytes = units * d * 2;
    const size_t i_bytes = units * 4;
    const Plan pl = plan_split(S, static_cast<int>(units), sm_count(dev), true, d, Hq / Hkv, true);
    const Layout L = scratch_layout(s, pl, 0);

    // Where each per-step buffer lives: device memory of this device is used
    // as is; page-locked host memory this device can address is read and
    // written in place (unless LF_HOST_ZEROCOPY=0); anything else is staged
    // in the handle's device memory with a copy each way per run.
    const char* zenv = std::getenv("LF_HOST_ZEROCOPY");
    const bool zero_copy = !(zenv && std::atoi(zenv) == 0);
    struct Io {
        const void* p;
        size_t bytes, align;
        bool input;
        const char* name;
        void* dev;      // the pointer the kernel uses (null: staged)
        size_t off;     // staging offset
    };
    Io io[6] = {{q, q_bytes, 16, true, "q", nullptr, 0},
                {new_k, kv_bytes, 16, true, "new_k", nullptr, 0},
                {new_v, kv_bytes, 16, true, "new_v", nullptr, 0},
                {write_slot, i_bytes, 4, true, "write_slot", nullptr, 0},
                {out, q_bytes, 16, false, "out", nullptr, 0},
                {next_slot, i_bytes, 4, false, "next_slot", nullptr, 0}};
    size_t staging = align_up(L.total, 256);
    for (Io& b : io) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, b.p) != cudaSuccess) {
            (void)cudaGetLastError();
            at.type = cudaMemoryTypeUnregistered;
        }
        if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
            if (at.device != dev)
                return fail(LF_ERR_INVALID_ARG, "%s is memory of device %d, not of the current device %d",
                            b.name, at.device, dev);
            if (!aligned(b.p, b.align))
                return fail(LF_ERR_INVALID_ARG, "%s is not %zu-byte aligned", b.name, b.align);
            b.dev = const_cast<void*>(b.p);
        } else if (zero_copy && at.type == cudaMemoryTypeHost && at.devicePointer &&
                   aligned(at.devicePointer, b.align)) {
            b.dev = at.devicePointer;
        } else {
            b.off = staging;
            staging = align_up(staging + b.bytes, 256);
        }
    }

    lf_step_handle* h = new (std::nothrow) lf_step_handle;
    if (!h) return fail(LF_ERR_NO_MEMORY, "out of host memory");
    h->dev = dev;
    h->stream = static_cast<cudaStream_t>(stream_v);
    if ((e = cudaMalloc(&h->mem, staging)) != cudaSuccess) {
        h->mem = nullptr;
        free_handle(h);
        return fail(LF_ERR_NO_MEMORY, "cudaMalloc(%zu bytes of scratch): %s", staging,
                    cudaGetErrorString(e));
    }
    const size_t words = lf::kCounterWordsPerUnit * units + 64;
    if ((e = cudaMalloc(&h->words, words * sizeof(uint32_t))) != cudaSuccess) {
        h->words = nullptr;
        free_handle(h);
        return fail(LF_ERR_NO_MEMORY, "cudaMalloc(counters): %s", cudaGetErrorString(e));
    }
    if ((e = cudaMemset(h->words, 0, words * sizeof(uint32_t))) != cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "cudaMemset");
    }
    h->dev_err = h->words + lf::kCounterWordsPerUnit * units;
    char* base = static_cast<char*>(h->mem);
    for (Io& b : io) {
        if (b.dev) continue;
        b.dev = base + b.off;
        if (b.input)
            h->h2d[h->n_h2d++] = {b.dev, b.p, b.bytes};
        else
            h->d2h[h->n_d2h++] = {const_cast<void*>(b.p), b.dev, b.bytes};
    }
    const StepArgs a{io[0].dev, k_cache, v_cache, mask, io[1].dev, io[2].dev,
                     static_cast<const int32_t*>(io[3].dev), io[4].dev,
                     static_cast<int32_t*>(io[5].dev), nullptr};
    if ((st = build_launch(a, s, base, h->words, h->dev_err, L, pl, &h->r)) != LF_OK) {
        free_handle(h);
        return st;
    }
    *handle = h;
    return LF_OK;
}

lf_status lf_step_run(lf_step_handle* h) {
    if (!h) return fail(LF_ERR_INVALID_ARG, "handle is NULL");
    cudaError_t e;
    for (int i = 0; i < h->n_h2d; ++i)
        if ((e = cudaMemcpyAsync(h->h2d[i].dst, h->h2d[i].src, h->h2d[i].bytes,
                                 cudaMemcpyHostToDevice, h->stream)) != cudaSuccess)
            return cuda_fail(e, "host-to-device copy");
    lf_status st = launch(h->r, h->stream);
    if (st != LF_OK) return st;
    for (int i = 0; i < h->n_d2h; ++i)
        if ((e = cudaMemcpyAsync(h->d2h[i].dst, h->d2h[i].src, h->d2h[i].bytes,
                                 cudaMemcpyDeviceToHost, h->stream)) != cudaSuccess)
            return cuda_fail(e, "device-to-host copy");
    return LF_OK;
}

lf_status lf_step_errors(lf_step_handle* h, uint32_t* flags, int clear) {
    if (!h || !flags) return fail(LF_ERR_INVALID_ARG, "handle or flags is NULL");
    *flags = 0;
    uint32_t v = 0;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(&v, h->dev_err, sizeof v, cudaMemcpyDeviceToHost, h->stream)) != cudaSuccess)
        return cuda_fail(e, "reading the device error word");
    if ((e = cudaStreamSynchronize(h->stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    *flags = v;
    if (clear && v) {
        if ((e = cudaMemsetAsync(h->dev_err, 0, sizeof v, h->stream)) != cudaSuccess)
            return cuda_fail(e, "cudaMemsetAsync");
        if ((e = cudaStreamSynchronize(h->stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    }
    return LF_OK;
}

lf_status lf_step_destroy(lf_step_handle* h) {
    if (!h) return LF_OK;
    // Work queued on the handle's stream may still use its memory.
    cudaError_t e = cudaStreamSynchronize(h->stream);
    free_handle(h);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return LF_OK;
}

lf_status lf_device_errors(void* stream_v, uint32_t* flags, int clear) {
    if (!flags) return fail(LF_ERR_INVALID_ARG, "flags is NULL");
    *flags = 0;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    // The word of the stream's scratch, and that of the allocation-free
    // entry point's static array once it has run on this device.
    uint32_t* words[2] = {nullptr, nullptr};
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_scratch.find({dev, stream});
        if (it != g_scratch.end()) words[0] = it->second.dev_err;
    }
    if (dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (g_static_base[dev])
            words[1] = reinterpret_cast<uint32_t*>(static_cast<char*>(g_static_base[dev]) +
                                                   kStaticErrOff);
    }
    for (uint32_t* word : words) {
        if (!word) continue;
        uint32_t v = 0;
        if ((e = cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
            return cuda_fail(e, "reading the device error word");
        if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
        *flags |= v;
        if (clear && v) {
            if ((e = cudaMemsetAsync(word, 0, sizeof v, stream)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
            if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
        }
    }
    return LF_OK;
}

lf_status lf_profile_enable(int enabled) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_on = enabled != 0;
    return LF_OK;
}

lf_status lf_profile_collect(int kernel_id, double* total_ms, int64_t* launches) {
    if (!total_ms || !launches) return fail(LF_ERR_INVALID_ARG, "NULL output");
    if (kernel_id < 0 || kernel_id >= LF_KERNEL_COUNT) return fail(LF_ERR_INVALID_ARG, "bad kernel id %d", kernel_id);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    double sum = 0.0;
    int64_t n = 0;
    std::vector<ProfRec> keep;
    for (const ProfRec& r : g_prof) {
        if (r.kernel != kernel_id) {
            keep.push_back(r);
            continue;
        }
        ++n;
        if (!r.start) continue;  // counted only
        cudaError_t e = cudaEventSynchronize(r.stop);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
        if (e != cudaSuccess) return cuda_fail(e, "profile event");
        sum += ms;
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_prof.swap(keep);
    *total_ms = sum;
    *launches = n;
    return LF_OK;
}

lf_status lf_release_workspace(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_scratch) {
        cudaSetDevice(kv.first.first);
        cudaDeviceSynchronize();
        if (kv.second.base) cudaFree(kv.second.base);
        if (kv.second.dev_err) cudaFree(kv.second.dev_err);
        if (kv.second.arrivals) cudaFree(kv.second.arrivals);
    }
    g_scratch.clear();
    cudaSetDevice(cur);
    return LF_OK;
}

const char* lf_status_string(lf_status status) {
    switch (status) {
        case LF_OK: return "LF_OK";
        case LF_ERR_INVALID_ARG: return "LF_ERR_INVALID_ARG: invalid argument";
        case LF_ERR_UNSUPPORTED: return "LF_ERR_UNSUPPORTED: shape not supported";
        case LF_ERR_CUDA: return "LF_ERR_CUDA: CUDA error";
        case LF_ERR_NO_MEMORY: return "LF_ERR_NO_MEMORY: scratch allocation failed";
    }
    return "unknown lf_status";
}

const char* lf_last_error(void) { return g_last_error; }

int lf_version(void) { return kVersion; }

}  // extern "C"
