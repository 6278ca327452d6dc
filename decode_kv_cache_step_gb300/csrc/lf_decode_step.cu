// Instantiations of the decode-step kernel that merge in the unit's last CTA
// (2- and 3-stage TMA rings, score on or off), the split-finish scoring
// kernel, and the launch dispatch; the thread-block-cluster instantiations
// live in lf_decode_step_cluster.cu so that the two compile in parallel.
#include "lf_step_kernel.cuh"

namespace lf {
namespace {

// ------------------------------------------------------ split finish --
//
// For long units the last CTA's scan of every slot sits on the step's tail,
// and while the other SMs stream K and V it gets about one SM's share of the
// memory system. With a split finish the decode-step kernel stops after the
// merge (publishing c_h per unit and raising the unit's ready flag) and this
// kernel, launched behind it with programmatic dependent launch, scores every
// chunk of every unit in parallel, each unit as soon as its flag is up:
// log2 I_j from the terms t_hj + c_h, the same arithmetic in the same order
// as the single-kernel scan, so scores and choices are bit-identical. The
// lexicographic (I_j, j) argmin is an atomic maximum over the complemented
// 64-bit key (ordered log2 I_j, slot), empty slots (fill-empty-first) taking
// score key 0; the last CTA of the unit reads and clears it. Units below
// split_from (the first ones of a grid of many waves) scan in their last
// CTA instead, and this grid covers only the others.
constexpr int kScoreThreads = 128;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kScoreTilesPerWarp = 2;  // tiles a warp loads per round trip (4 slots per lane)
constexpr int kScoreMaxChunks = 1024;

// CTA (part, y) scores the chunks [part * per, (part + 1) * per) of unit
// u = split_from + y, per = ceil(nchunk / parts) (one chunk by default). Warps take whole
// 64-slot tiles, so a tile's chunk and liveness are warp-uniform and a tile
// of a chunk without a live slot costs no load.
template <int G>
__global__ void __launch_bounds__(kScoreThreads, G >= 8 ? 4 : 8) lf_score_kernel(const StepParams p, int parts) {
    // Launched behind the decode-step kernel with programmatic dependent
    // launch, this grid starts only once every decode-step CTA has passed its
    // own dependency wait: all of them run or have run, and none waits on
    // this kernel, so every unit's flag goes up. Instead of waiting for the
    // whole decode-step grid to finish, each CTA waits for its own unit's
    // flag (acquire; every write the flag releases is then visible), so the
    // early units are scored while the decode-step kernel's tail still runs.
    // The next kernel of the stream may launch at once: it waits for this
    // grid to finish before its first global read.
    allow_dependent_launch();
    __shared__ unsigned char s_live[kScoreMaxChunks];
    __shared__ unsigned long long s_red[kScoreWarps];
    const int part = blockIdx.x;
    const int u = p.split_from + static_cast<int>(blockIdx.y);
    const int tid = threadIdx.x;
    if (tid == 0) {
        if (ld_acquire_gpu(p.ready + u) == 0u) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu(p.ready + u) == 0u) {
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                __nanosleep(100);
            }
        }
    }
    __syncthreads();
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int S = p.S;
    const int nchunk = p.nchunk;
    const int ct = p.chunk_tiles;
    const int per = (nchunk + parts - 1) / parts;
    const int c0 = part * per;
    const int c1 = min(nchunk, c0 + per);
    float* scores = p.scores ? p.scores + static_cast<size_t>(u) * S : nullptr;
    const bool fill_first = (p.flags & kFlagFillEmptyFirst) != 0;
    const bool all = fill_first || scores != nullptr;
    const float* stash = p.stash + static_cast<size_t>(u) * S * G;
    const int32_t* age = p.mask + static_cast<size_t>(u) * S;
    // A chunk whose softmax maximum is -inf holds no live slot: no scored
    // candidate there (empty slots and scores are still visited when wanted).
    for (int c = c0 + tid; c < c1; c += kScoreThreads)
        s_live[c - c0] = all || __ldcg(&p.part_ml[(static_cast<size_t>(u) * nchunk + c) * G].x) != -INFINITY;
    float cf[G];
#pragma unroll
    for (int h = 0; h < G; ++h) cf[h] = __ldcg(&p.cfold[static_cast<size_t>(u) * G + h]);
    __syncthreads();

    // Each lane keeps its best (score key, slot). A lane visits its slots in
    // increasing order, so a strict "<" on the key alone keeps the lowest slot
    // among equal keys. Key: ordered_key(log2 I_j) (the order of the scores
    // at any scale, below fp32's normal range included), 0 for an empty slot
    // under fill-empty-first, ~0u for none.
    uint32_t bkey = 0xffffffffu;
    int bj = 0x7fffffff;
    const int tlo = c0 * ct;
    const int thi = min((S + kTile - 1) / kTile, c1 * ct);
    // tile / ct by a multiply-high: exact for ct <= 32 and any tile of an int S
    // (the rounding error of the reciprocal stays below tile / 2^32 < 1 / ct).
    const uint32_t ct_inv = ct > 1 ? static_cast<uint32_t>((0x100000000ull + ct - 1) / ct) : 0u;
    const int W = p.W;
    constexpr int kSlots = 2 * kScoreTilesPerWarp;  // per lane and round trip
    for (int tb = tlo + warp * kScoreTilesPerWarp; tb < thi;
         tb += kScoreWarps * kScoreTilesPerWarp) {
        int a[kSlots];
        float t[kSlots][G];
        bool in[kScoreTilesPerWarp];
#pragma unroll
        for (int q = 0; q < kScoreTilesPerWarp; ++q) {
            const int tile = tb + q;
            const int c = ct > 1 ? static_cast<int>(__umulhi(static_cast<uint32_t>(tile), ct_inv)) : tile;
            in[q] = tile < thi && s_live[c - c0];  // warp-uniform
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int j = tile * kTile + r * 32 + lane;
                const bool ok = in[q] && j < S;
                a[2 * q + r] = ok ? __ldcg(age + j) : -1;
                if (ok) load_terms<G>(stash + j * G, t[2 * q + r]);
            }
        }
#pragma unroll
        for (int q = 0; q < kScoreTilesPerWarp; ++q) {
            if (!in[q]) continue;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int j = (tb + q) * kTile + r * 32 + lane;
                const int aa = a[2 * q + r];
                const float L = log2_score<G>(t[2 * q + r], cf);
                const bool live = aa >= 0;
                const bool cand = live ? (aa >= W && L == L) : fill_first;
                const uint32_t key = live ? ordered_key(L) : 0u;
                if (cand && j < S && key < bkey) {
                    bkey = key;
                    bj = j;
                }
                if (scores && j < S)
                    scores[j] = live ? exported_score<G>(p, L, t[2 * q + r], cf) : INFINITY;
            }
        }
    }
    // (key, slot) minimum of the CTA, as the complemented 64-bit word.
    unsigned long long best = bkey == 0xffffffffu
                                  ? 0ull
                                  : ~((static_cast<unsigned long long>(bkey) << 32) |
                                      static_cast<uint32_t>(bj));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
    }
    if (lane == 0) s_red[warp] = best;
    __syncthreads();
    if (tid == 0) {
#pragma unroll
        for (int w = 1; w < kScoreWarps; ++w) best = s_red[w] > best ? s_red[w] : best;
        bool last = true;
        if (parts > 1) {
            // The maximum needs no returned value; the acquire-release add
            // orders it before this CTA's arrival, and the unit's last CTA
            // acquires every other CTA's maximum with its own add.
            if (best) red_max_relaxed_gpu(&p.best[u], best);
            last = atom_add_acq_rel_gpu(&p.score_arrivals[u], 1u) ==
                   static_cast<uint32_t>(parts - 1);
            if (last) {
                p.score_arrivals[u] = 0u;
                best = atomicExch(&p.best[u], 0ull);
            }
        }
        if (last) {
            p.ready[u] = 0u;  // every CTA of the unit has seen the flag
            const int slot = best ? static_cast<int>(static_cast<uint32_t>(~best)) : -1;
            p.next_slot[u] = slot;
            if (slot >= 0 && (p.flags & kFlagMaskEvicted))
                p.mask[static_cast<size_t>(u) * S + slot] = -1;
        }
    }
    // Every read of these chunks' score terms is done: drop the lines.
    const int cs = ct * kTile;
    for (int c = c0; c < c1; ++c)
        if (s_live[c - c0])
            discard_range(stash + static_cast<size_t>(c) * cs * G,
                          static_cast<size_t>(min(S, (c + 1) * cs) - c * cs) * G * 4, tid,
                          kScoreThreads);
    // This grid waits for no unit of the decode-step grid that it does not
    // score, and its other CTAs wait only for flags: the grid's last CTA
    // also waits for the decode-step grid to complete, so that this grid
    // completes after it and the next kernel's dependency wait covers both
    // (the units that scan in their last CTA, and the decode CTAs' last
    // stores after their flags).
    if (tid == 0 && blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1)
        grid_dependency_wait();
}

template <int D, int G>
cudaError_t launch_dg(const CUtensorMap& tmK, const CUtensorMap& tmV, const StepParams& p,
                      int units, cudaStream_t stream, int stages, bool score, bool pdl) {
    if (!score) return launch_t<D, G, 2, false, false>(tmK, tmV, p, units, stream, pdl);
    return stages == 2 ? launch_t<D, G, 2, true, false>(tmK, tmV, p, units, stream, pdl)
                       : launch_t<D, G, 3, true, false>(tmK, tmV, p, units, stream, pdl);
}

template <int G>
cudaError_t launch_score_t(const StepParams& p, int units, cudaStream_t stream, bool pdl) {
    // One CTA per chunk: the CTAs of a unit wait for its flag, not for each
    // other or for the grid, so the grid need not be resident at once, and
    // the finest split scores each unit soonest after its merge (measured on
    // the 16K-slot workload: 4 CTAs per unit 203.9 us per step, 8: 200.5,
    // 16 (one per chunk): 199.6).
    int parts = p.nchunk;
    if (const char* env = std::getenv("LF_SCORE_PARTS")) parts = std::atoi(env);  // tests, tuning
    parts = std::max(1, std::min(p.nchunk, parts));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(parts, units - p.split_from);
    cfg.blockDim = dim3(kScoreThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lf_score_kernel<G>, p, parts);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool step_fits(int D, int G, int stages, bool score, int nchunk, int topk) {
    const size_t need = finish_smem_bytes(nchunk, G, score ? topk : 1);
    size_t have;
    if (stages == kDeepStages)
        have = D == 64 ? StepSmem<64, kDeepStages>::kBarOff : StepSmem<128, kDeepStages>::kBarOff;
    else if (stages == 2 || !score)
        have = D == 64 ? StepSmem<64, 2>::kBarOff : StepSmem<128, 2>::kBarOff;
    else
        have = D == 64 ? StepSmem<64, 3>::kBarOff : StepSmem<128, 3>::kBarOff;
    return need <= have;
}

size_t step_smem_bytes(int D, int stages) {
    if (stages == kDeepStages)
        return D == 64 ? StepSmem<64, kDeepStages>::kAlloc : StepSmem<128, kDeepStages>::kAlloc;
    if (stages == 2) return D == 64 ? StepSmem<64, 2>::kAlloc : StepSmem<128, 2>::kAlloc;
    return D == 64 ? StepSmem<64, 3>::kAlloc : StepSmem<128, 3>::kAlloc;
}

cudaError_t launch_decode_step(int D, int G, int stages, bool score, bool cluster,
                               const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const StepParams& p, int units, cudaStream_t stream) {
    // Programmatic dependent launch overlaps this step's launch and set-up
    // with the tail of the previous kernel in the stream (LF_PDL=0: off).
    const char* env = std::getenv("LF_PDL");
    const bool pdl = !(env && std::atoi(env) == 0);
    if (cluster) return launch_decode_step_cluster(D, G, stages, score, tmK, tmV, p, units, stream, pdl);
#define LF_STEP_CASE(DD, GG) \
    if (D == DD && G == GG)  \
        return launch_dg<DD, GG>(tmK, tmV, p, units, stream, stages, score, pdl);
    LF_STEP_CASE(64, 1) LF_STEP_CASE(64, 2) LF_STEP_CASE(64, 4) LF_STEP_CASE(64, 8)
    LF_STEP_CASE(128, 1) LF_STEP_CASE(128, 2) LF_STEP_CASE(128, 4) LF_STEP_CASE(128, 8)
#undef LF_STEP_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_score(int G, const StepParams& p, int units, cudaStream_t stream) {
    if (p.chunk_tiles > kMaxChunkTiles || p.nchunk > kScoreMaxChunks) return cudaErrorInvalidValue;
    const char* env = std::getenv("LF_PDL");
    const bool pdl = !(env && std::atoi(env) == 0);
    switch (G) {
        case 1: return launch_score_t<1>(p, units, stream, pdl);
        case 2: return launch_score_t<2>(p, units, stream, pdl);
        case 4: return launch_score_t<4>(p, units, stream, pdl);
        case 8: return launch_score_t<8>(p, units, stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lf
