// Internal interface between the C-ABI host code (lf_api.cu) and the kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lf {

constexpr int kTile = 64;           // cache slots per pipeline tile
constexpr int kMaxChunkTiles = 32;  // tiles per chunk (split of the slot axis) at most
constexpr int kBoxCols = 64;        // bf16 columns per 128-byte swizzled TMA box row

// One decode step. Grid (nchunk, units): CTA (c, u) performs the slot write
// and mask ageing for chunk c of unit u, attends over the chunk's live tiles
// and leaves softmax partials and per-slot score terms in scratch. The last
// CTA of a unit to finish merges them: output row, LongFlowScore, argmin
// (with split set, the scoring kernel does the last two).
struct StepParams {
    const __nv_bfloat16* q;      // [B][Hq][D]
    __nv_bfloat16* k_cache;      // [units][S][D] (row write_slot is written)
    __nv_bfloat16* v_cache;      // [units][S][D]
    int32_t* mask;               // [units][S]   ages, aged in place
    const __nv_bfloat16* new_k;  // [units][D]
    const __nv_bfloat16* new_v;  // [units][D]
    const int32_t* write_slot;   // [units]
    __nv_bfloat16* out;          // [B][Hq][D]
    int32_t* next_slot;          // [units][topk] slots to overwrite, ascending (score, slot)
    float* scores;               // [units][S] or nullptr
    // scratch
    float* part_o;               // [units][nchunk][G][D]  unnormalised output, base m
    float2* part_ml;             // [units][nchunk][G]     (m, l), log2 domain
    // [units][nchunk]: bit t set when tile t of the chunk holds a live slot
    // (written by the chunk's CTA; nullptr: not kept)
    uint32_t* part_tiles = nullptr;
    float* stash;                // [units][S][G]          log2(exp(s) * ||v||_1) per live slot
    uint32_t* arrivals;          // [units] chunk arrival counters, 0 between steps
    uint32_t* dev_err;           // LF_DEVERR_* bits
    // Split finish (top-1 only): the last CTA publishes c_h = log2(1/l_h) - m_h
    // and raises the unit's ready flag; a second kernel scores the unit's
    // chunks in parallel as soon as the flag is up.
    float* cfold = nullptr;                // [units][G]
    unsigned long long* best = nullptr;    // [units] ~(score key, slot) maximum, 0 between steps
    uint32_t* score_arrivals = nullptr;    // [units] arrival counters of the scoring kernel
    uint32_t* ready = nullptr;             // [units] 1 once the unit is merged, 0 between steps
    int split = 0;
    // With split set, units below this one still scan in their last CTA
    // (their score terms are still in L2 when they merge); the scoring kernel
    // takes the units from here on.
    int split_from = 0;
    int Hq, Hkv, S, W, nchunk, chunk_tiles;
    float scale_log2;            // scale * log2(e)
    int topk;                    // slots returned per unit (1 = the argmin)
    int flags;                   // kFlag* bits
    // Limit of the pipeline waits; drains of copies in flight always allow 1 s.
    uint64_t wait_limit_ns;
    // CTAs whose linear index is below this issue their chunk's first tiles
    // before the mask tells which tiles hold a live slot (the grid's first
    // wave; set by the launch).
    int spec_ctas = 0;
};

constexpr int kFlagFillEmptyFirst = 1;  // empty (masked) slots are returned before any score
constexpr int kFlagMaskEvicted = 2;     // returned slots are masked (-1) in place
constexpr int kFlagLog2Scores = 4;      // the score export holds log2 I_j
constexpr int kMaxTopK = 1024;
constexpr int kMaxClusterChunks = 16;   // chunks of a unit run as one cluster up to this
                                        // (above 8: a non-portable cluster size)
constexpr int kDeepStages = 6;          // TMA ring of the one-CTA-per-SM cluster variant
// Counter words per unit in a step's scratch, all zero between steps: the
// chunk arrival counter, the scoring kernel's arrival counter, the 64-bit
// argmin word and the ready flag, each in an array of its own.
constexpr int kCounterWordsPerUnit = 5;

// Dynamic shared memory the kernel needs for head dim D and a TMA ring of
// `stages` tiles (2 or 3).
size_t step_smem_bytes(int D, int stages);

// Whether finish-stage shared memory (chunk weights, top-k list) fits.
bool step_fits(int D, int G, int stages, bool score, int nchunk, int topk);

// score = false runs the attention-only variant: the slot write (the written
// slot becomes live; no other age changes) and the attention output, without
// LongFlowScore or eviction. next_slot, scores and topk are then unused.
// cluster = true launches each unit's nchunk (<= kMaxClusterChunks) CTAs as
// one thread-block cluster that merges through distributed shared memory
// (2-stage ring, topk == 1 only); otherwise the unit's last CTA merges.
cudaError_t launch_decode_step(int D, int G, int stages, bool score, bool cluster,
                               const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const StepParams& p, int units, cudaStream_t stream);

// The cluster instantiations (lf_decode_step_cluster.cu); stages is 2 or
// kDeepStages.
cudaError_t launch_decode_step_cluster(int D, int G, int stages, bool score,
                                       const CUtensorMap& tmK, const CUtensorMap& tmV,
                                       const StepParams& p, int units, cudaStream_t stream,
                                       bool pdl);

// How many clusters of csize CTAs (one unit each) of the cluster instance
// (stages 2 or kDeepStages) can be resident at once on the current device;
// 0 if none can or the query fails. Cached per device and instance.
int max_active_clusters(int D, int G, int stages, bool score, int csize);

// Slots of a chunk whose score terms the deep-ring cluster instance keeps
// in shared memory (the plan gives that ring no longer chunks).
int deep_term_slots(int D, int G);

// The scoring kernel of a split finish: grid (parts, units - split_from);
// CTA (c, y) takes unit u = split_from + y: it waits for unit u's ready flag, scores its chunks from the ages, the score
// terms and c_h, and the unit's last CTA writes next_slot (and masks it with
// kFlagMaskEvicted). It does not wait for the decode-step grid as a whole.
cudaError_t launch_score(int G, const StepParams& p, int units, cudaStream_t stream);


}  // namespace lf
