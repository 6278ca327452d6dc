// Internal interface between the C-ABI host code (lf_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lf {

constexpr int kTile = 64;           // cache slots per pipeline tile
constexpr int kMaxChunkTiles = 32;  // tiles per split (chunk) at most
constexpr int kBoxCols = 64;        // bf16 columns per 128-byte swizzled TMA box row

// Split attention: one CTA per (chunk of slots, unit). Performs the slot
// write and mask ageing for its chunk, attends over its live tiles and
// leaves per-chunk softmax partials plus per-slot score terms in scratch.
struct SplitParams {
    const __nv_bfloat16* q;      // [B][Hq][D]
    __nv_bfloat16* k_cache;      // [units][S][D] (row write_slot is written)
    __nv_bfloat16* v_cache;      // [units][S][D]
    int32_t* mask;               // [units][S]   ages, aged in place
    const __nv_bfloat16* new_k;  // [units][D]
    const __nv_bfloat16* new_v;  // [units][D]
    const int32_t* write_slot;   // [units]
    float* part_o;               // [units][nchunk][G][D]  unnormalised output, base m
    float2* part_ml;             // [units][nchunk][G]     (m, l), log2 domain
    float* stash;                // [units][S][G]          log2(p~ * ||v||_1) per live slot
    uint32_t* dev_err;           // LF_DEVERR_* bits
    int Hq, Hkv, S, W, nchunk, chunk_tiles;
    float scale_log2;            // scale * log2(e)
};

// Combine: one CTA per unit. Merges the chunks' partials into the output,
// finishes LongFlowScore for every live slot and reduces the argmin.
struct CombineParams {
    const float* part_o;
    const float2* part_ml;
    const float* stash;
    const int32_t* mask;         // aged mask written by the split kernel
    __nv_bfloat16* out;          // [B][Hq][D]
    int32_t* next_slot;          // [units]
    float* scores;               // [units][S] or nullptr
    int Hq, Hkv, S, W, nchunk;
};

// Dynamic shared memory the split kernel needs for head dim D.
size_t split_smem_bytes(int D);

cudaError_t launch_attn_split(int D, int G, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              const SplitParams& p, int units, cudaStream_t stream);

cudaError_t launch_combine(int D, int G, const CombineParams& p, int units,
                           cudaStream_t stream);

}  // namespace lf
