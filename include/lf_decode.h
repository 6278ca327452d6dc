/*
 * lf_decode.h - C ABI of the GB300 (sm_103a) LongFlow decode-step library.
 *
 * One call performs one decode step of "LongFlow: Efficient KV Cache
 * Compression for Reasoning Models" for every (sequence b, KV head kvh) unit
 * of a batch:
 *
 *   1. Slot write (Fig. 2, Left): the current token's K/V row replaces the
 *      cache slot chosen at the previous step (write_slot). That slot's age
 *      becomes 0, every other live slot of the unit ages by one.
 *   2. Attention (Fig. 2, Middle): the g = Hq / Hkv query heads of the unit
 *      attend over the static, mask-gated cache with softmax(scale * q.k).
 *   3. LongFlowScore and eviction (Fig. 2, Right; Fig. 1 caption): P.V is
 *      split into G[h][j][c] = p[h][j] * v[j][c] and O = sum_j G. The paper
 *      prints no formula for the score; this library uses
 *          I_j = sum over the unit's heads h, sum over c, of |p[h][j] * v[j][c]|
 *      with p the final normalised weight. The returned slot is the argmin of
 *      I_j over live slots whose age is at least W (the W most recent tokens
 *      are protected), ties to the lowest index.
 *
 * Conventions shared by every entry point:
 *   - bf16 arrays are raw IEEE bfloat16 (uint16 bit patterns), row-major,
 *     contiguous. Layouts:
 *        q, out          [B][Hq][d]
 *        k_cache,v_cache [B][Hkv][S][d]
 *        new_k, new_v    [B][Hkv][d]
 *        mask            [B][Hkv][S] int32
 *        write_slot,
 *        next_slot       [B][Hkv]   int32
 *   - Query head h belongs to KV head floor(h / g).
 *   - mask: a negative entry marks an empty/masked slot (never attended, never
 *     returned); an entry >= 0 is the slot's age in decode steps.
 *   - write_slot = -1 means "no write" (a priming call: nothing ages). A value
 *     in [0, S) is written even into a masked slot, which becomes live with
 *     age 0 (that is how a caller fills an empty cache). Any other value is
 *     ignored and raises LF_DEVERR_BAD_WRITE_SLOT in the device error word.
 *   - next_slot = -1 when no slot is eligible.
 *   - A unit with no live slot writes an all-zero output row.
 *   - All device pointers belong to the caller and must stay valid until the
 *     stream reaches the end of the call's work. bf16 arrays must be 16-byte
 *     aligned, int32 arrays 4-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Results are valid once the stream has synchronised.
 *   - The library owns a per-(device, stream) scratch buffer that it grows on
 *     demand with cudaMalloc (released by lf_release_workspace). Calls on the
 *     same stream are ordered; calls on different streams use different
 *     scratch. A prepared step (lf_step_prepare) owns its own scratch.
 *   - Argument errors are detected on the host before anything is enqueued;
 *     the kernels never trap.
 *
 * Supported shapes: d in {64, 128}; g in {1, 2, 4, 8}; 1 <= S <= 2^20;
 * B * Hkv <= 65535. Anything else returns LF_ERR_UNSUPPORTED.
 *
 * Environment switches, read at every call (tuning and tests; every setting
 * stays within the same tolerances of the exact result, and LF_SPLIT,
 * LF_SPLIT_TAIL, LF_SCORE_PARTS, LF_SPEC and LF_PDL change no result bit):
 *   LF_CHUNK_TILES=n   64-slot tiles per chunk of the slot axis (1..32);
 *                      a cluster merge may still re-chunk to its size cap
 *   LF_STAGES=3        three-stage TMA ring (two CTAs per SM) instead of two
 *   LF_CLUSTER=0|1     thread-block-cluster merge off / on wherever one
 *                      cluster of the split can be placed
 *   LF_CLUSTER_MAX=n   largest cluster tried, 2..16 CTAs (default 16, a
 *                      non-portable size; smaller ones where it cannot be
 *                      placed)
 *   LF_DEEP=0|1        cluster grids keep the 2-stage TMA ring / take the
 *                      deep one (one CTA per SM) whenever its clusters all
 *                      fit (default: the shorter modelled step)
 *   LF_PDL=0           programmatic dependent launch off
 *   LF_SPEC=0          the grid's first wave waits for the live-tile list
 *                      before loading tiles (no speculative first tiles)
 *   LF_SPLIT=0|1       split finish off / on for every top-1 step without
 *                      clusters (default: units of at least 8192 slots)
 *   LF_SPLIT_TAIL=n    in a split finish, the scoring kernel takes the last
 *                      n units and the others scan in their last CTA
 *                      (default: all units, or the last 5/8 of them when
 *                      the grid runs at least four waves)
 *   LF_SCORE_PARTS=n   scoring-kernel CTAs per unit in a split finish
 *   LF_WAIT_LIMIT_NS=n limit of the pipeline waits (diagnostic)
 *   LF_HOST_ZEROCOPY=0 lf_decode_step_host stages every host buffer
 */
#ifndef LF_DECODE_H
#define LF_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lf_status {
    LF_OK = 0,
    LF_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, Hq % Hkv != 0, W < 0, ... */
    LF_ERR_UNSUPPORTED = 2, /* valid request outside the supported shapes */
    LF_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    LF_ERR_NO_MEMORY = 4    /* scratch allocation failed */
} lf_status;

/* Bits of the device error word (lf_device_errors). */
#define LF_DEVERR_BAD_WRITE_SLOT 0x1u /* a write_slot outside [-1, S) was ignored */
#define LF_DEVERR_WAIT_TIMEOUT 0x2u   /* a pipeline wait gave up; that step's results are invalid */

/*
 * Kernel ids for lf_profile_collect. A decode step is one launch of the
 * decode-step kernel, followed, for top-1 steps over long units (a "split
 * finish"), by one launch of the scoring kernel: the decode-step kernel then
 * stops after each unit's merge and the scoring kernel computes LongFlowScore
 * and the argmin of every chunk in parallel, each unit as soon as the
 * decode-step kernel has merged it (the two kernels overlap).
 */
#define LF_KERNEL_DECODE_STEP 0 /* slot write, mask ageing, attention (+ score, eviction) */
#define LF_KERNEL_ATTENTION 1   /* lf_decode_attention: slot write and attention only */
#define LF_KERNEL_SCORE 2       /* split finish: LongFlowScore and eviction */
#define LF_KERNEL_COUNT 3

/* Flags of lf_decode_step_ex. */
#define LF_STEP_FILL_EMPTY_FIRST 0x1 /* return empty (masked) slots, lowest first, before any score */
#define LF_STEP_MASK_EVICTED 0x2     /* mask (-1) the returned slots in place */
#define LF_STEP_LOG2_SCORES 0x4      /* the score export holds log2 I_j instead of I_j */
#define LF_MAX_TOPK 1024             /* largest k of lf_decode_step_ex */

/*
 * One decode step (all three stages above) on device buffers.
 *
 * q         in   bf16 [B][Hq][d]       current queries (post-RoPE; the op applies none)
 * k_cache   in/out bf16 [B][Hkv][S][d] static K cache; row write_slot is overwritten
 * v_cache   in/out bf16 [B][Hkv][S][d] static V cache; row write_slot is overwritten
 * mask      in/out int32 [B][Hkv][S]   ages (>= 0) or masked (< 0); aged in place
 * new_k     in   bf16 [B][Hkv][d]      the current token's K row per unit
 * new_v     in   bf16 [B][Hkv][d]      the current token's V row per unit
 * write_slot in  int32 [B][Hkv]        slot to overwrite (the previous next_slot), or -1
 * out       out  bf16 [B][Hq][d]       attention output, round-to-nearest-even
 * next_slot out  int32 [B][Hkv]        slot to overwrite at the next step, or -1
 * W              protected window: slots with age < W are never returned (W >= 0)
 * scale          logit multiplier (typically 1/sqrt(d)); must be finite
 * stream         cudaStream_t to enqueue on
 */
lf_status lf_decode_step(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                         const void* new_k, const void* new_v, const int32_t* write_slot,
                         void* out, int32_t* next_slot, int B, int Hq, int Hkv, int d, int S,
                         int W, float scale, void* stream);

/*
 * lf_decode_step plus the per-slot LongFlowScore, for inspection and tests.
 * scores out float [B][Hkv][S]: I_j on every live slot (protected ones
 * included), +inf on masked slots. Same semantics otherwise.
 * I_j is fp32: a score below its normal range (about 1.2e-38, a slot whose
 * weight lies some 87 nats or more under the unit's maximum logit) reads 0.
 * The selection does not depend on that: every entry point ranks candidates
 * by log2 I_j, which fp32 holds at any such scale, and lf_decode_step_ex
 * with LF_STEP_LOG2_SCORES exports those values.
 */
lf_status lf_decode_step_scores(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                                const void* new_k, const void* new_v,
                                const int32_t* write_slot, void* out, int32_t* next_slot,
                                float* scores, int B, int Hq, int Hkv, int d, int S, int W,
                                float scale, void* stream);

/*
 * lf_decode_step with a choice of what to return.
 *
 * next_slots out int32 [B][Hkv][k]: the k candidates with the lowest
 *     (LongFlowScore, slot) per unit, ascending; -1 past the last candidate.
 *     k = 1 is lf_decode_step's argmin. Candidates are live slots with
 *     age >= W, plus empty (masked) slots with LF_STEP_FILL_EMPTY_FIRST.
 * k      1 <= k <= LF_MAX_TOPK. A k > 1 returns k slots at once: the
 *        periodic compression that the paper's baselines run every 128 steps
 *        (Fig. 3 caption), built on LongFlowScore instead of per-step argmin.
 * flags  LF_STEP_FILL_EMPTY_FIRST: while a unit has empty slots, return them
 *        (lowest index first) before any scored slot, i.e. fill the budget
 *        before evicting (the cache-fill phase before the budget is full).
 *        LF_STEP_MASK_EVICTED: set the mask of every returned slot to -1, so
 *        it is not attended again until a later step writes into it.
 *        LF_STEP_LOG2_SCORES: scores holds log2 I_j on live slots (-inf for
 *        a zero score) instead of I_j; masked slots still read +inf.
 * scores optional float [B][Hkv][S] as in lf_decode_step_scores (NULL = none).
 * The other arguments are those of lf_decode_step. A combination of k and
 * slot-axis split that does not fit in shared memory returns
 * LF_ERR_UNSUPPORTED.
 */
lf_status lf_decode_step_ex(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                            const void* new_k, const void* new_v, const int32_t* write_slot,
                            void* out, int32_t* next_slots, int k, int flags, float* scores,
                            int B, int Hq, int Hkv, int d, int S, int W, float scale,
                            void* stream);

/*
 * Decode attention alone, with the same kernel pipeline and no LongFlowScore:
 * the current K/V row is written into write_slot (which becomes live with age
 * 0 if it was empty; no other mask entry changes), then the g query heads of
 * each unit attend over the mask-gated cache. No score, no eviction, no
 * ageing. This is the baseline that measures what the score and eviction
 * cost on top of attention (the abstract calls it negligible).
 */
lf_status lf_decode_attention(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                              const void* new_k, const void* new_v, const int32_t* write_slot,
                              void* out, int B, int Hq, int Hkv, int d, int S, float scale,
                              void* stream);

/*
 * One decode step whose per-step inputs and outputs live in HOST memory, for
 * callers that drive decoding from the CPU. The caches and the mask stay on
 * the device (device pointers), as they are the decoder's resident state.
 * Each host buffer (q, new_k, new_v, write_slot in; out, next_slot out) is
 * used one of two ways, chosen per buffer at every call:
 *   - page-locked memory that the current device can address (cudaHostAlloc
 *     or cudaHostRegister; reported by cudaPointerGetAttributes with a device
 *     pointer) and aligned like the device arrays (16 bytes for bf16, 4 for
 *     int32) is read or written by the kernel in place, with no copy (on
 *     GB300 over NVLink-C2C);
 *   - any other buffer is copied through device staging in the library's
 *     scratch (host -> device before the step, device -> host after it, on
 *     `stream`). LF_HOST_ZEROCOPY=0 stages every buffer.
 * The host inputs must not change, and the outputs must not be read, until
 * the stream has synchronised.
 */
lf_status lf_decode_step_host(const void* q_host, void* k_cache, void* v_cache, int32_t* mask,
                              const void* new_k_host, const void* new_v_host,
                              const int32_t* write_slot_host, void* out_host,
                              int32_t* next_slot_host, int B, int Hq, int Hkv, int d, int S,
                              int W, float scale, void* stream);

/*
 * lf_decode_step for callers that cannot allocate device memory. The paper has
 * no counterpart; this entry point exists for embedding. A serving engine that
 * reserves all free GPU memory for its own pools at start-up has nothing left
 * for cudaMalloc (and a real-time loop may not accept the device-wide
 * synchronisation cudaMalloc and cudaFree can cause), yet lf_decode_step needs
 * scratch and grows it on demand. This variant instead uses a fixed 16 MiB
 * scratch array compiled into the library: it calls no cudaMalloc, cudaFree or
 * other allocating routine. Same arguments, semantics and results as
 * lf_decode_step.
 *   - Limit: the shape's scratch (softmax partials, per-slot score terms of
 *     B * Hkv * S slots in fp32 per query head, counters) must fit in 16 MiB,
 *     roughly B * Hq * S <= 3 million for d = 128; larger shapes return
 *     LF_ERR_UNSUPPORTED with the bytes needed.
 *   - Every device that loads the library holds the 16 MiB until exit.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array; calls whose work overlaps on
 *     the GPU (other streams, other host threads) race and corrupt each other.
 *     Serialise them on one stream. Each call zeroes the counters it needs.
 *   - Device error bits (an ignored out-of-range write_slot, a pipeline wait
 *     that gave up) go to one error word in the static array, shared by every
 *     call on the device and never cleared by a call: lf_device_errors,
 *     given the stream these calls ran on, reports (and may clear) them.
 */
lf_status lf_decode_step_noalloc(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                                 const void* new_k, const void* new_v,
                                 const int32_t* write_slot, void* out, int32_t* next_slot,
                                 int B, int Hq, int Hkv, int d, int S, int W, float scale,
                                 void* stream);

/*
 * Prepared steps: lf_decode_step (top-1, score on) with its buffers, shape,
 * launch plan and stream fixed once, for a serving loop that runs the same
 * layer's step token after token. lf_step_prepare checks the arguments
 * (errors as for lf_decode_step), takes the plan and the K/V tensor maps,
 * and resolves where each per-step buffer lives: q, new_k, new_v,
 * write_slot, out and next_slot may each be device memory of the current
 * device (used as is), page-locked host memory the device can address (read
 * and written by the kernel in place, as lf_decode_step_host does) or any
 * other host memory (staged through the handle's device memory, one copy
 * each way per run). k_cache, v_cache and mask are device memory.
 *   - The handle owns its scratch, counters and error word (about
 *     B * Hkv * S * (Hq / Hkv) * 4 bytes of per-slot score terms plus
 *     partials); no other call or handle shares them.
 *   - The handle keeps the pointers: the buffers must outlive it, and their
 *     contents are read and written at each run (the caller writes the next
 *     token's inputs into the same buffers; next_slot of one run is usually
 *     the write_slot buffer of the next, through a second handle whose
 *     write_slot and next_slot buffers are swapped).
 *   - lf_step_run enqueues one step on the prepare-time stream with the
 *     prepare-time device current: the staging copies, one or two kernel
 *     launches (two with the split finish), the copies back. No argument
 *     checks, allocation, plan or pointer queries: the cost of the call is
 *     the launches. Runs of one handle must not overlap (they share its
 *     scratch); they may be captured in a CUDA graph on that stream.
 *   - LF_* switches are read at prepare time. lf_step_prepare allocates
 *     (cudaMalloc, cudaMemset) and lf_step_destroy synchronises: call both
 *     outside any stream capture.
 *   - lf_step_errors reads (and with clear != 0 clears) the handle's device
 *     error word (LF_DEVERR_* bits), synchronising its stream.
 *   - lf_step_destroy synchronises the stream and frees the handle (NULL is
 *     a no-op).
 */
typedef struct lf_step_handle lf_step_handle;
lf_status lf_step_prepare(const void* q, void* k_cache, void* v_cache, int32_t* mask,
                          const void* new_k, const void* new_v, const int32_t* write_slot,
                          void* out, int32_t* next_slot, int B, int Hq, int Hkv, int d, int S,
                          int W, float scale, void* stream, lf_step_handle** handle);
lf_status lf_step_run(lf_step_handle* handle);
lf_status lf_step_errors(lf_step_handle* handle, uint32_t* flags, int clear);
lf_status lf_step_destroy(lf_step_handle* handle);

/*
 * Read (and optionally clear) the device error word of `stream`'s scratch
 * and, on the current device, the error word of lf_decode_step_noalloc's
 * static array (once that entry point has run there). Both are read through
 * `stream` after synchronising it, so pass the stream the steps ran on.
 * *flags receives an OR of LF_DEVERR_* bits, 0 if no step has set one.
 */
lf_status lf_device_errors(void* stream, uint32_t* flags, int clear);

/*
 * The launch plan lf_decode_step / lf_decode_step_ex (k = topk, score on)
 * take for this shape on the current device under the present LF_*
 * environment switches. Launches nothing; queries the device's SM count and
 * cluster occupancy (and sets the kernels' function attributes) on first use.
 * plan (host, 6 entries, written on LF_OK):
 *   [0] chunks per unit (CTAs per unit)   [1] 64-slot tiles per chunk
 *   [2] TMA ring stages                   [3] 1: a unit's chunks run as one
 *                                             thread-block cluster
 *   [4] 1: split finish (scoring kernel)  [5] how many clusters of the
 *       plan's size can be resident at once (without a cluster merge: of
 *       the largest size tried; -1: clusters not considered)
 * Errors: LF_ERR_INVALID_ARG / LF_ERR_UNSUPPORTED as for a step of this
 * shape; LF_ERR_CUDA without a usable device.
 */
lf_status lf_step_plan(int B, int Hq, int Hkv, int d, int S, int topk, int32_t* plan);

/*
 * Kernel timing. While enabled, every kernel launch of the library is
 * bracketed by CUDA events recorded on its own stream, except that a split
 * finish's two launches share one pair: its time, from the decode-step
 * kernel's start to the scoring kernel's end, is reported under
 * LF_KERNEL_DECODE_STEP, and the scoring launch is counted under
 * LF_KERNEL_SCORE with no time of its own (events between the two would
 * serialise them). lf_profile_collect synchronises the events and returns,
 * for one kernel id, the summed event time in milliseconds and the number of
 * launches since the last collect for that id, then forgets them.
 */
lf_status lf_profile_enable(int enabled);
lf_status lf_profile_collect(int kernel_id, double* total_ms, int64_t* launches);

/* Free every scratch buffer (after synchronising the device of each). */
lf_status lf_release_workspace(void);

/* Static description of a status code. */
const char* lf_status_string(lf_status status);

/* Message of the last failed call on this thread ("" if none). */
const char* lf_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int lf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LF_DECODE_H */
