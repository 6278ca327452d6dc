// The LongFlow decode-step kernel (sm_103a): slot write, split-KV attention,
// LongFlowScore and eviction in one launch.
//
// "LongFlow: Efficient KV Cache Compression for Reasoning Models":
//   Fig. 2 (Left)   the current K/V covers the slot chosen at the previous step,
//                   then the static KV and Mask go to the kernel with Q, which
//                   returns the output and the slot to cover next;
//   Fig. 2 (Middle) K, V and the Mask stream from HBM into on-chip memory by
//                   block and the attention runs there;
//   Fig. 2 (Right)  P.V is split in two: G = p * v (per slot) and O = sum_j G.
//                   LongFlowScore is read off G. With the score
//                   I_j = sum_h sum_c |p_hj v_jc| = (sum_h p_hj) * ||v_j||_1
//                   (p >= 0), G never has to exist: each live slot leaves
//                   t_hj = log2(exp(s_hj) * ||v_j||_1) per head, and the final
//                   I_j = sum_h 2^(t_hj - m_h) / l_h once m_h, l_h are known;
//   Fig. 1 caption  one token is evicted after every attention call.
//
// Grid (nchunk, units). CTA (c, u) owns chunk c (up to 32 tiles of 64 slots)
// of unit u = (b, kvh):
//   warp 4, lane 0 : producer. TMA-loads the K and V tiles of the chunk's
//                    live tiles (128-byte swizzled boxes, 2- or 3-stage
//                    mbarrier ring, L2 evict-first: each byte is read once
//                    per step).
//   warps 0..3     : consumers. Warp w owns rows 16w..16w+15 of every tile
//                    and keeps its own online-softmax state. Per 16 slots:
//        S^T[16 x 8]  = K[16 x D] . Q^T[D x 8]       (mma m16n8k16, heads as N)
//        N  [16 x 8]  = |V|[16 x D] . 1[D x 8]        (row L1 norms on the MMA)
//        O^T[D x 8]  += V^T[D x 16] . P^T[16 x 8]     (P^T via movmatrix)
//   GQA folding: the g <= 8 query heads of the unit share each K/V byte.
//   Masked slots are removed by select (logit -inf, V columns zeroed), so
//   NaN or Inf in masked rows never reaches the output.
// The CTA then publishes its chunk's (m, l, O) and counts itself in. The last
// CTA of the unit merges the chunks, writes the output row, finishes
// LongFlowScore for every live slot, selects the slots to evict and drops the
// unit's scratch lines from L2 without writing them back. The selection is
// the lexicographic (I_j, j) argmin over slots with age >= W, or, for k > 1,
// the k smallest by an 8-bit radix select on the score keys (then on the slot
// index among equal scores) and a bitonic sort of the k winners; the periodic
// k-at-once compression of the Fig. 3 caption. Candidates are compared by an
// order-preserving key of log2 I_j, so slots whose scores lie far below
// fp32's normal range (weights hundreds of nats under the unit's maximum)
// are still told apart. Empty slots can rank first
// (cache-fill phase) and the chosen slots can be masked in place.
// Long units stream their score terms through shared memory with bulk copies
// for that scan, or, for top-1 steps over units of thousands of slots, leave
// the scan to a second kernel (the split finish, lf_score_kernel in
// lf_decode_step.cu) that scores every chunk of every unit in parallel once
// the step's memory traffic is over. Shorter ragged units scan only the tiles
// that hold a live slot (top-1; the chunk CTAs publish their live-tile
// masks). When every unit's cluster (up to 16 CTAs) can be resident at once,
// a unit's chunks run as one thread-block cluster instead (kCluster): the
// CTAs push their merged states into one another's shared memory with
// asynchronous remote stores counted on mbarriers (cluster_merge_push), each
// writes the part of the output row it owns and scores its own chunk, and
// rank 0 reduces the argmin (top-1 only). A cluster grid of at most one CTA
// per SM uses a kDeepStages-deep TMA ring, so every tile of a short chunk is
// in flight at once.
// An attention-only instantiation (kScore = false) drops the row norms, the
// score terms, the ageing and the selection: the baseline for the overhead.
// Launches use programmatic dependent launch: a CTA lets the next kernel of
// the stream start launching as soon as it starts, and waits for the previous
// one before its first global read.
#pragma once

#include <limits.h>
#include <math.h>
#include <stdlib.h>

#include <algorithm>
#include <type_traits>

#include "../../include/lf_decode.h"
#include "lf_kernels.h"
#include "lf_ptx.cuh"

namespace lf {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr uint32_t kOnesBf16x2 = 0x3F803F80u;   // (1.0, 1.0) in bf16
constexpr uint32_t kAbsBf16x2 = 0x7FFF7FFFu;
constexpr int kSlotLive = 1;  // slot flag: age >= 0 after the step's ageing
constexpr int kSlotOld = 2;   // slot flag: age >= W (may be evicted)

// The chunk's per-slot state in shared memory: cluster instances keep the
// two flags in a byte; the others keep the age itself (measured: flag bytes
// cost the last-CTA instances 0.5% on the full batches).
template <bool kCluster>
using SlotState = typename std::conditional<kCluster, uint8_t, int32_t>::type;

__device__ __forceinline__ uint8_t slot_state(int a, int W, uint8_t*) {
    return static_cast<uint8_t>((a >= 0 ? kSlotLive : 0) | (a >= W ? kSlotOld : 0));
}
__device__ __forceinline__ int32_t slot_state(int a, int, int32_t*) { return a; }
__device__ __forceinline__ bool slot_live(uint8_t f) { return (f & kSlotLive) != 0; }
__device__ __forceinline__ bool slot_live(int32_t a) { return a >= 0; }

// Shared memory of one CTA: the TMA ring, the chunk's slot states
// (SlotState: a flag byte per slot in cluster instances, the age in the
// others), misc words and barriers.
template <int D, int kStages, bool kCluster = false>
struct StepSmem {
    static constexpr int kBoxes = D / kBoxCols;
    static constexpr int kBoxBytes = kTile * 128;              // 64 rows x 128 B
    static constexpr int kTensorBytes = kBoxes * kBoxBytes;    // K (or V) of one tile
    static constexpr int kStageBytes = 2 * kTensorBytes;       // K + V
    static constexpr int kFlagsOff = kStages * kStageBytes;
    static constexpr int kFlagsBytes = kMaxChunkTiles * kTile * (kCluster ? 1 : 4);
    static constexpr int kMiscOff = kFlagsOff + kFlagsBytes;
    static constexpr int kBarOff = kMiscOff + 16;
    static constexpr int kScanBarOff = kBarOff + 2 * kStages * 8;  // the finish's 2 barriers
    static constexpr int kBytes = kScanBarOff + 16;
    static constexpr int kAlloc = kBytes + 1024;               // slack for 1024-B alignment
};

// Receive buffers of the push merge (cluster grids, cluster_merge_push).
// Each CTA first merges its four warps' states in shared memory; then every
// consumer thread stores one 16-byte piece of the CTA's unnormalised output
// row (g x d floats, head-major) into the CTA that owns that piece, and the
// CTA's (m, l) per head go to every CTA; rank 0 also receives every CTA's
// best (key, slot). The bytes land through asynchronous remote stores
// counted on an mbarrier of the receiving CTA, so no CTA reads another's
// shared memory and no cluster barrier follows the main loop.
template <int D, int G>
struct PushSmem {
    static constexpr int kElems = G * D;  // floats of a unit's output row
    // CTA c of nchunk owns elements [c * per, (c + 1) * per), per a multiple of 4.
    static constexpr int per(int nchunk) { return (kElems / 4 + nchunk - 1) / nchunk * 4; }
    static constexpr int recv_max() {
        int m = 0;
        for (int n = 1; n <= kMaxClusterChunks; ++n) m = n * per(n) > m ? n * per(n) : m;
        return m;
    }
    static constexpr int kOOff = 0;                                     // float [source][per]
    static constexpr int kMlOff = kOOff + recv_max() * 4;               // float2 [source][head]
    static constexpr int kBestOff = kMlOff + kMaxClusterChunks * G * 8; // uint2 [source]
    static constexpr int kWOff = kBestOff + kMaxClusterChunks * 8;      // float [source][head]
    static constexpr int kMOff = kWOff + kMaxClusterChunks * G * 4;     // float [head]
    static constexpr int kIlOff = kMOff + G * 4;                        // float [head]
    static constexpr int kRedOff = kIlOff + G * 4;                      // 2 x [4 warps]
    static constexpr int kBarOff = (kRedOff + 2 * kConsumerWarps * 4 + 7) & ~7;
    static constexpr int kBytes = kBarOff + 24;  // (m, l), output and best barriers
    // The four warps' states, staged in the drained TMA ring (the deep ring:
    // beside the receive buffers): output rows with a padded stride
    // (conflict-free stores), then (m, l).
    static constexpr int kStride = D + 4;
    static constexpr int kStageBytes = (kConsumerWarps * G * kStride + 2 * kConsumerWarps * G) * 4;
};

// Shared-memory plan of one instantiation: cluster instances add the push
// merge's receive buffers (kPush: they fit at the instance's occupancy).
template <int D, int G, int kStages, bool kCluster>
struct StepAlloc {
    using L = StepSmem<D, kStages, kCluster>;
    using P = PushSmem<D, G>;
    static constexpr int kPushOff = (L::kBytes + 15) & ~15;
    // The deep ring also stages the four warps' states beside the receive
    // buffers, outside the ring (cluster_merge_push).
    static constexpr int kStageOff = kPushOff + ((P::kBytes + 15) & ~15);
    static constexpr int kTermOff =
        kStageOff + ((kStages == kDeepStages ? P::kStageBytes : 0) + 15) / 16 * 16;
    static constexpr int kPushAlloc = kTermOff + 1024;
    static constexpr int kPerSm = kStages == 2 ? 3 : (kStages == 3 ? 2 : 1);
    // 227 KB per CTA at most; 228 KB per SM, 1 KB of it reserved per CTA.
    static constexpr bool kPush =
        kCluster && kPushAlloc <= 232448 && kPerSm * (kPushAlloc + 1024) <= 233472;
    // The deep ring (one CTA per SM) keeps the chunk's score terms in what is
    // left of shared memory: [n][G] floats for chunks of up to kTermSlots
    // slots (the plan gives it no longer chunks).
    static constexpr bool kSmemTerms = kPush && kStages == kDeepStages;
    static constexpr int term_bytes() {
        const int m = (232448 - kPushAlloc) / 16 * 16;
        const int most = kMaxChunkTiles * kTile * G * 4;
        return m < 0 ? 0 : (m < most ? m : most);
    }
    static constexpr int kTermBytes = kSmemTerms ? term_bytes() : 0;
    static constexpr int kTermSlots = kTermBytes / (G * 4);
    static constexpr int kAlloc = kPush ? kPushAlloc + kTermBytes : L::kAlloc;
};

__device__ __forceinline__ void consumer_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Consumer barrier that also returns whether any consumer passed `pred`.
__device__ __forceinline__ bool consumer_bar_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "n"(kConsumers)
        : "memory");
    return r != 0;
}

// Byte offset of 16-byte chunk `cg` (8 bf16 columns) of tile row `row` in a
// swizzled K or V tile buffer.
constexpr int kBoxBytes = kTile * 128;  // one 64-row x 128-byte swizzled box

__device__ __forceinline__ uint32_t swz_off(int row, int cg) {
    return (cg >> 3) * kBoxBytes + row * 128 + (((cg & 7) ^ (row & 7)) << 4);
}

// log2 I_j of a live slot from its score terms, x_h = t_hj + c_h:
// I_j = sum_h 2^(x_h) = 2^M * sum_h 2^(x_h - M) with M = max_h x_h, so
// log2 I_j = M + log2(sum_h 2^(x_h - M)), the sum in [1, g]. fp32 holds this
// far below the range where I_j itself flushes to zero (a slot whose weight
// is hundreds of nats under the unit's maximum still has its own value).
// -inf for a zero score (every term -inf: a zero V row); NaN propagates. The
// "+ 0" turns a -0 into +0, so equal values have equal keys.
template <int G>
__device__ __forceinline__ float log2_score(const float (&t)[G], const float (&c)[G]) {
    float x[G];
    float M = -INFINITY;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        x[h] = t[h] + c[h];
        M = fmaxf(M, x[h]);
    }
    const float Mu = (M == -INFINITY || M == INFINITY) ? 0.f : M;
    float s = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) s += ex2_approx(x[h] - Mu);
    return Mu + __log2f(s) + 0.f;
}

// The linear score I_j = sum_h 2^(x_h) in fp32 (0 once below the normal
// range), for the score export.
template <int G>
__device__ __forceinline__ float linear_score(const float (&t)[G], const float (&c)[G]) {
    float I = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) I += ex2_approx(t[h] + c[h]);
    return I;
}

// Selection key of a live slot: the bits of log2 I_j mapped so that unsigned
// order is float order (negative values complemented, the sign bit set on
// the others). -inf maps to 0x007fffff and +inf to 0xff800000, which leaves
// key 0 for an empty slot ranked first (fill-empty-first) and 0xffffffff for
// "no candidate".
__device__ __forceinline__ uint32_t ordered_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// What the score export holds for a live slot: I_j, or log2 I_j with
// kFlagLog2Scores.
template <int G>
__device__ __forceinline__ float exported_score(const StepParams& p, float L, const float (&t)[G],
                                                const float (&c)[G]) {
    return (p.flags & kFlagLog2Scores) ? L : linear_score<G>(t, c);
}

template <int G>
__device__ __forceinline__ void load_terms(const float* t, float (&v)[G]) {
    if constexpr (G == 1) {
        v[0] = __ldcg(t);
    } else if constexpr (G == 2) {
        const float2 a = __ldcg(reinterpret_cast<const float2*>(t));
        v[0] = a.x;
        v[1] = a.y;
    } else {
#pragma unroll
        for (int q = 0; q < G / 4; ++q) {
            const float4 a = __ldcg(reinterpret_cast<const float4*>(t) + q);
            v[4 * q] = a.x;
            v[4 * q + 1] = a.y;
            v[4 * q + 2] = a.z;
            v[4 * q + 3] = a.w;
        }
    }
}

// The same from the chunk's term array in shared memory.
template <int G>
__device__ __forceinline__ void load_terms_smem(const float* t, float (&v)[G]) {
    if constexpr (G == 1) {
        v[0] = t[0];
    } else if constexpr (G == 2) {
        const float2 a = *reinterpret_cast<const float2*>(t);
        v[0] = a.x;
        v[1] = a.y;
    } else {
#pragma unroll
        for (int q = 0; q < G / 4; ++q) {
            const float4 a = reinterpret_cast<const float4*>(t)[q];
            v[4 * q] = a.x;
            v[4 * q + 1] = a.y;
            v[4 * q + 2] = a.z;
            v[4 * q + 3] = a.w;
        }
    }
}

// Drops the 128-byte lines lying wholly inside [p, p + bytes).
__device__ __forceinline__ void discard_range(const void* p, size_t bytes, int tid, int nthreads) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uintptr_t first = (a + 127) & ~static_cast<uintptr_t>(127);
    const uintptr_t end = (a + bytes) & ~static_cast<uintptr_t>(127);
    for (uintptr_t line = first + static_cast<uintptr_t>(tid) * 128; line < end;
         line += static_cast<uintptr_t>(nthreads) * 128)
        discard_l2_line(reinterpret_cast<const void*>(line));
}

// Lexicographic (key, slot) order of selection candidates.
__device__ __forceinline__ bool key_less(uint32_t ka, int ja, uint32_t kb, int jb) {
    return ka < kb || (ka == kb && ja < jb);
}

// One 8-bit radix-select pass over the unit's candidate keys: among values v
// with (v & pmask) == prefix, finds the digit (v >> shift) & 255 holding the
// `remaining`-th smallest and returns the rank left inside that digit. With
// by_slot the value is the slot index of keys equal to `tie_key`.
__device__ __forceinline__ int radix_pass(const uint32_t* keys, int stride, int S, int shift,
                                          uint32_t pmask, uint32_t prefix, int remaining,
                                          bool by_slot, uint32_t tie_key, int* hist,
                                          int* s_out, int tid, uint32_t* digit_out) {
    for (int i = tid; i < 256; i += kConsumers) hist[i] = 0;
    consumer_bar_sync();
    for (int j = tid; j < S; j += kConsumers) {
        const uint32_t key = __ldcg(keys + static_cast<size_t>(j) * stride);
        if (key == 0xffffffffu) continue;
        const uint32_t v = by_slot ? static_cast<uint32_t>(j) : key;
        if (by_slot && key != tie_key) continue;
        if ((v & pmask) == prefix) atomicAdd(&hist[(v >> shift) & 255], 1);
    }
    consumer_bar_sync();
    if (tid == 0) {
        int cum = 0, d = 255;
        for (int b = 0; b < 256; ++b) {
            if (cum + hist[b] >= remaining) {
                d = b;
                break;
            }
            cum += hist[b];
        }
        s_out[0] = d;
        s_out[1] = remaining - cum;
    }
    consumer_bar_sync();
    *digit_out = static_cast<uint32_t>(s_out[0]);
    return s_out[1];
}

// Shared memory of select_topk: histogram, scalars, the winners' keys and slots.
constexpr int kTopKAreaBytes = (256 + 4) * 4 + 2 * kMaxTopK * 4;

// The k smallest (key, slot) pairs of a unit, ascending, into next_slot[u][k]
// (-1 past the number of candidates). Keys were written one per slot (stride
// `stride` words); 0xffffffff marks a slot that is not a candidate.
__device__ void select_topk(const StepParams& p, int u, const uint32_t* keys, int stride,
                            int ncand, uint8_t* area, int tid) {
    const int S = p.S;
    const int k = p.topk;
    int* hist = reinterpret_cast<int*>(area);              // [256]
    int* s_out = hist + 256;                               // [4]
    uint32_t* l_key = reinterpret_cast<uint32_t*>(s_out + 4);  // [kMaxTopK]
    int* l_idx = reinterpret_cast<int*>(l_key + kMaxTopK);     // [kMaxTopK]
    const int keff = min(k, ncand);
    int32_t* out = p.next_slot + static_cast<size_t>(u) * k;
    if (keff > 0) {
        // Threshold key T: the keff-th smallest key.
        uint32_t prefix = 0, pmask = 0;
        int remaining = keff;
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            uint32_t dgt;
            remaining = radix_pass(keys, stride, S, shift, pmask, prefix, remaining, false, 0u,
                                   hist, s_out, tid, &dgt);
            prefix |= dgt << shift;
            pmask |= 0xffu << shift;
        }
        const uint32_t T = prefix;
        // Among keys equal to T, the `remaining` lowest slots: slot threshold J.
        uint32_t iprefix = 0, ipmask = 0;
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = 16 - 8 * pass;
            uint32_t dgt;
            remaining = radix_pass(keys, stride, S, shift, ipmask, iprefix, remaining, true, T,
                                   hist, s_out, tid, &dgt);
            iprefix |= dgt << shift;
            ipmask |= 0xffu << shift;
        }
        const int J = static_cast<int>(iprefix);
        if (tid == 0) s_out[2] = 0;
        consumer_bar_sync();
        for (int j = tid; j < S; j += kConsumers) {
            const uint32_t key = __ldcg(keys + static_cast<size_t>(j) * stride);
            if (key == 0xffffffffu) continue;
            if (key < T || (key == T && j <= J)) {
                const int pos = atomicAdd(&s_out[2], 1);
                if (pos < kMaxTopK) {
                    l_key[pos] = key;
                    l_idx[pos] = j;
                }
            }
        }
        consumer_bar_sync();
        // Bitonic sort of the keff winners by (key, slot).
        int n2 = 1;
        while (n2 < keff) n2 <<= 1;
        for (int i = keff + tid; i < n2; i += kConsumers) {
            l_key[i] = 0xffffffffu;
            l_idx[i] = 0x7fffffff;
        }
        consumer_bar_sync();
        for (int size = 2; size <= n2; size <<= 1) {
            for (int stride2 = size >> 1; stride2 > 0; stride2 >>= 1) {
                for (int i = tid; i < n2; i += kConsumers) {
                    const int ixj = i ^ stride2;
                    if (ixj > i) {
                        const bool up = (i & size) == 0;
                        const bool swap = up ? key_less(l_key[ixj], l_idx[ixj], l_key[i], l_idx[i])
                                             : key_less(l_key[i], l_idx[i], l_key[ixj], l_idx[ixj]);
                        if (swap) {
                            const uint32_t tk = l_key[i];
                            const int ti = l_idx[i];
                            l_key[i] = l_key[ixj];
                            l_idx[i] = l_idx[ixj];
                            l_key[ixj] = tk;
                            l_idx[ixj] = ti;
                        }
                    }
                }
                consumer_bar_sync();
            }
        }
    }
    for (int i = tid; i < k; i += kConsumers) {
        const int slot = (i < keff) ? l_idx[i] : -1;
        out[i] = slot;
        if (slot >= 0 && (p.flags & kFlagMaskEvicted))
            p.mask[static_cast<size_t>(u) * S + slot] = -1;
    }
}

template <int G>
__device__ void score_and_select(const StepParams& p, int u, const float* s_m, const float* s_il,
                                 float* red_v, int* red_j, int* s_ncand, const int* s_live,
                                 uint8_t* topk_area, uint8_t* scan_area, int scan_bytes,
                                 uint64_t* scan_bars, int tid);

// Merge of the unit's chunks by its last CTA (consumer threads only). The
// shared memory below `usable` is free; scan_bars are two spare mbarriers.
template <int D, int G, bool kScore>
__device__ void finish_unit(const StepParams& p, int u, uint8_t* smem, int usable,
                            uint64_t* scan_bars, int tid) {
    const int nchunk = p.nchunk;
    float* s_w = reinterpret_cast<float*>(smem);  // [nchunk][G]: 2^(m_c - m) / l
    float* s_m = s_w + nchunk * G;                // [G]
    float* s_il = s_m + G;                        // [G]
    float* red_v = s_il + G;                      // [4]
    int* red_j = reinterpret_cast<int*>(red_v + kConsumerWarps);
    int* s_ncand = red_j + kConsumerWarps;
    // [nchunk]: the chunk's live-tile bit mask (0: no live slot; all ones
    // when the masks were not kept)
    int* s_live = s_ncand + 4;
    uint8_t* topk_area = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(s_live + nchunk) + 15) & ~static_cast<uintptr_t>(15));
    uint8_t* scan_area = topk_area + (p.topk > 1 ? kTopKAreaBytes : 0);
    const int scan_bytes = usable - static_cast<int>(scan_area - smem);
    const float2* ml = p.part_ml + static_cast<size_t>(u) * nchunk * G;
    const int b = u / p.Hkv;
    const int kvh = u - b * p.Hkv;
    const float* po = p.part_o + static_cast<size_t>(u) * nchunk * G * D;
    __nv_bfloat16* out = p.out + (static_cast<size_t>(b) * p.Hq + kvh * G) * D;

    // The partial outputs of the first four chunks are requested first: they
    // do not depend on (m, l), so their round trip overlaps the weights'.
    constexpr int kPerT = (G * D + kConsumers - 1) / kConsumers;
    float v0[4][kPerT];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const int c = min(cc, nchunk - 1);
#pragma unroll
        for (int k = 0; k < kPerT; ++k) {
            const int e = tid + k * kConsumers;
            v0[cc][k] = (e < G * D) ? __ldcg(&po[static_cast<size_t>(c) * G * D + e]) : 0.f;
        }
    }

    // Chunk liveness for the score scan: the chunks' live-tile masks when
    // they were kept (0: no live slot), else from m_c below.
    // (Loaded into a register now, stored after the (m, l) loads are issued.)
    const bool kept = p.part_tiles && !(p.split && u >= p.split_from);
    const uint32_t* ptl = kept ? p.part_tiles + static_cast<size_t>(u) * nchunk : nullptr;
    const uint32_t my_tiles = (kScore && ptl && tid < nchunk) ? __ldcg(&ptl[tid]) : 0u;

    // Per head: m = max_c m_c, l = sum_c l_c 2^(m_c - m), weights
    // w_c = 2^(m_c - m) / l. Up to kFastChunks chunks thread h loads all of
    // its head's (m_c, l_c) at once and writes the weights itself.
    constexpr int kFastChunks = 16;
    const bool fast = nchunk <= kFastChunks;
    if (tid < G) {
        if (fast) {
            float2 mlv[kFastChunks];
#pragma unroll
            for (int c = 0; c < kFastChunks; ++c)
                if (c < nchunk) mlv[c] = __ldcg(&ml[c * G + tid]);
            float m = -INFINITY;
#pragma unroll
            for (int c = 0; c < kFastChunks; ++c)
                if (c < nchunk) m = fmaxf(m, mlv[c].x);
            float l = 0.f;
#pragma unroll
            for (int c = 0; c < kFastChunks; ++c)
                if (c < nchunk && mlv[c].x != -INFINITY) l += mlv[c].y * exp2f(mlv[c].x - m);
            const float il = (l > 0.f) ? 1.f / l : 0.f;
            s_m[tid] = m;
            s_il[tid] = il;
#pragma unroll
            for (int c = 0; c < kFastChunks; ++c) {
                if (c < nchunk) {
                    s_w[c * G + tid] = (mlv[c].x == -INFINITY) ? 0.f : exp2f(mlv[c].x - m) * il;
                    if (tid == 0 && !(kScore && ptl))
                        s_live[c] = mlv[c].x != -INFINITY ? -1 : 0;  // m = -inf: no live slot
                }
            }
        } else {
            float m = -INFINITY;
            for (int c = 0; c < nchunk; ++c) m = fmaxf(m, __ldcg(&ml[c * G + tid]).x);
            float l = 0.f;
            for (int c = 0; c < nchunk; ++c) {
                const float2 v = __ldcg(&ml[c * G + tid]);
                if (v.x != -INFINITY) l += v.y * exp2f(v.x - m);
            }
            s_m[tid] = m;
            s_il[tid] = (l > 0.f) ? 1.f / l : 0.f;
        }
    }
    if (kScore && ptl) {
        if (tid < nchunk) s_live[tid] = static_cast<int>(my_tiles);
        for (int c = tid + kConsumers; c < nchunk; c += kConsumers)
            s_live[c] = static_cast<int>(__ldcg(&ptl[c]));
    }
    if (tid == 0) s_ncand[0] = 0;
    consumer_bar_sync();
    if (!fast) {
        for (int e = tid; e < nchunk * G; e += kConsumers) {
            const float2 v = __ldcg(&ml[e]);
            const int h = e % G;
            s_w[e] = (v.x == -INFINITY) ? 0.f : exp2f(v.x - s_m[h]) * s_il[h];
            if (h == 0 && !(kScore && ptl))
                s_live[e / G] = v.x != -INFINITY ? -1 : 0;  // m = -inf: no live slot
        }
        consumer_bar_sync();
    }

    // Output: O_h = sum_c w_ch * O_ch, rounded to bf16. Four chunks' loads
    // are in flight at a time; a chunk that had no live tile has weight 0 and
    // its (unwritten) partial is selected away.
    float o[kPerT];
#pragma unroll
    for (int k = 0; k < kPerT; ++k) o[k] = 0.f;
    for (int c0 = 0; c0 < nchunk; c0 += 4) {
        float v[4][kPerT];
        if (c0 == 0) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int k = 0; k < kPerT; ++k) v[cc][k] = v0[cc][k];
        } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int c = min(c0 + cc, nchunk - 1);
#pragma unroll
                for (int k = 0; k < kPerT; ++k) {
                    const int e = tid + k * kConsumers;
                    v[cc][k] = (e < G * D) ? __ldcg(&po[static_cast<size_t>(c) * G * D + e]) : 0.f;
                }
            }
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c = c0 + cc;
            if (c >= nchunk) break;
#pragma unroll
            for (int k = 0; k < kPerT; ++k) {
                const int e = tid + k * kConsumers;
                const float w = (e < G * D) ? s_w[c * G + e / D] : 0.f;
                o[k] += (w != 0.f) ? w * v[cc][k] : 0.f;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kPerT; ++k) {
        const int e = tid + k * kConsumers;
        if (e < G * D) out[e] = __float2bfloat16_rn(o[k]);
    }
    if constexpr (kScore) {
        if (p.split && u >= p.split_from) {
            // The scoring kernel that follows scores the chunks in parallel
            // once the unit's flag is up: publish c_h, then release the flag
            // after every write it reads (c_h, and through the arrival
            // counter, the chunks' score terms and ages).
            if (tid < G) p.cfold[static_cast<size_t>(u) * G + tid] = __log2f(s_il[tid]) - s_m[tid];
            consumer_bar_sync();
            if (tid == 0) st_release_gpu(p.ready + u, 1u);  // after the barrier: the CTA's writes
        } else {
            score_and_select<G>(p, u, s_m, s_il, red_v, red_j, s_ncand, s_live, topk_area,
                                scan_area, scan_bytes, scan_bars, tid);
        }
    }
    consumer_bar_sync();
    // Every read of the unit's scratch is done: drop the lines, no write-back.
    discard_range(po, static_cast<size_t>(nchunk) * G * D * sizeof(float), tid, kConsumers);
}

// Segments of a unit's slot axis that the score scan visits, in order: pieces
// of at most `seg` slots of the runs of consecutive chunks that hold a live
// slot (of all chunks when `all` is set). The same walk runs in every
// consumer thread.
struct SegWalk {
    int j0;    // first slot of the current segment (>= S: done)
    int rend;  // end of the current run of chunks
};

__device__ __forceinline__ int next_chunk(int c, int nchunk, const int* s_live, bool all) {
    while (c < nchunk && !(all || s_live[c])) ++c;
    return c;
}

// Starts a run at chunk c (or ends the walk when c == nchunk).
__device__ __forceinline__ SegWalk seg_run(int c, int cs, int S, int nchunk, const int* s_live,
                                           bool all) {
    if (c >= nchunk) return SegWalk{S, S};
    int e = c;
    while (e + 1 < nchunk && (all || s_live[e + 1])) ++e;
    return SegWalk{c * cs, min((e + 1) * cs, S)};
}

__device__ __forceinline__ int seg_end(const SegWalk& w, int seg) { return min(w.j0 + seg, w.rend); }

__device__ __forceinline__ void seg_advance(SegWalk& w, int cs, int seg, int S, int nchunk,
                                            const int* s_live, bool all) {
    const int e = seg_end(w, seg);
    if (e < w.rend)
        w.j0 = e;
    else
        w = seg_run(next_chunk((w.rend + cs - 1) / cs, nchunk, s_live, all), cs, S, nchunk,
                    s_live, all);
}

// Units with more slots to score than this stream them through shared memory.
constexpr int kBulkScanMinSlots = 4096;
// The live-tile list of the top-1 register scan holds at most this many tiles.
constexpr int kMaxScanTiles = 1024;

// LongFlowScore of every live slot of unit u and the selection of the slots to
// evict, by the unit's last CTA once the final (m_h, l_h) are known.
template <int G>
__device__ void score_and_select(const StepParams& p, int u, const float* s_m, const float* s_il,
                                 float* red_v, int* red_j, int* s_ncand, const int* s_live,
                                 uint8_t* topk_area, uint8_t* scan_area, int scan_bytes,
                                 uint64_t* scan_bars, int tid) {
    // Candidates: live slots with age >= W and, with kFlagFillEmptyFirst,
    // empty slots (ranked before every score, lowest slot first).
    // I_j = sum_h 2^(t_hj - m_h) / l_h = sum_h 2^(t_hj + c_h), c_h = log2(1/l_h) - m_h.
    float c[G];
#pragma unroll
    for (int h = 0; h < G; ++h) c[h] = __log2f(s_il[h]) - s_m[h];
    const int S = p.S;
    const int nchunk = p.nchunk;
    const int cs = p.chunk_tiles * kTile;
    const int32_t* age = p.mask + static_cast<size_t>(u) * S;
    float* stash = p.stash + static_cast<size_t>(u) * S * G;
    // For top-k the slot's first stash word is reused for its selection key.
    uint32_t* keys = reinterpret_cast<uint32_t*>(stash);
    float* scores = p.scores ? p.scores + static_cast<size_t>(u) * S : nullptr;
    const bool fill_first = (p.flags & kFlagFillEmptyFirst) != 0;
    const bool top1 = p.topk == 1;
    // Chunks without a live slot hold no scored candidate; they are visited
    // only when empty slots are candidates or every score is wanted.
    const bool all = fill_first || scores != nullptr;
    const int W = p.W;
    // Selection key of a candidate: ordered_key(log2 I_j), 0 for an empty
    // slot under fill-empty-first; ~0u: none.
    uint32_t bkey = 0xffffffffu;  // top-1: this thread's best (key, slot)
    int bestj = 0x7fffffff;
    int ncand = 0;

    auto visit = [&](int j, int a, const float (&t)[G]) {
        const float L = log2_score<G>(t, c);
        const bool live = a >= 0;
        const bool cand = live ? (a >= W && L == L) : fill_first;
        const uint32_t key = live ? ordered_key(L) : 0u;
        if (top1) {
            // A thread visits its slots in increasing order, so a strict "<"
            // keeps the lowest slot among equal keys.
            if (cand && key < bkey) {
                bkey = key;
                bestj = j;
            }
        } else {
            keys[static_cast<size_t>(j) * G] = cand ? key : 0xffffffffu;
            ncand += cand ? 1 : 0;
        }
        if (scores) scores[j] = live ? exported_score<G>(p, L, t, c) : INFINITY;
    };

    if (!all && !top1) {
        // Top-k reads a key for every slot: skipped chunks hold no candidate.
        for (int c = 0; c < nchunk; ++c)
            if (!s_live[c])
                for (int j = c * cs + tid; j < min(S, (c + 1) * cs); j += kConsumers)
                    keys[static_cast<size_t>(j) * G] = 0xffffffffu;
    }

    // A long scan streams each segment's ages and score terms into shared memory
    // with bulk copies, two segments in flight, so it runs at L2 bandwidth
    // instead of one round trip per slot.
    constexpr int kSlotBytes = (G + 1) * 4;
    int seg = (scan_bytes / 2) / kSlotBytes;
    seg = min(2048, seg & ~(kConsumers - 1));
    // Short units are cheaper with loads batched in registers (one or two
    // round trips); long ones stream through shared memory.
    int nlive = 0;
    int live_tiles = 0;  // (from the live-tile masks when they were kept)
    for (int c = 0; c < nchunk; ++c) {
        nlive += (all || s_live[c]) ? 1 : 0;
        live_tiles += __popc(static_cast<uint32_t>(s_live[c]));
    }
    const bool bulk = seg >= kConsumers && nlive * cs > kBulkScanMinSlots && (S & 3) == 0 &&
                      (reinterpret_cast<uintptr_t>(p.mask) & 15) == 0;
    if (bulk) {
        const int half = seg * kSlotBytes;
        uint8_t* buf0 = reinterpret_cast<uint8_t*>(
            (reinterpret_cast<uintptr_t>(scan_area) + 15) & ~static_cast<uintptr_t>(15));
        if (tid == 0) {
            mbar_init(&scan_bars[0], 1);
            mbar_init(&scan_bars[1], 1);
            fence_barrier_init();
            // The ages and score terms were written through the generic proxy
            // (here and by the unit's other CTAs); the copies read them through
            // the async proxy.
            asm volatile("fence.proxy.async;" ::: "memory");
        }
        consumer_bar_sync();
        SegWalk wi = seg_run(next_chunk(0, nchunk, s_live, all), cs, S, nchunk, s_live, all);
        SegWalk wc = wi;
        int issued = 0;
        auto issue = [&](int s_idx) {
            const int j1 = seg_end(wi, seg);
            const int n = j1 - wi.j0;
            uint8_t* b = buf0 + (s_idx & 1) * half;
            uint64_t* bar = &scan_bars[s_idx & 1];
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * kSlotBytes));
            bulk_load(b, age + wi.j0, static_cast<uint32_t>(n * 4), bar);
            bulk_load(b + seg * 4, stash + static_cast<size_t>(wi.j0) * G,
                      static_cast<uint32_t>(n * G * 4), bar);
            seg_advance(wi, cs, seg, S, nchunk, s_live, all);
        };
        if (tid == 0) {
            for (; issued < 2 && wi.j0 < S; ++issued) issue(issued);
        }
        int s_idx = 0;
        for (; wc.j0 < S; ++s_idx) {
            const int b = s_idx & 1;
            const bool timed_out = !mbar_wait(&scan_bars[b], (s_idx >> 1) & 1, p.wait_limit_ns);
            if (consumer_bar_or(timed_out)) {
                if (tid == 0) {
                    atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);
                    // Copies still in flight land before the CTA retires.
                    for (int q = s_idx; q < issued; ++q)
                        (void)mbar_wait(&scan_bars[q & 1], (q >> 1) & 1);
                }
                break;
            }
            const int32_t* s_age = reinterpret_cast<const int32_t*>(buf0 + b * half);
            const float* s_t = reinterpret_cast<const float*>(buf0 + b * half + seg * 4);
            const int n = seg_end(wc, seg) - wc.j0;
#pragma unroll 4
            for (int i = tid; i < n; i += kConsumers) {
                float t[G];
                if constexpr (G >= 4) {
#pragma unroll
                    for (int q4 = 0; q4 < G / 4; ++q4) {
                        const float4 v = reinterpret_cast<const float4*>(s_t + i * G)[q4];
                        t[4 * q4] = v.x;
                        t[4 * q4 + 1] = v.y;
                        t[4 * q4 + 2] = v.z;
                        t[4 * q4 + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < G; ++h) t[h] = s_t[i * G + h];
                }
                visit(wc.j0 + i, s_age[i], t);
            }
            consumer_bar_sync();  // everyone is done with buffer b
            if (tid == 0 && wi.j0 < S) issue(issued++);
            seg_advance(wc, cs, seg, S, nchunk, s_live, all);
        }
    } else if (top1 && !all && p.part_tiles && nlive * p.chunk_tiles <= kMaxScanTiles &&
               live_tiles < (S + kTile - 1) / kTile) {
        // Top-1 over live tiles only, when some tile holds no live slot: the
        // chunks' live-tile masks are expanded into a list of tile indices,
        // and the batches walk the slots of the listed tiles (a ragged unit
        // scans its live part, not all S slots). A thread still visits its
        // slots in increasing order.
        constexpr int kBatch = 8;
        int* s_tl = reinterpret_cast<int*>(
            (reinterpret_cast<uintptr_t>(scan_area) + 15) & ~static_cast<uintptr_t>(15));
        if (tid < 32) {
            int nt = 0;
            for (int c = 0; c < nchunk; ++c) {
                const uint32_t bits = static_cast<uint32_t>(s_live[c]);
                if (!bits) continue;
                if (tid < p.chunk_tiles && ((bits >> tid) & 1u))
                    s_tl[nt + __popc(bits & ((1u << tid) - 1u))] = c * p.chunk_tiles + tid;
                nt += __popc(bits);
            }
            if (tid == 0) s_ncand[1] = nt;
        }
        consumer_bar_sync();
        const int nslots = s_ncand[1] * kTile;
        for (int i0 = tid; i0 < nslots; i0 += kBatch * kConsumers) {
            int a[kBatch];
            int jj[kBatch];
            float t[kBatch][G];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int i = i0 + k * kConsumers;
                jj[k] = (i < nslots) ? s_tl[i >> 6] * kTile + (i & (kTile - 1)) : S;
                a[k] = (jj[k] < S) ? __ldcg(&age[jj[k]]) : -1;
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k)
                if (jj[k] < S) load_terms<G>(stash + static_cast<size_t>(jj[k]) * G, t[k]);
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (jj[k] >= S) break;
                visit(jj[k], a[k], t[k]);
            }
        }
    } else {
        // Batches of loads in flight per thread (also for slot counts that
        // break the 16-byte copy alignment): 13 per thread covers a
        // 3200-slot unit in two round trips without spilling (g <= 4).
        constexpr int kBatch = G <= 4 ? 13 : 8;
        for (int j0 = tid; j0 < S; j0 += kBatch * kConsumers) {
            int a[kBatch];
            float t[kBatch][G];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int j = j0 + k * kConsumers;
                a[k] = (j < S) ? __ldcg(&age[j]) : -1;
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int j = j0 + k * kConsumers;
                if (j < S) load_terms<G>(stash + static_cast<size_t>(j) * G, t[k]);
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int j = j0 + k * kConsumers;
                if (j >= S) break;
                visit(j, a[k], t[k]);  // a slot of a chunk with no live slot is no candidate
            }
        }
    }

    if (top1) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const uint32_t ok = __shfl_xor_sync(0xffffffffu, bkey, off);
            const int oj = __shfl_xor_sync(0xffffffffu, bestj, off);
            if (key_less(ok, oj, bkey, bestj)) {
                bkey = ok;
                bestj = oj;
            }
        }
        uint32_t* red_k = reinterpret_cast<uint32_t*>(red_v);
        if ((tid & 31) == 0) {
            red_k[tid >> 5] = bkey;
            red_j[tid >> 5] = bestj;
        }
        consumer_bar_sync();
        if (tid == 0) {
            for (int w = 1; w < kConsumerWarps; ++w)
                if (key_less(red_k[w], red_j[w], bkey, bestj)) {
                    bkey = red_k[w];
                    bestj = red_j[w];
                }
            const int slot = (bkey == 0xffffffffu) ? -1 : bestj;
            p.next_slot[u] = slot;
            if (slot >= 0 && (p.flags & kFlagMaskEvicted))
                p.mask[static_cast<size_t>(u) * S + slot] = -1;
        }
    } else {
        if (ncand) atomicAdd(s_ncand, ncand);
        consumer_bar_sync();
        select_topk(p, u, keys, G, s_ncand[0], topk_area, tid);
    }
    consumer_bar_sync();
    discard_range(stash, static_cast<size_t>(S) * G * sizeof(float), tid, kConsumers);
}

// Shared-memory bytes finish_unit needs (it reuses the pipeline buffers).
__host__ __device__ constexpr size_t finish_smem_bytes(int nchunk, int G, int topk) {
    return (static_cast<size_t>(nchunk) * (G + 1) + 2 * G + 2 * kConsumerWarps + 4) * 4 + 16 +
           (topk > 1 ? kTopKAreaBytes : 0);
}

// Score terms of the cluster epilogues' first scan batch, requested before
// the merge so that their round trip overlaps it.
constexpr int kScoreBatch = 8;

template <int G>
__device__ __forceinline__ void preload_terms(const StepParams& p, int u, int slot0, int n,
                                              const uint8_t* sflags, int tid,
                                              float (&t0)[kScoreBatch][G]) {
    const float* stash0 = p.stash + (static_cast<size_t>(u) * p.S + slot0) * G;
#pragma unroll
    for (int k = 0; k < kScoreBatch; ++k) {
        const int i = tid + k * kConsumers;
        if (i < n && (sflags[i] & kSlotLive))
            load_terms<G>(stash0 + static_cast<size_t>(i) * G, t0[k]);
    }
}

// LongFlowScore of the chunk's slots slot0 .. slot0 + n - 1 (consumer thread
// tid takes slots tid, tid + 128, ...) from their score terms and c_h, the
// score export, and the thread's best candidate (key, slot): key 0xffffffff
// and slot 0x7fffffff when it has none. t0 holds the first batch when
// kPreloaded.
template <int G, bool kPreloaded, bool kSmemTerms = false>
__device__ __forceinline__ void score_chunk(const StepParams& p, int u, int slot0, int n,
                                            const uint8_t* sflags, const float (&cexp)[G],
                                            const float (&t0)[kScoreBatch][G], int tid,
                                            uint32_t& bkey, int& bestj,
                                            const float* sterm = nullptr) {
    const int S = p.S;
    const float* stash = p.stash + static_cast<size_t>(u) * S * G;
    float* scores = p.scores ? p.scores + static_cast<size_t>(u) * S : nullptr;
    const bool fill_first = (p.flags & kFlagFillEmptyFirst) != 0;
    // A thread visits its slots in increasing order, so a strict "<" on
    // the key (ordered_key(log2 I_j); 0 for an empty slot under
    // fill-empty-first) keeps the lowest slot among equal keys.
    bkey = 0xffffffffu;
    bestj = 0x7fffffff;
    if constexpr (kSmemTerms) {
        // Terms in shared memory: two slots per thread and round, both
        // computed without a branch between them, so their dependent chains
        // interleave (one warp per SM sub-partition hides no latency here).
        constexpr int kB = 2;
        for (int i0 = tid; i0 < n; i0 += kB * kConsumers) {
            float L[kB], t[kB][G];
            int f[kB];
#pragma unroll
            for (int k = 0; k < kB; ++k) {
                const int i = i0 + k * kConsumers;
                f[k] = (i < n) ? sflags[i] : 0;
                if (f[k] & kSlotLive) {
                    load_terms_smem<G>(sterm + i * G, t[k]);
                } else {
#pragma unroll
                    for (int h = 0; h < G; ++h) t[k][h] = -INFINITY;
                }
                L[k] = log2_score<G>(t[k], cexp);
            }
#pragma unroll
            for (int k = 0; k < kB; ++k) {
                const int i = i0 + k * kConsumers;
                if (i < n) {
                    const int j = slot0 + i;
                    const bool live = (f[k] & kSlotLive) != 0;
                    const bool cand = live ? ((f[k] & kSlotOld) && L[k] == L[k]) : fill_first;
                    const uint32_t key = live ? ordered_key(L[k]) : 0u;
                    if (cand && key < bkey) {
                        bkey = key;
                        bestj = j;
                    }
                    if (scores)
                        scores[j] = live ? exported_score<G>(p, L[k], t[k], cexp) : INFINITY;
                }
            }
        }
    } else {
        for (int i0 = tid; i0 < n; i0 += kScoreBatch * kConsumers) {
            float t[kScoreBatch][G];
            if (kPreloaded && i0 == tid) {
#pragma unroll
                for (int k = 0; k < kScoreBatch; ++k)
#pragma unroll
                    for (int h = 0; h < G; ++h) t[k][h] = t0[k][h];
            } else {
#pragma unroll
                for (int k = 0; k < kScoreBatch; ++k) {
                    const int i = i0 + k * kConsumers;
                    if (i < n && (sflags[i] & kSlotLive))
                        load_terms<G>(stash + static_cast<size_t>(slot0 + i) * G, t[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < kScoreBatch; ++k) {
                const int i = i0 + k * kConsumers;
                if (i >= n) break;
                const int f = sflags[i];
                const int j = slot0 + i;
                const float L = log2_score<G>(t[k], cexp);
                const bool live = (f & kSlotLive) != 0;
                const bool cand = live ? ((f & kSlotOld) && L == L) : fill_first;
                const uint32_t key = live ? ordered_key(L) : 0u;
                if (cand && key < bkey) {
                    bkey = key;
                    bestj = j;
                }
                if (scores) scores[j] = live ? exported_score<G>(p, L, t[k], cexp) : INFINITY;
            }
        }
    }
}

// The warp's lexicographic (key, slot) minimum, in every lane, by two warp
// reductions: the least key, then the least slot among the lanes holding it.
__device__ __forceinline__ void warp_best_redux(uint32_t& bkey, int& bestj) {
    const uint32_t kmin = __reduce_min_sync(0xffffffffu, bkey);
    const uint32_t jmin = __reduce_min_sync(
        0xffffffffu, bkey == kmin ? static_cast<uint32_t>(bestj) : 0xffffffffu);
    bkey = kmin;
    bestj = static_cast<int>(jmin);
}

// Merge of a cluster unit by pushes (StepAlloc::kPush). The CTA merges its
// four warps' online-softmax states in shared memory, then sends the CTA's
// (m, l) per head into every CTA and, one 16-byte piece per consumer thread,
// its merged output row into the CTAs that own the pieces (PushSmem), with
// asynchronous remote stores counted on the receiver's (m, l) and output
// barriers; each warp arrives on its own CTA's barriers for the stores it
// made locally. With every chunk's (m, l) a CTA scores its own chunk with
// c_h = log2(1/l_h) - m_h and sends its best (key, slot) to rank 0 while the
// output pieces land; then it writes the output elements it owns, and rank 0
// reduces the cluster's argmin. No cluster barrier follows the main loop:
// every store into a CTA is counted on one of its barriers, and a CTA leaves
// only after its own have completed.
template <int D, int G, int kStages, bool kScore, bool kSmemTerms>
__device__ __forceinline__ void cluster_merge_push(const StepParams& p, int u, int slot0, int n,
                                                   const uint8_t* sflags, uint8_t* smem,
                                                   uint8_t* pbase, uint8_t* wstage,
                                                   const float* sterm,
                                                   const float (&acc)[D / 16][4],
                                                   float m0, float m1, float l0, float l1,
                                                   int tid) {
    using P = PushSmem<D, G>;
    constexpr int kElems = P::kElems;
    constexpr int kStride = P::kStride;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int nchunk = p.nchunk;
    const int rank = static_cast<int>(cluster_ctarank());
    const int per = P::per(nchunk);
    float* recv_o = reinterpret_cast<float*>(pbase + P::kOOff);
    float2* recv_ml = reinterpret_cast<float2*>(pbase + P::kMlOff);
    uint2* recv_best = reinterpret_cast<uint2*>(pbase + P::kBestOff);
    float* s_w = reinterpret_cast<float*>(pbase + P::kWOff);
    float* s_m = reinterpret_cast<float*>(pbase + P::kMOff);
    float* s_il = reinterpret_cast<float*>(pbase + P::kIlOff);
    uint32_t* red_k = reinterpret_cast<uint32_t*>(pbase + P::kRedOff);
    int* red_j = reinterpret_cast<int*>(red_k + kConsumerWarps);
    uint64_t* bar_ml = reinterpret_cast<uint64_t*>(pbase + P::kBarOff);
    uint64_t* bar_o = bar_ml + 1;
    uint64_t* bar_best = bar_ml + 2;
    // The deep ring stages the warps' states outside the ring, so they need
    // no barrier before it; the others wait until every warp is done with
    // the ring.
    constexpr bool kStageOutside = kStages == kDeepStages;
    float* wO = reinterpret_cast<float*>(kStageOutside ? wstage : smem);  // [4][G][kStride]
    float* wm = wO + kConsumerWarps * G * kStride;                        // [4][G]
    float* wl = wm + kConsumerWarps * G;                                  // [4][G]
    const float NEG = -INFINITY;

    // The chunk's first batch of score terms, requested before the merge
    // (held across it only where registers allow). Every slot's terms were
    // stored by the warp that owns its row: a barrier orders them before
    // these loads.
    constexpr bool kPreload = kScore && !kSmemTerms && (G <= 4 || kStages == kDeepStages);
    float t0[kScoreBatch][G];
    if constexpr (!kStageOutside) {
        consumer_bar_sync();
        if constexpr (kPreload) preload_terms<G>(p, u, slot0, n, sflags, tid, t0);
    }

    // The four warps' states: lane (r, pair) holds heads h0 = 2 pair, h0 + 1
    // of rows mt * 16 + r and + 8 of every 16-row block.
    {
        const int r = lane >> 2;
        const int h0 = 2 * (lane & 3);
        if (r == 0) {
            if (h0 < G) { wm[warp * G + h0] = m0; wl[warp * G + h0] = l0; }
            if (h0 + 1 < G) { wm[warp * G + h0 + 1] = m1; wl[warp * G + h0 + 1] = l1; }
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int dd = mt * 16 + r;
            if (h0 < G) {
                wO[(warp * G + h0) * kStride + dd] = acc[mt][0];
                wO[(warp * G + h0) * kStride + dd + 8] = acc[mt][2];
            }
            if (h0 + 1 < G) {
                wO[(warp * G + h0 + 1) * kStride + dd] = acc[mt][1];
                wO[(warp * G + h0 + 1) * kStride + dd + 8] = acc[mt][3];
            }
        }
    }
    consumer_bar_sync();
    if constexpr (kStageOutside && kPreload) preload_terms<G>(p, u, slot0, n, sflags, tid, t0);

    // Every CTA of the cluster has initialised its barriers (the split
    // barrier begun at kernel start).
    cluster_wait();

    // The CTA's (m, l) of head h to CTA c (thread c * G + h), then its merged
    // output row, 4 elements per thread, each piece to the CTA that owns it.
    if (tid < nchunk * G) {
        const int c = tid / G;
        const int h = tid - c * G;
        float mh = NEG, l = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) mh = fmaxf(mh, wm[w * G + h]);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = wm[w * G + h];
            if (mw != NEG) l += wl[w * G + h] * exp2f(mw - mh);
        }
        float2* dst = &recv_ml[rank * G + h];
        if (c == rank)
            *dst = make_float2(mh, l);
        else
            st_async_v2(dsmem_addr(dst, c), __float_as_uint(mh), __float_as_uint(l),
                        dsmem_addr(bar_ml, c));
    }
    for (int e = 4 * tid; e < kElems; e += 4 * kConsumers) {
        const int h = e / D;
        const int d = e - h * D;
        float mw[kConsumerWarps];
        float mh = NEG;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            mw[w] = wm[w * G + h];
            mh = fmaxf(mh, mw[w]);
        }
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            if (mw[w] != NEG) {
                const float ew = exp2f(mw[w] - mh);
                const float4 v = *reinterpret_cast<const float4*>(&wO[(w * G + h) * kStride + d]);
                o.x += v.x * ew;
                o.y += v.y * ew;
                o.z += v.z * ew;
                o.w += v.w * ew;
            }
        }
        const int c = e / per;
        float* dst = &recv_o[rank * per + (e - c * per)];
        if (c == rank)
            *reinterpret_cast<float4*>(dst) = o;
        else
            st_async_v4(dsmem_addr(dst, c), o.x, o.y, o.z, o.w, dsmem_addr(bar_o, c));
    }
    __syncwarp();
    if (lane == 0) {  // this warp's local stores
        mbar_arrive(bar_ml);
        mbar_arrive(bar_o);
    }
    // These barriers complete only when every store into this CTA has
    // landed, so they take the full limit even under a shortened diagnostic
    // one: the CTA must not leave while a peer's stores are in flight. (A
    // main loop that gave up still stores its partial state, so they end.)
    if (!mbar_wait_cluster(bar_ml, 0) && lane == 0) atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);

    // Per head (warp h): m_h over the chunks, l_h and every chunk's weight
    // 2^(m_c - m_h) / l_h.
    for (int h = warp; h < G; h += kConsumerWarps) {
        const float2 a = (lane < nchunk) ? recv_ml[lane * G + h] : make_float2(NEG, 0.f);
        float m = a.x;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float ea = (a.x == NEG) ? 0.f : exp2f(a.x - m);
        float l = a.y * ea;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        const float il = (l > 0.f) ? 1.f / l : 0.f;
        if (lane < nchunk) s_w[lane * G + h] = ea * il;
        if (lane == 0) {
            s_m[h] = m;
            s_il[h] = il;
        }
    }
    consumer_bar_sync();

    // The chunk's scores and its best candidate, sent to rank 0.
    uint32_t bkey = 0xffffffffu;
    int bestj = 0x7fffffff;
    if constexpr (kScore) {
        float cexp[G];
#pragma unroll
        for (int h = 0; h < G; ++h) cexp[h] = __log2f(s_il[h]) - s_m[h];
        // (Terms in shared memory: the barrier after the staging ordered them.)
        score_chunk<G, kPreload, kSmemTerms>(p, u, slot0, n, sflags, cexp, t0, tid, bkey, bestj,
                                             sterm);
        warp_best_redux(bkey, bestj);
        if (lane == 0) {
            red_k[warp] = bkey;
            red_j[warp] = bestj;
        }
        consumer_bar_sync();
        if (tid == 0) {
            for (int w = 1; w < kConsumerWarps; ++w)
                if (key_less(red_k[w], red_j[w], bkey, bestj)) {
                    bkey = red_k[w];
                    bestj = red_j[w];
                }
            if (rank != 0)
                st_async_v2(dsmem_addr(&recv_best[rank], 0u), bkey, static_cast<uint32_t>(bestj),
                            dsmem_addr(bar_best, 0u));
        }
    }

    // The output elements this CTA owns: O_h = sum_c w_ch O_ch.
    if (!mbar_wait_cluster(bar_o, 0) && lane == 0) atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);
    {
        const int b = u / p.Hkv;
        const int kvh = u - b * p.Hkv;
        __nv_bfloat16* out = p.out + (static_cast<size_t>(b) * p.Hq + kvh * G) * D;
        const int e0 = rank * per;
        const int cnt = min(per, kElems - e0);
        for (int e = tid; e < cnt; e += kConsumers) {
            const int h = (e0 + e) / D;
            // Every chunk's weight and partial are loaded before the first is
            // used (a predicated unroll over the largest cluster), then summed
            // in chunk order.
            float wv[kMaxClusterChunks], ov[kMaxClusterChunks];
#pragma unroll
            for (int c = 0; c < kMaxClusterChunks; ++c) {
                wv[c] = (c < nchunk) ? s_w[c * G + h] : 0.f;
                ov[c] = (c < nchunk) ? recv_o[c * per + e] : 0.f;
            }
            float o = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxClusterChunks; ++c) o += (wv[c] != 0.f) ? wv[c] * ov[c] : 0.f;
            out[e0 + e] = __float2bfloat16_rn(o);
        }
    }

    if constexpr (kScore) {
        if (tid == 0 && rank == 0) {
            if (nchunk > 1 && !mbar_wait_cluster(bar_best, 0))  // full limit, as above
                atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);
            for (int c = 1; c < nchunk; ++c) {
                const uint2 v = recv_best[c];
                if (key_less(v.x, static_cast<int>(v.y), bkey, bestj)) {
                    bkey = v.x;
                    bestj = static_cast<int>(v.y);
                }
            }
            const int slot = (bestj == 0x7fffffff) ? -1 : bestj;
            p.next_slot[u] = slot;
            if (slot >= 0 && (p.flags & kFlagMaskEvicted))
                p.mask[static_cast<size_t>(u) * p.S + slot] = -1;
        }
        // This chunk's score terms are read: drop them from L2, no write-back.
        if constexpr (!kSmemTerms) {
            const float* stash = p.stash + (static_cast<size_t>(u) * p.S + slot0) * G;
            discard_range(stash, static_cast<size_t>(n) * G * 4, tid, kConsumers);
        }
    }
}

// Arms a receive barrier for `bytes` bytes of remote stores (a plain arrival
// when there are none).
__device__ __forceinline__ void arm_receive(uint64_t* bar, uint32_t bytes) {
    if (bytes > 0)
        mbar_arrive_expect_tx(bar, bytes);
    else
        mbar_arrive(bar);
}

// The push merge's barriers, armed at kernel start with the bytes the other
// nchunk - 1 CTAs store: their (m, l) per head, the output elements this CTA
// owns and, at rank 0, their (key, slot) pairs. The (m, l) and output
// barriers also count the four consumer warps' arrivals for their local
// stores.
template <int D, int G, bool kScore>
__device__ __forceinline__ void push_barriers_init(uint8_t* pbase, int nchunk) {
    using P = PushSmem<D, G>;
    uint64_t* bar_ml = reinterpret_cast<uint64_t*>(pbase + P::kBarOff);
    uint64_t* bar_o = bar_ml + 1;
    uint64_t* bar_best = bar_ml + 2;
    const int rank = static_cast<int>(cluster_ctarank());
    mbar_init(bar_ml, 1 + kConsumerWarps);
    mbar_init(bar_o, 1 + kConsumerWarps);
    mbar_init(bar_best, 1);
    const int per = P::per(nchunk);
    const uint32_t own = static_cast<uint32_t>(max(0, min(per, P::kElems - rank * per)));
    const uint32_t peers = static_cast<uint32_t>(nchunk - 1);
    arm_receive(bar_ml, peers * G * 8u);
    arm_receive(bar_o, peers * own * 4u);
    if (kScore && rank == 0) arm_receive(bar_best, peers * 8u);
}

// kStages-deep TMA ring; 3 stages run 2 CTAs per SM, 2 stages run 3.
// kScore = false is the attention-only variant (no ageing, score or eviction).
// kCluster: the grid is launched in clusters of nchunk CTAs (one per unit).
template <int D, int G, int kStages, bool kScore, bool kCluster>
__global__ void __launch_bounds__(kThreads, kStages == 2 ? 3 : (kStages == 3 ? 2 : 1))
    lf_decode_step_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const StepParams p) {
    using L = StepSmem<D, kStages, kCluster>;
    using A = StepAlloc<D, G, kStages, kCluster>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    using Slot = SlotState<kCluster>;
    Slot* sflags = reinterpret_cast<Slot*>(smem + L::kFlagsOff);  // [n]
    // The deep ring's score terms stay in shared memory ([n][G]).
    float* sterm = reinterpret_cast<float*>(smem + A::kTermOff);
    // [0] bit mask of the chunk's tiles that hold a live slot, [1] abort flag,
    // [2] last-CTA flag
    volatile int32_t* misc = reinterpret_cast<int32_t*>(smem + L::kMiscOff);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* empty = full + kStages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int chunk = blockIdx.x;
    const int u = blockIdx.y;
    const int S = p.S;
    const int slot0 = chunk * p.chunk_tiles * kTile;
    const int slot_end = min(slot0 + p.chunk_tiles * kTile, S);
    const int n = slot_end - slot0;
    const int ntiles = (n + kTile - 1) / kTile;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        misc[0] = 0;
        misc[1] = 0;
        if constexpr (kCluster) push_barriers_init<D, G, kScore>(smem + A::kPushOff, p.nchunk);
        fence_barrier_init();
    }
    // The barriers are initialised before any thread may use them (the
    // producer can issue copies before the prologue's barriers below).
    __syncthreads();
    // Push merge: peers may store into this CTA once every CTA of the
    // cluster has passed this point (waited for after the main loop).
    if constexpr (kCluster) cluster_arrive_relaxed();
    // With programmatic dependent launch this CTA may start while the previous
    // kernel of the stream (often the previous decode step) is still running:
    // everything above touches only this CTA's shared memory; every global
    // read comes after the wait. The next kernel may begin launching as soon
    // as every CTA of this one has started. With a split finish, the next
    // kernel is the scoring kernel, which watches this step's ready flags
    // without waiting for this grid: it may start only once every CTA here
    // has passed its own wait, so the previous step's scoring kernel (which
    // lowers the flags) is over.
    // Speculative first tiles. The CTAs of the grid's first wave all start
    // at once, when nothing else streams: they issue their chunk's first
    // nspec tiles before the mask round trip tells which tiles hold a live
    // slot, so the copies overlap it (a dead tile among them is processed as
    // fully masked and contributes nothing, so the results are the same bits).
    // Later CTAs start while their SM's other CTAs stream, and wait for the
    // live-tile list instead. Cluster grids are a single wave: all speculate.
    // A cluster CTA that starts before the previous kernel has finished
    // (programmatic dependent launch) already asks L2 for those tiles: a
    // prefetch into L2 reads no data into the CTA, so it needs no ordering
    // after the previous kernel, and the copies after the wait then find the
    // lines in L2 (measured per step: the Qwen3 3200-slot shape at batch 8
    // and 16, 19.9 -> 18.9 and 37.2 -> 35.9 us; the full batches unchanged
    // or slower, where the first wave's speculative tiles of empty chunks
    // would then compete with the previous step's last wave).
    const int lin = static_cast<int>(blockIdx.y) * static_cast<int>(gridDim.x) + chunk;
    const int nspec = (lin < p.spec_ctas) ? min(kStages, ntiles) : 0;
    if (kCluster && warp == kConsumerWarps && lane == 0) {
        for (int i = 0; i < nspec; ++i) {
            const int y = slot0 + i * kTile;
#pragma unroll
            for (int bx = 0; bx < L::kBoxes; ++bx) {
                tma_prefetch_l2_3d(&tmK, bx * kBoxCols, y, u);
                tma_prefetch_l2_3d(&tmV, bx * kBoxCols, y, u);
            }
        }
    }

    if (!p.split) allow_dependent_launch();
    grid_dependency_wait();
    if (p.split) allow_dependent_launch();

    if (warp == kConsumerWarps && lane == 0) {
        const uint64_t pol = l2_policy_evict_first();
        for (int i = 0; i < nspec; ++i) {
            uint8_t* kb = smem + i * L::kStageBytes;
            uint8_t* vb = kb + L::kTensorBytes;
            mbar_arrive_expect_tx(&full[i], L::kStageBytes);
            const int y = slot0 + i * kTile;
#pragma unroll
            for (int bx = 0; bx < L::kBoxes; ++bx) {
                tma_load_3d(kb + bx * L::kBoxBytes, &tmK, bx * kBoxCols, y, u, &full[i], pol);
                tma_load_3d(vb + bx * L::kBoxBytes, &tmV, bx * kBoxCols, y, u, &full[i], pol);
            }
        }
    }

    // The write slot, q and the chunk's mask are all loaded before the slot
    // is checked, so they share one round trip.
    int ws = p.write_slot[u];

    // Q^T as the B operand of S^T = K . Q^T, loaded early so its latency
    // overlaps the mask prologue: b0 = (d = 16kk + h0 .. +1, head r), b1 = d + 8.
    const int b = u / p.Hkv;
    const int kvh = u - b * p.Hkv;
    const int r = lane >> 2;          // fragment row (slot) 0..7
    const int h0 = 2 * (lane & 3);    // fragment columns (heads) h0, h0+1
    uint32_t qf[D / 16][2];
    if (warp < kConsumerWarps) {
        const bool valid = r < G;
        const __nv_bfloat16* qrow =
            p.q + (static_cast<size_t>(b) * p.Hq + kvh * G + (valid ? r : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int dc = kk * 16 + h0;
            qf[kk][0] = valid ? *reinterpret_cast<const uint32_t*>(qrow + dc) : 0u;
            qf[kk][1] = valid ? *reinterpret_cast<const uint32_t*>(qrow + dc + 8) : 0u;
        }
    }

    // Slot write, part 1 (Fig. 2 Left): age the chunk's mask. The written slot
    // gets age 0 (and becomes live); other live slots age by one. Every load
    // is issued before any store, so the chunk's mask costs one round trip.
    // The aged entries are stored evict-last: the next step reads them again,
    // and between the two the K/V stream passes through L2 evict-first.
    // Only the consumer threads age: the consumer barrier and the
    // acquire-release add on the unit's arrival counter (below) then also
    // publish the aged mask to the unit's last CTA, and nothing delays the
    // start of the pipeline. (Cluster CTAs read the slot flags from shared
    // memory only.)
    constexpr int kPer = (kMaxChunkTiles * kTile + kConsumers - 1) / kConsumers;
    int32_t* mrow = p.mask + static_cast<size_t>(u) * S + slot0;
    const uint64_t mask_pol = l2_policy_evict_last();
    const bool ager = tid < kConsumers;
    uint32_t live_bits = 0u;  // tiles of this thread's slots that hold a live slot
    int av[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = tid + k * kConsumers;
        av[k] = (ager && i < n) ? mrow[i] : -1;
    }
    if (ws < -1 || ws >= S) {
        if (tid == 0 && chunk == 0) atomicOr(p.dev_err, LF_DEVERR_BAD_WRITE_SLOT);
        ws = -1;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = tid + k * kConsumers;
        if (ager && i < n) {
            int a = av[k];
            if (ws >= 0) {
                int na;
                if constexpr (kScore)
                    na = (slot0 + i == ws) ? 0 : ((a >= 0 && a != 0x7fffffff) ? a + 1 : a);
                else
                    na = (slot0 + i == ws && a < 0) ? 0 : a;  // the written slot is live
                if (na != a) st_global_hint(mrow + i, na, mask_pol);
                a = na;
            }
            sflags[i] = slot_state(a, p.W, sflags);
            if (a >= 0) live_bits |= 1u << (i / kTile);
        }
    }
    // The chunk's live tiles, gathered while ageing: one OR per warp.
    if (ager) {
        live_bits = __reduce_or_sync(0xffffffffu, live_bits);
        if (lane == 0 && live_bits)
            atomicOr(const_cast<int*>(reinterpret_cast<volatile int*>(&misc[0])),
                     static_cast<int>(live_bits));
    }
    __syncthreads();

    // Tiles with no live slot are never loaded (ragged fills stream only
    // their live part), apart from speculative ones. The ring order: the
    // nspec speculative tiles, then the other live tiles in increasing order;
    // the producer and the consumers walk the same bits. The live tiles, as a
    // bit mask, also tell the unit's last CTA which tiles its score scan can
    // skip.
    const uint32_t live_tiles = static_cast<uint32_t>(misc[0]);
    const uint32_t rest_tiles = live_tiles & ~((1u << nspec) - 1u);  // nspec <= kStages < 32
    const int nlist = nspec + __popc(rest_tiles);  // tiles the ring delivers
    const int cnt = __popc(live_tiles);            // tiles holding a live slot
    if (kScore && !kCluster && tid == 0 && p.part_tiles && !(p.split && u >= p.split_from))
        p.part_tiles[static_cast<size_t>(u) * p.nchunk + chunk] = live_tiles;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int issued = nspec;
            uint32_t rest = rest_tiles;
            for (int i = nspec; i < nlist; ++i) {
                const int t = __ffs(rest) - 1;  // the next live tile
                rest &= rest - 1u;
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, p.wait_limit_ns)) {
                    atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);
                    misc[1] = 1;
                    break;
                }
                if (misc[1]) break;
                uint8_t* kb = smem + s * L::kStageBytes;
                uint8_t* vb = kb + L::kTensorBytes;
                mbar_arrive_expect_tx(&full[s], L::kStageBytes);
                const int y = slot0 + t * kTile;
#pragma unroll
                for (int bx = 0; bx < L::kBoxes; ++bx) {
                    tma_load_3d(kb + bx * L::kBoxBytes, &tmK, bx * kBoxCols, y, u, &full[s], pol);
                    tma_load_3d(vb + bx * L::kBoxBytes, &tmV, bx * kBoxCols, y, u, &full[s], pol);
                }
                ++issued;
            }
            // Every issued copy has landed before the CTA may retire.
            for (int i = max(0, issued - kStages); i < issued; ++i)
                (void)mbar_wait(&full[i % kStages], (i / kStages) & 1);
        }
        if constexpr (kCluster) cluster_wait();  // the split barrier begun at kernel start
        return;
    }

    // --------------------------------------------------------- consumers --
    const bool hv0 = h0 < G;
    const bool hv1 = h0 + 1 < G;
    const float NEG = -INFINITY;

    float acc[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    float m0 = NEG, m1 = NEG, l0 = 0.f, l1 = 0.f;
    const float sl = p.scale_log2;
    const int wrow0 = warp * 16;

    uint32_t rest = rest_tiles;
    for (int i = 0; i < nlist; ++i) {
        const int s = i % kStages;
        int t = i;  // speculative tiles first, then the live tiles in order
        if (i >= nspec) {
            t = __ffs(rest) - 1;
            rest &= rest - 1u;
        }
        if (!mbar_wait(&full[s], (i / kStages) & 1, p.wait_limit_ns)) {
            if (lane == 0) atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);
            misc[1] = 1;
            break;
        }
        uint8_t* kb = smem + s * L::kStageBytes;
        uint8_t* vb = kb + L::kTensorBytes;
        const int tslot0 = slot0 + t * kTile;

        // Slot write, part 2: the owning warp substitutes the current token's
        // row in shared memory and stores it to the cache.
        if (ws >= tslot0 + wrow0 && ws < tslot0 + wrow0 + 16) {
            const int row = ws - tslot0;
            const int cg = lane & 15;
            const bool is_v = lane >= 16;
            if (cg < D / 8) {
                const __nv_bfloat16* src = (is_v ? p.new_v : p.new_k) + static_cast<size_t>(u) * D;
                const uint4 val = reinterpret_cast<const uint4*>(src)[cg];
                *reinterpret_cast<uint4*>((is_v ? vb : kb) + swz_off(row, cg)) = val;
                __nv_bfloat16* dst =
                    (is_v ? p.v_cache : p.k_cache) + (static_cast<size_t>(u) * S + ws) * D;
                reinterpret_cast<uint4*>(dst)[cg] = val;
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        const int iA = tslot0 - slot0 + wrow0 + r;
        const int iB = iA + 8;
        const bool liveA = iA < n && slot_live(sflags[iA]);
        const bool liveB = iB < n && slot_live(sflags[iB]);

        // Logits S^T and row norms ||v||_1 for this warp's 16 slots.
        // Grids of many waves split each product into two accumulator chains
        // (even and odd k-steps), which halves the dependent MMA chain a warp
        // runs while it holds the ring stage (measured -0.4 to -0.8 us per
        // step on the large batches); the latency-bound cluster grids keep
        // one chain (measured +0.1 us with two), and so does g = 1, where
        // two would spill at d = 128.
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        float nv[4] = {0.f, 0.f, 0.f, 0.f};
        {
            constexpr int kChains = (kCluster || G == 1) ? 1 : 2;
            float sc1[4] = {0.f, 0.f, 0.f, 0.f};
            float nv1[4] = {0.f, 0.f, 0.f, 0.f};
            const int lrow = wrow0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const uint32_t kbase = smem_u32(kb);
            const uint32_t vbase = smem_u32(vb);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const bool odd = kChains == 2 && (kk & 1);
                const uint32_t off = swz_off(lrow, 2 * kk + (lane >> 4));
                uint32_t a[4];
                ldsm_x4(kbase + off, a);
                mma_bf16_16816(odd ? sc1 : sc, a, qf[kk][0], qf[kk][1]);
                if constexpr (kScore) {
                    uint32_t v[4];
                    ldsm_x4(vbase + off, v);
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] &= kAbsBf16x2;
                    mma_bf16_16816(odd ? nv1 : nv, v, kOnesBf16x2, kOnesBf16x2);
                }
            }
            if constexpr (kChains == 2) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sc[e] += sc1[e];
                    nv[e] += nv1[e];
                }
            }
        }

        // Logits in the log2 domain; masked rows and padding heads -> -inf.
        const float x0 = (liveA && hv0) ? sc[0] * sl : NEG;
        const float x1 = (liveA && hv1) ? sc[1] * sl : NEG;
        const float x2 = (liveB && hv0) ? sc[2] * sl : NEG;
        const float x3 = (liveB && hv1) ? sc[3] * sl : NEG;

        // Per-slot score terms t = log2(exp(s) * ||v||_1).
        if (kScore && hv0) {
            const int slotA = tslot0 + wrow0 + r;
            float* st = A::kSmemTerms
                            ? sterm + (slotA - slot0) * G + h0
                            : p.stash + (static_cast<size_t>(u) * S + slotA) * G + h0;
            if (liveA) {
                const float lv = __log2f(nv[0]);
                if (G == 1) st[0] = x0 + lv;
                else *reinterpret_cast<float2*>(st) = make_float2(x0 + lv, x1 + lv);
            }
            if (liveB) {
                const float lv = __log2f(nv[2]);
                if (G == 1) st[8 * G] = x2 + lv;
                else *reinterpret_cast<float2*>(st + 8 * G) = make_float2(x2 + lv, x3 + lv);
            }
        }

        // Online softmax per head (columns h0, h0+1), across the warp's rows.
        float mx0 = fmaxf(x0, x2);
        float mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0);
        const float mn1 = fmaxf(m1, mx1);
        const float mu0 = (mn0 == NEG) ? 0.f : mn0;
        const float mu1 = (mn1 == NEG) ? 0.f : mn1;
        const float al0 = exp2f(m0 - mu0);
        const float al1 = exp2f(m1 - mu1);
        const float p0 = exp2f(x0 - mu0);
        const float p1 = exp2f(x1 - mu1);
        const float p2 = exp2f(x2 - mu0);
        const float p3 = exp2f(x3 - mu1);
        l0 = l0 * al0 + p0 + p2;
        l1 = l1 * al1 + p1 + p3;
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            acc[mt][0] *= al0;
            acc[mt][1] *= al1;
            acc[mt][2] *= al0;
            acc[mt][3] *= al1;
        }
        // P^T (slots x heads) as the B operand of the P.V step.
        const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));

        // V^T columns of masked slots are zeroed (select, never multiply).
        const uint32_t bl = __ballot_sync(0xffffffffu, liveA);
        const uint32_t bh = __ballot_sync(0xffffffffu, liveB);
        const int k0 = 2 * (lane & 3);
        const uint32_t mlo = (((bl >> (4 * k0)) & 1u) ? 0x0000ffffu : 0u) |
                             (((bl >> (4 * k0 + 4)) & 1u) ? 0xffff0000u : 0u);
        const uint32_t mhi = (((bh >> (4 * k0)) & 1u) ? 0x0000ffffu : 0u) |
                             (((bh >> (4 * k0 + 4)) & 1u) ? 0xffff0000u : 0u);
        {
            const int lrow = wrow0 + (lane & 7) + (lane >> 4) * 8;
            const uint32_t vbase = smem_u32(vb);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                uint32_t a[4];
                ldsm_x4_trans(vbase + swz_off(lrow, 2 * mt + ((lane >> 3) & 1)), a);
                a[0] &= mlo;
                a[1] &= mlo;
                a[2] &= mhi;
                a[3] &= mhi;
                mma_bf16_16816(acc[mt], a, pb0, pb1);
            }
        }
        // The stage goes back to the producer as the iteration's last step,
        // after every use of what was loaded from it. (A variant that released
        // it earlier and stored the score terms after the release, with their
        // norms loaded from this stage, gave outputs that differed from run to
        // run in the last bits; a block fence before the release removed it.)
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ------------------------------------------ merge the 4 warps' state --
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if constexpr (kCluster) {
        static_assert(A::kPush, "a cluster instance without room for the push merge");
        static_assert(PushSmem<D, G>::kStageBytes <= L::kFlagsOff, "warp states exceed the TMA ring");
        cluster_merge_push<D, G, kStages, kScore, A::kSmemTerms>(
            p, u, slot0, n, sflags, smem, smem + A::kPushOff, smem + A::kStageOff, sterm, acc, m0,
            m1, l0, l1, tid);
        return;
    }
    consumer_bar_sync();  // every consumer is done with the stage buffers
    float* wO = reinterpret_cast<float*>(smem);  // [4][G][D]
    float* wm = wO + kConsumerWarps * G * D;     // [4][G]
    float* wl = wm + kConsumerWarps * G;         // [4][G]
    if (r == 0) {
        if (hv0) { wm[warp * G + h0] = m0; wl[warp * G + h0] = l0; }
        if (hv1) { wm[warp * G + h0 + 1] = m1; wl[warp * G + h0 + 1] = l1; }
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int dd = mt * 16 + r;
        if (hv0) {
            wO[(warp * G + h0) * D + dd] = acc[mt][0];
            wO[(warp * G + h0) * D + dd + 8] = acc[mt][2];
        }
        if (hv1) {
            wO[(warp * G + h0 + 1) * D + dd] = acc[mt][1];
            wO[(warp * G + h0 + 1) * D + dd + 8] = acc[mt][3];
        }
    }
    consumer_bar_sync();

    const size_t pidx = static_cast<size_t>(u) * p.nchunk + chunk;
    if (cnt > 0) {
        float* po = p.part_o + pidx * G * D;
        for (int e = tid; e < G * D; e += kConsumers) {
            const int h = e / D;
            float mh = NEG;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) mh = fmaxf(mh, wm[w * G + h]);
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = wm[w * G + h];
                if (mw != NEG) o += wO[w * G * D + e] * exp2f(mw - mh);
            }
            po[e] = o;
        }
    }
    if (tid < G) {
        float mh = NEG;
        float l = 0.f;
        if (cnt > 0) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) mh = fmaxf(mh, wm[w * G + tid]);
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = wm[w * G + tid];
                if (mw != NEG) l += wl[w * G + tid] * exp2f(mw - mh);
            }
        }
        p.part_ml[pidx * G + tid] = make_float2(mh, l);
    }

    // ---------------------------------------- last CTA of the unit merges --
    // One acquire-release add on the unit's arrival counter after a CTA
    // barrier releases every consumer's writes (partials, score terms, aged
    // mask entries) to the unit's last CTA, whose same add acquires all the
    // other chunks' (its barrier below passes that on to its threads); no
    // thread waits for a fence of its own.
    consumer_bar_sync();
    if (tid == 0) {
        int last = 1;
        if (p.nchunk > 1) {
            const uint32_t prev = atom_add_acq_rel_gpu(&p.arrivals[u], 1u);
            last = (prev == static_cast<uint32_t>(p.nchunk - 1));
            if (last) p.arrivals[u] = 0u;  // every chunk of the unit has arrived
        }
        misc[2] = last;
    }
    consumer_bar_sync();
    if (!misc[2]) return;
    finish_unit<D, G, kScore>(p, u, smem, L::kBarOff,
                              reinterpret_cast<uint64_t*>(smem + L::kScanBarOff), tid);
}

// Sets the kernel's function attributes (shared memory above 48 KB; cluster
// instances: clusters of more than 8 CTAs, an opt-in size) once per device.
template <int D, int G, int kStages, bool kScore, bool kCluster>
cudaError_t configure_t() {
    using A = StepAlloc<D, G, kStages, kCluster>;
    auto kernel = lf_decode_step_kernel<D, G, kStages, kScore, kCluster>;
    static int configured_for = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_for != dev) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, A::kAlloc);
        if (e != cudaSuccess) return e;
        if constexpr (kCluster) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        configured_for = dev;
    }
    return cudaSuccess;
}

// How many clusters of `csize` CTAs of the cluster instance can be resident
// at once on the current device (0: none, or the query failed).
template <int D, int G, int kStages, bool kScore>
int max_active_clusters_t(int csize) {
    if (configure_t<D, G, kStages, kScore, true>() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = StepAlloc<D, G, kStages, true>::kAlloc;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(csize);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, lf_decode_step_kernel<D, G, kStages, kScore, true>,
                                       &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// How many CTAs of the (non-cluster) instance are resident at once on the
// current device: the grid's first wave. Cached per device.
template <int D, int G, int kStages, bool kScore>
int first_wave_t() {
    static int cached_for = -1;
    static int ctas = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cached_for != dev) {
        int per_sm = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm, lf_decode_step_kernel<D, G, kStages, kScore, false>, kThreads,
                StepAlloc<D, G, kStages, false>::kAlloc) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        ctas = per_sm * sms;
        cached_for = dev;
    }
    return ctas;
}

template <int D, int G, int kStages, bool kScore, bool kCluster>
cudaError_t launch_t(const CUtensorMap& tmK, const CUtensorMap& tmV, const StepParams& p_in,
                     int units, cudaStream_t stream, bool pdl) {
    using L = StepSmem<D, kStages>;
    if (finish_smem_bytes(p_in.nchunk, G, kScore ? p_in.topk : 1) > static_cast<size_t>(L::kBarOff))
        return cudaErrorInvalidConfiguration;
    auto kernel = lf_decode_step_kernel<D, G, kStages, kScore, kCluster>;
    cudaError_t e = configure_t<D, G, kStages, kScore, kCluster>();
    if (e != cudaSuccess) return e;
    // Speculative first tiles in the first wave (LF_SPEC=0: off; cluster
    // grids, one wave by construction, always speculate).
    StepParams p = p_in;
    const char* spec_env = std::getenv("LF_SPEC");
    const bool spec = !(spec_env && std::atoi(spec_env) == 0);
    if constexpr (kCluster)
        p.spec_ctas = spec ? INT_MAX : 0;
    else
        p.spec_ctas = spec ? first_wave_t<D, G, kStages, kScore>() : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nchunk, units);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = StepAlloc<D, G, kStages, kCluster>::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if constexpr (kCluster) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(p.nchunk);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kernel, tmK, tmV, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace
}  // namespace lf
