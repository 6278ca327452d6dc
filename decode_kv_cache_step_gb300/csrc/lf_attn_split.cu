// Split attention kernel of the LongFlow decode step (sm_103a).
//
// "LongFlow: Efficient KV Cache Compression for Reasoning Models":
//   Fig. 2 (Left)   the current K/V covers the slot chosen at the previous step;
//   Fig. 2 (Middle) K, V and the Mask stream from HBM into on-chip memory by
//                   block and the attention runs there;
//   Fig. 2 (Right)  P.V is split in two: G = p * v (per slot) and O = sum_j G.
//                   LongFlowScore is read off G. With the score
//                   I_j = sum_h sum_c |p_hj v_jc| = (sum_h p_hj) * ||v_j||_1
//                   (p >= 0), G never has to exist: each live slot leaves
//                   log2(p~_hj) + log2(||v_j||_1) per head, relative to this
//                   chunk's final max, and the combine kernel rescales it.
//
// One CTA = one chunk (up to 32 tiles of 64 slots) of one (b, kvh) unit.
//   warp 4, lane 0 : producer. TMA-loads the K and V tiles of the chunk's
//                    live tiles (128-byte swizzled, 3-stage mbarrier ring,
//                    L2 evict-first: every byte is read once per step).
//   warps 0..3     : consumers. Warp w owns rows 16w..16w+15 of every tile
//                    and keeps its own online-softmax state. Per 16 slots:
//        S^T[16 x 8]  = K[16 x D] . Q^T[D x 8]       (mma m16n8k16, heads as N)
//        N  [16 x 8]  = |V|[16 x D] . 1[D x 8]        (row L1 norms on the MMA)
//        O^T[D x 8]  += V^T[D x 16] . P^T[16 x 8]     (P^T via movmatrix)
//   GQA folding: the g <= 8 query heads of the unit share each K/V byte.
//   Masked slots are removed by select (logit -inf, V columns zeroed), so
//   NaN or Inf in masked rows never reaches the output.
#include <math.h>

#include "../../include/lf_decode.h"
#include "lf_kernels.h"
#include "lf_ptx.cuh"

namespace lf {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr uint32_t kOnesBf16x2 = 0x3F803F80u;   // (1.0, 1.0) in bf16
constexpr uint32_t kAbsBf16x2 = 0x7FFF7FFFu;

template <int D>
struct SplitSmem {
    static constexpr int kBoxes = D / kBoxCols;
    static constexpr int kBoxBytes = kTile * 128;              // 64 rows x 128 B
    static constexpr int kTensorBytes = kBoxes * kBoxBytes;    // K (or V) of one tile
    static constexpr int kStageBytes = 2 * kTensorBytes;       // K + V
    static constexpr int kAgesOff = kStages * kStageBytes;
    static constexpr int kAgesBytes = kMaxChunkTiles * kTile * 4;
    static constexpr int kListOff = kAgesOff + kAgesBytes;
    static constexpr int kMiscOff = kListOff + kMaxChunkTiles * 4;
    static constexpr int kBarOff = kMiscOff + 16;
    static constexpr int kBytes = kBarOff + 2 * kStages * 8;
    static constexpr int kAlloc = kBytes + 1024;               // slack for 1024-B alignment
};

__device__ __forceinline__ void consumer_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Byte offset of 16-byte chunk `cg` (8 bf16 columns) of tile row `row` in a
// swizzled K or V tile buffer.
template <int D>
__device__ __forceinline__ uint32_t swz_off(int row, int cg) {
    return (cg >> 3) * SplitSmem<D>::kBoxBytes + row * 128 + (((cg & 7) ^ (row & 7)) << 4);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2)
    lf_attn_split_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    using L = SplitSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    int32_t* ages = reinterpret_cast<int32_t*>(smem + L::kAgesOff);
    int32_t* list = reinterpret_cast<int32_t*>(smem + L::kListOff);
    volatile int32_t* misc = reinterpret_cast<int32_t*>(smem + L::kMiscOff);  // [0] count, [1] abort
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

    int ws = p.write_slot[u];
    if (ws < -1 || ws >= S) {
        if (tid == 0 && chunk == 0) atomicOr(p.dev_err, LF_DEVERR_BAD_WRITE_SLOT);
        ws = -1;
    }

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        misc[1] = 0;
        fence_barrier_init();
    }

    // Slot write, part 1 (Fig. 2 Left): age the chunk's mask. The written slot
    // gets age 0 (and becomes live); other live slots age by one.
    int32_t* mrow = p.mask + static_cast<size_t>(u) * S;
    for (int i = tid; i < n; i += kThreads) {
        const int j = slot0 + i;
        int a = mrow[j];
        if (ws >= 0) {
            const int na = (j == ws) ? 0 : ((a >= 0 && a != 0x7fffffff) ? a + 1 : a);
            if (na != a) mrow[j] = na;
            a = na;
        }
        ages[i] = a;
    }
    __syncthreads();

    // Tiles with no live slot are never loaded (ragged fills stream only
    // their live prefix).
    if (warp == 0) {
        int cnt = 0;
        for (int t = 0; t < ntiles; ++t) {
            const int i0 = t * kTile + lane;
            const int i1 = i0 + 32;
            const bool live = (i0 < n && ages[i0] >= 0) || (i1 < n && ages[i1] >= 0);
            if (__any_sync(0xffffffffu, live)) {
                if (lane == 0) list[cnt] = t;
                ++cnt;
            }
        }
        if (lane == 0) misc[0] = cnt;
    }
    __syncthreads();
    const int cnt = misc[0];

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int issued = 0;
            for (int i = 0; i < cnt; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1)) {
                    atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);
                    misc[1] = 1;
                    break;
                }
                if (misc[1]) break;
                uint8_t* kb = smem + s * L::kStageBytes;
                uint8_t* vb = kb + L::kTensorBytes;
                mbar_arrive_expect_tx(&full[s], L::kStageBytes);
                const int y = slot0 + list[i] * kTile;
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
        return;
    }

    // --------------------------------------------------------- consumers --
    const int b = u / p.Hkv;
    const int kvh = u - b * p.Hkv;
    const int r = lane >> 2;          // fragment row (slot) 0..7
    const int h0 = 2 * (lane & 3);    // fragment columns (heads) h0, h0+1
    const bool hv0 = h0 < G;
    const bool hv1 = h0 + 1 < G;
    const float NEG = -INFINITY;

    // Q^T as the B operand: b0 = (d = 16kk + h0 .. +1, head r), b1 = d + 8.
    uint32_t qf[D / 16][2];
    {
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

    float acc[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    float m0 = NEG, m1 = NEG, l0 = 0.f, l1 = 0.f;
    const float sl = p.scale_log2;
    const int wrow0 = warp * 16;

    for (int i = 0; i < cnt; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&full[s], (i / kStages) & 1)) {
            if (lane == 0) atomicOr(p.dev_err, LF_DEVERR_WAIT_TIMEOUT);
            misc[1] = 1;
            break;
        }
        uint8_t* kb = smem + s * L::kStageBytes;
        uint8_t* vb = kb + L::kTensorBytes;
        const int tslot0 = slot0 + list[i] * kTile;

        // Slot write, part 2: the owning warp substitutes the current token's
        // row in shared memory and stores it to the cache.
        if (ws >= tslot0 + wrow0 && ws < tslot0 + wrow0 + 16) {
            const int row = ws - tslot0;
            const int cg = lane & 15;
            const bool is_v = lane >= 16;
            if (cg < D / 8) {
                const __nv_bfloat16* src = (is_v ? p.new_v : p.new_k) + static_cast<size_t>(u) * D;
                const uint4 val = reinterpret_cast<const uint4*>(src)[cg];
                *reinterpret_cast<uint4*>((is_v ? vb : kb) + swz_off<D>(row, cg)) = val;
                __nv_bfloat16* dst =
                    (is_v ? p.v_cache : p.k_cache) + (static_cast<size_t>(u) * S + ws) * D;
                reinterpret_cast<uint4*>(dst)[cg] = val;
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        const int iA = tslot0 - slot0 + wrow0 + r;
        const int iB = iA + 8;
        const bool liveA = iA < n && ages[iA] >= 0;
        const bool liveB = iB < n && ages[iB] >= 0;

        // Logits S^T and row norms ||v||_1 for this warp's 16 slots.
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        float nv[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int lrow = wrow0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const uint32_t kbase = smem_u32(kb);
            const uint32_t vbase = smem_u32(vb);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = swz_off<D>(lrow, 2 * kk + (lane >> 4));
                uint32_t a[4], v[4];
                ldsm_x4(kbase + off, a);
                ldsm_x4(vbase + off, v);
                mma_bf16_16816(sc, a, qf[kk][0], qf[kk][1]);
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] &= kAbsBf16x2;
                mma_bf16_16816(nv, v, kOnesBf16x2, kOnesBf16x2);
            }
        }

        // Logits in the log2 domain; masked rows and padding heads -> -inf.
        const float x0 = (liveA && hv0) ? sc[0] * sl : NEG;
        const float x1 = (liveA && hv1) ? sc[1] * sl : NEG;
        const float x2 = (liveB && hv0) ? sc[2] * sl : NEG;
        const float x3 = (liveB && hv1) ? sc[3] * sl : NEG;

        // Per-slot score terms: log2(exp(s) * ||v||_1), rebased by the combine.
        if (hv0) {
            const int slotA = tslot0 + wrow0 + r;
            float* st = p.stash + (static_cast<size_t>(u) * S + slotA) * G + h0;
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
                ldsm_x4_trans(vbase + swz_off<D>(lrow, 2 * mt + ((lane >> 3) & 1)), a);
                a[0] &= mlo;
                a[1] &= mlo;
                a[2] &= mhi;
                a[3] &= mhi;
                mma_bf16_16816(acc[mt], a, pb0, pb1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ------------------------------------------------ merge the 4 warps --
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
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
        for (int e = tid; e < G * D; e += kConsumerWarps * 32) {
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
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) mh = fmaxf(mh, wm[w * G + tid]);
        float l = 0.f;
        if (cnt > 0) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = wm[w * G + tid];
                if (mw != NEG) l += wl[w * G + tid] * exp2f(mw - mh);
            }
        } else {
            mh = NEG;
        }
        p.part_ml[pidx * G + tid] = make_float2(mh, l);
    }
}

template <int D, int G>
cudaError_t launch_split_t(const CUtensorMap& tmK, const CUtensorMap& tmV, const SplitParams& p,
                           int units, cudaStream_t stream) {
    static int configured_for = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_for != dev) {
        e = cudaFuncSetAttribute(lf_attn_split_kernel<D, G>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SplitSmem<D>::kAlloc);
        if (e != cudaSuccess) return e;
        configured_for = dev;
    }
    dim3 grid(p.nchunk, units);
    lf_attn_split_kernel<D, G><<<grid, kThreads, SplitSmem<D>::kAlloc, stream>>>(tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace

size_t split_smem_bytes(int D) {
    return D == 64 ? SplitSmem<64>::kAlloc : SplitSmem<128>::kAlloc;
}

cudaError_t launch_attn_split(int D, int G, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              const SplitParams& p, int units, cudaStream_t stream) {
#define LF_SPLIT_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_split_t<DD, GG>(tmK, tmV, p, units, stream);
    LF_SPLIT_CASE(64, 1) LF_SPLIT_CASE(64, 2) LF_SPLIT_CASE(64, 4) LF_SPLIT_CASE(64, 8)
    LF_SPLIT_CASE(128, 1) LF_SPLIT_CASE(128, 2) LF_SPLIT_CASE(128, 4) LF_SPLIT_CASE(128, 8)
#undef LF_SPLIT_CASE
    return cudaErrorInvalidValue;
}

}  // namespace lf
