// Combine kernel of the LongFlow decode step (sm_103a).
//
// One CTA per (b, kvh) unit, after the split kernel:
//   - merges the chunks' softmax partials (m, l, unnormalised O) into the
//     output, rounded to bf16 (nearest even);
//   - finishes LongFlowScore for every live slot from its per-head terms
//       I_j = sum_h 2^(t_hj - m_h) / l_h,  t_hj = log2(exp(s_hj) * ||v_j||_1)
//     which is sum_h p_hj * ||v_j||_1 = sum_h sum_c |G_hjc| with the final
//     normalised p ("LongFlow: Efficient KV Cache Compression for Reasoning
//     Models", Fig. 2 Right: the score is read off G);
//   - reduces (I_j, j) lexicographically over live slots with age >= W: the
//     slot the next step overwrites (Fig. 2 Left, Fig. 1 caption).
#include <math.h>

#include "lf_kernels.h"

namespace lf {
namespace {

constexpr int kThreads = 256;

template <int G>
__device__ __forceinline__ void load_terms(const float* t, float (&v)[G]) {
    if constexpr (G == 1) {
        v[0] = t[0];
    } else if constexpr (G == 2) {
        const float2 a = *reinterpret_cast<const float2*>(t);
        v[0] = a.x; v[1] = a.y;
    } else {
#pragma unroll
        for (int q = 0; q < G / 4; ++q) {
            const float4 a = *reinterpret_cast<const float4*>(t + 4 * q);
            v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
        }
    }
}

__device__ __forceinline__ bool better(float v, int j, float bv, int bj) {
    return v < bv || (v == bv && j < bj);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) lf_combine_kernel(const CombineParams p) {
    extern __shared__ float s_w[];  // [nchunk][G]: exp2(m_c - m) / l
    __shared__ float s_m[G];
    __shared__ float s_il[G];
    __shared__ float red_v[kThreads / 32];
    __shared__ int red_j[kThreads / 32];

    const int u = blockIdx.x;
    const int tid = threadIdx.x;
    const int nchunk = p.nchunk;
    const float2* ml = p.part_ml + static_cast<size_t>(u) * nchunk * G;

    if (tid < G) {
        float m = -INFINITY;
        for (int c = 0; c < nchunk; ++c) m = fmaxf(m, ml[c * G + tid].x);
        float l = 0.f;
        for (int c = 0; c < nchunk; ++c) {
            const float2 v = ml[c * G + tid];
            if (v.x != -INFINITY) l += v.y * exp2f(v.x - m);
        }
        s_m[tid] = m;
        s_il[tid] = (l > 0.f) ? 1.f / l : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < nchunk * G; e += kThreads) {
        const float2 v = ml[e];
        const int h = e % G;
        s_w[e] = (v.x == -INFINITY) ? 0.f : exp2f(v.x - s_m[h]) * s_il[h];
    }
    __syncthreads();

    // Output: O_h = sum_c w_ch * O_ch.
    const int b = u / p.Hkv;
    const int kvh = u - b * p.Hkv;
    const float* po = p.part_o + static_cast<size_t>(u) * nchunk * G * D;
    __nv_bfloat16* out = p.out + (static_cast<size_t>(b) * p.Hq + kvh * G) * D;
    for (int e = tid; e < G * D; e += kThreads) {
        const int h = e / D;
        float o = 0.f;
        for (int c = 0; c < nchunk; ++c) {
            const float w = s_w[c * G + h];
            if (w != 0.f) o += w * po[static_cast<size_t>(c) * G * D + e];
        }
        out[e] = __float2bfloat16_rn(o);
    }

    // LongFlowScore of every live slot, argmin over the eligible ones.
    float m[G], il[G];
#pragma unroll
    for (int h = 0; h < G; ++h) { m[h] = s_m[h]; il[h] = s_il[h]; }
    const int S = p.S;
    const int32_t* age = p.mask + static_cast<size_t>(u) * S;
    const float* stash = p.stash + static_cast<size_t>(u) * S * G;
    float* scores = p.scores ? p.scores + static_cast<size_t>(u) * S : nullptr;
    float best = INFINITY;
    int bestj = 0x7fffffff;
    for (int j = tid; j < S; j += kThreads) {
        const int a = age[j];
        float I = INFINITY;
        if (a >= 0) {
            float t[G];
            load_terms<G>(stash + static_cast<size_t>(j) * G, t);
            I = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) I += exp2f(t[h] - m[h]) * il[h];
            if (a >= p.W && better(I, j, best, bestj)) { best = I; bestj = j; }
        }
        if (scores) scores[j] = I;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, off);
        const int oj = __shfl_xor_sync(0xffffffffu, bestj, off);
        if (better(ov, oj, best, bestj)) { best = ov; bestj = oj; }
    }
    if ((tid & 31) == 0) { red_v[tid >> 5] = best; red_j[tid >> 5] = bestj; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kThreads / 32; ++w)
            if (better(red_v[w], red_j[w], best, bestj)) { best = red_v[w]; bestj = red_j[w]; }
        p.next_slot[u] = (bestj == 0x7fffffff) ? -1 : bestj;
    }
}

template <int D, int G>
cudaError_t launch_combine_t(const CombineParams& p, int units, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(p.nchunk) * G * sizeof(float);
    lf_combine_kernel<D, G><<<units, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(int D, int G, const CombineParams& p, int units,
                           cudaStream_t stream) {
#define LF_COMBINE_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_combine_t<DD, GG>(p, units, stream);
    LF_COMBINE_CASE(64, 1) LF_COMBINE_CASE(64, 2) LF_COMBINE_CASE(64, 4) LF_COMBINE_CASE(64, 8)
    LF_COMBINE_CASE(128, 1) LF_COMBINE_CASE(128, 2) LF_COMBINE_CASE(128, 4) LF_COMBINE_CASE(128, 8)
#undef LF_COMBINE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace lf
