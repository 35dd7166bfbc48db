// router_finish.cuh -- the per-token end of the router, shared by the CUDA-core routers
// (router.cu) and the fused tensor-core router (router_tc.cu): softmax over all experts, top-k
// in descending order with ties to the lower expert index, the near-tie gap, renormalisation.
// Page "混合专家 MoE", section "实现：逐 token 与按专家分组", MoE.route.
#pragma once

#include <float.h>
#include <limits.h>

#include "moe_internal.cuh"

namespace moe {
namespace router_detail {

// Unsigned key with the order of the float (negative floats bit-flipped, -0 made +0); a NaN
// gets the lowest key, so like the comparisons it stands for it never wins over a number.
static __device__ __forceinline__ uint32_t order_key(float v) {
    const float f = v == 0.f ? 0.f : v;
    const uint32_t u = __float_as_uint(f);
    return (f != f) ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
}
static __device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Warp arg-max over (value desc, index asc); every lane ends with the same pair: the maximum key
// is one warp reduction and the lowest index among the lanes holding it a second.
static __device__ __forceinline__ void warp_argmax(float& v, int& i) {
    const uint32_t key = order_key(v);
    const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
    i = (int)__reduce_min_sync(0xffffffffu, key == mk ? (uint32_t)i : 0xffffffffu);
    v = key_value(mk);
}

// Softmax, top-k, gap and renormalisation of one token held by one warp.  v[i] is the logit of
// expert lane + 32 i (ignored for experts >= E).  Adds the probabilities into pacc.
// bias_mode 1: b_r is added to the logits; 2: the top-k is chosen on p + b_r (rounded once to
// fp32) while the weights and probabilities stay unbiased ("混合专家 MoE", 负载均衡: the
// DeepSeek-V3 bias only picks the experts).
template <int NV>
__device__ __forceinline__ void finish_token(float (&v)[NV], const float* __restrict__ b_r,
                                             int bias_mode, int E, int k, int renorm, int64_t tok,
                                             int32_t* __restrict__ idx_out,
                                             float* __restrict__ w_out,
                                             float* __restrict__ gap_out,
                                             float* __restrict__ lse_out,
                                             float* __restrict__ probs_out, float (&pacc)[NV]) {
    const int lane = threadIdx.x & 31;
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        if (e < E) {
            if (bias_mode == 1) v[i] += b_r[e];
            m = fmaxf(m, v[i]);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? expf(v[i] - m) : 0.f;
        s += v[i];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0 && lse_out) lse_out[tok] = m + logf(s);   // log-sum-exp of the logits (z-loss)
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? v[i] / s : -1.f;   // -1: never selected
        if (e < E) pacc[i] += v[i];
        if (e < E && probs_out) probs_out[tok * E + e] = v[i];
    }
    // selection scores: the probabilities, or p + b for the selection-only bias
    float sv[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        sv[i] = (bias_mode == 2 && e < E) ? v[i] + b_r[e] : v[i];
    }
    float my_val = 0.f, kth = 0.f, sel_sum = 0.f;
    int my_idx = 0;
    const int rounds = k < E ? k + 1 : k;
    if constexpr (NV <= 8) {
        // Each lane sorts its NV candidates once by (score desc, expert asc); every round the
        // lanes offer their heads, two warp reductions pick the winner (the same order as a
        // full arg-max over the untaken experts) and the winning lane pops its head.
        uint32_t key[NV];
        int ex[NV];
        float pr[NV];
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int e = lane + 32 * i;
            key[i] = e < E ? order_key(sv[i]) : 0u;
            ex[i] = e < E ? e : INT_MAX;
            pr[i] = v[i];
        }
#pragma unroll
        for (int a = 1; a < NV; a++)
#pragma unroll
            for (int b = a; b > 0; b--)
                if (key[b] > key[b - 1]) {   // strict: equal keys keep the lower expert first
                    const uint32_t tk = key[b]; key[b] = key[b - 1]; key[b - 1] = tk;
                    const int te = ex[b]; ex[b] = ex[b - 1]; ex[b - 1] = te;
                    const float tp = pr[b]; pr[b] = pr[b - 1]; pr[b - 1] = tp;
                }
        for (int j = 0; j < rounds; j++) {
            const uint32_t mk = __reduce_max_sync(0xffffffffu, key[0]);
            const int bi =
                (int)__reduce_min_sync(0xffffffffu, key[0] == mk ? (uint32_t)ex[0] : 0xffffffffu);
            const float bv = key_value(mk);
            if (j < k) {
                const int wl = bi & 31;
                const float pv = __shfl_sync(0xffffffffu, pr[0], wl);
                const bool pop = lane == wl;
#pragma unroll
                for (int i = 0; i + 1 < NV; i++) {
                    key[i] = pop ? key[i + 1] : key[i];
                    ex[i] = pop ? ex[i + 1] : ex[i];
                    pr[i] = pop ? pr[i + 1] : pr[i];
                }
                if (pop) {
                    key[NV - 1] = 0u;
                    ex[NV - 1] = INT_MAX;
                }
                if (lane == j) {
                    my_val = pv;
                    my_idx = bi;
                }
                sel_sum += pv;   // slot order, identical on every lane
                kth = bv;
            } else if (lane == 0 && gap_out) {
                gap_out[tok] = kth - bv;
            }
        }
    } else {
    uint32_t taken = 0;
    for (int j = 0; j < rounds; j++) {
        float bv = -FLT_MAX;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int e = lane + 32 * i;
            if (e < E && !(taken & (1u << i)) && (sv[i] > bv || (sv[i] == bv && e < bi))) {
                bv = sv[i];
                bi = e;
            }
        }
        warp_argmax(bv, bi);
        if (j < k) {
            // the probability of the chosen expert, from the lane that holds it
            float pv = 0.f;
#pragma unroll
            for (int i = 0; i < NV; i++)
                if (i == (bi >> 5)) pv = v[i];
            pv = __shfl_sync(0xffffffffu, pv, bi & 31);
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == j) {
                my_val = pv;
                my_idx = bi;
            }
            sel_sum += pv;   // slot order, identical on every lane
            kth = bv;
        } else if (lane == 0 && gap_out) {
            gap_out[tok] = kth - bv;
        }
    }
    }
    if (k >= E && lane == 0 && gap_out) gap_out[tok] = __int_as_float(0x7f800000);
    if (lane < k) {
        idx_out[tok * k + lane] = my_idx;
        w_out[tok * k + lane] = renorm ? my_val / sel_sum : my_val;
    }
}

}  // namespace router_detail
}  // namespace moe
