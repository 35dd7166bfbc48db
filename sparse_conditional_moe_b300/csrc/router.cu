// router.cu -- fused router: logits (fp32 CUDA-core GEMM) + softmax + top-k + renormalise.
//
// Page "混合专家 MoE", section "实现：逐 token 与按专家分组", MoE.route: a linear layer d -> E
// scores every expert, softmax over the E scores, the k largest kept in descending order,
// and the k weights divided by their sum.  The router stays fp32 end to end.
//
// One block = BT tokens x all E experts.  The d-loop stages a DK-wide slice of x (widened to
// fp32) and of W_r in shared memory; every thread computes a TT x TE register tile, each slice
// as an fp32 FMA chain in increasing-d order, slices added to the running logit with
// compensated (Kahan) summation, so the logit error stays near u*sqrt(DK) for any d.  The
// logits then go through shared memory to the
// epilogue, where each warp owns whole tokens: max / sum by warp shuffles, top-k by k rounds
// of a warp arg-max on (probability desc, expert index asc), the (k+1)-th for the near-tie
// gap, and per-block column sums of the probabilities (deterministic, no float atomics).
#include <float.h>
#include <limits.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRouterThreads = 256;

template <int EP>
struct RouterTile {
    static constexpr int TE_THREADS = EP < 32 ? EP : 32;                  // threads along experts
    static constexpr int TE = EP / TE_THREADS;                            // experts per thread
    static constexpr int TT_THREADS = kRouterThreads / TE_THREADS;        // threads along tokens
    static constexpr int TT = EP >= 1024 ? 1 : (EP >= 512 ? 2 : (EP >= 16 ? 4 : 2));
    static constexpr int BT = TT_THREADS * TT;                            // tokens per block
    static constexpr int DK = EP >= 1024 ? 8 : (EP >= 512 ? 16 : 32);     // d-slice per stage
    static constexpr int XS = BT * (DK + 1);                              // x slice [BT][DK+1]
    static constexpr int WS = DK * EP;                                    // W slice [DK][EP]
    static constexpr int LS = BT * (EP + 1);                              // logits [BT][EP+1]
    static constexpr int SMEM_FLOATS = (XS + WS) > LS ? (XS + WS) : LS;
    static constexpr int NV = EP >= 32 ? EP / 32 : 1;                     // values per lane
};

__device__ __forceinline__ float load_x(const float* x, int64_t i) { return x[i]; }
__device__ __forceinline__ float load_x(const __nv_bfloat16* x, int64_t i) {
    return __bfloat162float(x[i]);
}

// Warp arg-max over (value desc, index asc); every lane ends with the same pair.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, off);
        int oi = __shfl_xor_sync(0xffffffffu, i, off);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

template <int EP, typename T>
__global__ void __launch_bounds__(kRouterThreads)
router_kernel(const T* __restrict__ x, const float* __restrict__ W_r, const float* __restrict__ b_r,
              int64_t N, int d, int E, int k, int renorm, int32_t* __restrict__ idx_out,
              float* __restrict__ w_out, float* __restrict__ gap_out, float* __restrict__ p_part) {
    using Tl = RouterTile<EP>;
    constexpr int TT = Tl::TT, TE = Tl::TE, BT = Tl::BT, DK = Tl::DK;
    constexpr int TEn = Tl::TE_THREADS, TTn = Tl::TT_THREADS, NV = Tl::NV;
    static_assert(Tl::SMEM_FLOATS >= (kRouterThreads / 32) * EP, "P table must fit the staging buffer");
    __shared__ float sm[Tl::SMEM_FLOATS];
    float* Xs = sm;             // [BT][DK+1]
    float* Ws = sm + Tl::XS;    // [DK][EP]

    const int tid = threadIdx.x;
    const int tx = tid % TEn, ty = tid / TEn;
    const int64_t t0 = (int64_t)blockIdx.x * BT;

    // acc: running logit; cmp: its compensation term (Kahan), so that the only rounding left
    // of any size is inside each DK-long slice (fp32 FMA chain over DK products).
    float acc[TT][TE], cmp[TT][TE];
#pragma unroll
    for (int i = 0; i < TT; i++)
#pragma unroll
        for (int j = 0; j < TE; j++) acc[i][j] = cmp[i][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += DK) {
        // stage x[t0 .. t0+BT) x [k0 .. k0+DK) as fp32 (zero outside the batch / past d)
        for (int v = tid; v < BT * DK; v += kRouterThreads) {
            int t = v / DK, kk = v % DK;
            int64_t tok = t0 + t;
            float val = 0.f;
            if (tok < N && k0 + kk < d) val = load_x(x, tok * d + k0 + kk);
            Xs[t * (DK + 1) + kk] = val;
        }
        // stage W_r[0 .. EP) x [k0 .. k0+DK) transposed to [DK][EP] (zero for padded experts)
        for (int v = tid; v < EP * DK; v += kRouterThreads) {
            int e = v % EP, kk = v / EP;
            float val = 0.f;
            if (e < E && k0 + kk < d) val = W_r[(int64_t)e * d + k0 + kk];
            Ws[kk * EP + e] = val;
        }
        __syncthreads();
        float part[TT][TE];
#pragma unroll
        for (int i = 0; i < TT; i++)
#pragma unroll
            for (int j = 0; j < TE; j++) part[i][j] = 0.f;
#pragma unroll 4
        for (int kk = 0; kk < DK; kk++) {
            float xv[TT], wv[TE];
#pragma unroll
            for (int i = 0; i < TT; i++) xv[i] = Xs[(ty + i * TTn) * (DK + 1) + kk];
#pragma unroll
            for (int j = 0; j < TE; j++) wv[j] = Ws[kk * EP + tx + j * TEn];
#pragma unroll
            for (int i = 0; i < TT; i++)
#pragma unroll
                for (int j = 0; j < TE; j++) part[i][j] = fmaf(xv[i], wv[j], part[i][j]);
        }
#pragma unroll
        for (int i = 0; i < TT; i++)
#pragma unroll
            for (int j = 0; j < TE; j++) {
                const float y = part[i][j] - cmp[i][j];
                const float t = acc[i][j] + y;
                cmp[i][j] = (t - acc[i][j]) - y;
                acc[i][j] = t;
            }
        __syncthreads();
    }

    // logits -> shared [BT][EP+1]
    float* Ls = sm;
#pragma unroll
    for (int i = 0; i < TT; i++)
#pragma unroll
        for (int j = 0; j < TE; j++) Ls[(ty + i * TTn) * (EP + 1) + tx + j * TEn] = acc[i][j];
    __syncthreads();

    const int warp = tid / 32, lane = tid % 32;
    constexpr int kWarps = kRouterThreads / 32;
    float pacc[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) pacc[i] = 0.f;

    for (int t = warp; t < BT; t += kWarps) {
        const int64_t tok = t0 + t;
        if (tok >= N) break;
        float v[NV];
        float m = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            int e = lane + 32 * i;
            if (e < E) {
                float l = Ls[t * (EP + 1) + e];
                if (b_r) l += b_r[e];
                v[i] = l;
                m = fmaxf(m, l);
            } else {
                v[i] = -FLT_MAX;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            int e = lane + 32 * i;
            v[i] = (e < E) ? expf(v[i] - m) : 0.f;
            s += v[i];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
#pragma unroll
        for (int i = 0; i < NV; i++) {
            int e = lane + 32 * i;
            v[i] = (e < E) ? v[i] / s : -1.f;   // -1: never selected
            if (e < E) pacc[i] += v[i];
        }
        // top-k (+ the next one for the gap)
        uint32_t taken = 0;
        float my_val = 0.f;
        int my_idx = 0;
        float kth = 0.f, sel_sum = 0.f;
        const int rounds = k < E ? k + 1 : k;
        for (int j = 0; j < rounds; j++) {
            float bv = -2.f;
            int bi = INT_MAX;
#pragma unroll
            for (int i = 0; i < NV; i++) {
                int e = lane + 32 * i;
                if (!(taken & (1u << i)) && (v[i] > bv || (v[i] == bv && e < bi))) {
                    bv = v[i];
                    bi = e;
                }
            }
            warp_argmax(bv, bi);
            if (j < k) {
                if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
                if (lane == j) {
                    my_val = bv;
                    my_idx = bi;
                }
                sel_sum += bv;   // slot order, identical on every lane
                kth = bv;
            } else if (lane == 0 && gap_out) {
                gap_out[tok] = kth - bv;
            }
        }
        if (k >= E && lane == 0 && gap_out) gap_out[tok] = __int_as_float(0x7f800000);
        if (lane < k) {
            idx_out[tok * k + lane] = my_idx;
            w_out[tok * k + lane] = renorm ? my_val / sel_sum : my_val;
        }
    }

    // per-block column sums of the probabilities, combined across warps in warp order
    __syncthreads();             // every warp is done reading the logits
    float* Pw = sm;              // [warps][EP]
#pragma unroll
    for (int i = 0; i < NV; i++) {
        int e = lane + 32 * i;
        if (e < EP) Pw[warp * EP + e] = pacc[i];
    }
    __syncthreads();
    for (int e = tid; e < E; e += kRouterThreads) {
        float sacc = 0.f;
        for (int w = 0; w < kWarps; w++) sacc += Pw[w * EP + e];
        p_part[(int64_t)blockIdx.x * E + e] = sacc;
    }
}

__global__ void reduce_p_kernel(const float* __restrict__ p_part, int blocks, int E,
                                float* __restrict__ P_sum) {
    int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float s = 0.f;
    for (int b = 0; b < blocks; b++) s += p_part[(int64_t)b * E + e];
    P_sum[e] = s;
}

int pad_experts(int E) {
    int ep = 8;
    while (ep < E) ep *= 2;
    return ep;
}

template <int EP>
cudaError_t launch_ep(const moe_cfg& c, const void* x, const float* W_r, const float* b_r,
                      int32_t* idx, float* w, float* gap, float* p_part, cudaStream_t s) {
    using Tl = RouterTile<EP>;
    int blocks = (int)((c.N + Tl::BT - 1) / Tl::BT);
    const float* bias = c.bias_mode == 1 ? b_r : nullptr;
    if (c.act_dtype == MOE_BF16)
        router_kernel<EP, __nv_bfloat16><<<blocks, kRouterThreads, 0, s>>>(
            (const __nv_bfloat16*)x, W_r, bias, c.N, c.d, c.E, c.k, c.renorm, idx, w, gap, p_part);
    else
        router_kernel<EP, float><<<blocks, kRouterThreads, 0, s>>>(
            (const float*)x, W_r, bias, c.N, c.d, c.E, c.k, c.renorm, idx, w, gap, p_part);
    return cudaGetLastError();
}

}  // namespace

int router_block_tokens(int E) {
    switch (pad_experts(E)) {
        case 8: return RouterTile<8>::BT;
        case 16: return RouterTile<16>::BT;
        case 32: return RouterTile<32>::BT;
        case 64: return RouterTile<64>::BT;
        case 128: return RouterTile<128>::BT;
        case 256: return RouterTile<256>::BT;
        case 512: return RouterTile<512>::BT;
        default: return RouterTile<1024>::BT;
    }
}

int router_blocks(int64_t N, int E) {
    int bt = router_block_tokens(E);
    return (int)((N + bt - 1) / bt);
}

cudaError_t launch_router(const moe_cfg& c, const void* x, const float* W_r, const float* b_r,
                          int32_t* idx, float* w, float* gap, float* p_part, float* P_sum,
                          cudaStream_t s) {
    cudaError_t err = cudaSuccess;
    if (c.N > 0) {
        switch (pad_experts(c.E)) {
            case 8: err = launch_ep<8>(c, x, W_r, b_r, idx, w, gap, p_part, s); break;
            case 16: err = launch_ep<16>(c, x, W_r, b_r, idx, w, gap, p_part, s); break;
            case 32: err = launch_ep<32>(c, x, W_r, b_r, idx, w, gap, p_part, s); break;
            case 64: err = launch_ep<64>(c, x, W_r, b_r, idx, w, gap, p_part, s); break;
            case 128: err = launch_ep<128>(c, x, W_r, b_r, idx, w, gap, p_part, s); break;
            case 256: err = launch_ep<256>(c, x, W_r, b_r, idx, w, gap, p_part, s); break;
            case 512: err = launch_ep<512>(c, x, W_r, b_r, idx, w, gap, p_part, s); break;
            default: err = launch_ep<1024>(c, x, W_r, b_r, idx, w, gap, p_part, s); break;
        }
        if (err != cudaSuccess) return err;
    }
    int blocks = router_blocks(c.N, c.E);
    reduce_p_kernel<<<(c.E + 255) / 256, 256, 0, s>>>(p_part, blocks, c.E, P_sum);
    return cudaGetLastError();
}

}  // namespace moe
