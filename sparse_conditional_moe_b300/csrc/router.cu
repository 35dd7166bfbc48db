// router.cu -- router: logits, softmax over all experts, top-k, renormalisation.
//
// Page "混合专家 MoE", section "实现：逐 token 与按专家分组", MoE.route: a linear layer d -> E
// scores every expert, softmax over the E scores, the k largest kept in descending order,
// and the k weights divided by their sum.  The router stays fp32 end to end: the logits are
// fp32 sums of exact products, and the top-k decision is taken on fp32 probabilities.
//
// Three ways to get the logits, one epilogue:
//   E <= 32      router_gemv_kernel: a warp per two tokens, lanes split d in 8-wide chunks,
//                each lane accumulates E short fp32 chains, a butterfly shuffle sums them;
//   E > 32, bf16 the tensor-core router of router_tc.cu: for E <= 512 and batches whose d is
//                not split, one fused launch (logits on chip, the tokens finished by the
//                cluster of expert-block CTAs); otherwise fp32 logits [N, E] (split over d for
//                small N), then logits_topk_kernel finishes each token, one per warp;
//   E > 32, fp32 router_tiled_kernel: BT tokens x all experts per block, DK-wide slices of x
//                and W_r in shared memory, each slice an fp32 FMA chain, slices added to the
//                running logit with compensated (Kahan) summation.
// finish_token() is the common epilogue: each warp owns a token, lane l holds the logits of
// experts l, l+32, ...; max and sum by warp shuffles; top-k by k rounds of a warp arg-max on
// (probability desc, expert index asc) -- each lane sorts its candidates once and offers its
// head, two warp reductions pick the winner; the (k+1)-th gives the near-tie gap; per-block
// column sums of the probabilities go to p_part (deterministic, no float atomics).
#include "router_finish.cuh"

namespace moe {
namespace {

using namespace router_detail;

constexpr int kRouterThreads = 256;
constexpr int kWarps = kRouterThreads / 32;

__device__ __forceinline__ float load_x(const float* x, int64_t i) { return x[i]; }
__device__ __forceinline__ float load_x(const __nv_bfloat16* x, int64_t i) {
    return __bfloat162float(x[i]);
}

// Column sums of the probabilities of this block's tokens, combined across warps in warp order.
template <int NV>
__device__ __forceinline__ void write_p_part(const float (&pacc)[NV], float* sm /*[kWarps][32NV]*/,
                                             int E, float* __restrict__ p_part) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int EPW = 32 * NV;
#pragma unroll
    for (int i = 0; i < NV; i++) sm[warp * EPW + lane + 32 * i] = pacc[i];
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kRouterThreads) {
        float sacc = 0.f;
        for (int w = 0; w < kWarps; w++) sacc += sm[w * EPW + e];
        p_part[(int64_t)blockIdx.x * E + e] = sacc;
    }
}

// ------------------------------------------------------------------ E <= 32: GEMV

constexpr int kGemvTokensPerWarp = 2;
constexpr int kGemvTokensPerBlock = kWarps * kGemvTokensPerWarp;

template <typename T>
struct Chunk8;
template <>
struct Chunk8<__nv_bfloat16> {
    __device__ static void load(const __nv_bfloat16* p, float (&f)[8]) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
};
template <>
struct Chunk8<float> {
    __device__ static void load(const float* p, float (&f)[8]) {
        float4 a = __ldg(reinterpret_cast<const float4*>(p));
        float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

template <int EP, typename T>
__global__ void __launch_bounds__(kRouterThreads)
router_gemv_kernel(const T* __restrict__ x, const float* __restrict__ W_r,
                   const float* __restrict__ b_r, int bias_mode, int64_t N, int d, int E, int k, int renorm,
                   int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                   float* __restrict__ gap_out, float* __restrict__ lse_out,
                   float* __restrict__ probs_out, float* __restrict__ p_part) {
    __shared__ float sm[kWarps * 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)blockIdx.x * kGemvTokensPerBlock + warp * kGemvTokensPerWarp;
    float pacc[1] = {0.f};
    float acc[kGemvTokensPerWarp][EP];
#pragma unroll
    for (int t = 0; t < kGemvTokensPerWarp; t++)
#pragma unroll
        for (int e = 0; e < EP; e++) acc[t][e] = 0.f;
    bool live[kGemvTokensPerWarp];
#pragma unroll
    for (int t = 0; t < kGemvTokensPerWarp; t++) live[t] = t0 + t < N;
    const int d8 = d & ~7;
    // unrolled so that several chunks' loads of x are in flight at once (the loop is
    // latency-bound otherwise: one x load per token per iteration)
#pragma unroll 4
    for (int c = lane * 8; c < d8; c += 256) {
        float xv[kGemvTokensPerWarp][8];
#pragma unroll
        for (int t = 0; t < kGemvTokensPerWarp; t++) {
            if (live[t]) Chunk8<T>::load(x + (t0 + t) * d + c, xv[t]);
            else
#pragma unroll
                for (int i = 0; i < 8; i++) xv[t][i] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < EP; e++) {
            if (e < E) {
                float wv[8];
                Chunk8<float>::load(W_r + (int64_t)e * d + c, wv);
#pragma unroll
                for (int t = 0; t < kGemvTokensPerWarp; t++)
#pragma unroll
                    for (int i = 0; i < 8; i++) acc[t][e] = fmaf(xv[t][i], wv[i], acc[t][e]);
            }
        }
    }
    for (int c = d8 + lane; c < d; c += 32) {   // d not a multiple of 8 (fp32 layers)
#pragma unroll
        for (int e = 0; e < EP; e++) {
            if (e < E) {
                const float wv = W_r[(int64_t)e * d + c];
#pragma unroll
                for (int t = 0; t < kGemvTokensPerWarp; t++)
                    if (live[t]) acc[t][e] = fmaf(load_x(x, (t0 + t) * d + c), wv, acc[t][e]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kGemvTokensPerWarp; t++) {
#pragma unroll
        for (int e = 0; e < EP; e++)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                acc[t][e] += __shfl_xor_sync(0xffffffffu, acc[t][e], off);
        if (!live[t]) continue;    // warp-uniform
        float v[1] = {0.f};
#pragma unroll
        for (int e = 0; e < EP; e++)
            if (e == lane) v[0] = acc[t][e];
        finish_token<1>(v, b_r, bias_mode, E, k, renorm, t0 + t, idx_out, w_out, gap_out, lse_out, probs_out, pacc);
    }
    write_p_part<1>(pacc, sm, E, p_part);
}

// ------------------------------------------------------------------ logits -> top-k

constexpr int kTopkTokensPerBlock = 8;   // one token per warp: latency is hidden by occupancy

template <int NV>
__global__ void __launch_bounds__(kRouterThreads)
logits_topk_kernel(const float* __restrict__ logits, const float* __restrict__ b_r, int bias_mode,
                   int64_t N,
                   int E, int k, int renorm, int32_t* __restrict__ idx_out,
                   float* __restrict__ w_out, float* __restrict__ gap_out,
                   float* __restrict__ lse_out, float* __restrict__ probs_out,
                   float* __restrict__ p_part) {
    __shared__ float sm[kWarps * 32 * NV];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float pacc[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) pacc[i] = 0.f;
    for (int t = warp; t < kTopkTokensPerBlock; t += kWarps) {
        const int64_t tok = (int64_t)blockIdx.x * kTopkTokensPerBlock + t;
        if (tok >= N) break;
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int e = lane + 32 * i;
            v[i] = e < E ? logits[tok * E + e] : 0.f;
        }
        finish_token<NV>(v, b_r, bias_mode, E, k, renorm, tok, idx_out, w_out, gap_out, lse_out, probs_out, pacc);
    }
    write_p_part<NV>(pacc, sm, E, p_part);
}

// ------------------------------------------------------------------ E > 32, fp32: tiled

template <int EP>
struct RouterTile {
    static constexpr int TE = EP / 32;                                    // experts per thread
    static constexpr int TT = EP >= 1024 ? 1 : (EP >= 512 ? 2 : 4);       // tokens per thread
    static constexpr int BT = kWarps * TT;                                // tokens per block
    static constexpr int DK = EP >= 1024 ? 8 : (EP >= 512 ? 16 : 32);     // d-slice per stage
    static constexpr int XS = BT * (DK + 1);                              // x slice [BT][DK+1]
    static constexpr int WS = DK * EP;                                    // W slice [DK][EP]
    static constexpr int LS = BT * (EP + 1);                              // logits [BT][EP+1]
    static constexpr int SMEM_FLOATS = (XS + WS) > LS ? (XS + WS) : LS;
    static constexpr int NV = EP / 32;
};

template <int EP, typename T>
__global__ void __launch_bounds__(kRouterThreads)
router_tiled_kernel(const T* __restrict__ x, const float* __restrict__ W_r,
                    const float* __restrict__ b_r, int bias_mode, int64_t N, int d, int E, int k, int renorm,
                    int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                    float* __restrict__ gap_out, float* __restrict__ lse_out,
                   float* __restrict__ probs_out, float* __restrict__ p_part) {
    using Tl = RouterTile<EP>;
    constexpr int TT = Tl::TT, TE = Tl::TE, BT = Tl::BT, DK = Tl::DK, NV = Tl::NV;
    static_assert(Tl::SMEM_FLOATS >= kWarps * EP, "P table must fit the staging buffer");
    __shared__ float sm[Tl::SMEM_FLOATS];
    float* Xs = sm;             // [BT][DK+1]
    float* Ws = sm + Tl::XS;    // [DK][EP]

    const int tid = threadIdx.x;
    const int tx = tid % 32, ty = tid / 32;
    const int64_t t0 = (int64_t)blockIdx.x * BT;

    // acc: running logit; cmp: its compensation term (Kahan), so that the only rounding left
    // of any size is inside each DK-long slice (fp32 FMA chain over DK products).
    float acc[TT][TE], cmp[TT][TE];
#pragma unroll
    for (int i = 0; i < TT; i++)
#pragma unroll
        for (int j = 0; j < TE; j++) acc[i][j] = cmp[i][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += DK) {
        for (int v = tid; v < BT * DK; v += kRouterThreads) {
            const int t = v / DK, kk = v % DK;
            const int64_t tok = t0 + t;
            float val = 0.f;
            if (tok < N && k0 + kk < d) val = load_x(x, tok * d + k0 + kk);
            Xs[t * (DK + 1) + kk] = val;
        }
        for (int v = tid; v < EP * DK; v += kRouterThreads) {
            const int e = v % EP, kk = v / EP;
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
            for (int i = 0; i < TT; i++) xv[i] = Xs[(ty + i * kWarps) * (DK + 1) + kk];
#pragma unroll
            for (int j = 0; j < TE; j++) wv[j] = Ws[kk * EP + tx + j * 32];
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

    // logits -> shared [BT][EP+1]; thread (ty, tx) owns tokens ty + i*8 and experts tx + j*32
    float* Ls = sm;
#pragma unroll
    for (int i = 0; i < TT; i++)
#pragma unroll
        for (int j = 0; j < TE; j++) Ls[(ty + i * kWarps) * (EP + 1) + tx + j * 32] = acc[i][j];
    __syncthreads();

    const int warp = tid >> 5, lane = tid & 31;
    float pacc[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) pacc[i] = 0.f;
    for (int t = warp; t < BT; t += kWarps) {
        const int64_t tok = t0 + t;
        if (tok >= N) break;
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; i++) v[i] = Ls[t * (EP + 1) + lane + 32 * i];
        finish_token<NV>(v, b_r, bias_mode, E, k, renorm, tok, idx_out, w_out, gap_out, lse_out, probs_out, pacc);
    }
    __syncthreads();             // every warp is done reading the logits
    write_p_part<NV>(pacc, sm, E, p_part);
}

// P_sum[e] = sum over router blocks b of p_part[b][e], in a fixed order (deterministic): one
// block of 32 warps per 32 experts, lane = expert (coalesced rows); warp w adds blocks w, w + 32,
// ... in order, then warp 0 adds the 32 warp sums in warp order.  Only E / 32 blocks run, so the
// kernel is bound by load latency: each warp keeps 32 loads in flight (8 took 8 us on 2048
// partial rows, four rounds of latency).
__global__ void __launch_bounds__(1024) reduce_p_kernel(const float* __restrict__ p_part, int blocks,
                                                        int E, float* __restrict__ P_sum) {
    __shared__ float part[32][33];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    float s = 0.f;
    if (e < E) {
        constexpr int kInFlight = 32;
        int b = warp;
        for (; b + (kInFlight - 1) * 32 < blocks; b += kInFlight * 32) {
            float v[kInFlight];
#pragma unroll
            for (int i = 0; i < kInFlight; i++) v[i] = p_part[(int64_t)(b + 32 * i) * E + e];
#pragma unroll
            for (int i = 0; i < kInFlight; i++) s += v[i];
        }
        for (; b < blocks; b += 32) s += p_part[(int64_t)b * E + e];
    }
    part[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && e < E) {
        float t = 0.f;
        for (int w = 0; w < 32; w++) t += part[w][lane];
        P_sum[e] = t;
    }
}

int pad_experts(int E) {
    int ep = 8;
    while (ep < E) ep *= 2;
    return ep;
}

template <typename Kernel, typename T>
void launch_k(Kernel kern, int blocks, cudaStream_t s, const T* x, const float* W_r,
              const float* bias, const moe_cfg& c, int32_t* idx, float* w, float* gap,
              float* lse, float* probs, float* p_part) {
    kern<<<blocks, kRouterThreads, 0, s>>>(x, W_r, bias, c.bias_mode, c.N, c.d, c.E, c.k, c.renorm, idx, w,
                                           gap, lse, probs, p_part);
}

template <int EP, typename T>
int launch_gemv(const moe_cfg& c, const T* x, const float* W_r, const float* bias, int32_t* idx,
                float* w, float* gap, float* lse, float* probs, float* p_part, cudaStream_t s) {
    const int blocks = (int)((c.N + kGemvTokensPerBlock - 1) / kGemvTokensPerBlock);
    launch_k(router_gemv_kernel<EP, T>, blocks, s, x, W_r, bias, c, idx, w, gap, lse, probs, p_part);
    return blocks;
}

template <int EP, typename T>
int launch_tiled(const moe_cfg& c, const T* x, const float* W_r, const float* bias, int32_t* idx,
                 float* w, float* gap, float* lse, float* probs, float* p_part, cudaStream_t s) {
    const int blocks = (int)((c.N + RouterTile<EP>::BT - 1) / RouterTile<EP>::BT);
    launch_k(router_tiled_kernel<EP, T>, blocks, s, x, W_r, bias, c, idx, w, gap, lse, probs, p_part);
    return blocks;
}

template <int NV>
int launch_topk(const moe_cfg& c, const float* logits, const float* bias, int32_t* idx, float* w,
                float* gap, float* lse, float* probs, float* p_part, cudaStream_t s) {
    const int blocks = (int)((c.N + kTopkTokensPerBlock - 1) / kTopkTokensPerBlock);
    logits_topk_kernel<NV><<<blocks, kRouterThreads, 0, s>>>(logits, bias, c.bias_mode, c.N, c.E, c.k, c.renorm,
                                                             idx, w, gap, lse, probs, p_part);
    return blocks;
}

template <typename T>
int dispatch_simt(const moe_cfg& c, const T* x, const float* W_r, const float* bias, int32_t* idx,
                  float* w, float* gap, float* lse, float* probs, float* p_part, cudaStream_t s) {
    switch (pad_experts(c.E)) {
        case 8: return launch_gemv<8>(c, x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        case 16: return launch_gemv<16>(c, x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        case 32: return launch_gemv<32>(c, x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        case 64: return launch_tiled<64>(c, x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        case 128: return launch_tiled<128>(c, x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        case 256: return launch_tiled<256>(c, x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        case 512: return launch_tiled<512>(c, x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        default: return launch_tiled<1024>(c, x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
    }
}

}  // namespace

bool router_uses_tensor_cores(const moe_cfg& c) { return c.act_dtype == MOE_BF16 && c.E > 32; }

int64_t router_part_rows(int64_t N) { return (N + 7) / 8 + 1; }

cudaError_t launch_router(const moe_cfg& c, const void* x, const float* W_r, const float* b_r,
                          int32_t* idx, float* w, float* gap, float* lse, float* p_part,
                          float* P_sum, __nv_bfloat16* w3, float* logits, int32_t* err,
                          cudaStream_t s, float* probs, bool w3_ready) {
    const float* bias = c.bias_mode != 0 ? b_r : nullptr;
    int blocks = 0;
    if (c.N > 0) {
        if (router_uses_tensor_cores(c)) {
            cudaError_t e = cudaSuccess;
            if (!w3_ready) e = tc_router_split(W_r, c.E, c.d, w3, s);
            if (e != cudaSuccess) return e;
            if (router_tc_fused(c.N, c.d, c.E)) {
                e = tc_router_fused((const __nv_bfloat16*)x, c.N, c.d, w3, c.E, bias, c.bias_mode,
                                    c.k, c.renorm, idx, w, gap, lse, probs, p_part, err, s);
                if (e != cudaSuccess) return e;
                reduce_p_kernel<<<(c.E + 31) / 32, 1024, 0, s>>>(
                    p_part, router_tc_part_rows(c.N, c.E), c.E, P_sum);
                return cudaGetLastError();
            }
            e = tc_router_logits((const __nv_bfloat16*)x, c.N, c.d, w3, c.E, logits, err, s);
            if (e != cudaSuccess) return e;
            switch (pad_experts(c.E) / 32) {
                case 1: case 2: blocks = launch_topk<2>(c, logits, bias, idx, w, gap, lse, probs, p_part, s); break;
                case 4: blocks = launch_topk<4>(c, logits, bias, idx, w, gap, lse, probs, p_part, s); break;
                case 8: blocks = launch_topk<8>(c, logits, bias, idx, w, gap, lse, probs, p_part, s); break;
                case 16: blocks = launch_topk<16>(c, logits, bias, idx, w, gap, lse, probs, p_part, s); break;
                default: blocks = launch_topk<32>(c, logits, bias, idx, w, gap, lse, probs, p_part, s); break;
            }
        } else if (c.act_dtype == MOE_BF16) {
            blocks = dispatch_simt(c, (const __nv_bfloat16*)x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        } else {
            blocks = dispatch_simt(c, (const float*)x, W_r, bias, idx, w, gap, lse, probs, p_part, s);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    reduce_p_kernel<<<(c.E + 31) / 32, 1024, 0, s>>>(p_part, blocks, c.E, P_sum);
    return cudaGetLastError();
}

}  // namespace moe
