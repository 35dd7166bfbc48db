// combine_stats.cu -- weighted combine back to token order, the GEMM tile plan, and the
// load-balance statistics.
//
// Combine (page "混合专家 MoE", section "结构": y = sum_i w_i Expert_i(x), plus the shared
// expert; forward_grouped scatters the weighted rows back with index_add_): each token
// gathers its k grouped rows (already multiplied by their routing weight in the down-GEMM
// epilogue) in slot order, skips dropped slots (pos = -1), adds the shared experts' rows,
// sums in fp32 and rounds once.  This is a deterministic gather-reduce, not a scatter with
// atomics.
//
// Statistics (same page, section "负载均衡", aux_loss): f_e = counts_e / (N k),
// P_e = sum_t p[t,e] / N, L_aux = E sum_e f_e P_e, plus dropped / fully-dropped / near-tie
// counters (integer atomics only, so the result is deterministic).
#include "moe_internal.cuh"

namespace moe {
namespace {

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void add(const __nv_bfloat16* p, float (&a)[8]) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 f = __bfloat1622float2(h[i]);
            a[2 * i] += f.x;
            a[2 * i + 1] += f.y;
        }
    }
    __device__ static void store(__nv_bfloat16* p, const float (&a)[8]) {
        uint4 v;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = v;
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void add(const float* p, float (&a)[4]) {
        float4 v = __ldg(reinterpret_cast<const float4*>(p));
        a[0] += v.x;
        a[1] += v.y;
        a[2] += v.z;
        a[3] += v.w;
    }
    __device__ static void store(float* p, const float (&a)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(a[0], a[1], a[2], a[3]);
    }
};

// A warp takes one (token, column segment) unit at a time, lanes over 16-byte vectors, two
// vectors per lane per pass (2 (k + S) independent loads in flight).  Large batches use one
// segment per token (the whole row); a decode batch of a few dozen tokens splits each row into
// `segs` segments so that enough warps run to cover the memory latency.
template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ y, const int32_t* __restrict__ pos, const T* __restrict__ ysh,
               int S, int64_t N, int d, int k, int64_t R, int segs, T* __restrict__ out,
               int32_t* err) {
    constexpr int V = Vec<T>::N;
    const int lane = threadIdx.x & 31;
    const int64_t warp_global = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int chunks = d / V;
    const int span = ((chunks + segs - 1) / segs + 63) / 64 * 64;   // vectors per segment
    const int64_t units = N * segs;   // < 2^32 (checked by the host)
    for (int64_t u = warp_global; u < units; u += warps) {
        const uint32_t t32 = (uint32_t)u / (uint32_t)segs;
        const int sg = (int)((uint32_t)u - t32 * (uint32_t)segs);
        const int64_t t = t32;
        const int c_end = min(chunks, (sg + 1) * span);
        int32_t p[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
            p[j] = -1;
            if (j < k) {
                int32_t v = pos[t * k + j];
                if (v >= R) {
                    if (lane == 0 && sg == 0) atomicOr(err, MOE_DEVERR_BOUNDS);
                    v = -1;
                }
                p[j] = v;
            }
        }
        int c = sg * span + lane;
        for (; c + 32 < c_end; c += 64) {   // two vectors per pass
            float a[V], b[V];
#pragma unroll
            for (int i = 0; i < V; i++) a[i] = b[i] = 0.f;
#pragma unroll
            for (int j = 0; j < 16; j++)
                if (j < k && p[j] >= 0) {
                    Vec<T>::add(y + (int64_t)p[j] * d + c * V, a);
                    Vec<T>::add(y + (int64_t)p[j] * d + (c + 32) * V, b);
                }
            for (int s2 = 0; s2 < S; s2++) {
                Vec<T>::add(ysh + ((int64_t)s2 * N + t) * d + c * V, a);
                Vec<T>::add(ysh + ((int64_t)s2 * N + t) * d + (c + 32) * V, b);
            }
            Vec<T>::store(out + t * d + c * V, a);
            Vec<T>::store(out + t * d + (c + 32) * V, b);
        }
        for (; c < c_end; c += 32) {
            float a[V];
#pragma unroll
            for (int i = 0; i < V; i++) a[i] = 0.f;
#pragma unroll
            for (int j = 0; j < 16; j++)
                if (j < k && p[j] >= 0) Vec<T>::add(y + (int64_t)p[j] * d + c * V, a);
            for (int s2 = 0; s2 < S; s2++) Vec<T>::add(ysh + ((int64_t)s2 * N + t) * d + c * V, a);
            Vec<T>::store(out + t * d + c * V, a);
        }
    }
}

// mtile_off[i] = sum_{i' < i} ceil(kept[g(i')] / bm), one block, E <= 1024, where g is the
// identity or, with zigzag, the order 0, E-1, 1, E-2, ... (zigzag_group).
__global__ void __launch_bounds__(1024)
plan_kernel(const int32_t* __restrict__ kept, int E, int bm, int zigzag,
            int32_t* __restrict__ mtile_off) {
    __shared__ int tmp[33];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    const int v = e < E ? (kept[zigzag ? zigzag_group(e, E) : e] + bm - 1) / bm : 0;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) tmp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int wv = tmp[lane];
        int winc = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, winc, off);
            if (lane >= off) winc += o;
        }
        tmp[lane] = winc - wv;
        if (lane == 31) tmp[32] = winc;
    }
    __syncthreads();
    if (e < E) mtile_off[e] = tmp[warp] + inc - v;
    if (e == 0) mtile_off[E] = tmp[32];
}

// counters[0] fully dropped tokens, [1] near-tie tokens (counters zeroed by the caller)
__global__ void stats_tokens_kernel(const int32_t* __restrict__ pos, const float* __restrict__ gap,
                                    int64_t N, int k, int32_t* counters) {
    int fd = 0, nt = 0;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < N;
         t += (int64_t)gridDim.x * blockDim.x) {
        bool any = false;
        for (int j = 0; j < k; j++) any |= pos[t * k + j] >= 0;
        fd += !any;
        if (gap && gap[t] < MOE_TIE_EPS) nt++;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        fd += __shfl_xor_sync(0xffffffffu, fd, off);
        nt += __shfl_xor_sync(0xffffffffu, nt, off);
    }
    if ((threadIdx.x & 31) == 0) {
        if (fd) atomicAdd(&counters[0], fd);
        if (nt) atomicAdd(&counters[1], nt);
    }
}

// stats_f layout: f[E], P[E], then aux, dropped (as float bits of int: see host), ...
__global__ void __launch_bounds__(1024)
stats_final_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ kept,
                   const float* __restrict__ P_sum, int64_t N, int E, int k,
                   float* __restrict__ stats_f, int32_t* counters) {
    __shared__ float red[32];
    __shared__ int ired[2][32];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    float fp = 0.f;
    int kp = 0, touched = 0;
    if (e < E) {
        const float f = N > 0 ? (float)counts[e] / (float)(N * k) : 0.f;
        const float P = N > 0 ? P_sum[e] / (float)N : 0.f;
        stats_f[e] = f;
        stats_f[E + e] = P;
        fp = f * P;
        kp = kept[e];
        touched = kept[e] > 0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        fp += __shfl_xor_sync(0xffffffffu, fp, off);
        kp += __shfl_xor_sync(0xffffffffu, kp, off);
        touched += __shfl_xor_sync(0xffffffffu, touched, off);
    }
    if (lane == 0) {
        red[warp] = fp;
        ired[0][warp] = kp;
        ired[1][warp] = touched;
    }
    __syncthreads();
    if (e == 0) {
        float s = 0.f;
        int ks = 0, ts = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); w++) {
            s += red[w];
            ks += ired[0][w];
            ts += ired[1][w];
        }
        stats_f[2 * E] = (float)E * s;
        counters[2] = ks;   // kept rows
        counters[3] = ts;   // touched experts
    }
}

// z-loss: block b sums lse^2 over its fixed token range in double (thread-strided, then a
// fixed tree), so the partials and their order do not depend on timing.
__global__ void __launch_bounds__(256)
z_partial_kernel(const float* __restrict__ lse, int64_t N, double* __restrict__ z_part) {
    __shared__ double sm[256];
    const int64_t per = (N + gridDim.x - 1) / gridDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * per;
    const int64_t t1 = t0 + per < N ? t0 + per : N;
    double s = 0.0;
    for (int64_t t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
        const double v = (double)lse[t];
        s += v * v;
    }
    sm[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) sm[threadIdx.x] += sm[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) z_part[blockIdx.x] = sm[0];
}

// importance: one warp per expert sums the weights of its segment of the expert-sorted slots
// (lanes strided, fixed butterfly).
__global__ void __launch_bounds__(256)
importance_kernel(const float* __restrict__ w, const int32_t* __restrict__ perm,
                  const int32_t* __restrict__ offsets, int E, double* __restrict__ imp) {
    const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (e >= E) return;
    double s = 0.0;
    for (int64_t i = offsets[e] + lane; i < offsets[e + 1]; i += 32) s += (double)w[perm[i]];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) imp[e] = s;
}

}  // namespace

cudaError_t launch_combine(const moe_cfg& c, const void* y_perm, const int32_t* pos,
                           const void* y_sh, void* out, int32_t* err, cudaStream_t s) {
    if (c.N <= 0) return cudaSuccess;
    const int64_t R = grouped_rows(c);
    // segments per token: 1 unless the batch is too small to give the GPU an eighth of the
    // warps it can hold (measured: splitting a 4096- or 8192-token batch is slower)
    const int vec = c.act_dtype == MOE_BF16 ? 8 : 4;
    const int64_t resident = (int64_t)device_sm_count() * 64;   // warps the GPU holds at once
    const int max_segs = (int)(((int64_t)c.d / vec + 63) / 64);
    int64_t segs = c.N * 8 >= resident ? 1 : (resident + c.N - 1) / c.N;
    if (segs > max_segs) segs = max_segs;
    if (segs < 1) segs = 1;
    if (c.N * segs >= (int64_t)1 << 32) return cudaErrorInvalidValue;
    const int64_t want = (c.N * segs + 7) / 8;   // 8 warps per block
    const int64_t cap = (int64_t)device_sm_count() * 16;
    const int blocks = (int)(want < cap ? want : cap);
    if (c.act_dtype == MOE_BF16)
        combine_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            (const __nv_bfloat16*)y_perm, pos, (const __nv_bfloat16*)y_sh, c.n_shared, c.N, c.d,
            c.k, R, (int)segs, (__nv_bfloat16*)out, err);
    else
        combine_kernel<float><<<blocks, 256, 0, s>>>((const float*)y_perm, pos, (const float*)y_sh,
                                                     c.n_shared, c.N, c.d, c.k, R, (int)segs,
                                                     (float*)out, err);
    return cudaGetLastError();
}

cudaError_t launch_plan_mtiles(const int32_t* kept, int E, int bm, int32_t* mtile_off,
                               cudaStream_t s, bool zigzag) {
    plan_kernel<<<1, 1024, 0, s>>>(kept, E, bm, zigzag ? 1 : 0, mtile_off);
    return cudaGetLastError();
}

cudaError_t launch_router_stats(int64_t N, int E, int k, const float* lse, const float* w,
                                const int32_t* perm, const int32_t* offsets, double* z_part,
                                double* imp, cudaStream_t s) {
    z_partial_kernel<<<kRouterStatBlocks, 256, 0, s>>>(lse, N, z_part);
    importance_kernel<<<(E + 7) / 8, 256, 0, s>>>(w, perm, offsets, E, imp);
    return cudaGetLastError();
    (void)k;
}

cudaError_t launch_stats(const moe_cfg& c, const int32_t* counts, const int32_t* kept,
                         const float* P_sum, const int32_t* pos, const float* gap,
                         int32_t* counters, float* stats_f, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(counters, 0, 4 * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    if (c.N > 0) {
        int64_t want = (c.N + 255) / 256;
        int blocks = (int)(want < 148 * 4 ? want : 148 * 4);
        stats_tokens_kernel<<<blocks, 256, 0, s>>>(pos, gap, c.N, c.k, counters);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    stats_final_kernel<<<1, 1024, 0, s>>>(counts, kept, P_sum, c.N, c.E, c.k, stats_f, counters);
    return cudaGetLastError();
}

}  // namespace moe
