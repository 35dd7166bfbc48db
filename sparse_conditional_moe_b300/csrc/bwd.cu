// bwd.cu -- backward pass of the layer: gradients of sum <dout, out> + aux_coef L_aux +
// z_coef L_z with respect to x, W_r, the logit bias and every expert matrix.
//
// The chain rule through page "混合专家 MoE" (实现: MoE.route, Expert.forward, forward_grouped;
// 负载均衡: aux_loss) and the z-loss of "混合专家模型 (MoE)：大规模稀疏条件计算的架构与工程实践"
// section 三.3.  Readings (shared with the oracle): no gradient through the top-k choice or a
// capacity drop, none for the selection-only bias (bias_mode 2), f_e of L_aux is a count, the
// bf16 rounding of h passes the gradient.  Steps, on the forward's workspace:
//   1. the router again (bit-identical) with its probabilities [N, E];
//   2. plans: every expert's kept rows in a zero-padded segment starting at a multiple of 128
//      (so reductions over rows never mix experts), one segment per shared expert;
//   3. gathers: dout and x rows into those segments;
//   4. per expert group (grouped_gemm_bwd.cu): dh and dw (G1), SwiGLU backward (G2), dX (G3),
//      dW_down (G4), dW_gate / dW_up (G5); the same for the shared experts;
//   5. router backward per token: dw -> dp through the renormalisation, + aux term, softmax
//      backward, + z term -> dl [N, E]; db = sum_t dl (bias_mode 1);
//   6. dW_r = dl^T x and the router's part of dx = dl W_r (tensor cores, fp32 operands split
//      into bf16 pieces);
//   7. dx per token: its kept rows of dX + the shared experts' dX + the router part (fp32).
#include "bwd_internal.cuh"

namespace moe {
namespace {

constexpr int kPad = 128;

__device__ __forceinline__ int find_group(const int32_t* off, int G, int64_t r) {
    int lo = 0, hi = G;   // largest g with off[g] <= r
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= r) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Routed plan: c_off = exclusive prefix of roundup(kept, 128) (one block, E <= 1024).
__global__ void __launch_bounds__(1024) plan_routed_kernel(const int32_t* __restrict__ kept, int E,
                                                           int32_t* __restrict__ c_off) {
    __shared__ int32_t sm[1024];
    const int e = threadIdx.x;
    const int v = e < E ? (kept[e] + kPad - 1) / kPad * kPad : 0;
    sm[e] = v;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {       // inclusive Hillis-Steele scan
        const int add = e >= off ? sm[e - off] : 0;
        __syncthreads();
        sm[e] += add;
        __syncthreads();
    }
    if (e < E) c_off[e + 1] = sm[e];
    if (e == 0) c_off[0] = 0;
}

// Shared plan: S groups of N rows, segments Np apart; A rows shared (offset 0).
__global__ void plan_shared_kernel(int S, int N, int Np, int32_t* rows, int32_t* zero_off,
                                   int32_t* c_off, int32_t* dense_off) {
    const int s = threadIdx.x;
    if (s <= S) {
        zero_off[s] = 0;
        c_off[s] = s * Np;
    }
    if (s < S) {
        rows[s] = N;
        dense_off[s] = s * N;
    }
}

// One warp per padded row: dout and x rows of routed groups (zeros in the padding), both read
// through the grouped row's token.
__global__ void __launch_bounds__(256)
gather_routed_kernel(const int32_t* __restrict__ c_off, const int32_t* __restrict__ kept,
                     const int32_t* __restrict__ kept_off, const int32_t* __restrict__ row_token,
                     int E, int64_t rows_bound, int d, const __nv_bfloat16* __restrict__ dout,
                     const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ dout_pad,
                     __nv_bfloat16* __restrict__ x_pad) {
    const int64_t pr = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (pr >= rows_bound || pr >= c_off[E]) return;
    const int g = find_group(c_off, E, pr);
    const int64_t local = pr - c_off[g];
    const bool valid = local < kept[g];
    const int64_t dr = kept_off[g] + local;
    const uint4* src_d = valid ? reinterpret_cast<const uint4*>(dout + (int64_t)row_token[dr] * d) : nullptr;
    const uint4* src_x = valid ? reinterpret_cast<const uint4*>(x + (int64_t)row_token[dr] * d) : nullptr;
    uint4* dd = reinterpret_cast<uint4*>(dout_pad + pr * d);
    uint4* dx = reinterpret_cast<uint4*>(x_pad + pr * d);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int c = lane; c < d / 8; c += 32) {
        dd[c] = valid ? src_d[c] : z;
        dx[c] = valid ? src_x[c] : z;
    }
}

// dout and x rows for the shared experts: rows [0, N) then zeros up to Np.
__global__ void __launch_bounds__(256)
gather_shared_kernel(int64_t N, int64_t Np, int d, const __nv_bfloat16* __restrict__ dout,
                     const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ dout_pad,
                     __nv_bfloat16* __restrict__ x_pad) {
    const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= Np) return;
    const bool valid = r < N;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int c = lane; c < d / 8; c += 32) {
        reinterpret_cast<uint4*>(dout_pad + r * d)[c] =
            valid ? reinterpret_cast<const uint4*>(dout + r * d)[c] : z;
        reinterpret_cast<uint4*>(x_pad + r * d)[c] =
            valid ? reinterpret_cast<const uint4*>(x + r * d)[c] : z;
    }
}

// dw of each dense grouped row: the sum of its G1 tile partials, in column-tile order.
__global__ void dw_rows_kernel(const int32_t* __restrict__ kept_off, const int32_t* __restrict__ c_off,
                               int E, int64_t R, const float* __restrict__ part, int n_tiles,
                               float* __restrict__ dw_row) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R || r >= kept_off[E]) return;
    const int g = find_group(kept_off, E, r);
    const int64_t pr = c_off[g] + (r - kept_off[g]);
    float s = 0.f;
    for (int t = 0; t < n_tiles; t++) s += part[pr * n_tiles + t];
    dw_row[r] = s;
}

// Router backward, one warp per token; lanes own experts lane, lane + 32, ...
template <int NV>
__global__ void __launch_bounds__(256)
router_bwd_kernel(int64_t N, int E, int k, int renorm, const float* __restrict__ probs,
                  const int32_t* __restrict__ idx, const float* __restrict__ w,
                  const int32_t* __restrict__ pos, const float* __restrict__ dw_row,
                  const int32_t* __restrict__ counts, const float* __restrict__ lse,
                  float aux_scale, float z_scale, float* __restrict__ dl) {
    // aux_scale = aux_coef E / (N k N): dL_aux/dp_e = aux_scale * counts_e;
    // z_scale = 2 z_coef / N: dL_z/dl_e = z_scale * lse_t * p_e
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= N) return;
    float p[NV], dp[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        p[i] = e < E ? probs[t * E + e] : 0.f;
        dp[i] = e < E ? aux_scale * (float)counts[e] : 0.f;
    }
    // routing weights -> selected probabilities: lane j < k loads slot j, then warp sums
    int ej = 0;
    float wj = 0.f, dwj = 0.f, pj = 0.f;
    if (lane < k) {
        ej = idx[t * k + lane];
        const int posj = pos[t * k + lane];
        wj = w[t * k + lane];
        dwj = posj >= 0 ? dw_row[posj] : 0.f;
        pj = probs[t * E + ej];
    }
    float ssel = pj, wdw = wj * dwj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ssel += __shfl_xor_sync(0xffffffffu, ssel, off);
        wdw += __shfl_xor_sync(0xffffffffu, wdw, off);
    }
    const float addj = renorm ? (dwj - wdw) / ssel : dwj;
    for (int j = 0; j < k; j++) {
        const int e = __shfl_sync(0xffffffffu, ej, j);
        const float add = __shfl_sync(0xffffffffu, addj, j);
#pragma unroll
        for (int i = 0; i < NV; i++)
            if (lane + 32 * i == e) dp[i] += add;
    }
    // softmax backward + z-loss term
    float pdp = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) pdp += p[i] * dp[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) pdp += __shfl_xor_sync(0xffffffffu, pdp, off);
    const float zt = z_scale * lse[t];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        if (e < E) dl[t * E + e] = p[i] * (dp[i] - pdp) + zt * p[i];
    }
}

// The router GEMMs run on the tensor cores with fp32 operands split into bf16 pieces:
// v = hi + lo + O(2^-17 |v|) with hi = bf16(v), lo = bf16(v - hi) (v - hi is exact in fp32).
//   dx_r = dl W_r  ~ dl_hi W_hi + dl_hi W_lo + dl_lo W_hi   (K = 3E: A = [hi | hi | lo],
//                                                              B = [W_hi; W_lo; W_hi])
//   dW_r = dl^T x  = dl_hi^T x + dl_lo^T x                  (K = 2N: A = [hi; lo], B = [x; x])
// (x is bf16 already).  The products are exact; the fp32 accumulation matches a plain fp32
// GEMM to within its own rounding.
// Row widths are padded to multiples of 8 elements (16-byte TMA strides) with zeros:
// dl3 [N, K3], K3 = roundup(3E, 8); dlT2 [2N, Ep], Ep = roundup(E, 8); w3 [K3, d].
__host__ __device__ inline int pad8(int v) { return (v + 7) / 8 * 8; }

__global__ void split_dl_kernel(const float* __restrict__ dl, int64_t N, int E,
                                __nv_bfloat16* __restrict__ dl3, __nv_bfloat16* __restrict__ dlT2) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N * E) return;
    const int64_t t = i / E;
    const int e = (int)(i - t * E);
    const int K3 = pad8(3 * E), Ep = pad8(E);
    const float v = dl[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    dl3[t * K3 + e] = hi;
    dl3[t * K3 + E + e] = hi;
    dl3[t * K3 + 2 * E + e] = lo;
    dlT2[t * Ep + e] = hi;
    dlT2[(N + t) * Ep + e] = lo;
}

__global__ void split_wr_kernel(const float* __restrict__ W, int E, int d,
                                __nv_bfloat16* __restrict__ w3) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)E * d) return;
    const float v = W[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    w3[i] = hi;
    w3[(int64_t)E * d + i] = lo;
    w3[2 * (int64_t)E * d + i] = hi;
}

// x2 = [x; x] (2N rows)
__global__ void dup_rows_kernel(const uint4* __restrict__ x, int64_t n16, uint4* __restrict__ x2) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n16) return;
    const uint4 v = x[i];
    x2[i] = v;
    x2[n16 + i] = v;
}

// One group of `rows` rows at offset 0 (a_off = c_off = {0, pad}, dense_off = {0}).
__global__ void plan_single_kernel(int64_t rows, int64_t pad, int32_t* plan) {
    if (threadIdx.x == 0) {
        plan[0] = (int32_t)rows;
        plan[1] = 0;
        plan[2] = (int32_t)pad;
        plan[3] = 0;
    }
}

// db partials: block b sums its token chunk for every expert (threads over experts: coalesced),
// then db[e] = the partials in block order.
constexpr int kDbChunks = 64;
__global__ void db_part_kernel(const float* __restrict__ dl, int64_t N, int E,
                               double* __restrict__ part) {
    const int64_t per = (N + kDbChunks - 1) / kDbChunks;
    const int64_t t0 = (int64_t)blockIdx.x * per, t1 = t0 + per < N ? t0 + per : N;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        double s = 0.0;
        for (int64_t t = t0; t < t1; t++) s += (double)dl[t * E + e];
        part[(int64_t)blockIdx.x * E + e] = s;
    }
}

__global__ void db_final_kernel(const double* __restrict__ part, int E, float* __restrict__ db) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    double s = 0.0;
    for (int b = 0; b < kDbChunks; b++) s += part[(int64_t)b * E + e];
    db[e] = (float)s;
}

// dx[t] = sum over t's kept slots of dX[padded row] + sum_s dX_s[s * Np + t] + dx_r[t].
__global__ void __launch_bounds__(256)
dx_combine_kernel(int64_t N, int k, int d, int S, int64_t Np, const int32_t* __restrict__ idx,
                  const int32_t* __restrict__ pos, const int32_t* __restrict__ kept_off,
                  const int32_t* __restrict__ c_off, const float* __restrict__ dX,
                  const float* __restrict__ dXs, const float* __restrict__ dx_r,
                  float* __restrict__ dx) {
    const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= N) return;
    int64_t prow[16];
    for (int j = 0; j < k; j++) {
        const int p = pos[t * k + j];
        const int e = idx[t * k + j];
        prow[j] = p >= 0 ? c_off[e] + (p - kept_off[e]) : -1;
    }
    for (int c = lane; c < d / 4; c += 32) {
        float4 a = reinterpret_cast<const float4*>(dx_r + t * d)[c];
        for (int j = 0; j < k; j++) {
            if (prow[j] < 0) continue;
            const float4 v = reinterpret_cast<const float4*>(dX + prow[j] * d)[c];
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
        for (int s = 0; s < S; s++) {
            const float4 v = reinterpret_cast<const float4*>(dXs + (s * Np + t) * d)[c];
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
        reinterpret_cast<float4*>(dx + t * d)[c] = a;
    }
}

int router_nv(int E) {
    int nv = 1;
    while (nv * 32 < E) nv *= 2;
    return nv;
}

}  // namespace

int64_t bwd_padded_rows(const moe_cfg& c) { return grouped_rows(c) + (int64_t)kPad * c.E; }
int64_t bwd_shared_rows(const moe_cfg& c) { return (c.N + kPad - 1) / kPad * kPad; }

BwdLayout bwd_layout(const moe_cfg& c) {
    BwdLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += ((bytes ? bytes : 1) + 255) & ~(size_t)255;
        return o;
    };
    const int64_t N = c.N, E = c.E, d = c.d, F = c.d_ff, S = c.n_shared, Fs = c.d_ff_shared;
    const int64_t R = grouped_rows(c), Rp = bwd_padded_rows(c), Np = bwd_shared_rows(c);
    L.probs = take(4 * (size_t)(N * E));
    L.dl = take(4 * (size_t)(N * E));
    L.dx_r = take(4 * (size_t)(N * d));
    L.dw_row = take(4 * (size_t)R);
    L.c_off = take(4 * (size_t)(E + 1));
    L.s_plan = take(4 * (size_t)(4 * (S + 1)));
    L.dout_pad = take(2 * (size_t)(Rp * d));
    L.x_pad = take(2 * (size_t)(Rp * d));
    L.dh = take(2 * (size_t)(Rp * F));
    L.dgu = take(2 * (size_t)(Rp * 2 * F));
    L.hw = take(2 * (size_t)(Rp * F));
    L.dX = take(4 * (size_t)(Rp * d));
    L.dw_part = take(4 * (size_t)(Rp * (F / 128)));
    L.dout_s = take(2 * (size_t)(Np * d));
    L.x_s = take(2 * (size_t)(Np * d));
    L.dh_s = take(2 * (size_t)(S * Np * Fs));
    L.dgu_s = take(2 * (size_t)(S * Np * 2 * Fs));
    L.hw_s = take(2 * (size_t)(S * Np * Fs));
    L.dX_s = take(4 * (size_t)(S * Np * d));
    L.dw_part_s = take(4 * (size_t)(S * Np * (Fs > 0 ? Fs / 128 : 1)));
    L.r_plan = take(4 * 8);
    L.dl3 = take(2 * (size_t)(N * pad8(3 * (int)E)));
    L.dlT2 = take(2 * (size_t)(2 * N * pad8((int)E)));
    L.w3 = take(2 * (size_t)(pad8(3 * (int)E) * d));
    L.x2 = take(2 * (size_t)(2 * N * d));
    L.db_part = take(8 * (size_t)(kDbChunks * E));
    L.total = off;
    return L;
}

template <typename T>
static T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Runs the expert part (G1..G5) for one set of groups.
static cudaError_t expert_bwd(const TbParams& base, const int32_t* zero_off, int64_t rows_a,
                              int64_t rows_c, int d, int F, const __nv_bfloat16* dout_pad,
                              const __nv_bfloat16* x_pad, const __nv_bfloat16* Wg,
                              const __nv_bfloat16* Wu, const __nv_bfloat16* Wd,
                              const __nv_bfloat16* h_fwd, const float* row_weight,
                              __nv_bfloat16* dh, float* dw_part, __nv_bfloat16* dgu,
                              __nv_bfloat16* hw, float* dX, float* dWg, float* dWu, float* dWd,
                              cudaStream_t s) {
    cudaError_t e;
    // G1: dh = w dH', partial <dH', h>
    TbParams p = base;
    p.aux_bf16 = h_fwd;
    p.ld_aux = F;
    p.row_weight = row_weight;
    p.out_bf16 = dh;
    p.ld_bf16 = F;
    p.dw_part = dw_part;
    if ((e = tb_dh(p, dout_pad, rows_a, d, Wd, F, s)) != cudaSuccess) return e;
    // G2: recompute g, u; dG, dU, w h
    p = base;
    p.aux_bf16 = dh;
    p.ld_aux = F;
    p.row_weight = row_weight;
    p.out_bf16 = dgu;
    p.ld_bf16 = 2 * F;
    p.out2_bf16 = hw;
    if ((e = tb_swiglu_bwd(p, x_pad, rows_a, d, Wg, Wu, F, s)) != cudaSuccess) return e;
    // G3: dX rows (A = [dG | dU] lives at the output's row offsets)
    p = base;
    p.a_off = base.c_off;
    p.out_f32 = dX;
    if ((e = tb_dx(p, dgu, rows_c, F, Wg, Wu, d, s)) != cudaSuccess) return e;
    // G4: dW_d[g] [d, F] = sum_r dout_r (w h)_r^T  (A = dout rows at a_off, B = w h at c_off)
    p = base;
    p.split_m = d;
    p.out_f32 = dWd;
    p.out_f32b = dWd;
    if ((e = tb_wgrad(p, dout_pad, rows_a, d, hw, rows_c, F, s)) != cudaSuccess) return e;
    // G5: [dW_g; dW_u][g] [2F, d] = sum_r [dG | dU]_r^T x_r  (A at c_off, B = x at a_off)
    p = base;
    p.a_off = base.c_off;
    p.c_off = zero_off ? zero_off : base.c_off;
    p.split_m = F;
    p.out_f32 = dWg;
    p.out_f32b = dWu;
    return tb_wgrad(p, dgu, rows_c, 2 * F, x_pad, rows_a, d, s);
}

cudaError_t run_backward(const BwdArgs& a, cudaStream_t s) {
    const moe_cfg& c = *a.cfg;
    const BwdLayout L = bwd_layout(c);
    void* bw = a.bws;
    const int64_t N = c.N, d = c.d, F = c.d_ff, S = c.n_shared, Fs = c.d_ff_shared;
    const int E = c.E, k = c.k;
    const int64_t R = grouped_rows(c), Rp = bwd_padded_rows(c), Np = bwd_shared_rows(c);
    cudaError_t e;
    float* probs = at<float>(bw, L.probs);
    // 1. router again, with its probabilities
    if ((e = launch_router(c, a.x, a.W_r, a.b_r, a.idx, a.w, a.gap, a.lse, a.p_part, a.P_sum, a.w3,
                           a.logits, a.err, s, probs)) != cudaSuccess)
        return e;
    // 2. plans
    int32_t* c_off = at<int32_t>(bw, L.c_off);
    plan_routed_kernel<<<1, 1024, 0, s>>>(a.kept, E, c_off);
    int32_t* sp = at<int32_t>(bw, L.s_plan);
    int32_t *s_rows = sp, *s_zero = sp + (S + 1), *s_coff = sp + 2 * (S + 1), *s_dense = sp + 3 * (S + 1);
    if (S > 0) plan_shared_kernel<<<1, 32, 0, s>>>((int)S, (int)N, (int)Np, s_rows, s_zero, s_coff, s_dense);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3. gathers
    __nv_bfloat16* dout_pad = at<__nv_bfloat16>(bw, L.dout_pad);
    __nv_bfloat16* x_pad = at<__nv_bfloat16>(bw, L.x_pad);
    if (R > 0) {
        gather_routed_kernel<<<(unsigned)((Rp * 32 + 255) / 256), 256, 0, s>>>(
            c_off, a.kept, a.kept_off, a.row_token, E, Rp, (int)d, a.dout,
            (const __nv_bfloat16*)a.x, dout_pad, x_pad);
    }
    __nv_bfloat16* dout_s = at<__nv_bfloat16>(bw, L.dout_s);
    __nv_bfloat16* x_s = at<__nv_bfloat16>(bw, L.x_s);
    if (S > 0 && N > 0)
        gather_shared_kernel<<<(unsigned)((Np * 32 + 255) / 256), 256, 0, s>>>(N, Np, (int)d, a.dout,
                                                                              (const __nv_bfloat16*)a.x,
                                                                              dout_s, x_s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4. experts
    float* dw_row = at<float>(bw, L.dw_row);
    if (R > 0) {
        TbParams base{};
        base.G = E;
        base.rows = a.kept;
        base.a_off = c_off;
        base.c_off = c_off;
        base.dense_off = a.kept_off;
        base.max_mtiles = Rp / 128;
        base.err = a.err;
        if ((e = expert_bwd(base, nullptr, Rp, Rp, (int)d, (int)F, dout_pad, x_pad, a.Wg, a.Wu, a.Wd,
                            a.h_perm, a.row_weight, at<__nv_bfloat16>(bw, L.dh),
                            at<float>(bw, L.dw_part), at<__nv_bfloat16>(bw, L.dgu),
                            at<__nv_bfloat16>(bw, L.hw), at<float>(bw, L.dX), a.dWg, a.dWu, a.dWd,
                            s)) != cudaSuccess)
            return e;
        dw_rows_kernel<<<(unsigned)((R + 255) / 256), 256, 0, s>>>(a.kept_off, c_off, E, R,
                                                                   at<float>(bw, L.dw_part),
                                                                   tb_dh_tiles((int)F), dw_row);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else {
        cudaMemsetAsync(a.dWg, 0, sizeof(float) * (size_t)(E * F * d), s);
        cudaMemsetAsync(a.dWu, 0, sizeof(float) * (size_t)(E * F * d), s);
        cudaMemsetAsync(a.dWd, 0, sizeof(float) * (size_t)(E * F * d), s);
    }
    if (S > 0 && N > 0) {
        TbParams base{};
        base.G = (int)S;
        base.rows = s_rows;
        base.a_off = s_zero;
        base.c_off = s_coff;
        base.dense_off = s_dense;
        base.max_mtiles = S * Np / 128;
        base.err = a.err;
        if ((e = expert_bwd(base, s_zero, Np, S * Np, (int)d, (int)Fs, dout_s, x_s, a.Wsg, a.Wsu,
                            a.Wsd, a.h_sh, nullptr, at<__nv_bfloat16>(bw, L.dh_s),
                            at<float>(bw, L.dw_part_s), at<__nv_bfloat16>(bw, L.dgu_s),
                            at<__nv_bfloat16>(bw, L.hw_s), at<float>(bw, L.dX_s), a.dWsg, a.dWsu,
                            a.dWsd, s)) != cudaSuccess)
            return e;
    }
    // 5. router backward
    float* dl = at<float>(bw, L.dl);
    const float aux_scale =
        N > 0 ? (float)(a.aux_coef * (double)E / ((double)N * (double)k * (double)N)) : 0.f;
    const float z_scale = N > 0 ? (float)(2.0 * a.z_coef / (double)N) : 0.f;
    if (N > 0) {
        const unsigned blocks = (unsigned)((N * 32 + 255) / 256);
        switch (router_nv(E)) {
            case 1: router_bwd_kernel<1><<<blocks, 256, 0, s>>>(N, E, k, c.renorm, probs, a.idx, a.w, a.pos, dw_row, a.counts, a.lse, aux_scale, z_scale, dl); break;
            case 2: router_bwd_kernel<2><<<blocks, 256, 0, s>>>(N, E, k, c.renorm, probs, a.idx, a.w, a.pos, dw_row, a.counts, a.lse, aux_scale, z_scale, dl); break;
            case 4: router_bwd_kernel<4><<<blocks, 256, 0, s>>>(N, E, k, c.renorm, probs, a.idx, a.w, a.pos, dw_row, a.counts, a.lse, aux_scale, z_scale, dl); break;
            case 8: router_bwd_kernel<8><<<blocks, 256, 0, s>>>(N, E, k, c.renorm, probs, a.idx, a.w, a.pos, dw_row, a.counts, a.lse, aux_scale, z_scale, dl); break;
            case 16: router_bwd_kernel<16><<<blocks, 256, 0, s>>>(N, E, k, c.renorm, probs, a.idx, a.w, a.pos, dw_row, a.counts, a.lse, aux_scale, z_scale, dl); break;
            default: router_bwd_kernel<32><<<blocks, 256, 0, s>>>(N, E, k, c.renorm, probs, a.idx, a.w, a.pos, dw_row, a.counts, a.lse, aux_scale, z_scale, dl); break;
        }
    }
    if (a.db) {
        if (c.bias_mode == 1 && N > 0) {
            db_part_kernel<<<kDbChunks, 256, 0, s>>>(dl, N, E, at<double>(bw, L.db_part));
            db_final_kernel<<<(E + 255) / 256, 256, 0, s>>>(at<double>(bw, L.db_part), E, a.db);
        } else {
            cudaMemsetAsync(a.db, 0, sizeof(float) * (size_t)E, s);
        }
    }
    // 6. router GEMMs on the tensor cores (bf16 pieces of the fp32 operands)
    float* dx_r = at<float>(bw, L.dx_r);
    if (N > 0) {
        __nv_bfloat16* dl3 = at<__nv_bfloat16>(bw, L.dl3);
        __nv_bfloat16* dlT2 = at<__nv_bfloat16>(bw, L.dlT2);
        __nv_bfloat16* w3 = at<__nv_bfloat16>(bw, L.w3);
        __nv_bfloat16* x2 = at<__nv_bfloat16>(bw, L.x2);
        int32_t* rp = at<int32_t>(bw, L.r_plan);   // [0..3] dx_r group, [4..7] dW_r group
        const int K3 = pad8(3 * E), Ep = pad8(E);
        if (K3 != 3 * E) cudaMemsetAsync(dl3, 0, 2 * (size_t)(N * K3), s);
        if (Ep != E) cudaMemsetAsync(dlT2, 0, 2 * (size_t)(2 * N * Ep), s);
        if (K3 != 3 * E) cudaMemsetAsync(w3 + (size_t)3 * E * d, 0, 2 * (size_t)(K3 - 3 * E) * d, s);
        split_dl_kernel<<<(unsigned)((N * E + 255) / 256), 256, 0, s>>>(dl, N, E, dl3, dlT2);
        split_wr_kernel<<<(unsigned)(((int64_t)E * d + 255) / 256), 256, 0, s>>>(a.W_r, E, (int)d, w3);
        const int64_t n16 = N * d / 8;
        dup_rows_kernel<<<(unsigned)((n16 + 255) / 256), 256, 0, s>>>(
            reinterpret_cast<const uint4*>(a.x), n16, reinterpret_cast<uint4*>(x2));
        const int64_t Npad = (N + 127) / 128 * 128;
        plan_single_kernel<<<1, 32, 0, s>>>(N, Npad, rp);
        plan_single_kernel<<<1, 32, 0, s>>>(2 * N, 2 * N, rp + 4);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        TbParams p{};
        p.G = 1;
        p.rows = rp;
        p.a_off = rp + 1;
        p.c_off = rp + 1;
        p.dense_off = rp + 3;
        p.max_mtiles = Npad / 128;
        p.err = a.err;
        p.out_f32 = dx_r;
        if ((e = tb_rows_f32(p, dl3, N, K3, w3, (int)d, s)) != cudaSuccess) return e;
        TbParams q{};
        q.G = 1;
        q.rows = rp + 4;
        q.a_off = rp + 5;
        q.c_off = rp + 5;
        q.dense_off = rp + 7;
        q.split_m = E;
        q.out_f32 = a.dW_r;
        q.out_f32b = a.dW_r;
        q.err = a.err;
        if ((e = tb_wgrad(q, dlT2, 2 * N, E, x2, 2 * N, (int)d, s, Ep)) != cudaSuccess) return e;
        // 7. dx
        dx_combine_kernel<<<(unsigned)((N * 32 + 255) / 256), 256, 0, s>>>(
            N, k, (int)d, (int)S, Np, a.idx, a.pos, a.kept_off, c_off, at<float>(bw, L.dX),
            at<float>(bw, L.dX_s), dx_r, a.dx);
    } else {
        cudaMemsetAsync(a.dW_r, 0, sizeof(float) * (size_t)(E * d), s);
    }
    return cudaGetLastError();
}

}  // namespace moe
