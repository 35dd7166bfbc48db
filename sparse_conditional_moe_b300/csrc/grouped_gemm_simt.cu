// grouped_gemm_simt.cu -- fp32 grouped GEMMs of the expert FFNs on the CUDA cores, for layers
// whose activations and weights are fp32 (the tensor cores have no fp32-exact mode).
//
// Same operation and tile scheduling as the tcgen05 kernels (page "混合专家 MoE", section
// "实现：逐 token 与按专家分组": every expert multiplies all of its grouped rows at once):
//   gate/up : C[r, n] = silu(A_r . Wg[g,n]) * (A_r . Wu[g,n])
//   down    : C[r, n] = row_scale[r] * (A_r . Wd[g,n])
// 64 x 64 output tiles, 256 threads with 4 x 4 register tiles, k-slices of 16 in shared memory,
// a grid-stride loop over the same group-major tile list.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int SBM = 64, SBN = 64, SBK = 16, STHREADS = 256;

struct SimtTile {
    int g, mt, nt, rows;
    int64_t a_row0, c_row0;
};

__device__ __forceinline__ int simt_total(const GroupGeom& p, int n_tiles) {
    if (p.rows == nullptr) return p.G * ((p.uniform_rows + SBM - 1) / SBM) * n_tiles;
    return p.mtile_off[p.G] * n_tiles;
}

__device__ __forceinline__ SimtTile simt_decode(const GroupGeom& p, int n_tiles, int tile) {
    SimtTile t;
    if (p.rows == nullptr) {
        const int mtg = (p.uniform_rows + SBM - 1) / SBM;
        const int per = mtg * n_tiles;
        t.g = tile / per;
        const int local = tile - t.g * per;
        t.mt = local % mtg;
        t.nt = local / mtg;
        t.rows = p.uniform_rows;
        t.a_row0 = (int64_t)t.g * p.a_stride;
        t.c_row0 = (int64_t)t.g * p.c_stride;
    } else {
        int lo = 0, hi = p.G;
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (p.mtile_off[mid] * n_tiles <= tile) lo = mid;
            else hi = mid;
        }
        t.g = lo;
        const int mt0 = p.mtile_off[lo];
        const int mtg = p.mtile_off[lo + 1] - mt0;
        const int local = tile - mt0 * n_tiles;
        t.mt = local % mtg;
        t.nt = local / mtg;
        t.rows = p.rows[lo];
        t.a_row0 = t.c_row0 = p.row_off[lo];
    }
    return t;
}

// SWIGLU: two B matrices (gate, up) -> silu(g) * u ; otherwise one B, scaled by row_scale.
template <bool SWIGLU>
__global__ void __launch_bounds__(STHREADS)
simt_grouped_kernel(const GroupGeom p, const float* __restrict__ A, int K,
                    const float* __restrict__ B0, const float* __restrict__ B1, int b_rows,
                    int n_out, const float* __restrict__ row_scale, float* __restrict__ C) {
    __shared__ float As[SBK][SBM + 4];
    __shared__ float Bs0[SBK][SBN + 4];
    __shared__ float Bs1[SWIGLU ? SBK : 1][SWIGLU ? SBN + 4 : 1];
    const int n_tiles = (n_out + SBN - 1) / SBN;
    const int ntot = simt_total(p, n_tiles);
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    for (int tile = blockIdx.x; tile < ntot; tile += gridDim.x) {
        const SimtTile t = simt_decode(p, n_tiles, tile);
        const int m0 = t.mt * SBM, n0 = t.nt * SBN;
        float acc0[4][4] = {}, acc1[4][4] = {};
        for (int k0 = 0; k0 < K; k0 += SBK) {
            for (int v = threadIdx.x; v < SBM * SBK; v += STHREADS) {
                const int r = v / SBK, kk = v % SBK;
                float a = 0.f;
                if (m0 + r < t.rows && k0 + kk < K) a = A[(t.a_row0 + m0 + r) * K + k0 + kk];
                As[kk][r] = a;
                float b0 = 0.f, b1 = 0.f;
                if (n0 + r < n_out && k0 + kk < K) {
                    const int64_t bi = ((int64_t)t.g * b_rows + n0 + r) * K + k0 + kk;
                    b0 = B0[bi];
                    if (SWIGLU) b1 = B1[bi];
                }
                Bs0[kk][r] = b0;
                if (SWIGLU) Bs1[kk][r] = b1;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < SBK; kk++) {
                float a[4], b0[4], b1[4];
#pragma unroll
                for (int i = 0; i < 4; i++) a[i] = As[kk][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    b0[j] = Bs0[kk][tx + 16 * j];
                    if (SWIGLU) b1[j] = Bs1[kk][tx + 16 * j];
                }
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        acc0[i][j] = fmaf(a[i], b0[j], acc0[i][j]);
                        if (SWIGLU) acc1[i][j] = fmaf(a[i], b1[j], acc1[i][j]);
                    }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int r = m0 + ty + 16 * i;
            if (r >= t.rows) continue;
            const int64_t crow = t.c_row0 + r;
            const float sc = (!SWIGLU && row_scale) ? row_scale[crow] : 1.f;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int n = n0 + tx + 16 * j;
                if (n >= n_out) continue;
                float v;
                if (SWIGLU) {
                    const float g = acc0[i][j];
                    v = g / (1.f + expf(-g)) * acc1[i][j];
                } else {
                    v = acc0[i][j] * sc;
                }
                C[crow * n_out + n] = v;
            }
        }
    }
}

int simt_grid(const GroupGeom& g, int n_out) {
    const int n_tiles = (n_out + SBN - 1) / SBN;
    int64_t max_tiles;
    if (g.rows == nullptr)
        max_tiles = (int64_t)g.G * ((g.uniform_rows + SBM - 1) / SBM) * n_tiles;
    else
        max_tiles = ((g.max_rows + SBM - 1) / SBM + g.G) * (int64_t)n_tiles;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (max_tiles < 1) max_tiles = 1;
    return (int)(max_tiles < cap ? max_tiles : cap);
}

}  // namespace

int simt_block_rows() { return SBM; }

cudaError_t simt_gateup_f32(const GroupGeom& g, const float* A, int K, const float* Wg,
                            const float* Wu, int F, float* H, cudaStream_t s) {
    if (g.G <= 0) return cudaSuccess;
    simt_grouped_kernel<true><<<simt_grid(g, F), STHREADS, 0, s>>>(g, A, K, Wg, Wu, F, F, nullptr, H);
    return cudaGetLastError();
}

cudaError_t simt_down_f32(const GroupGeom& g, const float* H, int F, const float* Wd, int D,
                          const float* row_scale, float* Y, cudaStream_t s) {
    if (g.G <= 0) return cudaSuccess;
    simt_grouped_kernel<false><<<simt_grid(g, D), STHREADS, 0, s>>>(g, H, F, Wd, nullptr, D, D,
                                                                    row_scale, Y);
    return cudaGetLastError();
}

}  // namespace moe
