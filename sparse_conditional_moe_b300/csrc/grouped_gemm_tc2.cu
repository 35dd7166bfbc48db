// grouped_gemm_tc2.cu -- the grouped expert GEMMs of grouped_gemm_tc.cu on CTA pairs
// (tcgen05.mma.cta_group::2): one MMA covers 256 rows x 256 columns over the two SMs of a pair.
//
// Same operation as grouped_gemm_tc.cu (page "混合专家 MoE", section "实现：逐 token 与按专家分组":
// after grouping, a single grouped GEMM serves all experts; Expert.forward is
// down(silu(gate(x)) * up(x))).  What changes is the feed: each CTA of a pair stages its own 128
// rows of A and half of the 256 B rows (gate rows in the even CTA and the matching up rows in the
// odd CTA for gate/up; the two 128-row halves of the W_down tile for down), so every SM pulls
// 32 KB per 64-wide k-block instead of 48 KB for the same tensor work, and the shared-memory
// ring gets 6 stages instead of 4.  The even CTA of the pair issues the MMAs; both CTAs' TMA
// loads complete on its barrier; its commits free the ring slots and announce finished
// accumulators in both CTAs; each CTA's epilogue reads its own 128 TMEM lanes.
// A pair always works on two consecutive 128-row m-tiles of one group, so a group with an odd
// number of m-tiles leaves the odd CTA's rows of its last pair masked: the host uses this kernel
// only when groups are large (see moe_api.cu).
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;            // rows per CTA (256 per pair)
constexpr int BK = 64;
constexpr int BN = 256;            // MMA N
constexpr int STAGES = 6;
constexpr int A_STAGE = BM * BK * 2;        // 16 KB
constexpr int B_STAGE = (BN / 2) * BK * 2;  // 16 KB: this CTA's half of B
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

enum { EPI_SWIGLU = 0, EPI_SCALE = 1 };

struct Tc2Params {
    int G;
    const int32_t* rows;
    const int32_t* row_off;
    const int32_t* mpair_off;   // [G+1] prefix of 256-row m-pairs (non-uniform groups)
    int uniform_rows;
    int64_t a_stride, c_stride;
    int K, n_out, b_rows, n_tiles;
    __nv_bfloat16* C;
    int64_t ldc;
    const float* row_scale;
    int32_t* err;
};

struct PairTile {
    int g, mp, nt, rows;
    int64_t a_row0, c_row0;
};

__device__ __forceinline__ int total_pair_tiles(const Tc2Params& p) {
    if (p.rows == nullptr) return p.G * ((p.uniform_rows + 2 * BM - 1) / (2 * BM)) * p.n_tiles;
    return p.mpair_off[p.G] * p.n_tiles;
}

__device__ __forceinline__ PairTile decode_pair(const Tc2Params& p, int tile) {
    PairTile t;
    if (p.rows == nullptr) {
        const int mpg = (p.uniform_rows + 2 * BM - 1) / (2 * BM);
        const int per = mpg * p.n_tiles;
        t.g = tile / per;
        const int local = tile - t.g * per;
        raster_tile(local, mpg, p.n_tiles, t.mp, t.nt);
        t.rows = p.uniform_rows;
        t.a_row0 = (int64_t)t.g * p.a_stride;
        t.c_row0 = (int64_t)t.g * p.c_stride;
    } else {
        int lo = 0, hi = p.G;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.mpair_off[mid] * p.n_tiles <= tile) lo = mid;
            else hi = mid;
        }
        t.g = lo;
        const int m0 = p.mpair_off[lo];
        const int mpg = p.mpair_off[lo + 1] - m0;
        const int local = tile - m0 * p.n_tiles;
        raster_tile(local, mpg, p.n_tiles, t.mp, t.nt);
        t.rows = p.rows[lo];
        t.a_row0 = t.c_row0 = p.row_off[lo];
    }
    return t;
}

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
tc2_grouped_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const Tc2Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* full = bars;                 // [STAGES] leader: both CTAs' loads landed
    uint64_t* empty = bars + STAGES;       // [STAGES] both: the pair's MMAs released the slot
    uint64_t* tfull = bars + 2 * STAGES;   // [2] both: accumulator ready
    uint64_t* tempty = tfull + 2;          // [2] leader: both epilogues drained the accumulator
    uint64_t* drain = tempty + 2;          // [1] leader: MMA drain on exit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);     // 4 epilogue warps x 2 CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB0);
        if (EPI == EPI_SWIGLU) prefetch_tmap(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();     // the peer's barriers exist before anything is sent to them
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    const int ntiles = total_pair_tiles(p);
    const int nk = (p.K + BK - 1) / BK;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------- TMA producer (both CTAs)
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            const CUtensorMap* mb = (EPI == EPI_SWIGLU && !leader) ? &tmB1 : &tmB0;
            for (int tile = cluster; tile < ntiles && ok; tile += nclusters) {
                const PairTile t = decode_pair(p, tile);
                const int a_y = (int)(t.a_row0 + (int64_t)t.mp * 2 * BM + rank * BM);
                const int b_y = (EPI == EPI_SWIGLU) ? t.g * p.b_rows + t.nt * (BN / 2)
                                                    : t.g * p.b_rows + t.nt * BN + (int)rank * (BN / 2);
                for (int kb = 0; kb < nk; kb++) {
                    if (!wait1(&empty[s], ph ^ 1u, abort_flag, kWaitTimeoutNs, true)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(&full[s], 2 * STAGE_BYTES);
                    const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
                    const int kx = kb * BK;
                    tma_load_2d_pair(smem_u32(sA + s * A_STAGE), &tmA, fb, kx, a_y);
                    tma_load_2d_pair(smem_u32(sB + s * B_STAGE), mb, fb, kx, b_y);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {   // let copies in flight land before the pair can exit
                const uint64_t t0 = gtimer();
                while (gtimer() - t0 < 200000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------------------------------------- MMA issuer (leader CTA only)
            constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int it = 0;
            for (int tile = cluster; tile < ntiles && ok; tile += nclusters, ++it) {
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                if (!wait1(&tempty[acc], aph ^ 1u, abort_flag, kWaitTimeoutNs, true)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < nk; kb++) {
                    if (!wait1(&full[s], ph, abort_flag, kWaitTimeoutNs, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + s * A_STAGE);
                    const uint32_t b0 = smem_u32(sB + s * B_STAGE);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; kk++)
                        umma_bf16_pair(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32),
                                       idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    umma_commit_pair(&empty[s], 0x3);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) umma_commit_pair(&tfull[acc], 0x3);
            }
            umma_commit_pair(drain, 0x1);
            wait1(drain, 0, abort_flag, kDrainTimeoutNs, false);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------- epilogue (warps 2..5, both CTAs)
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
        const uint32_t tempty1 = mapa_shared(smem_u32(&tempty[1]), 0);
        int it = 0;
        for (int tile = cluster; tile < ntiles; tile += nclusters, ++it) {
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            if (!waitw(&tfull[acc], aph, abort_flag)) break;
            tc_fence_after();
            const PairTile t = decode_pair(p, tile);
            const int r = t.mp * 2 * BM + (int)rank * BM + row_in_tile;
            const bool valid = r < t.rows;
            const int64_t crow = t.c_row0 + r;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if (EPI == EPI_SWIGLU) {
                const int col0 = t.nt * (BN / 2);
#pragma unroll 1
                for (int c = 0; c < (BN / 2) / 32; c++) {
                    uint32_t g[32], u[32];
                    tmem_ld32(taddr + c * 32, g);
                    tmem_ld32(taddr + BN / 2 + c * 32, u);
                    tmem_ld_wait();
                    if (valid) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; j++) {
                            const float h0 = silu(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
                            const float h1 =
                                silu(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
                            pk[j] = pack_bf16(h0, h1);
                        }
                        const int col = col0 + c * 32;
                        __nv_bfloat16* dst = p.C + crow * p.ldc + col;
#pragma unroll
                        for (int v = 0; v < 4; v++)
                            if (col + v * 8 + 8 <= p.n_out)
                                *reinterpret_cast<uint4*>(dst + v * 8) =
                                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
            } else {
                const int col0 = t.nt * BN;
                const float sc = (valid && p.row_scale) ? p.row_scale[crow] : 1.f;
#pragma unroll 1
                for (int c = 0; c < BN / 32; c++) {
                    uint32_t a[32];
                    tmem_ld32(taddr + c * 32, a);
                    tmem_ld_wait();
                    if (valid) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; j++)
                            pk[j] = pack_bf16(__uint_as_float(a[2 * j]) * sc,
                                              __uint_as_float(a[2 * j + 1]) * sc);
                        const int col = col0 + c * 32;
                        __nv_bfloat16* dst = p.C + crow * p.ldc + col;
#pragma unroll
                        for (int v = 0; v < 4; v++)
                            if (col + v * 8 + 8 <= p.n_out)
                                *reinterpret_cast<uint4*>(dst + v * 8) =
                                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc ? tempty1 : tempty0);
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();     // neither CTA leaves while the other may still signal it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag && p.err) atomicOr(p.err, MOE_DEVERR_TIMEOUT);
}

Tc2Params base_params(const GroupGeom& g) {
    Tc2Params p{};
    p.G = g.G;
    p.rows = g.rows;
    p.row_off = g.row_off;
    p.mpair_off = g.mtile_off;
    p.uniform_rows = g.uniform_rows;
    p.a_stride = g.a_stride;
    p.c_stride = g.c_stride;
    return p;
}

int grid_for(const GroupGeom& g, int n_tiles) {
    int64_t max_tiles;
    if (g.rows == nullptr)
        max_tiles = (int64_t)g.G * ((g.uniform_rows + 2 * BM - 1) / (2 * BM)) * n_tiles;
    else
        max_tiles = ((g.max_rows + 2 * BM - 1) / (2 * BM) + g.G) * (int64_t)n_tiles;
    const int64_t pairs = device_sm_count() / 2;
    const int64_t use = max_tiles < pairs ? (max_tiles < 1 ? 1 : max_tiles) : pairs;
    return (int)(2 * use);
}

template <int EPI>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                   const Tc2Params& p, int grid, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(tc2_grouped_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    tc2_grouped_kernel<EPI><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(a, b0, b1, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t tc2_gateup(const GroupGeom& g, const __nv_bfloat16* A, int64_t a_rows, int K,
                       const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int F,
                       __nv_bfloat16* H, int32_t* err, cudaStream_t s) {
    if (g.G <= 0 || a_rows <= 0) return cudaSuccess;
    CUtensorMap ma, mg, mu;
    if (!make_map(&ma, A, a_rows, K, BM) || !make_map(&mg, Wg, (int64_t)g.G * F, K, BN / 2) ||
        !make_map(&mu, Wu, (int64_t)g.G * F, K, BN / 2))
        return cudaErrorInvalidValue;
    Tc2Params p = base_params(g);
    p.K = K;
    p.n_out = F;
    p.b_rows = F;
    p.n_tiles = (F + BN / 2 - 1) / (BN / 2);
    p.C = H;
    p.ldc = F;
    p.row_scale = nullptr;
    p.err = err;
    return launch<EPI_SWIGLU>(ma, mg, mu, p, grid_for(g, p.n_tiles), s);
}

cudaError_t tc2_down(const GroupGeom& g, const __nv_bfloat16* H, int64_t h_rows, int F,
                     const __nv_bfloat16* Wd, int D, const float* row_scale, __nv_bfloat16* Y,
                     int32_t* err, cudaStream_t s) {
    if (g.G <= 0 || h_rows <= 0) return cudaSuccess;
    CUtensorMap ma, mb;
    if (!make_map(&ma, H, h_rows, F, BM) || !make_map(&mb, Wd, (int64_t)g.G * D, F, BN / 2))
        return cudaErrorInvalidValue;
    Tc2Params p = base_params(g);
    p.K = F;
    p.n_out = D;
    p.b_rows = D;
    p.n_tiles = (D + BN - 1) / BN;
    p.C = Y;
    p.ldc = D;
    p.row_scale = row_scale;
    p.err = err;
    return launch<EPI_SCALE>(ma, mb, mb, p, grid_for(g, p.n_tiles), s);
}

}  // namespace moe
