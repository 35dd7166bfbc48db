// grouped_gemm_tc.cu -- grouped bf16 GEMMs of the expert FFNs on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// Page "混合专家 MoE", section "实现：逐 token 与按专家分组": after grouping, every expert
// multiplies all of its tokens at once and a single grouped GEMM serves all experts;
// Expert.forward is down(silu(gate(x)) * up(x)).  Two kernels:
//   gate/up : per group g, C[r, n] = silu(A_r . Wg[g,n]) * (A_r . Wu[g,n])   (bf16 out)
//   down    : per group g, C[r, n] = row_scale[r] * (A_r . Wd[g,n])          (bf16 out)
// A group owns a contiguous row range of A and C (its kept tokens in grouped order, or all
// tokens for a shared expert); empty groups own no tile.
//
// Design (one CTA per SM, persistent, warp-specialised, 192 threads):
//   warp 0      TMA producer (the warp runs the loop, an elected lane issues): A tile 128x64
//               and B tile 256x64 (bf16, 128-byte swizzle) per k-block into a 4-stage
//               shared-memory ring (48 KB per stage);
//   warp 1      allocates 512 TMEM columns; the warp runs the loop and an elected lane issues
//               tcgen05.mma (M=128, N=256, K=16, fp32 accumulate) and frees ring slots with
//               tcgen05.commit;
//   warps 2..5  epilogue: tcgen05.ld of the 128x256 fp32 accumulator (each warp its 32-lane
//               quarter), silu*mul or scale in fp32, one rounding to bf16, 16-byte stores.
// Two accumulators (2 x 256 columns) let the epilogue of tile i overlap the mainloop of i+1.
// For gate/up the B tile stacks 128 gate rows over the 128 matching up rows, so one MMA
// yields both projections of 128 hidden units side by side in TMEM.
// Tiles are ordered group-major, then n-tile, with the m-tiles of a group innermost, so the
// CTAs working at the same time share a weight tile through L2.
// The last m-tile of a group is usually ragged (a group of 257 rows needs a third tile for one
// row).  When it holds at most kSwapMaxRows rows it is computed transposed: the same shared
// memory stages feed two MMAs with the weight rows as M = 128 and the tile's rows, rounded up to
// 16, as N, and the epilogue writes the transposed accumulator (lane = output column).
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA raises an abort flag, the
// other roles stop at their next wait, in-flight copies and MMAs are drained with bounded
// waits, TMEM is freed and the device error word gets MOE_DEVERR_TIMEOUT.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BK = 64, BN = 256, STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;      // 16 KB: 128 rows of A
constexpr int B_STAGE = BN * BK * 2;      // 32 KB: 256 rows of B
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int NUM_THREADS = 192;
constexpr int STAGING_BYTES = 4 * 2 * 2048;   // epilogue: 4 warps x 2 buffers x 32x32 bf16
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*alignment*/ + 256 /*barriers*/;

enum { EPI_SWIGLU = 0, EPI_SCALE = 1 };

struct TcParams {
    int G;
    const int32_t* rows;
    const int32_t* row_off;
    const int32_t* mtile_off;
    int uniform_rows;
    int64_t a_stride, c_stride;
    int K;               // reduction length
    int n_out;           // valid output columns per group
    int b_rows;          // rows of B per group in its 2-D map (F for gate/up, d for down)
    int n_tiles;         // output column tiles per group
    __nv_bfloat16* C;
    int64_t ldc;
    const float* row_scale;
    int32_t* err;
};

// ---------------------------------------------------------------- tile scheduling

// The last m-tile of a group is usually ragged (a group of 257 rows needs a third tile for one
// row).  When it holds at most kSwapMaxRows rows it is computed with the operands swapped: the
// weight rows are the MMA's M = 128 side (two MMAs: gate and up, or the two 128-row halves of
// the down tile) and the tile's rows are its N side, rounded up to 16, so the MMA work shrinks
// with the rows present.
constexpr int kSwapMaxRows = 96;

struct TileInfo {
    int g, mt, nt, rows;
    int64_t a_row0, c_row0;
    int tr;       // valid rows of this m-tile (1..BM)
    bool swap;    // computed with the operands swapped (tr <= kSwapMaxRows)
};

__device__ __forceinline__ int total_tiles(const TcParams& p) {
    if (p.rows == nullptr) return p.G * ((p.uniform_rows + BM - 1) / BM) * p.n_tiles;
    return p.mtile_off[p.G] * p.n_tiles;
}

__device__ __forceinline__ TileInfo decode_tile(const TcParams& p, int tile) {
    TileInfo t;
    if (p.rows == nullptr) {
        const int mtg = (p.uniform_rows + BM - 1) / BM;
        const int per = mtg * p.n_tiles;
        t.g = tile / per;
        const int local = tile - t.g * per;
        raster_tile(local, mtg, p.n_tiles, t.mt, t.nt);
        t.rows = p.uniform_rows;
        t.a_row0 = (int64_t)t.g * p.a_stride;
        t.c_row0 = (int64_t)t.g * p.c_stride;
    } else {
        // largest g with mtile_off[g] * n_tiles <= tile (that group is non-empty)
        int lo = 0, hi = p.G;
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (p.mtile_off[mid] * p.n_tiles <= tile) lo = mid;
            else hi = mid;
        }
        t.g = lo;
        const int mt0 = p.mtile_off[lo];
        const int mtg = p.mtile_off[lo + 1] - mt0;
        const int local = tile - mt0 * p.n_tiles;
        raster_tile(local, mtg, p.n_tiles, t.mt, t.nt);
        t.rows = p.rows[lo];
        t.a_row0 = t.c_row0 = p.row_off[lo];
    }
    const int left = t.rows - t.mt * BM;
    t.tr = left < BM ? left : BM;
    t.swap = t.tr <= kSwapMaxRows;
    return t;
}

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------- epilogues (one warp each)

// Accumulator of rows in TMEM lanes: rows [row0 + q*32, +32) of the part, all 256 columns.
template <int EPI>
__device__ __forceinline__ void epi_rows(const TcParams& p, const CUtensorMap* tmC, uint32_t taddr,
                                         uint32_t stage0, int& nchunk, int q, int nt, int64_t row0,
                                         int nrows) {
    const int lane = threadIdx.x & 31;
    const int r = q * 32 + lane;
    const bool valid = r < nrows;
    const bool all_valid = q * 32 + 31 < nrows;   // warp-uniform
    const int64_t crow = row0 + r;
    const int32_t gy = (int32_t)(row0 + q * 32);
    if (EPI == EPI_SWIGLU) {
        const int col0 = nt * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < (BN / 2) / 32; c++, nchunk++) {
            uint32_t g[32], u[32];
            tmem_ld32(taddr + c * 32, g);
            tmem_ld32(taddr + BN / 2 + c * 32, u);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const float h0 = silu(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
                const float h1 = silu(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
                pk[j] = pack_bf16(h0, h1);
            }
            const int col = col0 + c * 32;
            store_chunk32(tmC, stage0 + (uint32_t)(nchunk & 1) * 2048u, pk, all_valid, valid,
                          p.C + crow * p.ldc + col, col, p.n_out, gy);
        }
    } else {
        const int col0 = nt * BN;
        const float sc = (valid && p.row_scale) ? p.row_scale[crow] : 1.f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; c++, nchunk++) {
            uint32_t a[32];
            tmem_ld32(taddr + c * 32, a);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; j++)
                pk[j] = pack_bf16(__uint_as_float(a[2 * j]) * sc, __uint_as_float(a[2 * j + 1]) * sc);
            const int col = col0 + c * 32;
            store_chunk32(tmC, stage0 + (uint32_t)(nchunk & 1) * 2048u, pk, all_valid, valid,
                          p.C + crow * p.ldc + col, col, p.n_out, gy);
        }
    }
}

// Swapped accumulator: TMEM lane = output column (this warp: 32 of them), TMEM column = row;
// columns [0, n16) hold the first 128 weight rows, [128, 128 + n16) the second 128.
template <int EPI>
__device__ __forceinline__ void epi_swapped(const TcParams& p, const CUtensorMap* tmC,
                                            uint32_t taddr, uint32_t stage0, int& nchunk, int q,
                                            int nt, int64_t row0, int nrows) {
    const int lane = threadIdx.x & 31;
    const int nch = (nrows + 31) >> 5;
    if (EPI == EPI_SWIGLU) {
        const int col = nt * (BN / 2) + q * 32;
        const bool col_ok = col + lane < p.n_out;
#pragma unroll 1
        for (int c = 0; c < nch; c++, nchunk++) {
            uint32_t g[32], u[32];
            tmem_ld32(taddr + c * 32, g);
            tmem_ld32(taddr + BN / 2 + c * 32, u);
            tmem_ld_wait();
            float h[32];
#pragma unroll
            for (int j = 0; j < 32; j++) h[j] = silu(__uint_as_float(g[j])) * __uint_as_float(u[j]);
            const int64_t gr = row0 + c * 32;
            store_chunk32_t(tmC, stage0 + (uint32_t)(nchunk & 1) * 2048u, h, nrows - c * 32,
                            p.C + gr * p.ldc + col + lane, p.ldc, col_ok, col, (int32_t)gr);
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < nch; c++) {
            const int64_t gr = row0 + c * 32;
            const float s_lane = (p.row_scale && c * 32 + lane < nrows) ? p.row_scale[gr + lane] : 1.f;
#pragma unroll 1
            for (int hh = 0; hh < 2; hh++, nchunk++) {
                uint32_t a[32];
                tmem_ld32(taddr + hh * (BN / 2) + c * 32, a);
                tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; j++)
                    v[j] = __uint_as_float(a[j]) * __shfl_sync(0xffffffffu, s_lane, j);
                const int col = nt * BN + hh * (BN / 2) + q * 32;
                store_chunk32_t(tmC, stage0 + (uint32_t)(nchunk & 1) * 2048u, v, nrows - c * 32,
                                p.C + gr * p.ldc + col + lane, p.ldc, col + lane < p.n_out, col,
                                (int32_t)gr);
            }
        }
    }
}

// ---------------------------------------------------------------- the kernel

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_grouped_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                  const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmC,
                  const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sA = smem;                          // [STAGES] x 16 KB
    uint8_t* sB = smem + STAGES * A_STAGE;       // [STAGES] x 32 KB
    uint8_t* sStage = smem + STAGES * STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + STAGING_BYTES);
    uint64_t* full = bars;                 // [STAGES]  TMA -> MMA
    uint64_t* empty = bars + STAGES;       // [STAGES]  MMA -> TMA
    uint64_t* tfull = bars + 2 * STAGES;   // [2]       MMA -> epilogue
    uint64_t* tempty = tfull + 2;          // [2]       epilogue -> MMA
    uint64_t* drain = tempty + 2;          // [1]       MMA drain on exit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB0);
        if (EPI == EPI_SWIGLU) prefetch_tmap(&tmB1);
        prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    const int ntiles = total_tiles(p);
    const int nk = (p.K + BK - 1) / BK;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer: the whole warp runs
        // the loop and the waits, one elected lane issues the copies
        int s = 0;
        uint32_t ph = 0;
        int last_ph[STAGES];
        for (int i = 0; i < STAGES; i++) last_ph[i] = -1;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const TileInfo t = decode_tile(p, tile);
            const int a_y = (int)(t.a_row0 + (int64_t)t.mt * BM);
            const int b_y = t.g * p.b_rows + t.nt * (EPI == EPI_SWIGLU ? BN / 2 : BN);
            for (int kb = 0; kb < nk; kb++) {
                if (!waitw(&empty[s], ph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                    const int kx = kb * BK;
                    tma_load_2d(smem_u32(sA + s * A_STAGE), &tmA, &full[s], kx, a_y);
                    if (EPI == EPI_SWIGLU) {
                        tma_load_2d(smem_u32(sB + s * B_STAGE), &tmB0, &full[s], kx, b_y);
                        tma_load_2d(smem_u32(sB + s * B_STAGE + B_STAGE / 2), &tmB1, &full[s], kx,
                                    b_y);
                    } else {
                        tma_load_2d(smem_u32(sB + s * B_STAGE), &tmB0, &full[s], kx, b_y);
                    }
                }
                __syncwarp();
                last_ph[s] = (int)ph;
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            // let every copy already issued land before the CTA can exit
            for (int i = 0; i < STAGES; i++)
                if (last_ph[i] >= 0)
                    wait1(&full[i], (uint32_t)last_ph[i], abort_flag, kDrainTimeoutNs, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer: the whole warp runs the
        // loop and the waits, one elected lane issues the MMAs and commits (one thread issuing
        // between mbarrier waits spends ~100-115 cycles per MMA); one k-loop per tile kind,
        // descriptors advanced by addition (+2 = 32 bytes = K 16 within a stage, the stage size
        // between stages)
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
        const uint64_t ad0 = sw128_desc(smem_u32(sA)), bd0 = sw128_desc(smem_u32(sB));
        uint64_t ad = ad0, bd = bd0;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        int it = 0;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            if (!waitw(&tempty[acc], aph ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            const TileInfo t = decode_tile(p, tile);
            // swapped: D0 = W[0:128) . A^T and D1 = W[128:256) . A^T, each 128 x n16
            const uint32_t idesc_sw = idesc_bf16_f32(BM, (t.tr + 15) & ~15);
            for (int kb = 0; kb < nk; kb++) {
                if (!waitw(&full[s], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    if (!t.swap) {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; kk++)
                            umma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc,
                                      (kb > 0 || kk > 0) ? 1u : 0u);
                    } else {
                        const uint64_t bd_hi = bd + (uint64_t)((B_STAGE / 2) >> 4);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; kk++) {
                            const uint32_t acc_in = (kb > 0 || kk > 0) ? 1u : 0u;
                            umma_bf16(d_tmem, bd + 2 * kk, ad + 2 * kk, idesc_sw, acc_in);
                            umma_bf16(d_tmem + BN / 2, bd_hi + 2 * kk, ad + 2 * kk, idesc_sw, acc_in);
                        }
                    }
                    umma_commit(&empty[s]);
                }
                __syncwarp();
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                    ad = ad0;
                    bd = bd0;
                } else {
                    ad += (uint64_t)(A_STAGE >> 4);
                    bd += (uint64_t)(B_STAGE >> 4);
                }
            }
            if (ok && elect_one()) umma_commit(&tfull[acc]);
            __syncwarp();
        }
        // every MMA issued by the elected lane completes before TMEM can be released
        if (elect_one()) {
            umma_commit(drain);
            wait1(drain, 0, abort_flag, kDrainTimeoutNs, false);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue (warps 2..5)
        const int q = warp & 3;   // TMEM lane quarter this warp may access
        const uint32_t stage0 = smem_u32(sStage) + (uint32_t)(warp - 2) * 4096u;
        int nchunk = 0;
        int it = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            if (!waitw(&tfull[acc], (uint32_t)(it >> 1) & 1u, abort_flag)) break;
            tc_fence_after();
            const TileInfo t = decode_tile(p, tile);
            const int64_t row0 = t.c_row0 + (int64_t)t.mt * BM;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if (t.swap)
                epi_swapped<EPI>(p, &tmC, taddr, stage0, nchunk, q, t.nt, row0, t.tr);
            else
                epi_rows<EPI>(p, &tmC, taddr, stage0, nchunk, q, t.nt, row0, t.tr);
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
        if (lane == 0) bulk_wait_all();   // staged stores done before the CTA can exit
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag && p.err) atomicOr(p.err, MOE_DEVERR_TIMEOUT);
}

// ---------------------------------------------------------------- host side

TcParams base_params(const GroupGeom& g) {
    TcParams p{};
    p.G = g.G;
    p.rows = g.rows;
    p.row_off = g.row_off;
    p.mtile_off = g.mtile_off;
    p.uniform_rows = g.uniform_rows;
    p.a_stride = g.a_stride;
    p.c_stride = g.c_stride;
    return p;
}

int grid_for(const GroupGeom& g, int n_tiles) {
    int64_t max_tiles;
    if (g.rows == nullptr)
        max_tiles = (int64_t)g.G * ((g.uniform_rows + BM - 1) / BM) * n_tiles;
    else
        max_tiles = ((g.max_rows + BM - 1) / BM + g.G) * (int64_t)n_tiles;
    int sms = device_sm_count();
    return (int)(max_tiles < sms ? (max_tiles < 1 ? 1 : max_tiles) : sms);
}

template <int EPI>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                   const CUtensorMap& c, const TcParams& p, int grid, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(tc_grouped_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    tc_grouped_kernel<EPI><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(a, b0, b1, c, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t tc_gateup(const GroupGeom& g, const __nv_bfloat16* A, int64_t a_rows, int K,
                      const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int F,
                      __nv_bfloat16* H, int64_t h_rows, int32_t* err, cudaStream_t s) {
    if (g.G <= 0 || a_rows <= 0) return cudaSuccess;
    CUtensorMap ma, mg, mu, mc;
    if (!make_map(&ma, A, a_rows, K, BM) || !make_map(&mg, Wg, (int64_t)g.G * F, K, BN / 2) ||
        !make_map(&mu, Wu, (int64_t)g.G * F, K, BN / 2) || !make_store_map(&mc, H, h_rows, F))
        return cudaErrorInvalidValue;
    TcParams p = base_params(g);
    p.K = K;
    p.n_out = F;
    p.b_rows = F;
    p.n_tiles = (F + BN / 2 - 1) / (BN / 2);
    p.C = H;
    p.ldc = F;
    p.row_scale = nullptr;
    p.err = err;
    return launch<EPI_SWIGLU>(ma, mg, mu, mc, p, grid_for(g, p.n_tiles), s);
}

cudaError_t tc_down(const GroupGeom& g, const __nv_bfloat16* H, int64_t h_rows, int F,
                    const __nv_bfloat16* Wd, int D, const float* row_scale,
                    __nv_bfloat16* Y, int64_t y_rows, int32_t* err, cudaStream_t s) {
    if (g.G <= 0 || h_rows <= 0) return cudaSuccess;
    CUtensorMap ma, mb, mc;
    if (!make_map(&ma, H, h_rows, F, BM) || !make_map(&mb, Wd, (int64_t)g.G * D, F, BN) ||
        !make_store_map(&mc, Y, y_rows, D))
        return cudaErrorInvalidValue;
    TcParams p = base_params(g);
    p.K = F;
    p.n_out = D;
    p.b_rows = D;
    p.n_tiles = (D + BN - 1) / BN;
    p.C = Y;
    p.ldc = D;
    p.row_scale = row_scale;
    p.err = err;
    return launch<EPI_SCALE>(ma, mb, mb, mc, p, grid_for(g, p.n_tiles), s);
}

}  // namespace moe
