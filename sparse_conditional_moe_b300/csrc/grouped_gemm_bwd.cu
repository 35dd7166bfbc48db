// grouped_gemm_bwd.cu -- the grouped GEMMs of the expert backward pass on tcgen05.
//
// Chain rule through Expert.forward = down(silu(gate(x)) * up(x)) of page "混合专家 MoE"
// (实现 section), per expert e over its kept rows r (the rows laid out in zero-padded segments
// that start at multiples of 128, so a reduction over rows never mixes two experts):
//   G1  dH'[r, :]   = dout[r, :] . W_d[e]            (B = W_d [d, F] as stored: MN-major)
//       epilogue: dw_r partial = <dH'_r, h_r> per 128-column tile, dh_r = w_r dH'_r (bf16)
//   G2  G, U        = x[r, :] . W_g[e]^T, W_u[e]^T   (recomputed, K-major like the forward)
//       epilogue: dg = dh u silu'(g), du = dh silu(g) into [dG | dU], and w_r h_r (bf16)
//   G3  dX[r, :]    = [dG | dU][r, :] . [W_g[e]; W_u[e]]   (B MN-major, K = 2F)
//   G4  dW_d[e]     = sum_r dout_r (w_r h_r)^T             (A, B MN-major, K = rows)
//   G5  [dW_g; dW_u][e] = sum_r [dG | dU]_r^T x_r          (A, B MN-major, K = rows)
// The same kernels serve the shared experts (one group of N rows each, weight 1).
//
// Design (one CTA per SM, persistent, warp-specialised, 192 threads), as the forward kernel:
//   warp 0      TMA producer (the warp runs the loop, an elected lane issues): A tile 128x64
//               and B tile 256x64 (bf16, 128-byte swizzle) per k-block into a 4-stage ring
//               (48 KB per stage).  A K-major operand is one box of its rows x 64; an MN-major
//               operand is boxes of 64 k-rows x 64 elements, 8 KB apart (two for A, four for B);
//   warp 1      allocates 512 TMEM columns; the warp runs the loop and an elected lane issues
//               tcgen05.mma (M=128, N=256, K=16) with the operands' majorness in the
//               instruction descriptor;
//   warps 2..5  epilogue: tcgen05.ld of the 128x256 fp32 accumulator, per-row arithmetic,
//               16-byte stores.  Two accumulators overlap epilogue and mainloop.
// Every wait is bounded (globaltimer); on expiry the CTA raises an abort flag, drains, frees
// TMEM and sets MOE_DEVERR_TIMEOUT.
#include "tc_ptx.cuh"
#include "bwd_internal.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;   // 16 KB
constexpr int B_STAGE = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int MN_BOX = 64 * BK * 2;    // one MN-major box: 64 k-rows x 64 elements, 8 KB
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int NUM_THREADS = 192;
constexpr int STAGE_BUF = 4096;         // per epilogue warp: 2 buffers of 32 rows x 128 B
constexpr int STAGING_BYTES = 4 * 2 * STAGE_BUF;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*alignment*/ + 256 /*barriers*/;

// MN-major operand, 128-byte swizzle: 64 elements (128 B) along M or N per row, one row per k,
// 8-row groups 1024 bytes apart (stride byte offset), the second 64-element column 8 KB away
// (leading byte offset).
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(MN_BOX >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

struct Tile {
    int g, mt, nt, nk;
};

__device__ __forceinline__ int total_tiles(const TbParams& p) {
    if (p.mode == TB_ROWS) return p.c_off[p.G] / BM * p.n_tiles;
    return p.G * p.m_tiles * p.n_tiles;
}

__device__ __forceinline__ Tile decode(const TbParams& p, int tile) {
    Tile t;
    if (p.mode == TB_ROWS) {
        int lo = 0, hi = p.G;   // largest g with (c_off[g] / BM) * n_tiles <= tile
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.c_off[mid] / BM * p.n_tiles <= tile) lo = mid;
            else hi = mid;
        }
        t.g = lo;
        const int mt0 = p.c_off[lo] / BM;
        const int mtg = p.c_off[lo + 1] / BM - mt0;
        raster_tile(tile - mt0 * p.n_tiles, mtg, p.n_tiles, t.mt, t.nt);
        t.nk = (p.K + BK - 1) / BK;
    } else {
        const int per = p.m_tiles * p.n_tiles;
        t.g = tile / per;
        const int local = tile - t.g * per;
        t.mt = local / p.n_tiles;
        t.nt = local - t.mt * p.n_tiles;
        t.nk = (p.rows[t.g] + BK - 1) / BK;
    }
    return t;
}

__device__ __forceinline__ float sigmoid(float z) { return 1.f / (1.f + expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// The warp's 32 rows x 32 fp32 (lane = row) to global memory through the warp's staging buffer
// (128-byte rows, 128-byte swizzle: conflict-free 16-byte stores) and one TMA store at (col,
// row0) of the output map; the map clips rows and columns outside the tensor.  The warp
// alternates between two buffers: the store that used a buffer two chunks ago must have finished
// reading it.
__device__ __forceinline__ void store_chunk_f32(const CUtensorMap* map, uint32_t buf,
                                                const uint32_t (&v)[32], int32_t col, int32_t row0) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    const uint32_t rowb = buf + (uint32_t)lane * 128u;
    const uint32_t sw = (uint32_t)lane & 7u;
#pragma unroll
    for (int c = 0; c < 8; c++)
        st_shared_v4(rowb + (((uint32_t)c ^ sw) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                     v[4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(map, buf, col, row0);
        bulk_commit();
    }
}

// The same for 32 rows x 16 words (32 bf16 per row, 64 bytes): two rows per store instruction.
__device__ __forceinline__ void store_rows16(uint32_t* buf, const uint32_t (&v)[16],
                                             uint32_t* row_dst) {
    const int lane = threadIdx.x & 31;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 16; j++) buf[lane * 17 + j] = v[j];
    __syncwarp();
    const uint64_t mine = reinterpret_cast<uint64_t>(row_dst);
    const int half = lane >> 4, wdx = lane & 15;
#pragma unroll 4
    for (int r2 = 0; r2 < 16; r2++) {
        const int r = 2 * r2 + half;
        const uint64_t pr = ((uint64_t)__shfl_sync(0xffffffffu, (uint32_t)(mine >> 32), r) << 32) |
                            __shfl_sync(0xffffffffu, (uint32_t)mine, r);
        if (pr != 0) reinterpret_cast<uint32_t*>(pr)[wdx] = buf[r * 17 + wdx];
    }
}

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tcb_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
           const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmC0,
           const __grid_constant__ CUtensorMap tmC1, const TbParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE;
    uint32_t* staging = reinterpret_cast<uint32_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + STAGING_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
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
        prefetch_tmap(&tmB1);
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

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer: the whole warp runs
        // the loop and the waits, one elected lane issues the copies
        int s = 0;
        uint32_t ph = 0;
        int last_ph[STAGES];
        for (int i = 0; i < STAGES; i++) last_ph[i] = -1;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const Tile t = decode(p, tile);
            for (int kb = 0; kb < t.nk; kb++) {
                if (!waitw(&empty[s], ph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                    const uint32_t a_dst = smem_u32(sA + s * A_STAGE);
                    const uint32_t b_dst = smem_u32(sB + s * B_STAGE);
                    const int kx = kb * BK;
                    const bool rows_mode = p.mode == TB_ROWS;
                    // A: K offset and M offset of this tile in A's 2-D map
                    const int a_k = (rows_mode ? 0 : p.a_off[t.g]) + kx;
                    const int a_m = (rows_mode ? p.a_off[t.g] : 0) + t.mt * BM;
                    if (A_MN) {                            // [K rows, M]: two 64-wide boxes
                        tma_load_2d(a_dst, &tmA, &full[s], a_m, a_k);
                        tma_load_2d(a_dst + MN_BOX, &tmA, &full[s], a_m + 64, a_k);
                    } else {                               // [M rows, K]: one box of BM rows
                        tma_load_2d(a_dst, &tmA, &full[s], a_k, a_m);
                    }
                    if (EPI == TBE_SWIGLU_BWD) {           // gate rows over up rows, K-major
                        const int y = t.g * p.b_rows + t.nt * (BN / 2);
                        tma_load_2d(b_dst, &tmB0, &full[s], kx, y);
                        tma_load_2d(b_dst + B_STAGE / 2, &tmB1, &full[s], kx, y);
                    } else if (B_MN) {                     // [K rows, N]: four 64-wide boxes
                        const bool second = rows_mode && kx >= p.k_split;
                        const CUtensorMap* m = second ? &tmB1 : &tmB0;
                        const int b_k = rows_mode ? t.g * p.b_rows + (second ? kx - p.k_split : kx)
                                                  : p.c_off[t.g] + kx;
#pragma unroll
                        for (int j = 0; j < BN / 64; j++)
                            tma_load_2d(b_dst + j * MN_BOX, m, &full[s], t.nt * BN + 64 * j, b_k);
                    } else {                               // [N rows, K]: one box of BN rows
                        const int b_k = (rows_mode ? 0 : p.c_off[t.g]) + kx;
                        const int b_n = (rows_mode ? t.g * p.b_rows : 0) + t.nt * BN;
                        tma_load_2d(b_dst, &tmB0, &full[s], b_k, b_n);
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
        if (!ok && lane == 0) {   // let the copies in flight land before the CTA can exit
            for (int i = 0; i < STAGES; i++)
                if (last_ph[i] >= 0)
                    wait1(&full[i], (uint32_t)last_ph[i], abort_flag, kDrainTimeoutNs, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer: the whole warp runs the
        // loop and the waits, one elected lane issues the MMAs and commits (one thread issuing
        // between mbarrier waits spends ~100-115 cycles per MMA); the ring descriptors advance by
        // adding the stage size to their address field
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN) | ((A_MN ? 1u : 0u) << 15) |
                                   ((B_MN ? 1u : 0u) << 16);
        // K 16 = 32 bytes (K-major) or 2048 bytes (MN-major): +2 or +128 in the address field
        constexpr uint64_t a_step = A_MN ? 128 : 2, b_step = B_MN ? 128 : 2;
        const uint64_t ad0 = A_MN ? sw128_mn_desc(smem_u32(sA)) : sw128_desc(smem_u32(sA));
        const uint64_t bd0 = B_MN ? sw128_mn_desc(smem_u32(sB)) : sw128_desc(smem_u32(sB));
        uint64_t ad = ad0, bd = bd0;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        int it = 0;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++it) {
            const Tile t = decode(p, tile);
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            if (!waitw(&tempty[acc], aph ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < t.nk; kb++) {
                if (!waitw(&full[s], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; kk++)
                        umma_bf16(d_tmem, ad + a_step * kk, bd + b_step * kk, idesc,
                                  (kb > 0 || kk > 0) ? 1u : 0u);
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
            // after the loop, so that a tile without k-blocks (an empty group) is released too
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
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        int it = 0;
        int nchunk = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            if (!waitw(&tfull[acc], aph, abort_flag)) break;
            tc_fence_after();
            const Tile t = decode(p, tile);
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            uint32_t* buf = staging + (warp - 2) * (2 * STAGE_BUF / 4);
            const uint32_t sbuf = smem_u32(buf);
            if (EPI == TBE_F32) {
                // weight gradient rows m of group g (every lane reads TMEM: the load is
                // warp-collective); a group without rows has no MMAs: its tile is zero
                // the warp's 32 rows: all in the first output (rows < split_m) or all in the
                // second (split_m is a multiple of 32); rows past M are clipped by the map
                const int m0 = t.mt * BM + q * 32;
                if (m0 < p.M) {
                    const bool first = m0 < p.split_m;
                    const CUtensorMap* map = first ? &tmC0 : &tmC1;
                    const int32_t row0 = first ? t.g * p.split_m + m0
                                               : t.g * (p.M - p.split_m) + (m0 - p.split_m);
#pragma unroll 1
                    for (int c = 0; c < BN / 32; c++) {
                        uint32_t a[32];
                        if (t.nk > 0) {
                            tmem_ld32(taddr + c * 32, a);
                            tmem_ld_wait();
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; j++) a[j] = 0u;
                        }
                        const int col = t.nt * BN + c * 32;
                        if (col >= p.N) continue;          // warp-uniform
                        store_chunk_f32(map, sbuf + (uint32_t)(nchunk++ & 1) * STAGE_BUF, a, col, row0);
                    }
                }
            } else {
                const int rl = t.mt * BM + row_in_tile;          // row within the group
                const bool valid = rl < p.rows[t.g];
                const int64_t pr = (int64_t)p.c_off[t.g] + rl;   // padded row
                const int64_t dr = (int64_t)p.dense_off[t.g] + rl;   // dense row (valid only)
                const float w = (valid && p.row_weight) ? p.row_weight[dr] : 1.f;
                if (EPI == TBE_DH) {
                    float part = 0.f;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; c++) {
                        uint32_t a[32];
                        tmem_ld32(taddr + c * 32, a);
                        tmem_ld_wait();
                        const int col = t.nt * BN + c * 32;
                        if (col >= p.N) continue;         // ragged last tile (F % 256 != 0)
                        uint32_t pk[16];
                        if (valid) {
                            const uint4* hp = reinterpret_cast<const uint4*>(p.aux_bf16 + dr * p.ld_aux + col);
#pragma unroll
                            for (int v = 0; v < 4; v++) {
                                const uint4 hv = hp[v];
                                const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
                                for (int i = 0; i < 4; i++) {
                                    const float a0 = __uint_as_float(a[8 * v + 2 * i]);
                                    const float a1 = __uint_as_float(a[8 * v + 2 * i + 1]);
                                    part = fmaf(a0, bf16_lo(hw[i]), part);
                                    part = fmaf(a1, bf16_hi(hw[i]), part);
                                    pk[4 * v + i] = pack_bf16(w * a0, w * a1);
                                }
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; j++) pk[j] = 0u;
                        }
                        store_rows16(buf, pk, reinterpret_cast<uint32_t*>(p.out_bf16 + pr * p.ld_bf16 + col));
                    }
                    p.dw_part[pr * p.n_tiles + t.nt] = valid ? part : 0.f;
                } else if (EPI == TBE_SWIGLU_BWD) {
                    const int f0 = t.nt * (BN / 2);
#pragma unroll 1
                    for (int c = 0; c < (BN / 2) / 32; c++) {
                        uint32_t g[32], u[32];
                        tmem_ld32(taddr + c * 32, g);
                        tmem_ld32(taddr + BN / 2 + c * 32, u);
                        tmem_ld_wait();
                        const int f = f0 + c * 32;
                        uint32_t pg[16], pu[16], ph[16];
                        if (valid) {
                            const uint4* dhp = reinterpret_cast<const uint4*>(p.aux_bf16 + pr * p.ld_aux + f);
#pragma unroll
                            for (int v = 0; v < 4; v++) {
                                const uint4 dv = dhp[v];
                                const uint32_t dw4[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                                for (int i = 0; i < 4; i++) {
                                    float rg[2], ru[2], rh[2];
#pragma unroll
                                    for (int e = 0; e < 2; e++) {
                                        const float gv = __uint_as_float(g[8 * v + 2 * i + e]);
                                        const float uv = __uint_as_float(u[8 * v + 2 * i + e]);
                                        const float dh = e ? bf16_hi(dw4[i]) : bf16_lo(dw4[i]);
                                        const float sg = sigmoid(gv);
                                        const float si = gv * sg;
                                        rg[e] = dh * uv * sg * (1.f + gv * (1.f - sg));
                                        ru[e] = dh * si;
                                        rh[e] = w * si * uv;
                                    }
                                    pg[4 * v + i] = pack_bf16(rg[0], rg[1]);
                                    pu[4 * v + i] = pack_bf16(ru[0], ru[1]);
                                    ph[4 * v + i] = pack_bf16(rh[0], rh[1]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; j++) pg[j] = pu[j] = ph[j] = 0u;
                        }
                        store_rows16(buf, pg, reinterpret_cast<uint32_t*>(p.out_bf16 + pr * p.ld_bf16 + f));
                        store_rows16(buf, pu, reinterpret_cast<uint32_t*>(p.out_bf16 + pr * p.ld_bf16 + p.F + f));
                        store_rows16(buf, ph, reinterpret_cast<uint32_t*>(p.out2_bf16 + pr * p.F + f));
                    }
                } else {   // TBE_ROWS_F32: fp32 rows (padding rows of a segment included; the
                           // output map clips rows past the buffer)
                    const int32_t row0 = p.c_off[t.g] + t.mt * BM + q * 32;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; c++) {
                        uint32_t a[32];
                        tmem_ld32(taddr + c * 32, a);
                        tmem_ld_wait();
                        const int col = t.nt * BN + c * 32;
                        if (col >= p.N) continue;         // warp-uniform
                        store_chunk_f32(&tmC0, sbuf + (uint32_t)(nchunk++ & 1) * STAGE_BUF, a, col, row0);
                    }
                }
            }
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

template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_tb(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                      const CUtensorMap& c0, const CUtensorMap& c1, const TbParams& p,
                      int64_t max_tiles, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tcb_kernel<A_MN, B_MN, EPI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int sms = device_sm_count();
    const int grid = (int)(max_tiles < sms ? (max_tiles < 1 ? 1 : max_tiles) : sms);
    tcb_kernel<A_MN, B_MN, EPI><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(a, b0, b1, c0, c1, p);
    return cudaGetLastError();
}

// 2-D bf16 maps.  K-major operand: box 64 (K) x box_rows rows.  MN-major operand: box 64
// elements x 64 k-rows.  Both 128-byte swizzle.
bool map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols,
              int box_rows) {
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn || rows <= 0 || cols <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output [rows, cols], box 32 x 32 (128-byte rows, 128-byte swizzle) for staged stores.
bool map_f32_store(CUtensorMap* m, const float* base, int64_t rows, int64_t cols) {
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn || rows <= 0 || cols <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int tb_dh_tiles(int F) { return (F + BN - 1) / BN; }

// G1: dh = w * (dout_pad . W_d), dw partials.  dout_pad [rows_a, d] (a_off rows), W_d [G*d, F].
cudaError_t tb_dh(const TbParams& p0, const __nv_bfloat16* dout_pad, int64_t rows_a, int d,
                  const __nv_bfloat16* Wd, int F, cudaStream_t s) {
    CUtensorMap ma, mb;
    if (!map_bf16(&ma, dout_pad, rows_a, d, 64, BM) || !map_bf16(&mb, Wd, (int64_t)p0.G * d, F, 64, 64))
        return cudaErrorInvalidValue;
    TbParams p = p0;
    p.mode = TB_ROWS;
    p.K = d;
    p.k_split = d;
    p.b_rows = d;
    p.N = F;
    p.n_tiles = tb_dh_tiles(F);
    return launch_tb<false, true, TBE_DH>(ma, mb, mb, ma, ma, p, p.max_mtiles * (int64_t)p.n_tiles, s);
}

// G2: recompute gate/up of x_pad, SwiGLU backward with dh_pad; writes [dG | dU] and w * h.
cudaError_t tb_swiglu_bwd(const TbParams& p0, const __nv_bfloat16* x_pad, int64_t rows_a, int d,
                          const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int F, cudaStream_t s) {
    CUtensorMap ma, mg, mu;
    if (!map_bf16(&ma, x_pad, rows_a, d, 64, BM) || !map_bf16(&mg, Wg, (int64_t)p0.G * F, d, 64, BN / 2) ||
        !map_bf16(&mu, Wu, (int64_t)p0.G * F, d, 64, BN / 2))
        return cudaErrorInvalidValue;
    TbParams p = p0;
    p.mode = TB_ROWS;
    p.K = d;
    p.k_split = d;
    p.b_rows = F;
    p.F = F;
    p.n_tiles = F / (BN / 2);
    return launch_tb<false, false, TBE_SWIGLU_BWD>(ma, mg, mu, ma, ma, p, p.max_mtiles * (int64_t)p.n_tiles, s);
}

// G3: dX = [dG | dU] . [W_g; W_u] (fp32 rows).  dgu [rows_a, 2F], W_g, W_u [G*F, d].
cudaError_t tb_dx(const TbParams& p0, const __nv_bfloat16* dgu, int64_t rows_a, int F,
                  const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int d, cudaStream_t s) {
    CUtensorMap ma, mg, mu;
    if (!map_bf16(&ma, dgu, rows_a, 2 * F, 64, BM) || !map_bf16(&mg, Wg, (int64_t)p0.G * F, d, 64, 64) ||
        !map_bf16(&mu, Wu, (int64_t)p0.G * F, d, 64, 64))
        return cudaErrorInvalidValue;
    CUtensorMap mc;
    if (!map_f32_store(&mc, p0.out_f32, rows_a, d)) return cudaErrorInvalidValue;
    TbParams p = p0;
    p.mode = TB_ROWS;
    p.K = 2 * F;
    p.k_split = F;
    p.b_rows = F;
    p.N = d;
    p.n_tiles = (d + BN - 1) / BN;
    return launch_tb<false, true, TBE_ROWS_F32>(ma, mg, mu, mc, mc, p, p.max_mtiles * (int64_t)p.n_tiles, s);
}

// Rows GEMM of one operand pair: out[r, :] (fp32) = A[a_off + r, :K] (K-major) . B[k, :N]
// (B [K rows, N], MN-major), for the group rows given in p (the router's part of dx).
cudaError_t tb_rows_f32(const TbParams& p0, const __nv_bfloat16* A, int64_t rows_a, int K,
                        const __nv_bfloat16* B, int N, cudaStream_t s) {
    CUtensorMap ma, mb, mc;
    if (!map_bf16(&ma, A, rows_a, K, 64, BM) || !map_bf16(&mb, B, K, N, 64, 64) ||
        !map_f32_store(&mc, p0.out_f32, rows_a, N))
        return cudaErrorInvalidValue;
    TbParams p = p0;
    p.mode = TB_ROWS;
    p.K = K;
    p.k_split = K;
    p.b_rows = 0;
    p.N = N;
    p.n_tiles = (N + BN - 1) / BN;
    return launch_tb<false, true, TBE_ROWS_F32>(ma, mb, mb, mc, mc, p, p.max_mtiles * (int64_t)p.n_tiles, s);
}

// Weight gradients: out[g] (M x N fp32, rows < split_m into out_f32, the rest into out_f32b)
// = sum over the group's padded rows r of A[a_off + r, m] * B[c_off + r, n].
// (a_cols >= M: A's row width in memory when its rows are padded; 0 = M.)
cudaError_t tb_wgrad(const TbParams& p0, const __nv_bfloat16* A, int64_t rows_a, int M,
                     const __nv_bfloat16* B, int64_t rows_b, int N, cudaStream_t s, int a_cols) {
    CUtensorMap ma, mb;
    if (!map_bf16(&ma, A, rows_a, a_cols > 0 ? a_cols : M, 64, 64) || !map_bf16(&mb, B, rows_b, N, 64, 64))
        return cudaErrorInvalidValue;
    // outputs: rows [0, split_m) of every group in out_f32, the rest in out_f32b
    CUtensorMap c0, c1;
    const int m1 = M - p0.split_m;
    if (!map_f32_store(&c0, p0.out_f32, (int64_t)p0.G * p0.split_m, N) ||
        !map_f32_store(&c1, p0.out_f32b, (int64_t)p0.G * (m1 > 0 ? m1 : p0.split_m), N))
        return cudaErrorInvalidValue;
    TbParams p = p0;
    p.mode = TB_WEIGHTS;
    p.M = M;
    p.N = N;
    p.m_tiles = (M + BM - 1) / BM;
    p.n_tiles = (N + BN - 1) / BN;
    return launch_tb<true, true, TBE_F32>(ma, mb, mb, c0, c1, p, (int64_t)p.G * p.m_tiles * p.n_tiles, s);
}

// One group, any operand majorness, fp32 out: the engine's self-test (see selftest.cu).
cudaError_t tb_selftest(bool a_mn, bool b_mn, int M, int N, int K, const __nv_bfloat16* A,
                        const __nv_bfloat16* B, float* C, const int32_t* plan, int32_t* err,
                        cudaStream_t s) {
    // plan: [rows = K][a_off 0, K][c_off 0, K][dense_off 0] on the device
    TbParams p{};
    p.mode = TB_WEIGHTS;
    p.G = 1;
    p.rows = plan;
    p.a_off = plan + 1;
    p.c_off = plan + 3;
    p.dense_off = plan + 5;
    p.M = M;
    p.N = N;
    p.split_m = M;
    p.out_f32 = C;
    p.out_f32b = C;
    p.m_tiles = (M + BM - 1) / BM;
    p.n_tiles = (N + BN - 1) / BN;
    p.err = err;
    CUtensorMap ma, mb;
    const bool okA = a_mn ? map_bf16(&ma, A, K, M, 64, 64) : map_bf16(&ma, A, M, K, 64, BM);
    const bool okB = b_mn ? map_bf16(&mb, B, K, N, 64, 64) : map_bf16(&mb, B, N, K, 64, BN);
    if (!okA || !okB) return cudaErrorInvalidValue;
    CUtensorMap mc;
    if (!map_f32_store(&mc, C, M, N)) return cudaErrorInvalidValue;
    const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
    if (a_mn && b_mn) return launch_tb<true, true, TBE_F32>(ma, mb, mb, mc, mc, p, tiles, s);
    if (a_mn) return launch_tb<true, false, TBE_F32>(ma, mb, mb, mc, mc, p, tiles, s);
    if (b_mn) return launch_tb<false, true, TBE_F32>(ma, mb, mb, mc, mc, p, tiles, s);
    return launch_tb<false, false, TBE_F32>(ma, mb, mb, mc, mc, p, tiles, s);
}

}  // namespace moe
