// permute.cu -- grouping of (token, slot) assignments by expert, with the capacity limit.
//
// Page "混合专家 MoE", section "实现：逐 token 与按专家分组": forward_grouped flattens the
// (token, slot) pairs (slot f = t*k + j), stably sorts them by expert, counts per expert
// (bincount) and walks the segments from their running start; the remark after the listing
// names the pieces: the counts are a histogram and the segment starts a prefix sum.  The
// capacity rule is from "混合专家模型 (MoE)", section 三.1: an expert keeps at most C
// assignments; the first C in the stable order are kept, the rest skip the experts.
//
// The stable sort is rebuilt from integer counting, so it is bit-identical to a stable
// argsort and does not depend on thread timing:
//   count   : block b counts its 2048 consecutive slots per expert (per-warp rows in
//             shared memory, warp-aggregated with __match_any_sync; the block's slots split
//             evenly over its warps, in order) -> blk_hist[b][e]
//   scan    : one block turns blk_hist into counts, offsets (exclusive scan over e),
//             kept = min(counts, C), kept_offsets, and blk_base[b][e] = offsets-free
//             prefix of blk_hist over blocks b' < b
//   scatter : block b recounts per warp, scans over warps, then each warp walks its slots in
//             order; rank r = blk_base + earlier warps + earlier lanes (__popc of the match
//             mask below the lane) + earlier steps.  perm[offsets[e] + r] = f,
//             pos[f] = kept_offsets[e] + r if r < kept[e] else -1
//   gather  : row r of x_perm = x[row_token[r]], 16-byte vector copies, warp per row.
// When the count blocks can all be resident at once, count, scan and scatter run as one
// cooperative kernel (perm_fused_kernel): after a grid barrier every block reads the whole
// per-block histogram and computes its own bases and the offsets itself, so the three passes
// cost one launch.
#include <cooperative_groups.h>

#include <atomic>
#include <cstdlib>
#include <cstring>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = kPermThreads / 32;

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
    if (err) atomicOr(err, bits);
}

// This warp's slots: the block's slots (kPermSlotsPerBlock, fewer in the last block) in equal
// consecutive runs of a multiple of 32, warp after warp, so a small last block (a decode batch
// has a few hundred slots) still spreads over all warps.  Returns the run length; *f0 its start.
__device__ __forceinline__ int warp_slots(int64_t A, int64_t* f0) {
    const int64_t b0 = (int64_t)blockIdx.x * kPermSlotsPerBlock;
    const int64_t left = A - b0;
    const int64_t in_block = left < kPermSlotsPerBlock ? left : kPermSlotsPerBlock;
    const int spw = (int)(((in_block + kWarps - 1) / kWarps + 31) / 32 * 32);
    *f0 = b0 + (int64_t)(threadIdx.x / 32) * spw;
    return spw;
}

// The expert of each of the warp's slots, all steps loaded at once (the loads' latency is
// paid once, not once per step): ev[step] for slot f_begin + 32 step + lane, -1 past A or for
// an index outside [0, E) (reported when err is given).
constexpr int kPermSteps = kPermSlotsPerWarp / 32;
__device__ __forceinline__ void load_slots(const int32_t* __restrict__ idx, int64_t A, int E,
                                           int64_t f_begin, int spw, int (&ev)[kPermSteps],
                                           int32_t* err) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int step = 0; step < kPermSteps; step++) {
        const int64_t f = f_begin + step * 32 + lane;
        ev[step] = (step < spw / 32 && f < A) ? idx[f] : 0;
    }
#pragma unroll
    for (int step = 0; step < kPermSteps; step++) {
        const int64_t f = f_begin + step * 32 + lane;
        if (!(step < spw / 32 && f < A)) {
            ev[step] = -1;
        } else if (ev[step] < 0 || ev[step] >= E) {
            if (err) set_err(err, MOE_DEVERR_BOUNDS);
            ev[step] = -1;
        }
    }
}

// Per-warp expert counts of the warp's slots into cnt[warp][e] (E entries per warp).
__device__ __forceinline__ void warp_count(const int (&ev)[kPermSteps], int spw, int* cnt_row) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int step = 0; step < kPermSteps; step++) {
        if (step >= spw / 32) break;
        const int e = ev[step];
        unsigned mask = __match_any_sync(0xffffffffu, e);
        int leader = __ffs(mask) - 1;
        if (e >= 0 && lane == leader) cnt_row[e] += __popc(mask);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kPermThreads)
perm_count_kernel(const int32_t* __restrict__ idx, int64_t A, int E, int32_t* __restrict__ blk_hist,
                  int32_t* err) {
    extern __shared__ int cnt[];   // [kWarps][E]
    const int warp = threadIdx.x / 32;
    for (int i = threadIdx.x; i < kWarps * E; i += kPermThreads) cnt[i] = 0;
    __syncthreads();
    int64_t f0 = 0;
    const int spw = warp_slots(A, &f0);
    int ev[kPermSteps];
    load_slots(idx, A, E, f0, spw, ev, err);
    warp_count(ev, spw, cnt + warp * E);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kPermThreads) {
        int s = 0;
        for (int w = 0; w < kWarps; w++) s += cnt[w * E + e];
        blk_hist[(int64_t)blockIdx.x * E + e] = s;
    }
}

// Exclusive scan of one value per thread over a 1024-thread block (deterministic).
__device__ int block_exclusive_scan(int v, int* tmp /*[32]*/, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) tmp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int wv = lane < (int)(blockDim.x >> 5) ? tmp[lane] : 0;
        int winc = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, winc, off);
            if (lane >= off) winc += o;
        }
        tmp[lane] = winc - wv;   // exclusive prefix of warp totals
        if (lane == 31) tmp[32] = winc;
    }
    __syncthreads();
    int res = tmp[warp] + inc - v;
    *total = tmp[32];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(1024)
perm_scan_kernel(const int32_t* __restrict__ blk_hist, int blocks, int E, int64_t cap,
                 int32_t* __restrict__ blk_base, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ kept,
                 int32_t* __restrict__ kept_off) {
    __shared__ int tmp[33];
    const int e = threadIdx.x;
    int c = 0;
    if (e < E) {
        for (int b = 0; b < blocks; b++) {
            int h = blk_hist[(int64_t)b * E + e];
            blk_base[(int64_t)b * E + e] = c;
            c += h;
        }
    }
    int kp = (cap >= 0 && c > cap) ? (int)cap : c;
    int total;
    int off = block_exclusive_scan(e < E ? c : 0, tmp, &total);
    int koff_total;
    int koff = block_exclusive_scan(e < E ? kp : 0, tmp, &koff_total);
    if (e < E) {
        counts[e] = c;
        offsets[e] = off;
        kept[e] = kp;
        kept_off[e] = koff;
    }
    if (e == 0) {
        offsets[E] = total;
        kept_off[E] = koff_total;
    }
}

// Scatter of this block's slots (their experts ev from load_slots) given the per-warp run bases
// in cnt[warp][e] and the offsets, kept counts and kept offsets per expert (shared by
// perm_scatter_kernel and perm_fused_kernel).  The slots' routing weights are loaded up front
// like their experts.
__device__ __forceinline__ void scatter_slots(const int (&ev)[kPermSteps],
                                              const float* __restrict__ w, int64_t A, int k,
                                              int64_t f0, int spw, int* base,
                                              const int32_t* offsets, const int32_t* kept,
                                              const int32_t* kept_off, int32_t* __restrict__ perm,
                                              int32_t* __restrict__ pos,
                                              int32_t* __restrict__ row_token,
                                              float* __restrict__ row_weight) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    float wv[kPermSteps];
#pragma unroll
    for (int step = 0; step < kPermSteps; step++) {
        const int64_t f = f0 + step * 32 + lane;
        wv[step] = (w && step < spw / 32 && f < A) ? w[f] : 1.f;
    }
#pragma unroll
    for (int step = 0; step < kPermSteps; step++) {
        if (step >= spw / 32) break;
        const int64_t f = f0 + step * 32 + lane;
        const int e = ev[step];
        unsigned mask = __match_any_sync(0xffffffffu, e);
        int r = 0;
        if (e >= 0) r = base[e] + __popc(mask & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(mask) - 1) base[e] += __popc(mask);
        __syncwarp();
        if (f < A) {
            if (e >= 0) {
                perm[offsets[e] + r] = (int32_t)f;
                if (r < kept[e]) {
                    int p = kept_off[e] + r;
                    pos[f] = p;
                    row_token[p] = (int32_t)(f / k);
                    row_weight[p] = wv[step];
                } else {
                    pos[f] = -1;
                }
            } else {
                pos[f] = -1;
            }
        }
    }
}

__global__ void __launch_bounds__(kPermThreads)
perm_scatter_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w, int64_t A, int k,
                    int E, const int32_t* __restrict__ blk_base, const int32_t* __restrict__ offsets,
                    const int32_t* __restrict__ kept, const int32_t* __restrict__ kept_off,
                    int32_t* __restrict__ perm, int32_t* __restrict__ pos,
                    int32_t* __restrict__ row_token, float* __restrict__ row_weight) {
    extern __shared__ int cnt[];   // [kWarps][E] counts, then running bases
    const int warp = threadIdx.x / 32;
    for (int i = threadIdx.x; i < kWarps * E; i += kPermThreads) cnt[i] = 0;
    __syncthreads();
    int64_t f0 = 0;
    const int spw = warp_slots(A, &f0);
    int ev[kPermSteps];
    load_slots(idx, A, E, f0, spw, ev, nullptr);
    warp_count(ev, spw, cnt + warp * E);
    __syncthreads();
    // per expert: exclusive scan over warps, starting at this block's base
    for (int e = threadIdx.x; e < E; e += kPermThreads) {
        int run = blk_base[(int64_t)blockIdx.x * E + e];
        for (int wv = 0; wv < kWarps; wv++) {
            int c = cnt[wv * E + e];
            cnt[wv * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    scatter_slots(ev, w, A, k, f0, spw, cnt + warp * E, offsets, kept, kept_off, perm, pos,
                  row_token, row_weight);
}

// count -> grid barrier -> scan -> scatter in one cooperative launch (every block resident).
// Shared memory: cnt [kWarps][E], then base, off, kept, koff [E] each.
__global__ void __launch_bounds__(kPermThreads)
perm_fused_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w, int64_t A, int k,
                  int E, int64_t cap, int32_t* __restrict__ blk_hist, int32_t* __restrict__ counts,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ kept,
                  int32_t* __restrict__ kept_off, int32_t* __restrict__ perm,
                  int32_t* __restrict__ pos, int32_t* __restrict__ row_token,
                  float* __restrict__ row_weight, int32_t* err) {
    extern __shared__ int sm[];
    int* cnt = sm;
    int* s_base = cnt + kWarps * E;
    int* s_off = s_base + E;
    int* s_kept = s_off + E;
    int* s_koff = s_kept + E;
    __shared__ int tmp[33];
    const int warp = threadIdx.x / 32;
    for (int i = threadIdx.x; i < kWarps * E; i += kPermThreads) cnt[i] = 0;
    __syncthreads();
    int64_t f0 = 0;
    const int spw = warp_slots(A, &f0);
    int ev[kPermSteps];   // kept in registers across the grid barrier for the scatter
    load_slots(idx, A, E, f0, spw, ev, err);
    warp_count(ev, spw, cnt + warp * E);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kPermThreads) {
        int sum = 0;
        for (int wv = 0; wv < kWarps; wv++) sum += cnt[wv * E + e];
        blk_hist[(int64_t)blockIdx.x * E + e] = sum;
    }
    cooperative_groups::this_grid().sync();
    // this block's base per expert (blocks before it) and the totals; thread t owns the
    // contiguous experts [t per, (t + 1) per), so the scans below run in expert order
    const int nb = (int)gridDim.x;
    const int per = (E + kPermThreads - 1) / kPermThreads;
    const int e_lo = min(E, (int)threadIdx.x * per), e_hi = min(E, e_lo + per);
    int loc_c = 0, loc_k = 0;
    for (int e = e_lo; e < e_hi; e++) {
        // sixteen loads in flight: the histogram's rows are read in rounds, not one by one
        int before = 0, total = 0, b = 0;
        for (; b + 16 <= nb; b += 16) {
            int h[16];
#pragma unroll
            for (int i = 0; i < 16; i++) h[i] = __ldcg(blk_hist + (int64_t)(b + i) * E + e);
#pragma unroll
            for (int i = 0; i < 16; i++) {
                if (b + i < (int)blockIdx.x) before += h[i];
                total += h[i];
            }
        }
        for (; b < nb; b++) {
            const int h = __ldcg(blk_hist + (int64_t)b * E + e);
            if (b < (int)blockIdx.x) before += h;
            total += h;
        }
        s_base[e] = before;
        s_off[e] = total;
        const int kp = (cap >= 0 && total > cap) ? (int)cap : total;
        s_kept[e] = kp;
        loc_c += total;
        loc_k += kp;
    }
    int tot_c, tot_k;
    const int ex_c = block_exclusive_scan(loc_c, tmp, &tot_c);
    const int ex_k = block_exclusive_scan(loc_k, tmp, &tot_k);
    {
        int rc = ex_c, rk = ex_k;
        for (int e = e_lo; e < e_hi; e++) {
            const int c = s_off[e], kp = s_kept[e];
            s_off[e] = rc;
            s_koff[e] = rk;
            if (blockIdx.x == 0) {
                counts[e] = c;
                offsets[e] = rc;
                kept[e] = kp;
                kept_off[e] = rk;
            }
            rc += c;
            rk += kp;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        offsets[E] = tot_c;
        kept_off[E] = tot_k;
    }
    __syncthreads();
    // per expert: exclusive scan over warps, starting at this block's base
    for (int e = threadIdx.x; e < E; e += kPermThreads) {
        int run = s_base[e];
        for (int wv = 0; wv < kWarps; wv++) {
            int c = cnt[wv * E + e];
            cnt[wv * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    scatter_slots(ev, w, A, k, f0, spw, cnt + warp * E, s_off, s_kept, s_koff, perm, pos,
                  row_token, row_weight);
}

// x_perm[r] = x[row_token[r]] for r < kept_off[E]; one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ row_token,
                   const int32_t* __restrict__ kept_off_end, int64_t N, int row_vecs,
                   uint4* __restrict__ xp, int32_t* err) {
    const int64_t rows = *kept_off_end;
    const int lane = threadIdx.x & 31;
    const int64_t warp_global = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = warp_global; r < rows; r += warps) {
        int64_t t = row_token[r];
        if (t < 0 || t >= N) {
            if (lane == 0) set_err(err, MOE_DEVERR_BOUNDS);
            continue;
        }
        const uint4* src = x + t * row_vecs;
        uint4* dst = xp + r * row_vecs;
        int v = lane;
        for (; v + 224 < row_vecs; v += 256) {   // eight 16-byte loads in flight per lane
            uint4 a[8];
#pragma unroll
            for (int i = 0; i < 8; i++) a[i] = __ldg(src + v + 32 * i);
#pragma unroll
            for (int i = 0; i < 8; i++) __stcs(dst + v + 32 * i, a[i]);   // streamed: read later by TMA
        }
        for (; v + 96 < row_vecs; v += 128) {   // four 16-byte loads in flight per lane
            const uint4 a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64),
                        e = __ldg(src + v + 96);
            __stcs(dst + v, a);
            __stcs(dst + v + 32, b);
            __stcs(dst + v + 64, c);
            __stcs(dst + v + 96, e);
        }
        for (; v < row_vecs; v += 32) __stcs(dst + v, __ldg(src + v));
    }
}

// Blocks of perm_fused_kernel the GPU holds at once (per device and shared-memory size); 0 with
// MOE_PERMUTE=unfused (read once per process), which keeps the three-launch form for comparisons.
// The cache holds (shared-memory bytes, capacity) in one atomic word per device, so threads
// forwarding at once never see one call's size with another's capacity.
int fused_capacity(size_t smem) {
    static std::atomic<int> unfused{-1};
    if (unfused.load(std::memory_order_relaxed) < 0) {
        const char* v = getenv("MOE_PERMUTE");
        unfused.store((v && strcmp(v, "unfused") == 0) ? 1 : 0, std::memory_order_relaxed);
    }
    if (unfused.load(std::memory_order_relaxed)) return 0;
    static std::atomic<uint64_t> cached[64];                // (smem << 32) | capacity, 0 = none
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const uint64_t hit = cached[dev].load(std::memory_order_acquire);
    if (hit != 0 && (hit >> 32) == (uint64_t)smem) return (int)(hit & 0xffffffffu);
    int per_sm = 0;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(perm_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, perm_fused_kernel, kPermThreads,
                                                      smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const int capn = per_sm * device_sm_count();
    cached[dev].store(((uint64_t)smem << 32) | (uint32_t)capn, std::memory_order_release);
    return capn;
}

}  // namespace

cudaError_t launch_permute_unfused(const moe_cfg& c, const int32_t* idx, const float* w,
                                   int32_t* counts, int32_t* offsets, int32_t* kept,
                                   int32_t* kept_off, int32_t* perm, int32_t* pos,
                                   int32_t* row_token, float* row_weight, int32_t* blk_hist,
                                   int32_t* blk_base, int32_t* err, cudaStream_t s);

cudaError_t launch_permute(const moe_cfg& c, const int32_t* idx, const float* w, const void* x,
                           int32_t* counts, int32_t* offsets, int32_t* kept, int32_t* kept_off,
                           int32_t* perm, int32_t* pos, int32_t* row_token, float* row_weight,
                           void* x_perm, int32_t* blk_hist, int32_t* blk_base, int32_t* err,
                           cudaStream_t s) {
    const int64_t A = c.N * c.k;
    const int E = c.E;
    const int blocks = perm_blocks(A);
    const size_t fused_smem = sizeof(int) * (kWarps + 4) * E;
    if (blocks > 0 && blocks <= fused_capacity(fused_smem)) {
        int64_t cap = capacity(c);
        int k = c.k, e = E;
        void* args[] = {(void*)&idx, (void*)&w, (void*)&A, (void*)&k, (void*)&e, (void*)&cap,
                        (void*)&blk_hist, (void*)&counts, (void*)&offsets, (void*)&kept,
                        (void*)&kept_off, (void*)&perm, (void*)&pos, (void*)&row_token,
                        (void*)&row_weight, (void*)&err};
        cudaError_t ef = cudaLaunchCooperativeKernel((const void*)perm_fused_kernel, dim3(blocks),
                                                     dim3(kPermThreads), args, fused_smem, s);
        if (ef != cudaSuccess) return ef;
    } else {
        cudaError_t eu = launch_permute_unfused(c, idx, w, counts, offsets, kept, kept_off, perm,
                                                pos, row_token, row_weight, blk_hist, blk_base,
                                                err, s);
        if (eu != cudaSuccess) return eu;
    }
    if (blocks == 0 || x_perm == nullptr) return cudaSuccess;
    {
        const int esz = c.act_dtype == MOE_BF16 ? 2 : 4;
        const int row_vecs = (int)((int64_t)c.d * esz / 16);
        const int64_t rows = grouped_rows(c);
        int64_t want = (rows + 7) / 8;     // 8 warps per block
        int gblocks = (int)(want < 148 * 16 ? want : 148 * 16);
        if (gblocks < 1) gblocks = 1;
        gather_rows_kernel<<<gblocks, 256, 0, s>>>((const uint4*)x, row_token, kept_off + E, c.N,
                                                   row_vecs, (uint4*)x_perm, err);
    }
    return cudaGetLastError();
}

// The three-launch form (count, one-block scan, scatter), for grids too large to be resident.
cudaError_t launch_permute_unfused(const moe_cfg& c, const int32_t* idx, const float* w,
                                   int32_t* counts, int32_t* offsets, int32_t* kept,
                                   int32_t* kept_off, int32_t* perm, int32_t* pos,
                                   int32_t* row_token, float* row_weight, int32_t* blk_hist,
                                   int32_t* blk_base, int32_t* err, cudaStream_t s) {
    const int64_t A = c.N * c.k;
    const int E = c.E;
    const int blocks = perm_blocks(A);
    const size_t smem = sizeof(int) * kWarps * E;
    if (blocks > 0) {
        perm_count_kernel<<<blocks, kPermThreads, smem, s>>>(idx, A, E, blk_hist, err);
        cudaError_t e1 = cudaGetLastError();
        if (e1 != cudaSuccess) return e1;
    }
    perm_scan_kernel<<<1, 1024, 0, s>>>(blk_hist, blocks, E, capacity(c), blk_base, counts,
                                        offsets, kept, kept_off);
    cudaError_t e2 = cudaGetLastError();
    if (e2 != cudaSuccess || blocks == 0) return e2;
    perm_scatter_kernel<<<blocks, kPermThreads, smem, s>>>(idx, w, A, c.k, E, blk_base, offsets,
                                                           kept, kept_off, perm, pos, row_token,
                                                           row_weight);
    return cudaGetLastError();
}

}  // namespace moe
