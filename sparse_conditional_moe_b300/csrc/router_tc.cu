// router_tc.cu -- router logits l = x W_r^T on the tensor cores, still fp32-accurate.
//
// Page "混合专家 MoE", section "实现：逐 token 与按专家分组", MoE.route: the router is a linear
// layer d -> E whose scores decide the top-k.  The router weight is fp32 and x is bf16.  Each
// fp32 weight w splits exactly into three bf16 numbers, w = hi + mid + lo (hi = bf16(w),
// mid = bf16(w - hi), lo = w - hi - mid, each subtraction exact), so every product x * part is
// exact in fp32 and l = x.hi + x.mid + x.lo loses nothing to the split.  The three parts are
// stacked as the N dimension of one MMA (N = 3 x 64 experts).
//
// Accuracy of the sum: TMEM accumulates in fp32 over 256-wide slices of d only; after each
// slice the epilogue reads the three partial sums, adds them smallest first, and adds the
// slice into the running logit with compensated (Kahan) summation.  The logit error therefore
// stays near the error of a 256-term fp32 sum, whatever d is.
//
// One CTA = 128 tokens x 64 experts, 320 threads:
//   warp 0      TMA producer: x tile 128x64 and the hi/mid/lo rows 3 x 64x64 per k-block,
//               4-stage ring (40 KB per stage, 128-byte swizzle);
//   warp 1      TMEM allocation (512 columns: two 192-column slice accumulators) and the
//               MMA issue (tcgen05.mma M=128, N=192, K=16) from one elected lane;
//   warps 2..9  two epilogue warpgroups, experts [0,32) and [32,64) of the tile.
// Fused form (d not split, 192 < E <= 512): the ceil(E/64) CTAs of one token tile run as a
// thread-block cluster.  Each CTA leaves its 128 x 64 logits in its shared memory (the drained ring); after a
// cluster barrier every CTA finishes 128 / cluster-size of the tile's tokens -- softmax, top-k,
// gap and renormalisation as in router.cu, one warp per token, all ten warps -- reading the
// token's E logits from the cluster's shared memory, and writes its column sums of the
// probabilities.  The logits never go to global memory.  A warp finishes a token in a chain of
// dependent shuffles and reductions (about a microsecond), so the fused form pays off only while a
// CTA finishes few tokens: with clusters of 2 (E <= 128, 64 tokens per CTA) the separate top-k
// kernel, whose thousands of warps hide that latency, is faster and is used instead.
// Unfused form: logits are written as fp32 [N, E] and router.cu finishes the tokens.  Small
// batches (N <= 1024, few CTAs) split d over blockIdx.z: each CTA writes the sum of every
// 256-wide slice it covers, and router_slices_kernel adds the slices in order with the same
// Kahan recurrence, so the logits are bit-identical to the unsplit kernel's.
#include "router_finish.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int RBM = 128;                 // tokens per tile
constexpr int REN = 64;                  // experts per tile
constexpr int RN = 3 * REN;              // MMA N: hi | mid | lo
constexpr int RBK = 64;
constexpr int RSTAGES = 4;
constexpr int SLICE_KB = 4;              // k-blocks per TMEM read-out (256 of d)
constexpr int RA_STAGE = RBM * RBK * 2;  // 16 KB
constexpr int RB_PART = REN * RBK * 2;   // 8 KB
constexpr int RB_STAGE = 3 * RB_PART;    // 24 KB
constexpr int RSTAGE = RA_STAGE + RB_STAGE;
constexpr int RTHREADS = 320;
constexpr uint32_t RTMEM_COLS = 512;
constexpr int RSMEM = RSTAGES * RSTAGE + 1024 + 256;
constexpr int LS_STRIDE = REN + 1;        // fused: logits [128][65] fp32 in the drained ring
constexpr int kFinishWarps = RTHREADS / 32;   // fused: every warp finishes tokens
static_assert(RBM * LS_STRIDE * 4 + kFinishWarps * 512 * 4 <= RSTAGES * RSTAGE,
              "fused finish buffers fit the ring");

// The fused router's per-token outputs (see launch_router for their meaning).
struct RouterFinish {
    const float* b_r;
    int bias_mode, k, renorm;
    int32_t* idx;
    float* w;
    float* gap;
    float* lse;
    float* probs;
    float* p_part;
};

static __device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__global__ void split3_kernel(const float* __restrict__ W, int64_t n, __nv_bfloat16* __restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float w = W[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        out[i] = hi;
        out[n + i] = mid;
        out[2 * n + i] = __float2bfloat16_rn(r2);
    }
}

// FNV = 0: logits to global memory; FNV > 0: fused finish, expert slots per lane = FNV.
template <int FNV>
__global__ void __launch_bounds__(RTHREADS, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 int64_t N, int d, int E, int slices_per_cta, float* __restrict__ logits,
                 float* __restrict__ slice_out, int32_t* err, const RouterFinish fin) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + RSTAGES * RA_STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RSTAGES * RSTAGE);
    uint64_t* full = bars;
    uint64_t* empty = bars + RSTAGES;
    uint64_t* tfull = bars + 2 * RSTAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * RBM;
    const int e0 = blockIdx.y * REN;
    const int nk = (d + RBK - 1) / RBK;
    const int nslices_all = (nk + SLICE_KB - 1) / SLICE_KB;
    // this CTA's slices of d: all of them, or (split over blockIdx.z) a contiguous run whose
    // per-slice sums go to slice_out for router_slices_kernel to add in order
    const int sl0 = blockIdx.z * slices_per_cta;
    const int sl1 = min(nslices_all, sl0 + slices_per_cta);
    const int nslices = sl1 > sl0 ? sl1 - sl0 : 0;
    const int kb0 = sl0 * SLICE_KB, kb1 = min(nk, sl1 * SLICE_KB);

    if (threadIdx.x == 0) {
        for (int s = 0; s < RSTAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 256);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), RTMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (warp == 0) {
        // TMA producer: the whole warp runs the loop and the waits, one elected lane issues
        int s = 0;
        uint32_t ph = 0;
        int last_ph[RSTAGES];
        for (int i = 0; i < RSTAGES; i++) last_ph[i] = -1;
        bool ok = true;
        for (int kb = kb0; kb < kb1; kb++) {
            if (!waitw(&empty[s], ph ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            if (elect_one()) {
                mbar_arrive_expect_tx(&full[s], RSTAGE);
                const int kx = kb * RBK;
                tma_load_2d(smem_u32(sA + s * RA_STAGE), &tmX, &full[s], kx, m0);
#pragma unroll
                for (int p = 0; p < 3; p++)
                    tma_load_2d(smem_u32(sB + s * RB_STAGE + p * RB_PART), &tmW, &full[s], kx,
                                p * E + e0);
            }
            __syncwarp();
            last_ph[s] = (int)ph;
            if (++s == RSTAGES) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok && lane == 0)
            for (int i = 0; i < RSTAGES; i++)
                if (last_ph[i] >= 0)
                    wait1(&full[i], (uint32_t)last_ph[i], abort_flag, kDrainTimeoutNs, false);
        __syncwarp();
    } else if (warp == 1) {
        // MMA issuer: the whole warp runs the loop and the waits, one elected lane issues the
        // MMAs and commits (a loop run by a single thread spends ~100 cycles per MMA once it
        // waits on an mbarrier between groups); the ring descriptors advance by the slot size
        constexpr uint32_t idesc = idesc_bf16_f32(RBM, RN);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        const uint64_t ad0 = sw128_desc(smem_u32(sA)), bd0 = sw128_desc(smem_u32(sB));
        uint64_t ad = ad0, bd = bd0;
        for (int sl = 0; sl < nslices && ok; sl++) {
            const int acc = sl & 1;
            const uint32_t aph = (uint32_t)(sl >> 1) & 1u;
            if (!waitw(&tempty[acc], aph ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
            const int kb_beg = kb0 + sl * SLICE_KB;
            const int kb_end = min(kb1, kb_beg + SLICE_KB);
            for (int kb = kb_beg; kb < kb_end; kb++) {
                if (!waitw(&full[s], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < RBK / 16; kk++)
                        umma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc,
                                  (kb > kb_beg || kk > 0) ? 1u : 0u);
                    umma_commit(&empty[s]);
                    if (kb == kb_end - 1) umma_commit(&tfull[acc]);
                }
                __syncwarp();
                if (++s == RSTAGES) {
                    s = 0;
                    ph ^= 1u;
                    ad = ad0;
                    bd = bd0;
                } else {
                    ad += (uint64_t)(RA_STAGE >> 4);
                    bd += (uint64_t)(RB_STAGE >> 4);
                }
            }
        }
        // every MMA issued by the elected lane completes before TMEM can be released
        if (elect_one()) {
            umma_commit(drain);
            wait1(drain, 0, abort_flag, kDrainTimeoutNs, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue: 2 warpgroups x 4 quarters
        const int q = warp & 3;
        const int wg = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        float acc[32], cmp[32];
#pragma unroll
        for (int j = 0; j < 32; j++) acc[j] = cmp[j] = 0.f;
        bool ok = true;
        for (int sl = 0; sl < nslices; sl++) {
            const int a = sl & 1;
            const uint32_t aph = (uint32_t)(sl >> 1) & 1u;
            if (!waitw(&tfull[a], aph, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t t = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * 256 + wg * 32);
            uint32_t p0[32], p1[32], p2[32];
            tmem_ld32(t, p0);
            tmem_ld32(t + REN, p1);
            tmem_ld32(t + 2 * REN, p2);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&tempty[a]);
            const int64_t tok = (int64_t)m0 + row;
            const int ebase = e0 + wg * 32;
            if (slice_out) {
                // split over d: this slice's sum, for router_slices_kernel
                if (tok < N) {
                    float* dst = slice_out + ((int64_t)(sl0 + sl) * N + tok) * E + ebase;
#pragma unroll
                    for (int j = 0; j < 32; j++)
                        if (ebase + j < E)
                            dst[j] = (__uint_as_float(p2[j]) + __uint_as_float(p1[j])) +
                                     __uint_as_float(p0[j]);
                }
                continue;
            }
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const float s = (__uint_as_float(p2[j]) + __uint_as_float(p1[j])) +
                                __uint_as_float(p0[j]);
                const float y = s - cmp[j];
                const float tt = acc[j] + y;
                cmp[j] = (tt - acc[j]) - y;
                acc[j] = tt;
            }
        }
        const int64_t tok = (int64_t)m0 + row;
        const int ebase = e0 + wg * 32;
        if (FNV > 0) {
            // the ring is drained (every MMA that read it has completed): the logits go there
            float* Ls = reinterpret_cast<float*>(smem);
#pragma unroll
            for (int j = 0; j < 32; j++) Ls[row * LS_STRIDE + wg * 32 + j] = acc[j];
        } else if (ok && !slice_out && tok < N) {
            float* dst = logits + tok * E + ebase;
            if (ebase + 32 <= E && (E & 3) == 0) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(dst + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; j++)
                    if (ebase + j < E) dst[j] = acc[j];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, RTMEM_COLS);
    }
    if constexpr (FNV > 0) {
        // every CTA of the cluster holds its experts' logits for the tile's 128 tokens
        cluster_sync_all();
        const int cy = (int)gridDim.y;                 // the cluster spans the expert blocks
        const int per = (RBM + cy - 1) / cy;
        const int t_beg = (int)blockIdx.y * per;
        const int t_end = min(RBM, t_beg + per);
        float* ptab = reinterpret_cast<float*>(smem) + RBM * LS_STRIDE;   // [8 warps][E]
        {
            using namespace router_detail;
            const int fw = warp;
            const uint32_t ls0 = smem_u32(smem);
            float pacc[FNV];
#pragma unroll
            for (int i = 0; i < FNV; i++) pacc[i] = 0.f;
            for (int t = t_beg + fw; t < t_end; t += kFinishWarps) {
                const int64_t tok = (int64_t)m0 + t;
                if (tok >= N) break;
                float v[FNV];
#pragma unroll
                for (int i = 0; i < FNV; i++) {
                    const int e = lane + 32 * i;
                    v[i] = e < E ? ld_cluster_f32(mapa_shared(ls0, (uint32_t)(e / REN)) +
                                                  (uint32_t)((t * LS_STRIDE + e % REN) * 4))
                                 : 0.f;
                }
                finish_token<FNV>(v, fin.b_r, fin.bias_mode, E, fin.k, fin.renorm, tok, fin.idx,
                                  fin.w, fin.gap, fin.lse, fin.probs, pacc);
            }
            // this CTA's column sums of the probabilities, added over its warps in warp order
#pragma unroll
            for (int i = 0; i < FNV; i++)
                if (lane + 32 * i < E) ptab[fw * E + lane + 32 * i] = pacc[i];
            asm volatile("bar.sync 1, %0;" ::"r"(kFinishWarps * 32) : "memory");
            const int64_t prow = (int64_t)blockIdx.x * cy + blockIdx.y;
            for (int e = threadIdx.x; e < E; e += kFinishWarps * 32) {
                float sacc = 0.f;
                for (int w2 = 0; w2 < kFinishWarps; w2++) sacc += ptab[w2 * E + e];
                fin.p_part[prow * E + e] = sacc;
            }
        }
        cluster_sync_all();   // no CTA leaves while a peer may still read its logits
    }
    if (threadIdx.x == 0 && *abort_flag && err) atomicOr(err, MOE_DEVERR_TIMEOUT);
}

// Split over d: logits[t, e] = the compensated (Kahan) sum of the slice sums in slice order,
// the same recurrence and order the unsplit kernel runs in its epilogue.
__global__ void router_slices_kernel(const float* __restrict__ slice_out, int nslices, int64_t NE,
                                     float* __restrict__ logits) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < NE;
         i += (int64_t)gridDim.x * blockDim.x) {
        float acc = 0.f, cmp = 0.f;
        for (int sl = 0; sl < nslices; sl++) {
            const float y = slice_out[(int64_t)sl * NE + i] - cmp;
            const float tt = acc + y;
            cmp = (tt - acc) - y;
            acc = tt;
        }
        logits[i] = acc;
    }
}

}  // namespace

int router_tc_split(int64_t N, int d, int E) {
    const int64_t ctas = ((N + RBM - 1) / RBM) * ((E + REN - 1) / REN);
    const int nslices = ((d + RBK - 1) / RBK + SLICE_KB - 1) / SLICE_KB;
    if (N > 1024 || ctas * 2 > device_sm_count() || nslices < 2) return 1;
    int64_t z = device_sm_count() / ctas;
    if (z > nslices) z = nslices;
    const int spc = (int)((nslices + z - 1) / z);
    return (nslices + spc - 1) / spc;
}

size_t router_tc_logits_floats(int64_t N, int d, int E) {
    const int nslices = ((d + RBK - 1) / RBK + SLICE_KB - 1) / SLICE_KB;
    return (size_t)N * E * (router_tc_split(N, d, E) > 1 ? 1 + nslices : 1);
}

cudaError_t tc_router_split(const float* W_r, int E, int d, __nv_bfloat16* w3, cudaStream_t s) {
    const int64_t n = (int64_t)E * d;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 148 * 8) blocks = 148 * 8;
    split3_kernel<<<blocks, 256, 0, s>>>(W_r, n, w3);
    return cudaGetLastError();
}

bool router_tc_fused(int64_t N, int d, int E) {
    return router_tc_split(N, d, E) == 1 && E > 3 * REN && E <= 8 * REN;
}

template <int FNV>
cudaError_t launch_fused(const CUtensorMap& mx, const CUtensorMap& mw, int64_t N, int d, int E,
                         int nslices, int32_t* err, const RouterFinish& fin, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<FNV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, RSMEM);
    if (e != cudaSuccess) return e;
    const int cy = (E + REN - 1) / REN;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + RBM - 1) / RBM), (unsigned)cy, 1);
    cfg.blockDim = dim3(RTHREADS, 1, 1);
    cfg.dynamicSmemBytes = RSMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = (unsigned)cy;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, router_tc_kernel<FNV>, mx, mw, N, d, E, nslices,
                              (float*)nullptr, (float*)nullptr, err, fin);
}

cudaError_t tc_router_fused(const __nv_bfloat16* x, int64_t N, int d, const __nv_bfloat16* w3,
                            int E, const float* b_r, int bias_mode, int k, int renorm,
                            int32_t* idx, float* w, float* gap, float* lse, float* probs,
                            float* p_part, int32_t* err, cudaStream_t s) {
    if (N <= 0) return cudaSuccess;
    CUtensorMap mx, mw;
    if (!make_map(&mx, x, N, d, RBM) || !make_map(&mw, w3, 3 * (int64_t)E, d, REN))
        return cudaErrorInvalidValue;
    const int nslices = ((d + RBK - 1) / RBK + SLICE_KB - 1) / SLICE_KB;
    const RouterFinish fin{b_r, bias_mode, k, renorm, idx, w, gap, lse, probs, p_part};
    if (E <= 64) return launch_fused<2>(mx, mw, N, d, E, nslices, err, fin, s);
    if (E <= 128) return launch_fused<4>(mx, mw, N, d, E, nslices, err, fin, s);
    if (E <= 256) return launch_fused<8>(mx, mw, N, d, E, nslices, err, fin, s);
    return launch_fused<16>(mx, mw, N, d, E, nslices, err, fin, s);
}

int router_tc_part_rows(int64_t N, int E) { return (int)((N + RBM - 1) / RBM) * ((E + REN - 1) / REN); }

cudaError_t tc_router_logits(const __nv_bfloat16* x, int64_t N, int d, const __nv_bfloat16* w3,
                             int E, float* logits, int32_t* err, cudaStream_t s) {
    if (N <= 0) return cudaSuccess;
    cudaError_t e;
    CUtensorMap mx, mw;
    if (!make_map(&mx, x, N, d, RBM) || !make_map(&mw, w3, 3 * (int64_t)E, d, REN))
        return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(router_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, RSMEM);
    if (e != cudaSuccess) return e;
    const int nslices = ((d + RBK - 1) / RBK + SLICE_KB - 1) / SLICE_KB;
    const int z = router_tc_split(N, d, E);
    const int spc = (nslices + z - 1) / z;
    float* slices = z > 1 ? logits + N * E : nullptr;   // the region is sized by router_tc_logits_floats
    dim3 grid((unsigned)((N + RBM - 1) / RBM), (unsigned)((E + REN - 1) / REN), (unsigned)z);
    router_tc_kernel<0><<<grid, RTHREADS, RSMEM, s>>>(mx, mw, N, d, E, spc, logits, slices, err,
                                                      RouterFinish{});
    e = cudaGetLastError();
    if (e != cudaSuccess || z == 1) return e;
    const int64_t NE = N * E;
    router_slices_kernel<<<(unsigned)((NE + 255) / 256), 256, 0, s>>>(slices, nslices, NE, logits);
    return cudaGetLastError();
}

}  // namespace moe
