// grouped_gemm_pair.cu -- the grouped bf16 GEMMs of the expert FFNs on CTA pairs
// (tcgen05.mma.cta_group::2) with the expert weights as the MMA's M side and the tokens as its
// N side.
//
// Page "混合专家 MoE", section "实现：逐 token 与按专家分组": after grouping, every expert
// multiplies all of its tokens at once and one grouped GEMM serves all experts;
// Expert.forward is down(silu(gate(x)) * up(x)).  Two kernels:
//   gate/up : per group g, H[r, f] = silu(Wg[g,f] . A_r) * (Wu[g,f] . A_r)     (bf16 out)
//   down    : per group g, Y[r, n] = row_scale[r] * (Wd[g,n] . H_r)            (bf16 out)
// computed as D = W . A^T: the accumulator's rows (TMEM lanes) are weight rows and its columns
// are the group's token rows.
//
// Why this orientation: the token count of a group is ragged (routing decides it), while an
// MMA's N may be any multiple of 16 up to 256 and its M is fixed (256 on a pair).  With tokens
// on N a group is cut into chunks of at most 256 rows (split evenly), each rounded up to 16, so
// at most 15 computed rows per chunk are padding, and every tile moves a full 256-row weight
// tile per k-block for all of its tokens.  On a pair each CTA stages its own 128 weight rows and
// half of the chunk's tokens, so an SM pulls at most 32 KB per 64-wide k-block for 128 x 256 x 64
// multiply-adds (a single-CTA 128 x 256 tile needs 48 KB for the same work), and 192 KB of
// shared memory hold 7 weight and 5 token k-blocks.
//
// Roles (384 threads per CTA, one CTA per SM, persistent over the pair's tiles):
//   warp 0      weight producer in each CTA: its weight rows into the weight ring (TMA); both
//               CTAs' copies complete on the leader CTA's barrier;
//   warp 10     token producer in each CTA: its half of the chunk's token rows into the token
//               ring, likewise;
//   warp 1      allocates 512 TMEM columns in each CTA (two 256-column accumulators); in the
//               leader CTA it issues the pair's MMAs (M = 256, N = chunk rows rounded up to 16,
//               K = 16) from one elected lane and frees ring slots in both CTAs with multicast
//               commits;
//   warps 2..9  epilogue in each CTA, two warps per TMEM lane quarter taking alternate 32-token
//               chunks (short tiles are otherwise bound by the epilogue): tcgen05.ld of its 128
//               weight rows, silu*mul or scale in fp32, one rounding to bf16, stores through
//               shared memory and TMA;
//   warp 11     tile scheduler in each CTA: decodes the pair's tiles (group, chunk, weight
//               tile, token rows) into a 4-entry queue in shared memory that the producers, the
//               MMA warp and the down GEMM's epilogue read.
// Gate/up: each CTA's 128 weight rows are 64 gate rows followed by the matching 64 up rows (two
// TMA boxes per k-block: every copy instruction has a fixed cost in the copy engine, so boxes stay
// large), so TMEM lanes 0-63 hold gate and lanes 64-127 up projections of the same 64 hidden
// units.  A warp reads only its own quarter of the lanes, so each up warp passes its values to the
// gate warp of the same units through shared memory (named barriers pace the handoff) and the
// gate warp finishes silu(g) * u and the store.
// Tiles run group-major, then by weight tile, with the chunks of a group innermost (in blocks of
// 16 chunks), so the pairs working at the same time share weight tiles and token chunks in L2.
// Routed groups run in the order 0, E-1, 1, E-2, ... so that, under a router that loads one end
// of the expert range (the Zipf-biased layer), tiles of heavy and light experts run side by side.
// The routed GEMMs of the large layers stream every expert's weights from HBM once, and their
// speed is set by how many bytes each SM keeps in flight: the rings fill 192 KB of shared memory
// (7 weight + 5 token slots of 16 KB; 10 + 8 in the decode-sized variant with 32-row token slots
// of 4 KB, used when no group has more than 64 rows).
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA raises an abort flag, the other
// roles stop at their next wait, TMEM is freed and the device error word gets
// MOE_DEVERR_TIMEOUT.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BK = 64;
constexpr int WROWS = 128;                 // weight rows per CTA (the pair's M = 256)
constexpr int TOK_MAX = 256;               // token rows per tile (the MMA's N)
constexpr int A_STAGE = WROWS * BK * 2;    // 16 KB
constexpr uint32_t TMEM_COLS = 2 * TOK_MAX;
constexpr int EPI_WARPS = 8;
constexpr int TOK_WARP = 2 + EPI_WARPS;    // the token producer, after the epilogue warps
constexpr int SCHED_WARP = TOK_WARP + 1;   // the tile scheduler
constexpr int NUM_THREADS = 32 * (SCHED_WARP + 1);
constexpr int QDEPTH = 4;                  // decoded tiles the scheduler may run ahead
constexpr int TQ_BYTES = 256;              // the decoded-tile queue (QDEPTH PTile entries)
// Epilogue shared memory: down = 8 warps x 2 staging buffers x 2 KB; gate/up = 4 exchange buffers
// (32 lanes x 32 floats, one per warp pair) + 4 gate warps x 2 staging buffers x 2 KB; + flags.
constexpr int EPI_BYTES = 32768 + 256;
// Token boxes per CTA: 8 rows, then 16..128 in steps of 16 (a tile needs n_mma / 2 rows).
constexpr int kTokBoxes = 9;
__host__ __device__ constexpr int tok_box_rows(int b) { return b == 0 ? 8 : 16 * b; }

enum { EPI_SWIGLU = 0, EPI_SCALE = 1 };

// Two rings, each with its own producer warp: weight k-blocks (read from HBM once per weight
// tile) in A_STAGES slots and token k-blocks (rows of A, re-read by every weight tile of a chunk,
// mostly L2 hits) in B_STAGES slots.  Measured on the DeepSeek-V3-shaped layer, both kinds of copy
// take several k-blocks to land under this load: with 128-row token slots 7 + 5 slots beat 8 + 4
// and 9 + 3 (2 or 3 token slots stall the MMAs) and match 6 + 6; with 32-row slots (decode)
// 10 + 8 beats 11 + 3 by 11% and matches 9 + 9.
template <int TOK_SLOT>
struct PairCfg {
    static constexpr int B_STAGE = TOK_SLOT * BK * 2;
    static constexpr int A_STAGES = TOK_SLOT >= 128 ? 7 : 10;
    static constexpr int B_STAGES = TOK_SLOT >= 128 ? 5 : 8;
    static constexpr int RING_BYTES = A_STAGES * A_STAGE + B_STAGES * B_STAGE;
    static constexpr int SMEM_BYTES = RING_BYTES + EPI_BYTES + 1024 + 512 + TQ_BYTES;
    static_assert(SMEM_BYTES <= 232448, "shared memory per block");
    static_assert(B_STAGE % 1024 == 0, "stages stay 1 KB aligned for the 128-byte swizzle");
    static_assert((2 * A_STAGES + 2 * B_STAGES + 5 + 2 * QDEPTH) * 8 + 8 <= 512, "barriers fit their area");
};

struct TokMaps {
    CUtensorMap m[kTokBoxes];
};

struct PairParams {
    int G;
    const int32_t* rows;        // [G] device, or nullptr for uniform groups
    const int32_t* row_off;     // [G] device (token row of the group's first row)
    const int32_t* chunk_off;   // [G+1] prefix of the groups' 256-row chunks (non-uniform),
                                // over the groups in zigzag_group order when zigzag is set
    int zigzag;
    int uniform_rows;
    int64_t a_stride, c_stride;
    int K;             // reduction length
    int n_out;         // valid output columns per group (F for gate/up, D for down)
    int w_rows;        // weight rows per group in the 2-D maps (F for gate/up, D for down)
    int n_wt;          // weight tiles per group
    __nv_bfloat16* C;
    int64_t ldc;
    const float* row_scale;
    int32_t* err;
};

struct PTile {
    int g, c, w;
    int nch;           // chunks of the group (how many tiles read each of its weight tiles)
    int rows;          // token rows of this chunk (1..256)
    int n_mma;         // rows rounded up to 16
    int box;           // token box index: tok_box_rows(box) rows per CTA
    int64_t a_row0;    // token row (in A) of the chunk's first row
    int64_t c_row0;    // output row of the chunk's first row
};

static_assert(QDEPTH * sizeof(PTile) <= TQ_BYTES, "the tile queue fits its area");

__device__ __forceinline__ int total_tiles(const PairParams& p) {
    if (p.rows == nullptr) return p.G * ((p.uniform_rows + TOK_MAX - 1) / TOK_MAX) * p.n_wt;
    return p.chunk_off[p.G] * p.n_wt;
}

// Called by all 32 lanes of a warp with the same tile.  The group is found by a 32-way search
// over chunk_off: each level is one coalesced load per lane and a ballot (two levels cover 1024
// groups), and the last level also loads every candidate's row count and row offset, so a tile
// costs two rounds of loads instead of the ten dependent ones of a binary search (measured at
// 1.4-1.8k cycles per tile in every role, a sixth of a short tile's time).
__device__ __forceinline__ PTile decode_tile(const PairParams& p, int tile, int lane) {
    PTile t;
    int nch, n, local;
    int64_t a0, c0;
    if (p.rows == nullptr) {
        nch = (p.uniform_rows + TOK_MAX - 1) / TOK_MAX;
        const int per = nch * p.n_wt;
        t.g = tile / per;
        local = tile - t.g * per;
        n = p.uniform_rows;
        a0 = (int64_t)t.g * p.a_stride;
        c0 = (int64_t)t.g * p.c_stride;
    } else {
        // the largest g with chunk_off[g] * n_wt <= tile (that group is non-empty); it lies in
        // [lo, hi), and chunk_off[lo] * n_wt <= tile holds throughout (chunk_off[0] = 0)
        int lo = 0, hi = p.G;
        while (hi - lo > 32) {
            const int step = (hi - lo + 31) >> 5;
            const int i = lo + lane * step;
            const bool le = i < hi && p.chunk_off[i] * p.n_wt <= tile;
            const int L = 31 - __clz(__ballot_sync(0xffffffffu, le));   // lane 0 always holds
            lo += L * step;
            hi = min(hi, lo + step);
        }
        const int i = lo + lane;
        int off0 = 0, off1 = 0, rows = 0, roff = 0;
        if (i < hi) {
            const int g = p.zigzag ? zigzag_group(i, p.G) : i;
            off0 = p.chunk_off[i];
            off1 = p.chunk_off[i + 1];
            rows = p.rows[g];
            roff = p.row_off[g];
        }
        const int L = 31 - __clz(__ballot_sync(0xffffffffu, i < hi && off0 * p.n_wt <= tile));
        lo += L;
        off0 = __shfl_sync(0xffffffffu, off0, L);
        off1 = __shfl_sync(0xffffffffu, off1, L);
        n = __shfl_sync(0xffffffffu, rows, L);
        a0 = c0 = __shfl_sync(0xffffffffu, roff, L);
        t.g = p.zigzag ? zigzag_group(lo, p.G) : lo;
        nch = off1 - off0;
        local = tile - off0 * p.n_wt;
    }
    raster_tile(local, nch, p.n_wt, t.c, t.w);
    t.nch = nch;
    // the group's rows split evenly over its chunks: the first n % nch chunks get one more
    const int base = n / nch, rem = n - base * nch;
    t.rows = base + (t.c < rem ? 1 : 0);
    const int start = t.c * base + (t.c < rem ? t.c : rem);
    t.n_mma = (t.rows + 15) & ~15;
    const int half = t.n_mma >> 1;
    t.box = half <= 8 ? 0 : (half + 15) >> 4;   // 8 rows, else the multiple of 16 >= half
    t.a_row0 = a0 + start;
    t.c_row0 = c0 + start;
    return t;
}

// The decoded-tile queue.  The scheduler warp pushes each of the pair's tiles (in the order every
// role walks them) and then an end marker (g < 0); a reader warp takes the next entry and frees
// the slot.  Returns 1 for a tile, 0 at the end, -1 when a wait gave up (abort).
__device__ __forceinline__ int pop_tile(const PTile* tq, uint64_t* q_full, uint64_t* q_empty, int& s,
                                        uint32_t& ph, PTile& t, volatile int* abort_flag) {
    if (!waitw(&q_full[s], ph, abort_flag)) return -1;
    t = tq[s];
    __syncwarp();
    if (elect_one()) mbar_arrive(&q_empty[s]);
    __syncwarp();
    if (++s == QDEPTH) {
        s = 0;
        ph ^= 1u;
    }
    return t.g >= 0 ? 1 : 0;
}

// silu(z) = z / (1 + e^-z) with the hardware exponential and division: their relative error
// (a few ulp of fp32) is far below the bf16 rounding that follows.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.f + __expf(-z)); }

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c,
                                             uint32_t& d) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr)
                 : "memory");
}

// ---------------------------------------------------------------- the kernel

template <int EPI, int TOK_SLOT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
pair_grouped_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                    const __grid_constant__ TokMaps tmT, const __grid_constant__ CUtensorMap tmC,
                    const PairParams p) {
    using Cfg = PairCfg<TOK_SLOT>;
    constexpr int SA = Cfg::A_STAGES, SB = Cfg::B_STAGES;
    constexpr int B_STAGE = Cfg::B_STAGE;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sA = smem;                              // [SA] x 16 KB weight rows
    uint8_t* sB = smem + SA * A_STAGE;               // [SB] x B_STAGE token rows
    uint8_t* sEpi = smem + Cfg::RING_BYTES;          // epilogue buffers (see EPI_BYTES)
    volatile int* xflag = reinterpret_cast<volatile int*>(sEpi + 32768);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + EPI_BYTES);
    uint64_t* full_a = bars;               // [SA] leader: both CTAs' weight copies landed
    uint64_t* empty_a = full_a + SA;       // [SA] both: the pair's MMAs released the slot
    uint64_t* full_b = empty_a + SA;       // [SB] leader: both CTAs' token copies landed
    uint64_t* empty_b = full_b + SB;       // [SB] both
    uint64_t* tfull = empty_b + SB;        // [2] both: accumulator ready
    uint64_t* tempty = tfull + 2;          // [2] leader: both CTAs' epilogues drained it
    uint64_t* drain = tempty + 2;          // [1] leader: MMA drain on exit
    uint64_t* q_full = drain + 1;          // [QDEPTH] a decoded tile is in the queue slot
    uint64_t* q_empty = q_full + QDEPTH;   // [QDEPTH] every consumer has read the slot
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_empty + QDEPTH);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    PTile* tq = reinterpret_cast<PTile*>(reinterpret_cast<uint8_t*>(bars) + 512);   // [QDEPTH]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; s++) {
            mbar_init(&full_a[s], 1);
            mbar_init(&empty_a[s], 1);
        }
        for (int s = 0; s < SB; s++) {
            mbar_init(&full_b[s], 1);
            mbar_init(&empty_b[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * EPI_WARPS);   // every epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        // the queue's readers: both producers, the MMA warp (leader CTA) and, in the down GEMM,
        // the epilogue warps (the gate/up epilogue paces its warp pairs itself, see below)
        const int readers = 2 + (leader ? 1 : 0) + (EPI == EPI_SCALE ? EPI_WARPS : 0);
        for (int i = 0; i < QDEPTH; i++) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], readers);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmW0);
        if (EPI == EPI_SWIGLU) prefetch_tmap(&tmW1);
        prefetch_tmap(&tmC);
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

    const int ntiles = total_tiles(p);
    const int nk = (p.K + BK - 1) / BK;
    // a chunk wider than the token slot (not produced by the host's variant choice) is skipped
    // by every role alike and reported
    constexpr int kMaxBox = TOK_SLOT / 16;

    if (warp == 0 || warp == TOK_WARP) {
        // ------------------------------------ TMA producers (both CTAs): warp 0 the weight ring,
        // the token warp the token ring.  The whole warp runs the loop and the waits; one elected
        // lane issues the copies, which complete on the leader CTA's barrier.
        const bool wts = warp == 0;
        const int nst = wts ? SA : SB;
        uint64_t* fullr = wts ? full_a : full_b;
        uint64_t* emptyr = wts ? empty_a : empty_b;
        int s = 0, qs = 0;
        uint32_t ph = 0, qph = 0;
        bool ok = true;
        // A chunk's token rows are re-read by every weight tile of its group, a weight tile by
        // the group's other chunks only.  For gate/up tiles of groups of at most two chunks the
        // weights are marked evict-first, so that the token rows stay in L2.  Groups of more
        // chunks (the Mixtral-shaped layer's four) re-read each weight tile too often for that,
        // and the down GEMM keeps the default policy: evict-first weights there slowed it and
        // the combine that reads its output.
        const uint64_t w_policy = policy_evict_first();
        while (ok) {
            PTile t;
            const int got = pop_tile(tq, q_full, q_empty, qs, qph, t, abort_flag);
            if (got <= 0) {
                ok = got == 0;
                break;
            }
            const int half = t.n_mma >> 1;
            const int tok_y = (int)(t.a_row0 + (int64_t)rank * half);
            const uint32_t tx = wts ? 2u * (uint32_t)A_STAGE : 2u * (uint32_t)(tok_box_rows(t.box) * BK * 2);
            // gate/up: this CTA's 64 hidden units; down: its 128 output rows
            const int wy = EPI == EPI_SWIGLU ? t.g * p.w_rows + t.w * 128 + (int)rank * 64
                                             : t.g * p.w_rows + t.w * 256 + (int)rank * 128;
            const CUtensorMap* mt = &tmT.m[t.box];
            for (int kb = 0; kb < nk; kb++) {
                if (!waitw(&emptyr[s], ph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    if (leader) mbar_arrive_expect_tx(&fullr[s], tx);
                    const uint32_t fb = mapa_shared(smem_u32(&fullr[s]), 0);
                    const int kx = kb * BK;
                    if (wts) {
                        const uint32_t a = smem_u32(sA + s * A_STAGE);
                        if (EPI == EPI_SWIGLU && t.nch <= 2) {
                            tma_load_2d_pair_hint(a, &tmW0, fb, kx, wy, w_policy);
                            tma_load_2d_pair_hint(a + A_STAGE / 2, &tmW1, fb, kx, wy, w_policy);
                        } else {
                            tma_load_2d_pair(a, &tmW0, fb, kx, wy);
                            if (EPI == EPI_SWIGLU) tma_load_2d_pair(a + A_STAGE / 2, &tmW1, fb, kx, wy);
                        }
                    } else {
                        tma_load_2d_pair(smem_u32(sB + s * B_STAGE), mt, fb, kx, tok_y);
                    }
                }
                __syncwarp();
                if (++s == nst) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {   // let copies in flight land before the pair can exit
            const uint64_t t0 = gtimer();
            while (gtimer() - t0 < 200000ull) {
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (leader) {
            // ---------------------------------------------- MMA issuer (leader CTA only)
            // The whole warp runs the loop and the waits; one elected lane issues the MMAs and
            // the commits (see elect_one).  The ring descriptors advance by adding the slot size
            // to their address field.
            int sa = 0, sb = 0, qs = 0;
            uint32_t pha = 0, phb = 0, qph = 0;
            bool ok = true;
            int it = 0;
            const uint64_t ad0 = sw128_desc(smem_u32(sA)), bd0 = sw128_desc(smem_u32(sB));
            uint64_t ad = ad0, bd = bd0;
            while (ok) {
                PTile t;
                if (pop_tile(tq, q_full, q_empty, qs, qph, t, abort_flag) <= 0) break;
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                ++it;
                if (!waitw(&tempty[acc], aph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * TOK_MAX);
                const uint32_t idesc = idesc_bf16_f32(2 * WROWS, t.n_mma);
                for (int kb = 0; kb < nk; kb++) {
                    if (!waitw(&full_a[sa], pha, abort_flag) || !waitw(&full_b[sb], phb, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; kk++)
                            umma_bf16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc,
                                           (kb > 0 || kk > 0) ? 1u : 0u);
                        umma_commit_pair(&empty_a[sa], 0x3);
                        umma_commit_pair(&empty_b[sb], 0x3);
                        if (kb == nk - 1) umma_commit_pair(&tfull[acc], 0x3);
                    }
                    __syncwarp();
                    if (++sa == SA) {
                        sa = 0;
                        pha ^= 1u;
                        ad = ad0;
                    } else {
                        ad += (uint64_t)(A_STAGE >> 4);
                    }
                    if (++sb == SB) {
                        sb = 0;
                        phb ^= 1u;
                        bd = bd0;
                    } else {
                        bd += (uint64_t)(B_STAGE >> 4);
                    }
                }
            }
            // every MMA issued by the elected lane completes before TMEM can be released
            if (elect_one()) {
                umma_commit_pair(drain, 0x1);
                wait1(drain, 0, abort_flag, kDrainTimeoutNs, false);
            }
        }
        __syncwarp();
    } else if (warp == SCHED_WARP) {
        // ---------------------------------- tile scheduler (both CTAs): decodes each tile once,
        // up to QDEPTH ahead of its readers (a decode is a few rounds of dependent loads and
        // integer divisions, about a thousand cycles that the producers and the MMA warp would
        // otherwise spend between tiles)
        int qs = 0;
        uint32_t qph = 0;
        bool ok = true;
        for (int tile = cluster; tile < ntiles && ok; tile += nclusters) {
            const PTile t = decode_tile(p, tile, lane);
            if (t.box > kMaxBox) {
                if (leader && lane == 0 && p.err) atomicOr(p.err, MOE_DEVERR_BOUNDS);
                continue;
            }
            if (!waitw(&q_empty[qs], qph ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                tq[qs] = t;
                mbar_arrive(&q_full[qs]);
            }
            __syncwarp();
            if (++qs == QDEPTH) {
                qs = 0;
                qph ^= 1u;
            }
        }
        if (ok && waitw(&q_empty[qs], qph ^ 1u, abort_flag)) {   // the end marker
            if (lane == 0) {
                tq[qs].g = -1;
                mbar_arrive(&q_full[qs]);
            }
        }
        __syncwarp();
    } else {
        // -------------------------------------------------- epilogue (warps 2..9, both CTAs)
        static_assert(TOK_WARP == 2 + EPI_WARPS, "warps 2 .. 1 + EPI_WARPS are the epilogue");
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int sub = (warp - 2) >> 2;     // chunks sub, sub + 2, ... of every tile
        const uint32_t te0 = mapa_shared(smem_u32(&tempty[0]), 0);
        const uint32_t te1 = mapa_shared(smem_u32(&tempty[1]), 0);
        if (EPI == EPI_SWIGLU) {
            // Warp pair wp (per sub): the up warp (quarter 2 + wp) hands each of its 32-token
            // chunks of 32 up values to the gate warp (quarter wp) of the same hidden units.  Named
            // barrier 1 + 2 wp: the chunk (or the stop message) is in the buffer; 2 + 2 wp: the
            // gate warp has read it.  Only the up warp waits on the accumulator barrier, so both
            // warps always take the same number of handoffs, and a stop message ends the gate warp.
            const int wp = sub * 2 + (q & 1);
            const bool up_warp = q >= 2;
            const int bar_full = 1 + 2 * wp, bar_free = 2 + 2 * wp;
            const uint32_t xb = smem_u32(sEpi) + (uint32_t)wp * 4096u + (uint32_t)lane * 128u;
            const uint32_t stage0 = smem_u32(sEpi) + 16384u + (uint32_t)wp * 4096u;
            int nchunk = 0, it = 0, sent = 0;
            bool stop = false;
            for (int tile = cluster; tile < ntiles && !stop; tile += nclusters) {
                const PTile t = decode_tile(p, tile, lane);
                if (t.box > kMaxBox) continue;
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                ++it;
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * TOK_MAX);
                const int nch = (t.rows + 31) >> 5;
                if (up_warp) {
                    if (!waitw(&tfull[acc], aph, abort_flag)) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = sub; ch < nch; ch += 2) {
                        uint32_t a[32];
                        tmem_ld32(taddr + ch * 32, a);
                        tmem_ld_wait();
                        if (sent > 0) named_sync(bar_free, 64);
#pragma unroll
                        for (int v = 0; v < 8; v++)
                            st_shared_v4(xb + (uint32_t)((v ^ (lane & 7)) << 4), a[4 * v], a[4 * v + 1],
                                         a[4 * v + 2], a[4 * v + 3]);
                        if (lane == 0) xflag[wp] = 0;
                        named_arrive(bar_full, 64);
                        ++sent;
                    }
                } else {
                    const int unit0 = t.w * 128 + (int)rank * 64 + q * 32;   // this warp's units
                    const bool warp_ok = unit0 < p.n_out;
#pragma unroll 1
                    for (int ch = sub; ch < nch; ch += 2, nchunk++) {
                        named_sync(bar_full, 64);
                        if (xflag[wp] != 0) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
                        uint32_t g[32], u[32];
                        tmem_ld32(taddr + ch * 32, g);
#pragma unroll
                        for (int v = 0; v < 8; v++)
                            ld_shared_v4(xb + (uint32_t)((v ^ (lane & 7)) << 4), u[4 * v], u[4 * v + 1],
                                         u[4 * v + 2], u[4 * v + 3]);
                        named_arrive(bar_free, 64);
                        tmem_ld_wait();
                        float h[32];
#pragma unroll
                        for (int j = 0; j < 32; j++)
                            h[j] = silu_fast(__uint_as_float(g[j])) * __uint_as_float(u[j]);
                        const int64_t gr = t.c_row0 + ch * 32;
                        if (warp_ok)
                            store_chunk32_t(&tmC, stage0 + (uint32_t)(nchunk & 1) * 2048u, h,
                                            t.rows - ch * 32, p.C + gr * p.ldc + unit0 + lane, p.ldc,
                                            unit0 + lane < p.n_out, unit0, (int32_t)gr);
                    }
                    if (stop) break;
                    // a gate warp with no chunk in this tile waited on nothing: its up warp, which
                    // waited for the accumulator, releases it on its behalf
                    if (nch <= sub) continue;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_cluster_relaxed(acc ? te1 : te0);
                    if (up_warp && nch <= sub) mbar_arrive_cluster_relaxed(acc ? te1 : te0);
                }
            }
            if (up_warp) {   // the stop message: the gate warp leaves its loop on it
                if (sent > 0) named_sync(bar_free, 64);
                if (lane == 0) xflag[wp] = 1;
                named_arrive(bar_full, 64);
            } else if (!stop) {
                named_sync(bar_full, 64);   // the stop message after the last tile
            }
            if (lane == 0) bulk_wait_all();   // staged stores done before the CTA can exit
            __syncwarp();
        } else {
            const uint32_t stage0 = smem_u32(sEpi) + (uint32_t)(warp - 2) * 4096u;
            int nchunk = 0, it = 0, qs = 0;
            uint32_t qph = 0;
            static_assert(TOK_MAX <= 2 * 4 * 32, "a warp takes at most 4 chunks of a tile");
            // One tile of lookahead: the next tile is taken from the queue, and the row scales of
            // this warp's (at most 4) chunks of it loaded, before the current tile's chunks are
            // written, so that the loads' latency (high while the rings stream) stays hidden.
            auto load_scales = [&](const PTile& u, float (&sc)[4]) {
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int r = (sub + 2 * i) * 32 + lane;
                    sc[i] = (p.row_scale && r < u.rows) ? p.row_scale[u.c_row0 + r] : 1.f;
                }
            };
            PTile t;
            float sc[4];
            int got = pop_tile(tq, q_full, q_empty, qs, qph, t, abort_flag);
            if (got > 0) load_scales(t, sc);
            while (got > 0) {
                PTile tn;
                float scn[4];
                const int gotn = pop_tile(tq, q_full, q_empty, qs, qph, tn, abort_flag);
                if (gotn > 0) load_scales(tn, scn);
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                ++it;
                if (!waitw(&tfull[acc], aph, abort_flag)) break;
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * TOK_MAX);
                const int nch = (t.rows + 31) >> 5;
                const int col = t.w * 256 + (int)rank * 128 + q * 32;
                const bool warp_ok = col < p.n_out;
                auto emit = [&](const uint32_t (&a)[32], int ch, float s_lane) {
                    const int left = t.rows - ch * 32;
                    const int64_t gr = t.c_row0 + ch * 32;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; j++)
                        v[j] = __uint_as_float(a[j]) * __shfl_sync(0xffffffffu, s_lane, j);
                    if (warp_ok)
                        store_chunk32_t(&tmC, stage0 + (uint32_t)(nchunk & 1) * 2048u, v, left,
                                        p.C + gr * p.ldc + col + lane, p.ldc, col + lane < p.n_out,
                                        col, (int32_t)gr);
                    ++nchunk;
                };
                // chunks sub, sub + 2, ...: the next chunk's TMEM load is in flight while the
                // current one is scaled and stored (two register sets, used in turn)
                uint32_t a0[32], a1[32];
                if (sub < nch) tmem_ld32(taddr + sub * 32, a0);
#pragma unroll 1
                for (int ch = sub, i = 0; ch < nch; ch += 4, i += 2) {
                    tmem_ld_wait();
                    if (ch + 2 < nch) tmem_ld32(taddr + (ch + 2) * 32, a1);
                    emit(a0, ch, i == 0 ? sc[0] : sc[2]);
                    if (ch + 2 >= nch) break;
                    tmem_ld_wait();
                    if (ch + 4 < nch) tmem_ld32(taddr + (ch + 4) * 32, a0);
                    emit(a1, ch + 2, i == 0 ? sc[1] : sc[3]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(acc ? te1 : te0);
                t = tn;
#pragma unroll
                for (int i = 0; i < 4; i++) sc[i] = scn[i];
                got = gotn;
            }
            if (lane == 0) bulk_wait_all();   // staged stores done before the CTA can exit
            __syncwarp();
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

// ---------------------------------------------------------------- host side

bool make_tok_maps(TokMaps* t, const void* A, int64_t a_rows, int K) {
    for (int b = 0; b < kTokBoxes; b++)
        if (!make_map(&t->m[b], A, a_rows, K, tok_box_rows(b))) return false;
    return true;
}

PairParams base_params(const GroupGeom& g) {
    PairParams p{};
    p.G = g.G;
    p.rows = g.rows;
    p.row_off = g.row_off;
    p.chunk_off = g.mtile_off;
    p.zigzag = g.zigzag ? 1 : 0;
    p.uniform_rows = g.uniform_rows;
    p.a_stride = g.a_stride;
    p.c_stride = g.c_stride;
    return p;
}

// Pairs that can be resident at once (one CTA per SM), per device and kernel variant.
template <int EPI, int TS>
int resident_pairs() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return device_sm_count() / 2;
    if (cached[dev] == 0) {
        int n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)device_sm_count(), 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = PairCfg<TS>::SMEM_BYTES;
        if (cudaOccupancyMaxActiveClusters(&n, pair_grouped_kernel<EPI, TS>, &cfg) != cudaSuccess ||
            n <= 0) {
            (void)cudaGetLastError();
            n = device_sm_count() / 2;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

template <int EPI, int TS>
cudaError_t launch(const CUtensorMap& w0, const CUtensorMap& w1, const TokMaps& tok,
                   const CUtensorMap& c, const PairParams& p, int64_t max_tiles, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(pair_grouped_kernel<EPI, TS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg<TS>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t pairs = resident_pairs<EPI, TS>();
    const int64_t use = max_tiles < pairs ? (max_tiles < 1 ? 1 : max_tiles) : pairs;
    pair_grouped_kernel<EPI, TS><<<(unsigned)(2 * use), NUM_THREADS, PairCfg<TS>::SMEM_BYTES, s>>>(
        w0, w1, tok, c, p);
    return cudaGetLastError();
}

int64_t max_tiles_of(const GroupGeom& g, int n_wt) {
    if (g.rows == nullptr)
        return (int64_t)g.G * ((g.uniform_rows + TOK_MAX - 1) / TOK_MAX) * n_wt;
    return ((g.max_rows + TOK_MAX - 1) / TOK_MAX + g.G) * (int64_t)n_wt;
}

}  // namespace

int pair_chunk_rows() { return TOK_MAX; }

cudaError_t pair_gateup(const GroupGeom& g, const __nv_bfloat16* A, int64_t a_rows, int K,
                        const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int F,
                        __nv_bfloat16* H, int64_t h_rows, int32_t* err, int64_t max_group_rows,
                        cudaStream_t s) {
    if (g.G <= 0 || a_rows <= 0) return cudaSuccess;
    CUtensorMap mg, mu, mc;
    TokMaps tok;
    if (!make_map(&mg, Wg, (int64_t)g.G * F, K, 64) || !make_map(&mu, Wu, (int64_t)g.G * F, K, 64) ||
        !make_tok_maps(&tok, A, a_rows, K) || !make_store_map(&mc, H, h_rows, F))
        return cudaErrorInvalidValue;
    PairParams p = base_params(g);
    p.K = K;
    p.n_out = F;
    p.w_rows = F;
    p.n_wt = (F + 127) / 128;
    p.C = H;
    p.ldc = F;
    p.row_scale = nullptr;
    p.err = err;
    const int64_t mt = max_tiles_of(g, p.n_wt);
    if (max_group_rows <= 64) return launch<EPI_SWIGLU, 32>(mg, mu, tok, mc, p, mt, s);
    return launch<EPI_SWIGLU, 128>(mg, mu, tok, mc, p, mt, s);
}

cudaError_t pair_down(const GroupGeom& g, const __nv_bfloat16* H, int64_t h_rows, int F,
                      const __nv_bfloat16* Wd, int D, const float* row_scale,
                      __nv_bfloat16* Y, int64_t y_rows, int32_t* err, int64_t max_group_rows,
                      cudaStream_t s) {
    if (g.G <= 0 || h_rows <= 0) return cudaSuccess;
    CUtensorMap mw, mc;
    TokMaps tok;
    if (!make_map(&mw, Wd, (int64_t)g.G * D, F, 128) || !make_tok_maps(&tok, H, h_rows, F) ||
        !make_store_map(&mc, Y, y_rows, D))
        return cudaErrorInvalidValue;
    PairParams p = base_params(g);
    p.K = F;
    p.n_out = D;
    p.w_rows = D;
    p.n_wt = (D + 255) / 256;
    p.C = Y;
    p.ldc = D;
    p.row_scale = row_scale;
    p.err = err;
    const int64_t mt = max_tiles_of(g, p.n_wt);
    if (max_group_rows <= 64) return launch<EPI_SCALE, 32>(mw, mw, tok, mc, p, mt, s);
    return launch<EPI_SCALE, 128>(mw, mw, tok, mc, p, mt, s);
}

}  // namespace moe
