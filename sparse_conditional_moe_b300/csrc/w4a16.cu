// w4a16.cu -- expert FFNs with 4-bit weights and bf16 activations (W4A16), for decode-sized
// layers whose cost is reading the expert weights.
//
// Page "混合专家模型 (MoE)：大规模稀疏条件计算的架构与工程实践", section 五.1: only the expert
// layers are quantised, weights to INT4 while activations stay 16-bit, and the arithmetic runs
// on dequantised values.  Format (the page fixes none; the plainest symmetric per-group choice):
// per weight row, groups of 128 consecutive inputs share one fp32 scale s = max|w| / 7 (scales
// stored group-major, [cols/128, rows]); a weight is the code q = round-half-even(w / s) clamped
// to [-8, 7], stored as a two's-complement nibble, two per byte with the even input in the low
// nibble.  A weight's value is q * s.
//
// Kernels:
//   w4_quantize_kernel  one warp per (row, group): bf16 weights -> codes + scale with the same
//                       fp32 operations as the format's definition, so codes are bit-exact;
//   w4_mma_kernel       the grouped SwiGLU gate/up and down products on the codes (below): TMA
//                       streams the codes, CUDA cores dequantise, mma.sync does the products.
// Every code byte of a touched expert is read once per pass of 8 token rows, so for decode (a
// few rows per expert) the expert weights cost a quarter of their bf16 bytes plus 1/32 for
// scales.
#include <atomic>
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kW4Group = 128;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(256)
w4_quantize_kernel(const __nv_bfloat16* __restrict__ W, int64_t rows, int cols,
                   uint8_t* __restrict__ q, float* __restrict__ s) {
    const int groups = cols / kW4Group;
    const int64_t warp_global = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    for (int64_t wg = warp_global; wg < rows * groups; wg += warps) {
        const int64_t r = wg / groups;
        const int g = (int)(wg % groups);
        const __nv_bfloat16* src = W + r * cols + (int64_t)g * kW4Group + lane * 4;
        float v[4], mx = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            v[i] = __bfloat162float(src[i]);
            mx = fmaxf(mx, fabsf(v[i]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float sc = mx / 7.0f;
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            int code = 0;
            if (sc > 0.f) {
                code = __float2int_rn(v[i] / sc);      // round half to even
                code = code < -8 ? -8 : (code > 7 ? 7 : code);
            }
            packed |= (uint32_t)(code & 15) << (4 * i);
        }
        *reinterpret_cast<uint16_t*>(q + (r * cols + (int64_t)g * kW4Group) / 2 + lane * 2) =
            (uint16_t)packed;
        if (lane == 0) s[(int64_t)g * rows + r] = sc;
    }
}

// ------------------------------------------------------------------ grouped W4A16 FFN
//
// Shapes: a group g (expert) owns `rows` token rows of A [*, K] (bf16) and J output features;
// its weight rows are [g*J, g*J + J) of the code matrices [G*J, K/2] and of the group-major
// scale matrices [K/128, G*J].  A block takes kMmaWarps warps x FPW features of one group; a
// warp computes kTiles 16-row weight tiles against kTokTile = 8 token rows per pass: for gate/up
// the gate and up rows of the same 32 features, for down 64 consecutive rows.
//   - codes and scales: each warp streams its rows group by group through its own
//     kStages-deep ring of shared memory: per ring item two boxes of 32 rows x 64 code bytes and
//     two boxes of 32 scales, so the loads run ahead of the arithmetic independently of registers;
//   - activations: the block stages x for the pass in chunks of kChunkK inputs as ready-made
//     mma B fragments (bf16 pairs in the weights' pair order, zeros for missing tokens), plus the
//     sum X of every token's 128 inputs of each group;
//   - per 128-input group a thread turns its code words into bf16 pairs with one LOP3 each
//     (0x4300 | (n ^ 8) is exactly 128 + q + 8 = q + 136), runs 8 mma.m16n8k16 per tile (fp32
//     accumulate) giving D = sum (q + 136) x, and adds s * (D - 136 X) to its accumulators.
// The dot product's input order is permuted consistently on both sides: a thread's pair p of a
// group covers inputs (32t + 8(p/4) + p%4) and that + 4, t = lane % 4, which is where one
// shift + mask of a 32-bit code word puts two nibbles.

// Tunables (compile-time; the defaults are the measured best on B300)
#ifndef MOE_W4_WARPS
#define MOE_W4_WARPS 8
#endif
#ifndef MOE_W4_STAGES
#define MOE_W4_STAGES 2
#endif
#ifndef MOE_W4_PREFETCH_X
#define MOE_W4_PREFETCH_X 0
#endif
#ifndef MOE_W4_MINBLOCKS
#define MOE_W4_MINBLOCKS 2
#endif
constexpr int kMmaWarps = MOE_W4_WARPS;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kStages = MOE_W4_STAGES;
constexpr int kTiles = 4;                               // 16-row tiles per warp
constexpr int kTileRows = 16;
constexpr int kBoxRows = kTiles / 2 * kTileRows;        // 32 rows per TMA box, two boxes
constexpr int kGroupBytes = kW4Group / 2;               // 64 code bytes per row per group
constexpr int kBoxBytes = kBoxRows * kGroupBytes;       // 2 KB
constexpr int kScaleBytes = kBoxRows * 4;               // 128 B: a box's scales of one group
constexpr int kStageTx = 2 * kBoxBytes + 2 * kScaleBytes;
constexpr int kStageBytes = kStageTx;                   // codes 0, codes 1, s 0, s 1
constexpr int kTokTile = 8;                             // tokens per pass (mma n = 8)
constexpr int kChunkK = 2048;                           // inputs staged per x chunk
constexpr int kUnitsPerThread = kTokTile * (kChunkK / 8) / kMmaThreads;  // 16 B units
constexpr int kRingBytes = kMmaWarps * kStages * kStageBytes;
constexpr int kXfragBytes = (kChunkK / kW4Group) * 4 * 32 * 16;        // 32 KB
constexpr int kXsumBytes = (kChunkK / kW4Group) * kTokTile * 4;        // 512 B
constexpr int kMmaSmem = kRingBytes + kXfragBytes + kXsumBytes + kMmaWarps * kStages * 8 + 16 + 1024;
static_assert(kChunkK % kW4Group == 0 && (kTokTile * (kChunkK / 8)) % kMmaThreads == 0,
              "a chunk is whole groups and splits evenly into 16-byte units per thread");
static_assert(kMmaSmem <= 232448, "shared memory per block");
static_assert(kStageBytes % 128 == 0 && kBoxBytes % 128 == 0 && kScaleBytes % 128 == 0,
              "TMA destinations must stay 128-byte aligned");

struct W4MmaArgs {
    int G;
    const int32_t* rows;      // [G] device, or nullptr for uniform rows
    const int32_t* row_off;   // [G] device, or nullptr
    int uniform_rows;
    int64_t a_stride, c_stride;
    const __nv_bfloat16* A;
    int K;
    int J;
    const float* row_scale;   // down: per output row, nullable
    __nv_bfloat16* C;         // [*, J]
    int32_t* err;
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

// Two nibbles n of w (bits 0-3 and 16-19, two's complement codes q) as the bf16 pair
// (q_lo + 136, q_hi + 136): 0x4300 | (n ^ 8) is 128 + (q + 8), exact.
__device__ __forceinline__ uint32_t nib_pair(uint32_t w) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(w), "r"(0x000F000Fu), "r"(0x43084308u));
    return r;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// NM = 2: box 0 = gate rows, box 1 = up rows of 32 features (FPW 32); NM = 1: 64 down rows.
template <int NM>
__global__ void __launch_bounds__(kMmaThreads, MOE_W4_MINBLOCKS)
w4_mma_kernel(const __grid_constant__ CUtensorMap tmQ0, const __grid_constant__ CUtensorMap tmQ1,
              const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
              const W4MmaArgs a) {
    using namespace tc;
    constexpr int FPW = NM == 2 ? kBoxRows : 2 * kBoxRows;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~(uintptr_t)1023);
    const int gi = blockIdx.y;
    const int rows = a.rows ? a.rows[gi] : a.uniform_rows;
    if (rows <= (int)blockIdx.z * kTokTile) return;          // uniform over the block
    const int64_t a_row0 = a.rows ? a.row_off[gi] : (int64_t)gi * a.a_stride;
    const int64_t c_row0 = a.rows ? a.row_off[gi] : (int64_t)gi * a.c_stride;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int j0 = (blockIdx.x * kMmaWarps + warp) * FPW;
    const bool active = j0 < a.J;
    const int groups = a.K / kW4Group;
    // this block's passes of kTokTile token rows: z, z + Z, z + 2Z, ... (Z = gridDim.z)
    const int zp = (int)blockIdx.z, Z = (int)gridDim.z;
    const int all_passes = (rows + kTokTile - 1) / kTokTile;
    const int passes = all_passes > zp ? (all_passes - zp + Z - 1) / Z : 0;
    const int total = passes * groups;                       // ring items per warp

    uint8_t* ring = smem + (size_t)warp * kStages * kStageBytes;
    uint8_t* xfrag = smem + kRingBytes;
    float* xsum = reinterpret_cast<float*>(smem + kRingBytes + kXfragBytes);     // [group][token]
    uint64_t* full =
        reinterpret_cast<uint64_t*>(smem + kRingBytes + kXfragBytes + kXsumBytes) + warp * kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(
        smem + kRingBytes + kXfragBytes + kXsumBytes + kMmaWarps * kStages * 8);

    if (lane == 0)
        for (int st = 0; st < kStages; st++) mbar_init(&full[st], 1);
    // a block that already gave up on a wait makes the rest of the grid return at once
    if (threadIdx.x == 0)
        *abort_flag = (*reinterpret_cast<volatile int32_t*>(a.err) & MOE_DEVERR_TIMEOUT) ? 1 : 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    if (*abort_flag) return;                                 // uniform: read after the barrier

    // box 0 rows: gate or the first 32 down rows; box 1: up rows or the next 32 down rows
    const int64_t wrow0 = (int64_t)gi * a.J + j0;
    const int64_t wrow1 = NM == 2 ? wrow0 : wrow0 + kBoxRows;
    // Ring item q (group q % groups of its pass) is four TMA boxes, one per lane 0..3, after
    // lane 0 has armed the stage's barrier with the byte count.  Every lane tracks the counters.
    int issued = 0, igrp = 0;
    const CUtensorMap* my_map = lane == 0 ? &tmQ0 : lane == 1 ? (NM == 2 ? &tmQ1 : &tmQ0)
                              : lane == 2 ? &tmS0 : (NM == 2 ? &tmS1 : &tmS0);
    const uint32_t my_off = lane == 0 ? 0u : lane == 1 ? (uint32_t)kBoxBytes
                          : lane == 2 ? 2u * kBoxBytes : 2u * kBoxBytes + kScaleBytes;
    const int32_t my_row = (int32_t)(lane == 0 || lane == 2 ? wrow0 : wrow1);
    auto issue = [&]() {                                     // called by all lanes
        const int st = issued % kStages;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], kStageTx);
        __syncwarp();
        if (lane < 4) {
            const uint32_t dst = smem_u32(ring + st * kStageBytes) + my_off;
            if (lane < 2)
                tma_load_2d(dst, my_map, &full[st], igrp * kGroupBytes, my_row);
            else
                tma_load_2d(dst, my_map, &full[st], my_row, igrp);
        }
        ++issued;
        if (++igrp == groups) igrp = 0;
    };
    if (active) {
        if (lane < 4) prefetch_tmap(my_map);
        while (issued < kStages && issued < total) issue();
    }

    bool ok = true;        // this warp's waits all succeeded
    bool stop = false;     // block-uniform: some warp gave up; read only right after a barrier
    int q = 0;

    // x rows of a chunk, 16 bytes per unit (token n, 8 inputs)
    uint4 xr[kUnitsPerThread];
    auto load_chunk = [&](int p0n, int k0n) {
        const int Tn = min(kTokTile, rows - p0n);
        const int blocks8 = min(kChunkK, a.K - k0n) / 8;
#pragma unroll
        for (int i = 0; i < kUnitsPerThread; i++) {
            const int u = threadIdx.x + i * kMmaThreads;
            const int n = u / blocks8, e8 = u % blocks8;
            xr[i] = make_uint4(0u, 0u, 0u, 0u);
            if (u < kTokTile * blocks8 && n < Tn)
                xr[i] = __ldg(reinterpret_cast<const uint4*>(a.A + (a_row0 + p0n + n) * a.K + k0n +
                                                            e8 * 8));
        }
    };
    // B fragments.  The 16 units of one (token, group) are 16 aligned lanes of one warp, and a
    // warp is wholly inside or wholly past the unit range (a chunk is a multiple of 128
    // inputs), so the shuffles below always see full warps.
    auto store_chunk = [&](int kc) {
        const int blocks8 = kc / 8;
#pragma unroll
        for (int i = 0; i < kUnitsPerThread; i++) {
            const int u = threadIdx.x + i * kMmaThreads;
            if (u >= kTokTile * blocks8) break;
            const int n = u / blocks8, e8 = u % blocks8;
            const uint4 v = xr[i];
            const int gl = e8 >> 4, t = (e8 >> 2) & 3, m = e8 & 3;
            const uint32_t dst = smem_u32(xfrag) + (((gl * 4 + m) * 32 + n * 4 + t) << 4);
            st_shared_v4(dst, __byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                         __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
            float part = 0.f;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vw[c]));
                part += f.x + f.y;
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if ((lane & 15) == 0) xsum[gl * kTokTile + n] = part;
        }
    };
    if (MOE_W4_PREFETCH_X && passes > 0) load_chunk(zp * kTokTile, 0);

    // thread's code rows within a box: tile m covers box m / 2, rows (m % 2) * 16 + g (+ 8)
    const uint32_t row_off_b = (uint32_t)(gq * kGroupBytes + tq * 16);
    for (int pass = 0; pass < passes; pass++) {
        const int p0 = (zp + pass * Z) * kTokTile;
        float acc[kTiles][4];
#pragma unroll
        for (int m = 0; m < kTiles; m++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[m][i] = 0.f;

        for (int k0 = 0; k0 < a.K; k0 += kChunkK) {
            const int kc = min(kChunkK, a.K - k0);
            __syncthreads();                                 // fragments of the last chunk read
            if (*abort_flag) {
                stop = true;
                break;
            }
            if (!MOE_W4_PREFETCH_X) load_chunk(p0, k0);
            store_chunk(kc);
            __syncthreads();
            if (MOE_W4_PREFETCH_X) {
                if (k0 + kChunkK < a.K) load_chunk(p0, k0 + kChunkK);
                else if (pass + 1 < passes) load_chunk(p0 + Z * kTokTile, 0);
            }
            if (!active || !ok) continue;

            const int ng = kc / kW4Group;
            for (int gl = 0; gl < ng; gl++, q++) {
                const int st = q % kStages;
                if (!waitw(&full[st], (uint32_t)((q / kStages) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = smem_u32(ring + st * kStageBytes);
                uint4 c[kTiles][2];                          // [tile][row g, row g + 8]
#pragma unroll
                for (int m = 0; m < kTiles; m++) {
                    const uint32_t base = sb + (m >> 1) * kBoxBytes + (m & 1) * kTileRows * kGroupBytes + row_off_b;
                    c[m][0] = lds128(base);
                    c[m][1] = lds128(base + 8 * kGroupBytes);
                }
                const float* scp = reinterpret_cast<const float*>(ring + st * kStageBytes + 2 * kBoxBytes);
                float sa[kTiles], sbv[kTiles];               // scales of rows g and g + 8
#pragma unroll
                for (int m = 0; m < kTiles; m++) {
                    const int r = (m >> 1) * kBoxRows + (m & 1) * kTileRows + gq;
                    sa[m] = scp[r];
                    sbv[m] = scp[r + 8];
                }
                __syncwarp();
                if (issued < total) {
                    fence_proxy_async_smem();
                    issue();
                }
                const uint32_t xb = smem_u32(xfrag) + ((gl * 4 * 32 + lane) << 4);
                float d[kTiles][4];
#pragma unroll
                for (int m = 0; m < kTiles; m++)
#pragma unroll
                    for (int i = 0; i < 4; i++) d[m][i] = 0.f;
#pragma unroll
                for (int j = 0; j < 4; j++) {                // code word j: steps 2j, 2j+1
                    const uint4 b = lds128(xb + j * 32 * 16);
#pragma unroll
                    for (int h = 0; h < 2; h++) {            // step 2j + h: shifts 8h, 8h + 4
                        const int sl = 8 * h, sh = 8 * h + 4;
                        const uint32_t b0 = h ? b.z : b.x, b1 = h ? b.w : b.y;
#pragma unroll
                        for (int m = 0; m < kTiles; m++) {
                            const uint32_t w0 = word(c[m][0], j), w1 = word(c[m][1], j);
                            mma_bf16_16816(d[m], nib_pair(w0 >> sl), nib_pair(w1 >> sl),
                                           nib_pair(w0 >> sh), nib_pair(w1 >> sh), b0, b1);
                        }
                    }
                }
                // D = sum (q + 136) x over the group: subtract 136 X per token column
                const float2 xs = *reinterpret_cast<const float2*>(xsum + gl * kTokTile + 2 * tq);
                const float cx0 = 136.f * xs.x, cx1 = 136.f * xs.y;
#pragma unroll
                for (int m = 0; m < kTiles; m++) {
                    acc[m][0] = fmaf(sa[m], d[m][0] - cx0, acc[m][0]);
                    acc[m][1] = fmaf(sa[m], d[m][1] - cx1, acc[m][1]);
                    acc[m][2] = fmaf(sbv[m], d[m][2] - cx0, acc[m][2]);
                    acc[m][3] = fmaf(sbv[m], d[m][3] - cx1, acc[m][3]);
                }
            }
            if (!ok) *abort_flag = 1;
        }
        if (stop) break;
        if (!ok || !active) continue;
        const int T = min(kTokTile, rows - p0);
        // ---- epilogue: thread holds rows (g, g+8) x tokens (2t, 2t+1) of every tile
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int r = gq + (i >> 1) * 8, n = 2 * tq + (i & 1);
            if (n >= T) continue;
            const int64_t crow = c_row0 + p0 + n;
            __nv_bfloat16* out = a.C + crow * a.J + j0 + r;
            if (NM == 2) {                                   // tiles 0, 1 gate; 2, 3 up
                out[0] = __float2bfloat16_rn(silu(acc[0][i]) * acc[2][i]);
                out[kTileRows] = __float2bfloat16_rn(silu(acc[1][i]) * acc[3][i]);
            } else {
                const float sc = a.row_scale ? a.row_scale[crow] : 1.f;
#pragma unroll
                for (int m = 0; m < kTiles; m++) out[m * kTileRows] = __float2bfloat16_rn(acc[m][i] * sc);
            }
        }
    }
    if (!ok || stop) {
        // let every copy this warp issued land before the block can exit
        if (active && lane == 0)
            for (int r = q; r < issued; r++)   // issued and q are the same on every lane
                wait1(&full[r % kStages], (uint32_t)((r / kStages) & 1), abort_flag,
                      kDrainTimeoutNs, false);
        if (threadIdx.x == 0) atomicOr(a.err, MOE_DEVERR_TIMEOUT);
    }
}

// 2-D map over packed codes [rows, K/2] bytes, box = 32 rows x 64 bytes (one group), no swizzle.
bool make_code_map(CUtensorMap* m, const uint8_t* q, int64_t rows, int K) {
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn || rows <= 0 || K <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {(cuuint32_t)kGroupBytes, (cuuint32_t)kBoxRows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Blocks along z split a group's token passes: enough to fill the GPU when there are few
// groups with many rows (shared experts), 1 for routed decode groups of a few rows each.
int w4_z_split(const W4Group& g, int J, int per_block, int64_t total_rows) {
    const int64_t avg_rows = g.G > 0 ? total_rows / g.G : 0;
    const int64_t passes = (avg_rows + kTokTile - 1) / kTokTile;
    const int64_t blocks_xy = (int64_t)g.G * ((J + per_block - 1) / per_block);
    const int64_t want = (2 * (int64_t)device_sm_count() + blocks_xy - 1) / blocks_xy;
    int64_t z = passes < want ? passes : want;
    return (int)(z < 1 ? 1 : (z > 64 ? 64 : z));
}

// 2-D map over group-major scales [K/128, rows] fp32, box = 32 rows of one group.
bool make_scale_map(CUtensorMap* m, const float* sc, int64_t rows, int K) {
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn || rows <= 0 || K <= 0 || rows % 4) return false;
    cuuint64_t dims[2] = {(cuuint64_t)rows, (cuuint64_t)(K / kW4Group)};
    cuuint64_t strides[1] = {(cuuint64_t)rows * 4};
    cuuint32_t box[2] = {(cuuint32_t)kBoxRows, 1u};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(sc), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NM>
cudaError_t launch_w4mma(const W4Group& g, const __nv_bfloat16* A, int K, const W4Mat& M0,
                         const W4Mat& M1, int J, const float* row_scale, __nv_bfloat16* C,
                         int32_t* err, int64_t total_rows, cudaStream_t s) {
    constexpr int FPW = NM == 2 ? kBoxRows : 2 * kBoxRows;
    if (g.G <= 0 || J <= 0) return cudaSuccess;
    const int z_split = w4_z_split(g, J, kMmaWarps * FPW, total_rows);
    if (K % kW4Group || J % FPW) return cudaErrorInvalidValue;
    const int64_t wrows = (int64_t)g.G * J;
    CUtensorMap m0, m1, s0, s1;
    if (!make_code_map(&m0, M0.q, wrows, K) || !make_code_map(&m1, NM == 2 ? M1.q : M0.q, wrows, K) ||
        !make_scale_map(&s0, M0.s, wrows, K) || !make_scale_map(&s1, NM == 2 ? M1.s : M0.s, wrows, K))
        return cudaErrorInvalidValue;
    // the shared-memory opt-in is per device: remember it per device
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_relaxed)) {
        cudaError_t e = cudaFuncSetAttribute(w4_mma_kernel<NM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_relaxed);
    }
    W4MmaArgs a{g.G, g.rows, g.row_off, g.uniform_rows, g.a_stride, g.c_stride, A, K,
                J, row_scale, C, err};
    const int per_block = kMmaWarps * FPW;
    dim3 grid((unsigned)((J + per_block - 1) / per_block), (unsigned)g.G, (unsigned)z_split);
    w4_mma_kernel<NM><<<grid, kMmaThreads, kMmaSmem, s>>>(m0, m1, s0, s1, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t w4_quantize(const __nv_bfloat16* W, int64_t rows, int cols, uint8_t* q, float* s,
                        cudaStream_t st) {
    const int64_t units = rows * (cols / kW4Group);
    if (units <= 0) return cudaSuccess;
    int64_t blocks = (units + kWarps - 1) / kWarps;
    if (blocks > 148 * 64) blocks = 148 * 64;
    w4_quantize_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(W, rows, cols, q, s);
    return cudaGetLastError();
}

cudaError_t w4_gateup(const W4Group& g, const __nv_bfloat16* A, int K, const W4Mat& Wg,
                      const W4Mat& Wu, int F, __nv_bfloat16* H, int32_t* err, int64_t total_rows,
                      cudaStream_t s) {
    return launch_w4mma<2>(g, A, K, Wg, Wu, F, nullptr, H, err, total_rows, s);
}

cudaError_t w4_down(const W4Group& g, const __nv_bfloat16* H, int F, const W4Mat& Wd, int D,
                    const float* row_scale, __nv_bfloat16* Y, int32_t* err, int64_t total_rows,
                    cudaStream_t s) {
    return launch_w4mma<1>(g, H, F, Wd, Wd, D, row_scale, Y, err, total_rows, s);
}

}  // namespace moe
