// tc_ptx.cuh -- inline-PTX wrappers for the tcgen05 / TMA / mbarrier kernels (sm_103a), the
// bounded mbarrier waits they use, and host-side TMA tensor-map encoding.
#pragma once

#include <cuda.h>

#include "moe_internal.cuh"

namespace moe {
namespace tc {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s per wait
constexpr uint64_t kDrainTimeoutNs = 100000000ull;   // 100 ms

// ---------------------------------------------------------------- PTX wrappers

static __device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
static __device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
static __device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
static __device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
static __device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
static __device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
static __device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
static __device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
static __device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
static __device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
static __device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
static __device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
static __device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, cta_group::1.
static __device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on an mbarrier once every tcgen05 op issued so far by this thread has completed.
static __device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
static __device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
static __device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- TMA stores

// Shared -> global tile store, tracked by the issuing thread's bulk groups.
static __device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                                    int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(src)
                 : "memory");
}
// L2 eviction policies for cache hints.
static __device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
static __device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
static __device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src,
                                                         int32_t c0, int32_t c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::
            "l"(reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(src), "l"(policy)
        : "memory");
}
static __device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map,
                                                        uint64_t* bar, int32_t c0, int32_t c1,
                                                        uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
static __device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups still read their shared-memory source.
template <int N>
static __device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
static __device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
static __device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
static __device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                                    uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// One epilogue warp writes its 32 rows x 32 bf16 columns (lane = row, pk = the row's 16 packed
// pairs).  A chunk whose 32 rows all belong to the group goes through the warp's 2 KB staging
// buffer (64-byte rows, 64-byte swizzle: conflict-free 16-byte stores) and one TMA store of
// whole lines; a chunk that crosses the end of the group is written row by row for its valid
// rows only, so rows of the next group are never touched.  Columns past n_out are clipped (TMA)
// or skipped (direct).  The warp alternates between two buffers; the TMA store that used a
// buffer two chunks ago must have finished reading it.
static __device__ __forceinline__ void store_chunk32(const CUtensorMap* tmC, uint32_t buf,
                                                     const uint32_t (&pk)[16], bool all_valid,
                                                     bool valid, __nv_bfloat16* dst, int col,
                                                     int n_out, int32_t gy) {
    const int lane = threadIdx.x & 31;
    if (all_valid) {
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        const uint32_t rowb = buf + (uint32_t)lane * 64u;
        const uint32_t sw = ((uint32_t)lane >> 1) & 3u;
#pragma unroll
        for (int v = 0; v < 4; v++)
            st_shared_v4(rowb + (((uint32_t)v ^ sw) << 4), pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                         pk[4 * v + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {   // the output is read once, later: keep it from evicting operands
            tma_store_2d_hint(tmC, buf, col, gy, policy_evict_first());
            bulk_commit();
        }
    } else if (valid) {
#pragma unroll
        for (int v = 0; v < 4; v++)
            if (col + v * 8 + 8 <= n_out)
                *reinterpret_cast<uint4*>(dst + v * 8) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
}

static __device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Transposed form of store_chunk32 for tiles computed with the operands swapped: lane = output
// column (col + lane), v[j] = the value of row gy + j.  The warp writes the same 32 x 32 block
// as store_chunk32: whole (nrows >= 32) through the staging buffer in its 64-byte-swizzled
// layout and one TMA store, otherwise the first nrows rows with 2-byte stores (a warp covers
// 64 contiguous bytes of one row per store); col_ok says whether this lane's column is < n_out.
static __device__ __forceinline__ void store_chunk32_t(const CUtensorMap* tmC, uint32_t buf,
                                                       const float (&v)[32], int nrows,
                                                       __nv_bfloat16* dst, int64_t ldc, bool col_ok,
                                                       int col, int32_t gy) {
    const int lane = threadIdx.x & 31;
    if (nrows >= 32) {
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        const uint32_t ch = (uint32_t)lane >> 3, cb = ((uint32_t)lane & 7u) * 2u;
#pragma unroll
        for (int j = 0; j < 32; j++) {
            const __nv_bfloat16 b = __float2bfloat16_rn(v[j]);
            st_shared_u16(buf + (uint32_t)j * 64u + ((ch ^ (((uint32_t)j >> 1) & 3u)) << 4) + cb,
                          *reinterpret_cast<const uint16_t*>(&b));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d_hint(tmC, buf, col, gy, policy_evict_first());
            bulk_commit();
        }
    } else if (col_ok) {
#pragma unroll
        for (int j = 0; j < 32; j++)
            if (j < nrows) dst[(int64_t)j * ldc] = __float2bfloat16_rn(v[j]);
    }
}

// ---------------------------------------------------------------- tile order inside a group

// Tile `local` of a group with mtg m-tiles and nt n-tiles -> (m-tile, n-tile).  m-tiles run in
// blocks of kMBlock: inside a block the m-tiles are innermost (CTAs working together share one
// weight tile through L2) and the block's n-tiles come one after another, so an A panel of
// kMBlock m-tiles stays in L2 while all n-tiles sweep it.  Groups with at most kMBlock m-tiles
// keep the plain m-innermost order.
constexpr int kMBlock = 16;
static __device__ __forceinline__ void raster_tile(int local, int mtg, int ntiles, int& mt, int& nt) {
    const int full = mtg / kMBlock;
    const int per_block = kMBlock * ntiles;
    const int mb = local / per_block;
    if (mb < full) {
        const int w = local - mb * per_block;
        nt = w / kMBlock;
        mt = mb * kMBlock + w % kMBlock;
    } else {
        const int rem = mtg - full * kMBlock;
        const int w = local - full * per_block;
        nt = w / rem;
        mt = full * kMBlock + w % rem;
    }
}

// ---------------------------------------------------------------- CTA pairs (cta_group::2)

static __device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of this cluster
static __device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
static __device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// Arrive on an mbarrier given by its shared::cluster address (own or peer CTA).
// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address) with no memory
// ordering, for a signal that orders nothing but tcgen05 work the caller has already waited for.
// The accumulator hand-back is one: the epilogue's tcgen05.ld have completed (tcgen05.wait::ld)
// and been fenced (tcgen05.fence::before_thread_sync), so the MMAs that follow the wait cannot
// touch data still being read.  A release at cluster scope would in addition wait until the
// warp's earlier output stores are visible cluster-wide, which was measured at 2-3 thousand
// cycles per tile while the rings stream, half the epilogue's time on short tiles.
static __device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an mbarrier that may
// live in the peer CTA (the pair's leader); bar_cluster is a shared::cluster address.
static __device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                        uint32_t bar_cluster, int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
// The same with an L2 eviction policy for the loaded lines.
static __device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map,
                                                             uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                             uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster), "l"(policy)
        : "memory");
}
static __device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
static __device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
static __device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D (M=256 over the pair) (+)= A (each CTA its 128 rows) * B (each CTA half of N)^T.
static __device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                      uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the mbarrier at this offset in every CTA of cta_mask once the pair's MMAs issued so
// far by this thread have completed.
static __device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row core-matrix groups 1024 bytes apart (stride byte offset), tile base 1024-aligned.
static __device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);       // start address >> 4      [0,14)
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset >> 4 [32,46)
    d |= (uint64_t)1 << 46;                          // descriptor version 0b001 [46,49)
    d |= (uint64_t)2 << 61;                          // layout: 128-byte swizzle [61,64)
    return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M x N.
static __host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- bounded waits

// One thread.  false when the abort flag is up (if honoured) or the wait timed out.
static __device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                      uint64_t timeout_ns, bool honour_abort) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = gtimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; i++)
            if (mbar_try_wait(a, parity)) return true;
        if (honour_abort && *abort_flag) return false;
        if (gtimer() - t0 > timeout_ns) {
            *abort_flag = 1;
            return false;
        }
    }
}

// elect.sync over the full warp: true on exactly one lane (the same lane while the warp is
// converged).  Measured on B300: a loop that waits on an mbarrier and then issues tcgen05.mma
// from one lane chosen by this instruction, with the whole warp running the loop, issues at the
// tensor rate; the same loop run by one thread (or with a `lane == 0` test) spends ~100 cycles
// per MMA and holds MMAs of N < 200 well below the tensor rate.
static __device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Whole warp, convergent; every lane returns the same answer.
static __device__ __forceinline__ bool waitw(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t timeout_ns = kWaitTimeoutNs) {
    const uint32_t a = smem_u32(bar);
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        bool ok = mbar_try_wait(a, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((it & 63) == 63) {
            int stop = 0;
            if (lane == 0) {
                uint64_t now = gtimer();
                if (t0 == 0) t0 = now;
                stop = (*abort_flag != 0) || (now - t0 > timeout_ns);
                if (stop) *abort_flag = 1;
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        }
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D bf16 map over a row-major [rows, cols] matrix, box = box_rows x 64 columns, 128B swizzle.
inline bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows <= 0 || cols <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};   // 64 bf16 = one 128-byte swizzle row
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map for epilogue stores: box = 32 rows x 32 columns (64-byte rows, 64-byte swizzle).
inline bool make_store_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows <= 0 || cols <= 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace moe
