// moe_api.cu -- the C ABI of libmoe.so: argument validation, workspace layout and the order of
// launches for each entry point declared in include/moe.h.
#include <atomic>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <unordered_map>

#include <nvtx3/nvToolsExt.h>

#include "bwd_internal.cuh"

namespace moe {

// NVTX range over a host-side scope (an entry point or a phase of the forward), for timeline
// tools; a no-op unless a profiler has injected its NVTX handler.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

int device_sm_count() {
    static std::atomic<int> cached[64];       // per device; 0 until first asked
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// The bf16 forward's grouped GEMMs run on the CTA-pair kernels of grouped_gemm_pair.cu;
// MOE_GROUPED_GEMM=single (read once per process) selects the single-CTA kernels of
// grouped_gemm_tc.cu instead, for comparisons.
bool use_pair_gemm() {
    static int enabled = -1;
    if (enabled < 0) {
        const char* e = getenv("MOE_GROUPED_GEMM");
        enabled = (e && strcmp(e, "single") == 0) ? 0 : 1;
    }
    return enabled == 1;
}

int64_t capacity(const moe_cfg& c) {
    if (!(c.capacity_factor > 0.f)) return -1;
    return (int64_t)ceil(c.capacity_factor * (double)c.N * (double)c.k / (double)c.E);
}

int64_t grouped_rows(const moe_cfg& c) {
    const int64_t A = c.N * c.k;
    const int64_t cap = capacity(c);
    if (cap < 0) return A;
    const int64_t lim = cap * c.E;
    return lim < A ? lim : A;
}

static size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

WsLayout ws_layout(const moe_cfg& c) {
    WsLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += up256(bytes ? bytes : 1);
        return o;
    };
    const int64_t N = c.N, E = c.E, A = c.N * c.k, R = grouped_rows(c);
    const int64_t S = c.n_shared, F = c.d_ff, Fs = c.d_ff_shared, d = c.d;
    const size_t esz = c.act_dtype == MOE_BF16 ? 2 : 4;
    L.err = take(256);
    L.p_part = take(4 * (size_t)router_part_rows(N) * E);
    const bool tc_router = router_uses_tensor_cores(c);
    L.router_w3 = take(tc_router ? 2 * 3 * (size_t)E * d : 0);
    L.logits = take(tc_router ? 4 * router_tc_logits_floats(N, (int)d, (int)E) : 0);
    L.blk_hist = take(4 * (size_t)perm_blocks(A) * E);
    L.blk_base = take(4 * (size_t)perm_blocks(A) * E);
    L.mtile_off = take(4 * (size_t)(E + 1));
    L.stats_f = take(4 * (size_t)(2 * E + 8));
    L.idx = take(4 * (size_t)A);
    L.w = take(4 * (size_t)A);
    L.gap = take(4 * (size_t)N);
    L.lse = take(4 * (size_t)N);
    L.rstat = take(8 * (size_t)(kRouterStatBlocks + E));
    L.P_sum = take(4 * (size_t)E);
    L.counts = take(4 * (size_t)E);
    L.offsets = take(4 * (size_t)(E + 1));
    L.kept = take(4 * (size_t)E);
    L.kept_offsets = take(4 * (size_t)(E + 1));
    L.perm = take(4 * (size_t)A);
    L.pos = take(4 * (size_t)A);
    L.row_token = take(4 * (size_t)R);
    L.row_weight = take(4 * (size_t)R);
    L.x_perm = take(esz * (size_t)R * d);
    L.h_perm = take(esz * (size_t)R * F);
    L.y_perm = take(esz * (size_t)R * d);
    L.h_sh = take(esz * (size_t)(S * N) * Fs);
    L.y_sh = take(esz * (size_t)(S * N) * d);
    L.total = off;
    return L;
}

}  // namespace moe

using namespace moe;

namespace {

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status check_cfg(const moe_cfg* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->N < 0 || c->d <= 0 || c->d_ff <= 0 || c->E <= 0 || c->k <= 0 || c->n_shared < 0)
        return MOE_ERR_INVALID_ARG;
    if (c->k > c->E) return MOE_ERR_INVALID_ARG;
    if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->renorm != 0 && c->renorm != 1) return MOE_ERR_INVALID_ARG;
    if (c->bias_mode < 0 || c->bias_mode > 2) return MOE_ERR_INVALID_ARG;
    if (c->n_shared > 0 && c->d_ff_shared <= 0) return MOE_ERR_INVALID_ARG;
    const int mult = c->act_dtype == MOE_BF16 ? 8 : 4;   // 16-byte rows
    if (c->d % mult || c->d_ff % mult || (c->n_shared > 0 && c->d_ff_shared % mult))
        return MOE_ERR_INVALID_ARG;
    if (isnan(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
    if (c->E > 1024 || c->k > 16 || c->n_shared > 8) return MOE_ERR_UNSUPPORTED;
    if (c->N * (int64_t)c->k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    if (grouped_rows(*c) * (int64_t)(c->d > c->d_ff ? c->d : c->d_ff) >= ((int64_t)1 << 40))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status check_ws(const moe_cfg* c, void* ws, size_t ws_bytes) {
    if (!ws || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(*c).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                         \
    do {                                      \
        moe_status _s = (expr);               \
        if (_s != MOE_OK) return _s;          \
    } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

moe_status need(const void* p, size_t align) {
    if (!p) return MOE_ERR_INVALID_ARG;
    return aligned(p, align) ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// --------------------------------------------------------------------- shared pieces

moe_status do_grouped_ffn(const moe_cfg* c, const void* x_perm, const int32_t* kept,
                          const int32_t* kept_offsets, const float* row_weight, const void* Wg,
                          const void* Wu, const void* Wd, void* y_perm, void* ws,
                          cudaStream_t s, void* const* ev) {
    const WsLayout L = ws_layout(*c);
    int32_t* err = at<int32_t>(ws, L.err);
    int32_t* mtile = at<int32_t>(ws, L.mtile_off);
    const int64_t R = grouped_rows(*c);
    const bool bf16 = c->act_dtype == MOE_BF16;
    const bool pair_gemm = bf16 && use_pair_gemm();
    // no group holds more rows than tokens (top-k picks distinct experts) or than the capacity
    const int64_t cap = capacity(*c);
    const int64_t max_group_rows = cap >= 0 && cap < c->N ? cap : c->N;
    GroupGeom g{};
    g.G = c->E;
    g.rows = kept;
    g.row_off = kept_offsets;
    g.mtile_off = mtile;
    g.max_rows = R;
    const int bm = pair_gemm ? pair_chunk_rows() : bf16 ? kTcBlockRows : simt_block_rows();
    g.zigzag = pair_gemm;
    MOE_CUDA(launch_plan_mtiles(kept, c->E, bm, mtile, s, g.zigzag));
    void* h = at<void>(ws, L.h_perm);
    if (pair_gemm) {
        MOE_CUDA(pair_gateup(g, (const __nv_bfloat16*)x_perm, R, c->d, (const __nv_bfloat16*)Wg,
                             (const __nv_bfloat16*)Wu, c->d_ff, (__nv_bfloat16*)h, R, err,
                             max_group_rows, s));
    } else if (bf16) {
        MOE_CUDA(tc_gateup(g, (const __nv_bfloat16*)x_perm, R, c->d, (const __nv_bfloat16*)Wg,
                           (const __nv_bfloat16*)Wu, c->d_ff, (__nv_bfloat16*)h, R, err, s));
    } else {
        MOE_CUDA(simt_gateup_f32(g, (const float*)x_perm, c->d, (const float*)Wg,
                                 (const float*)Wu, c->d_ff, (float*)h, s));
    }
    if (ev && ev[3]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[3], s));
    if (pair_gemm) {
        MOE_CUDA(pair_down(g, (const __nv_bfloat16*)h, R, c->d_ff, (const __nv_bfloat16*)Wd, c->d,
                           row_weight, (__nv_bfloat16*)y_perm, R, err, max_group_rows, s));
    } else if (bf16) {
        MOE_CUDA(tc_down(g, (const __nv_bfloat16*)h, R, c->d_ff, (const __nv_bfloat16*)Wd, c->d,
                         row_weight, (__nv_bfloat16*)y_perm, R, err, s));
    } else {
        MOE_CUDA(simt_down_f32(g, (const float*)h, c->d_ff, (const float*)Wd, c->d, row_weight,
                               (float*)y_perm, s));
    }
    if (ev && ev[4]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[4], s));
    return MOE_OK;
}

// The shared experts: Ysh = SwiGLU_s(x) for every token, into the workspace.
moe_status do_shared(const moe_cfg* c, const void* x, const void* Wsg, const void* Wsu,
                     const void* Wsd, void* ws, cudaStream_t s) {
    const WsLayout L = ws_layout(*c);
    int32_t* err = at<int32_t>(ws, L.err);
    void* hsh = at<void>(ws, L.h_sh);
    void* ysh = at<void>(ws, L.y_sh);
    const int S = c->n_shared, Fs = c->d_ff_shared;
    if (S > 0 && c->N > 0) {
        GroupGeom g{};
        g.G = S;
        g.uniform_rows = (int)c->N;
        g.max_rows = c->N;
        if (c->act_dtype == MOE_BF16 && use_pair_gemm()) {
            g.a_stride = 0;        // every shared expert reads all tokens of x
            g.c_stride = c->N;
            MOE_CUDA(pair_gateup(g, (const __nv_bfloat16*)x, c->N, c->d, (const __nv_bfloat16*)Wsg,
                                 (const __nv_bfloat16*)Wsu, Fs, (__nv_bfloat16*)hsh, S * c->N, err,
                                 c->N, s));
            g.a_stride = c->N;
            MOE_CUDA(pair_down(g, (const __nv_bfloat16*)hsh, S * c->N, Fs, (const __nv_bfloat16*)Wsd,
                               c->d, nullptr, (__nv_bfloat16*)ysh, S * c->N, err, c->N, s));
        } else if (c->act_dtype == MOE_BF16) {
            g.a_stride = 0;        // every shared expert reads all tokens of x
            g.c_stride = c->N;
            MOE_CUDA(tc_gateup(g, (const __nv_bfloat16*)x, c->N, c->d, (const __nv_bfloat16*)Wsg,
                               (const __nv_bfloat16*)Wsu, Fs, (__nv_bfloat16*)hsh, S * c->N, err, s));
            g.a_stride = c->N;
            MOE_CUDA(tc_down(g, (const __nv_bfloat16*)hsh, S * c->N, Fs, (const __nv_bfloat16*)Wsd,
                             c->d, nullptr, (__nv_bfloat16*)ysh, S * c->N, err, s));
        } else {
            g.a_stride = 0;
            g.c_stride = c->N;
            MOE_CUDA(simt_gateup_f32(g, (const float*)x, c->d, (const float*)Wsg, (const float*)Wsu,
                                     Fs, (float*)hsh, s));
            g.a_stride = c->N;
            MOE_CUDA(simt_down_f32(g, (const float*)hsh, Fs, (const float*)Wsd, c->d, nullptr,
                                   (float*)ysh, s));
        }
    }
    return MOE_OK;
}

// Shared experts (unless already run on the side stream) and the combine, on s.
moe_status do_shared_and_combine(const moe_cfg* c, const void* y_perm, const int32_t* pos,
                                 const void* x, const void* Wsg, const void* Wsu, const void* Wsd,
                                 void* out, void* ws, cudaStream_t s, void* const* ev,
                                 bool shared_done = false) {
    const WsLayout L = ws_layout(*c);
    if (!shared_done) MOE_TRY(do_shared(c, x, Wsg, Wsu, Wsd, ws, s));
    if (ev && ev[5]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[5], s));
    MOE_CUDA(launch_combine(*c, y_perm, pos, at<void>(ws, L.y_sh), out, at<int32_t>(ws, L.err), s));
    if (ev && ev[6]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[6], s));
    return MOE_OK;
}

// ------------------------------------------------------------------ prepared router splits
//
// moe_router_prepare records, per workspace, the W_r pointer (and E, d) whose exact bf16 split
// sits in the workspace; forwards and routes that pass the same pointer skip the split.
struct PreparedSplit {
    const float* W_r;
    int E, d;
};
std::mutex g_prepared_mu;
std::unordered_map<uintptr_t, PreparedSplit> g_prepared;

bool split_prepared(const moe_cfg& c, const float* W_r, const void* ws) {
    std::lock_guard<std::mutex> lock(g_prepared_mu);
    auto it = g_prepared.find(reinterpret_cast<uintptr_t>(ws));
    return it != g_prepared.end() && it->second.W_r == W_r && it->second.E == c.E &&
           it->second.d == c.d;
}
void forget_prepared(const void* ws) {
    std::lock_guard<std::mutex> lock(g_prepared_mu);
    g_prepared.erase(reinterpret_cast<uintptr_t>(ws));
}

// ------------------------------------------------------------------ side stream
//
// For a decode-sized batch the shared experts are a handful of tiles that would run alone with
// most SMs idle; they depend only on x, so they are forked onto a library-owned stream at the
// start of the forward and joined before the combine, overlapping the router, the permutation
// and the routed experts.  Larger batches keep them in line (their GEMMs fill the GPU).
// The side stream belongs to the calling thread (one per device and host thread, created on its
// first decode-sized forward and kept until the process exits), so forwards from different
// threads never meet on it: neither do they serialise there, nor does one thread's stream
// capture pull in another thread's shared-expert work.
constexpr int64_t kSideStreamMaxTokens = 128;

bool fork_shared(const moe_cfg& c) {
    return c.act_dtype == MOE_BF16 && c.n_shared > 0 && c.N > 0 && c.N <= kSideStreamMaxTokens;
}

cudaStream_t side_stream() {
    thread_local cudaStream_t streams[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
        streams[dev] = nullptr;
    return streams[dev];
}

// Fork: the side stream waits for everything issued to s so far, then runs the shared experts;
// *join is recorded after them.  The events are created per call (and destroyed by the caller
// once s waits on join), so concurrent callers never share an event.
moe_status fork_shared_begin(cudaStream_t s, cudaStream_t side, cudaEvent_t* join) {
    cudaEvent_t fork = nullptr;
    MOE_CUDA(cudaEventCreateWithFlags(&fork, cudaEventDisableTiming));
    cudaError_t e = cudaEventRecord(fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, fork, 0);
    cudaEventDestroy(fork);
    MOE_CUDA(e);
    MOE_CUDA(cudaEventCreateWithFlags(join, cudaEventDisableTiming));
    return MOE_OK;
}
moe_status fork_shared_end(cudaStream_t s, cudaStream_t side, cudaEvent_t join) {
    cudaError_t e = cudaEventRecord(join, side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, join, 0);
    cudaEventDestroy(join);
    MOE_CUDA(e);
    return MOE_OK;
}

// Joins a forked side stream back into s when it goes out of scope unless join() already did:
// an error return between the fork and the join still leaves no unjoined work behind (which
// under stream capture would turn the caller's error into cudaErrorStreamCaptureUnjoined).
struct ForkJoin {
    cudaStream_t s = nullptr, side = nullptr;
    cudaEvent_t ev = nullptr;
    bool open = false;
    moe_status begin(cudaStream_t s_, cudaStream_t side_) {
        s = s_;
        side = side_;
        MOE_TRY(fork_shared_begin(s, side, &ev));
        open = true;
        return MOE_OK;
    }
    moe_status join() {
        if (!open) return MOE_OK;
        open = false;
        return fork_shared_end(s, side, ev);
    }
    ~ForkJoin() { (void)join(); }
};

// ------------------------------------------------------------------ W4A16 pieces

moe_status check_w4_cfg(const moe_cfg* c) {
    if (c->act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (c->d % kW4GroupK || c->d_ff % kW4GroupK || (c->n_shared > 0 && c->d_ff_shared % kW4GroupK))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status need_w4(const moe_w4& m) {
    MOE_TRY(need(m.q, 16));
    return need(m.s, 16);
}

moe_status check_w4_layer(const moe_cfg* c, const moe_w4_layer* W, bool shared) {
    if (!W) return MOE_ERR_INVALID_ARG;
    MOE_TRY(need_w4(W->gate));
    MOE_TRY(need_w4(W->up));
    MOE_TRY(need_w4(W->down));
    if (shared && c->n_shared > 0) {
        MOE_TRY(need_w4(W->shared_gate));
        MOE_TRY(need_w4(W->shared_up));
        MOE_TRY(need_w4(W->shared_down));
    }
    return MOE_OK;
}

W4Mat w4m(const moe_w4& m) { return W4Mat{m.q, m.s}; }

moe_status do_grouped_ffn_w4(const moe_cfg* c, const void* x_perm, const int32_t* kept,
                             const int32_t* kept_offsets, const float* row_weight,
                             const moe_w4_layer& W, void* y_perm, void* ws, cudaStream_t s,
                             void* const* ev) {
    const WsLayout L = ws_layout(*c);
    W4Group g{c->E, kept, kept_offsets, 0, 0, 0};
    auto* h = at<__nv_bfloat16>(ws, L.h_perm);
    if (grouped_rows(*c) > 0)
        MOE_CUDA(w4_gateup(g, (const __nv_bfloat16*)x_perm, c->d, w4m(W.gate), w4m(W.up), c->d_ff,
                           h, at<int32_t>(ws, L.err), grouped_rows(*c), s));
    if (ev && ev[3]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[3], s));
    if (grouped_rows(*c) > 0)
        MOE_CUDA(w4_down(g, h, c->d_ff, w4m(W.down), c->d, row_weight, (__nv_bfloat16*)y_perm,
                         at<int32_t>(ws, L.err), grouped_rows(*c), s));
    if (ev && ev[4]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[4], s));
    return MOE_OK;
}

moe_status do_shared_w4(const moe_cfg* c, const void* x, const moe_w4_layer& W, void* ws,
                        cudaStream_t s) {
    const WsLayout L = ws_layout(*c);
    auto* hsh = at<__nv_bfloat16>(ws, L.h_sh);
    auto* ysh = at<__nv_bfloat16>(ws, L.y_sh);
    if (c->n_shared > 0 && c->N > 0) {
        // every shared expert reads all N tokens of x; its h and y blocks are N rows apart
        W4Group g{c->n_shared, nullptr, nullptr, (int)c->N, 0, c->N};
        MOE_CUDA(w4_gateup(g, (const __nv_bfloat16*)x, c->d, w4m(W.shared_gate),
                           w4m(W.shared_up), c->d_ff_shared, hsh, at<int32_t>(ws, L.err),
                           c->N * c->n_shared, s));
        g.a_stride = c->N;
        MOE_CUDA(w4_down(g, hsh, c->d_ff_shared, w4m(W.shared_down), c->d, nullptr, ysh,
                         at<int32_t>(ws, L.err), c->N * c->n_shared, s));
    }
    return MOE_OK;
}

moe_status do_shared_w4_and_combine(const moe_cfg* c, const void* y_perm, const int32_t* pos,
                                    const void* x, const moe_w4_layer& W, void* out, void* ws,
                                    cudaStream_t s, void* const* ev, bool shared_done) {
    const WsLayout L = ws_layout(*c);
    if (!shared_done) MOE_TRY(do_shared_w4(c, x, W, ws, s));
    if (ev && ev[5]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[5], s));
    MOE_CUDA(launch_combine(*c, y_perm, pos, at<__nv_bfloat16>(ws, L.y_sh), out,
                            at<int32_t>(ws, L.err), s));
    if (ev && ev[6]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[6], s));
    return MOE_OK;
}

moe_status check_weights(const moe_cfg* c, const void* Wg, const void* Wu, const void* Wd) {
    MOE_TRY(need(Wg, 16));
    MOE_TRY(need(Wu, 16));
    MOE_TRY(need(Wd, 16));
    return MOE_OK;
    (void)c;
}

moe_status check_shared(const moe_cfg* c, const void* a, const void* b, const void* d) {
    if (c->n_shared == 0) return MOE_OK;
    MOE_TRY(need(a, 16));
    MOE_TRY(need(b, 16));
    MOE_TRY(need(d, 16));
    return MOE_OK;
}

}  // namespace

// ===================================================================== C ABI

extern "C" {

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE_BOUNDS: return "device saw an out-of-range index";
        case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case MOE_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    }
    return "unknown status";
}

const char* moe_status_str(moe_status s) { return moe_status_string(s); }

int64_t moe_grouped_rows(const moe_cfg* cfg) {
    if (check_cfg(cfg) != MOE_OK) return -1;
    return grouped_rows(*cfg);
}

moe_status moe_workspace_size(const moe_cfg* cfg, size_t* bytes) {
    MOE_TRY(check_cfg(cfg));
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(*cfg).total;
    return MOE_OK;
}

moe_status moe_workspace_init(const moe_cfg* cfg, void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    forget_prepared(ws);
    MOE_CUDA(cudaMemsetAsync(ws, 0, 256, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_router_prepare(const moe_cfg* cfg, const float* W_r, void* ws, size_t ws_bytes,
                              void* stream) {
    NvtxRange nvtx_("moe_router_prepare");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    MOE_TRY(need(W_r, 16));
    if (!router_uses_tensor_cores(*cfg)) return MOE_OK;
    const WsLayout L = ws_layout(*cfg);
    forget_prepared(ws);
    MOE_CUDA(tc_router_split(W_r, cfg->E, cfg->d, at<__nv_bfloat16>(ws, L.router_w3),
                             (cudaStream_t)stream));
    std::lock_guard<std::mutex> lock(g_prepared_mu);
    g_prepared[reinterpret_cast<uintptr_t>(ws)] = PreparedSplit{W_r, cfg->E, cfg->d};
    return MOE_OK;
}

moe_status moe_route(const moe_cfg* cfg, const void* x, const float* W_r, const float* b_r,
                     int32_t* idx, float* w, float* P_sum, float* gap, void* ws, size_t ws_bytes,
                     void* stream) {
    NvtxRange nvtx_("moe_route");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    if (cfg->N > 0) {
        MOE_TRY(need(x, 16));
        MOE_TRY(need(idx, 4));
        MOE_TRY(need(w, 4));
    }
    MOE_TRY(need(W_r, 16));
    MOE_TRY(need(P_sum, 4));
    if (cfg->bias_mode != 0) MOE_TRY(need(b_r, 4));
    const WsLayout L = ws_layout(*cfg);
    const bool prepared = split_prepared(*cfg, W_r, ws);
    if (!prepared) forget_prepared(ws);
    MOE_CUDA(launch_router(*cfg, x, W_r, b_r, idx, w, gap, at<float>(ws, L.lse),
                           at<float>(ws, L.p_part), P_sum,
                           at<__nv_bfloat16>(ws, L.router_w3), at<float>(ws, L.logits),
                           at<int32_t>(ws, L.err), (cudaStream_t)stream, nullptr, prepared));
    return MOE_OK;
}

moe_status moe_permute(const moe_cfg* cfg, const int32_t* idx, const float* w, const void* x,
                       int32_t* counts, int32_t* offsets, int32_t* kept, int32_t* kept_offsets,
                       int32_t* perm, int32_t* pos, int32_t* row_token, float* row_weight,
                       void* x_perm, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_("moe_permute");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    MOE_TRY(need(counts, 4));
    MOE_TRY(need(offsets, 4));
    MOE_TRY(need(kept, 4));
    MOE_TRY(need(kept_offsets, 4));
    if (cfg->N > 0) {
        MOE_TRY(need(idx, 4));
        MOE_TRY(need(w, 4));
        MOE_TRY(need(x, 16));
        MOE_TRY(need(perm, 4));
        MOE_TRY(need(pos, 4));
        MOE_TRY(need(row_token, 4));
        MOE_TRY(need(row_weight, 4));
        MOE_TRY(need(x_perm, 16));
    }
    const WsLayout L = ws_layout(*cfg);
    MOE_CUDA(launch_permute(*cfg, idx, w, x, counts, offsets, kept, kept_offsets, perm, pos,
                            row_token, row_weight, x_perm, at<int32_t>(ws, L.blk_hist),
                            at<int32_t>(ws, L.blk_base), at<int32_t>(ws, L.err),
                            (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_grouped_ffn(const moe_cfg* cfg, const void* x_perm, const int32_t* kept,
                           const int32_t* kept_offsets, const float* row_weight,
                           const void* W_gate, const void* W_up, const void* W_down, void* y_perm,
                           void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_("moe_grouped_ffn");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    MOE_TRY(need(kept, 4));
    MOE_TRY(need(kept_offsets, 4));
    MOE_TRY(check_weights(cfg, W_gate, W_up, W_down));
    if (grouped_rows(*cfg) > 0) {
        MOE_TRY(need(x_perm, 16));
        MOE_TRY(need(y_perm, 16));
        if (row_weight) MOE_TRY(need(row_weight, 4));
    }
    return do_grouped_ffn(cfg, x_perm, kept, kept_offsets, row_weight, W_gate, W_up, W_down,
                          y_perm, ws, (cudaStream_t)stream, nullptr);
}

moe_status moe_combine(const moe_cfg* cfg, const void* y_perm, const int32_t* pos, const void* x,
                       const void* Ws_gate, const void* Ws_up, const void* Ws_down, void* out,
                       void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_("moe_combine");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    MOE_TRY(check_shared(cfg, Ws_gate, Ws_up, Ws_down));
    if (cfg->N > 0) {
        MOE_TRY(need(pos, 4));
        MOE_TRY(need(x, 16));
        MOE_TRY(need(out, 16));
        if (grouped_rows(*cfg) > 0) MOE_TRY(need(y_perm, 16));
    }
    return do_shared_and_combine(cfg, y_perm, pos, x, Ws_gate, Ws_up, Ws_down, out, ws,
                                 (cudaStream_t)stream, nullptr);
}

moe_status moe_forward_traced(const moe_cfg* cfg, const void* x, const float* W_r,
                              const float* b_r, const void* W_gate, const void* W_up,
                              const void* W_down, const void* Ws_gate, const void* Ws_up,
                              const void* Ws_down, void* out, void* ws, size_t ws_bytes,
                              void* stream, void* const* ev) {
    NvtxRange nvtx_("moe_forward_traced");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    MOE_TRY(need(W_r, 16));
    if (cfg->bias_mode != 0) MOE_TRY(need(b_r, 4));
    MOE_TRY(check_weights(cfg, W_gate, W_up, W_down));
    MOE_TRY(check_shared(cfg, Ws_gate, Ws_up, Ws_down));
    if (cfg->N > 0) {
        MOE_TRY(need(x, 16));
        MOE_TRY(need(out, 16));
    }
    cudaStream_t s = (cudaStream_t)stream;
    const WsLayout L = ws_layout(*cfg);
    int32_t* err = at<int32_t>(ws, L.err);
    if (ev && ev[0]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[0], s));
    // a forward that splits W_r itself overwrites the workspace's prepared split
    const bool prepared = split_prepared(*cfg, W_r, ws);
    if (!prepared) forget_prepared(ws);
    cudaStream_t side = fork_shared(*cfg) ? side_stream() : nullptr;
    ForkJoin fj;
    if (side) {
        MOE_TRY(fj.begin(s, side));
        MOE_TRY(do_shared(cfg, x, Ws_gate, Ws_up, Ws_down, ws, side));
    }
    MOE_CUDA(launch_router(*cfg, x, W_r, b_r, at<int32_t>(ws, L.idx), at<float>(ws, L.w),
                           at<float>(ws, L.gap), at<float>(ws, L.lse), at<float>(ws, L.p_part),
                           at<float>(ws, L.P_sum),
                           at<__nv_bfloat16>(ws, L.router_w3), at<float>(ws, L.logits), err, s,
                           nullptr, prepared));
    if (ev && ev[1]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[1], s));
    MOE_CUDA(launch_permute(*cfg, at<int32_t>(ws, L.idx), at<float>(ws, L.w), x,
                            at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
                            at<int32_t>(ws, L.kept), at<int32_t>(ws, L.kept_offsets),
                            at<int32_t>(ws, L.perm), at<int32_t>(ws, L.pos),
                            at<int32_t>(ws, L.row_token), at<float>(ws, L.row_weight),
                            at<void>(ws, L.x_perm), at<int32_t>(ws, L.blk_hist),
                            at<int32_t>(ws, L.blk_base), err, s));
    if (ev && ev[2]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[2], s));
    MOE_TRY(do_grouped_ffn(cfg, at<void>(ws, L.x_perm), at<int32_t>(ws, L.kept),
                           at<int32_t>(ws, L.kept_offsets), at<float>(ws, L.row_weight), W_gate,
                           W_up, W_down, at<void>(ws, L.y_perm), ws, s, ev));
    if (side) MOE_TRY(fj.join());
    MOE_TRY(do_shared_and_combine(cfg, at<void>(ws, L.y_perm), at<int32_t>(ws, L.pos), x, Ws_gate,
                                  Ws_up, Ws_down, out, ws, s, ev, side != nullptr));
    return MOE_OK;
}

moe_status moe_forward(const moe_cfg* cfg, const void* x, const float* W_r, const float* b_r,
                       const void* W_gate, const void* W_up, const void* W_down,
                       const void* Ws_gate, const void* Ws_up, const void* Ws_down, void* out,
                       void* ws, size_t ws_bytes, void* stream) {
    return moe_forward_traced(cfg, x, W_r, b_r, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, out,
                              ws, ws_bytes, stream, nullptr);
}

moe_status moe_quantize_w4(const void* W, int64_t rows, int32_t cols, uint8_t* q, float* s,
                           void* stream) {
    if (rows < 0 || cols <= 0 || cols % kW4GroupK) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (rows * (int64_t)cols >= ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED;
    MOE_TRY(need(W, 16));
    MOE_TRY(need(q, 16));
    MOE_TRY(need(s, 16));
    MOE_CUDA(w4_quantize((const __nv_bfloat16*)W, rows, cols, q, s, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_grouped_ffn_w4a16(const moe_cfg* cfg, const void* x_perm, const int32_t* kept,
                                 const int32_t* kept_offsets, const float* row_weight,
                                 const moe_w4_layer* W, void* y_perm, void* ws, size_t ws_bytes,
                                 void* stream) {
    NvtxRange nvtx_("moe_grouped_ffn_w4a16");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_w4_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    MOE_TRY(need(kept, 4));
    MOE_TRY(need(kept_offsets, 4));
    MOE_TRY(check_w4_layer(cfg, W, false));
    if (grouped_rows(*cfg) > 0) {
        MOE_TRY(need(x_perm, 16));
        MOE_TRY(need(y_perm, 16));
        if (row_weight) MOE_TRY(need(row_weight, 4));
    }
    return do_grouped_ffn_w4(cfg, x_perm, kept, kept_offsets, row_weight, *W, y_perm, ws,
                             (cudaStream_t)stream, nullptr);
}

moe_status moe_forward_w4a16(const moe_cfg* cfg, const void* x, const float* W_r, const float* b_r,
                             const moe_w4_layer* W, void* out, void* ws, size_t ws_bytes,
                             void* stream, void* const* ev) {
    NvtxRange nvtx_("moe_forward_w4a16");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_w4_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    MOE_TRY(need(W_r, 16));
    if (cfg->bias_mode != 0) MOE_TRY(need(b_r, 4));
    MOE_TRY(check_w4_layer(cfg, W, true));
    if (cfg->N > 0) {
        MOE_TRY(need(x, 16));
        MOE_TRY(need(out, 16));
    }
    cudaStream_t s = (cudaStream_t)stream;
    const WsLayout L = ws_layout(*cfg);
    int32_t* err = at<int32_t>(ws, L.err);
    if (ev && ev[0]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[0], s));
    // a forward that splits W_r itself overwrites the workspace's prepared split
    const bool prepared = split_prepared(*cfg, W_r, ws);
    if (!prepared) forget_prepared(ws);
    cudaStream_t side = fork_shared(*cfg) ? side_stream() : nullptr;
    ForkJoin fj;
    if (side) {
        MOE_TRY(fj.begin(s, side));
        MOE_TRY(do_shared_w4(cfg, x, *W, ws, side));
    }
    MOE_CUDA(launch_router(*cfg, x, W_r, b_r, at<int32_t>(ws, L.idx), at<float>(ws, L.w),
                           at<float>(ws, L.gap), at<float>(ws, L.lse), at<float>(ws, L.p_part),
                           at<float>(ws, L.P_sum),
                           at<__nv_bfloat16>(ws, L.router_w3), at<float>(ws, L.logits), err, s,
                           nullptr, prepared));
    if (ev && ev[1]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[1], s));
    MOE_CUDA(launch_permute(*cfg, at<int32_t>(ws, L.idx), at<float>(ws, L.w), x,
                            at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
                            at<int32_t>(ws, L.kept), at<int32_t>(ws, L.kept_offsets),
                            at<int32_t>(ws, L.perm), at<int32_t>(ws, L.pos),
                            at<int32_t>(ws, L.row_token), at<float>(ws, L.row_weight),
                            at<void>(ws, L.x_perm), at<int32_t>(ws, L.blk_hist),
                            at<int32_t>(ws, L.blk_base), err, s));
    if (ev && ev[2]) MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[2], s));
    MOE_TRY(do_grouped_ffn_w4(cfg, at<void>(ws, L.x_perm), at<int32_t>(ws, L.kept),
                              at<int32_t>(ws, L.kept_offsets), at<float>(ws, L.row_weight), *W,
                              at<void>(ws, L.y_perm), ws, s, ev));
    if (side) MOE_TRY(fj.join());
    MOE_TRY(do_shared_w4_and_combine(cfg, at<void>(ws, L.y_perm), at<int32_t>(ws, L.pos), x, *W,
                                     out, ws, s, ev, side != nullptr));
    return MOE_OK;
}

moe_status check_bwd_cfg(const moe_cfg* c) {
    if (c->act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (c->d % 64 || c->d_ff % 128 || (c->n_shared > 0 && c->d_ff_shared % 128))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status moe_backward_workspace_size(const moe_cfg* cfg, size_t* bytes) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_bwd_cfg(cfg));
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = bwd_layout(*cfg).total;
    return MOE_OK;
}

moe_status moe_backward(const moe_cfg* cfg, const void* x, const float* W_r, const float* b_r,
                        const void* W_gate, const void* W_up, const void* W_down,
                        const void* Ws_gate, const void* Ws_up, const void* Ws_down,
                        const void* dout, double aux_coef, double z_coef, float* dx, float* dW_r,
                        float* db, float* dW_gate, float* dW_up, float* dW_down, float* dWs_gate,
                        float* dWs_up, float* dWs_down, void* ws, size_t ws_bytes, void* bws,
                        size_t bws_bytes, void* stream) {
    NvtxRange nvtx_("moe_backward");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_bwd_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    if (!bws || !aligned(bws, 256) || bws_bytes < bwd_layout(*cfg).total) return MOE_ERR_WORKSPACE;
    if (isnan(aux_coef) || isnan(z_coef)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(need(W_r, 16));
    if (cfg->bias_mode != 0) MOE_TRY(need(b_r, 4));
    MOE_TRY(check_weights(cfg, W_gate, W_up, W_down));
    MOE_TRY(check_shared(cfg, Ws_gate, Ws_up, Ws_down));
    MOE_TRY(need(dW_r, 16));
    MOE_TRY(need(dW_gate, 16));
    MOE_TRY(need(dW_up, 16));
    MOE_TRY(need(dW_down, 16));
    if (db) MOE_TRY(need(db, 4));
    if (cfg->n_shared > 0) {
        MOE_TRY(need(dWs_gate, 16));
        MOE_TRY(need(dWs_up, 16));
        MOE_TRY(need(dWs_down, 16));
    }
    if (cfg->N > 0) {
        MOE_TRY(need(x, 16));
        MOE_TRY(need(dout, 16));
        MOE_TRY(need(dx, 16));
    }
    const WsLayout L = ws_layout(*cfg);
    forget_prepared(ws);   // the backward's router pass re-splits W_r into the workspace
    BwdArgs a{};
    a.cfg = cfg;
    a.x = x;
    a.W_r = W_r;
    a.b_r = cfg->bias_mode != 0 ? b_r : nullptr;
    a.Wg = (const __nv_bfloat16*)W_gate;
    a.Wu = (const __nv_bfloat16*)W_up;
    a.Wd = (const __nv_bfloat16*)W_down;
    a.Wsg = (const __nv_bfloat16*)Ws_gate;
    a.Wsu = (const __nv_bfloat16*)Ws_up;
    a.Wsd = (const __nv_bfloat16*)Ws_down;
    a.dout = (const __nv_bfloat16*)dout;
    a.aux_coef = aux_coef;
    a.z_coef = z_coef;
    a.dx = dx;
    a.dW_r = dW_r;
    a.db = db;
    a.dWg = dW_gate;
    a.dWu = dW_up;
    a.dWd = dW_down;
    a.dWsg = dWs_gate;
    a.dWsu = dWs_up;
    a.dWsd = dWs_down;
    a.idx = at<int32_t>(ws, L.idx);
    a.pos = at<int32_t>(ws, L.pos);
    a.counts = at<int32_t>(ws, L.counts);
    a.kept = at<int32_t>(ws, L.kept);
    a.kept_off = at<int32_t>(ws, L.kept_offsets);
    a.row_token = at<int32_t>(ws, L.row_token);
    a.err = at<int32_t>(ws, L.err);
    a.w = at<float>(ws, L.w);
    a.gap = at<float>(ws, L.gap);
    a.lse = at<float>(ws, L.lse);
    a.p_part = at<float>(ws, L.p_part);
    a.P_sum = at<float>(ws, L.P_sum);
    a.row_weight = at<float>(ws, L.row_weight);
    a.logits = at<float>(ws, L.logits);
    a.w3 = at<__nv_bfloat16>(ws, L.router_w3);
    a.h_perm = at<__nv_bfloat16>(ws, L.h_perm);
    a.h_sh = at<__nv_bfloat16>(ws, L.h_sh);
    a.bws = bws;
    MOE_CUDA(run_backward(a, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_forward_buffers(const moe_cfg* cfg, void* ws, size_t ws_bytes, moe_buffers* out) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    if (!out) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*cfg);
    out->idx = at<int32_t>(ws, L.idx);
    out->w = at<float>(ws, L.w);
    out->gap = at<float>(ws, L.gap);
    out->P_sum = at<float>(ws, L.P_sum);
    out->counts = at<int32_t>(ws, L.counts);
    out->offsets = at<int32_t>(ws, L.offsets);
    out->kept = at<int32_t>(ws, L.kept);
    out->kept_offsets = at<int32_t>(ws, L.kept_offsets);
    out->perm = at<int32_t>(ws, L.perm);
    out->pos = at<int32_t>(ws, L.pos);
    out->row_token = at<int32_t>(ws, L.row_token);
    out->row_weight = at<float>(ws, L.row_weight);
    out->x_perm = at<void>(ws, L.x_perm);
    out->y_perm = at<void>(ws, L.y_perm);
    out->lse = at<float>(ws, L.lse);
    return MOE_OK;
}

moe_status moe_router_stats(const moe_cfg* cfg, const float* lse, const float* w,
                            const int32_t* perm, const int32_t* offsets, float* importance_host,
                            moe_router_summary* summary, void* ws, size_t ws_bytes,
                            void* stream) {
    NvtxRange nvtx_("moe_router_stats");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    if (!summary) return MOE_ERR_INVALID_ARG;
    MOE_TRY(need(offsets, 4));
    if (cfg->N > 0) {
        MOE_TRY(need(lse, 4));
        MOE_TRY(need(w, 4));
        MOE_TRY(need(perm, 4));
    }
    cudaStream_t s = (cudaStream_t)stream;
    const WsLayout L = ws_layout(*cfg);
    double* zp = at<double>(ws, L.rstat);
    double* imp = zp + kRouterStatBlocks;
    MOE_CUDA(launch_router_stats(cfg->N, cfg->E, cfg->k, lse, w, perm, offsets, zp, imp, s));
    const int E = cfg->E;
    double* h = static_cast<double*>(malloc(sizeof(double) * (size_t)(kRouterStatBlocks + E)));
    if (!h) return MOE_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(h, zp, sizeof(double) * (size_t)(kRouterStatBlocks + E),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        free(h);
        return MOE_ERR_CUDA;
    }
    double z = 0.0, mean = 0.0, var = 0.0;
    for (int b = 0; b < kRouterStatBlocks; b++) z += h[b];
    for (int i = 0; i < E; i++) mean += h[kRouterStatBlocks + i];
    mean /= (double)E;
    for (int i = 0; i < E; i++) {
        const double dv = h[kRouterStatBlocks + i] - mean;
        var += dv * dv;
    }
    var /= (double)E;
    summary->z_loss = cfg->N > 0 ? z / (double)cfg->N : 0.0;
    summary->importance_mean = mean;
    summary->importance_cv2 = mean > 0.0 ? var / (mean * mean) : 0.0;
    if (importance_host)
        for (int i = 0; i < E; i++) importance_host[i] = (float)h[kRouterStatBlocks + i];
    free(h);
    return MOE_OK;
}

moe_status moe_stats(const moe_cfg* cfg, const int32_t* counts, const int32_t* kept,
                     const float* P_sum, const int32_t* pos, const float* gap, float* f_host,
                     float* P_host, moe_stats_summary* summary, void* ws, size_t ws_bytes,
                     void* stream) {
    NvtxRange nvtx_("moe_stats");
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    MOE_TRY(need(counts, 4));
    MOE_TRY(need(kept, 4));
    MOE_TRY(need(P_sum, 4));
    if (cfg->N > 0) MOE_TRY(need(pos, 4));
    if (!summary) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const WsLayout L = ws_layout(*cfg);
    int32_t* errw = at<int32_t>(ws, L.err);
    int32_t* counters = errw + 8;
    float* sf = at<float>(ws, L.stats_f);
    MOE_CUDA(launch_stats(*cfg, counts, kept, P_sum, pos, gap, counters, sf, s));
    const int E = cfg->E;
    int32_t hc[9];
    float hscal = 0.f;
    MOE_CUDA(cudaMemcpyAsync(hc, errw, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    MOE_CUDA(cudaMemcpyAsync(hc + 1, counters, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    MOE_CUDA(cudaMemcpyAsync(&hscal, sf + 2 * E, sizeof(float), cudaMemcpyDeviceToHost, s));
    if (f_host) MOE_CUDA(cudaMemcpyAsync(f_host, sf, E * sizeof(float), cudaMemcpyDeviceToHost, s));
    if (P_host)
        MOE_CUDA(cudaMemcpyAsync(P_host, sf + E, E * sizeof(float), cudaMemcpyDeviceToHost, s));
    MOE_CUDA(cudaStreamSynchronize(s));
    summary->aux = hscal;
    summary->device_error = hc[0];
    summary->fully_dropped = hc[1];
    summary->near_tie = hc[2];
    summary->kept_rows = hc[3];
    summary->touched_experts = hc[4];
    summary->dropped = cfg->N * cfg->k - (int64_t)hc[3];
    return MOE_OK;
}

moe_status moe_device_error(void* ws, size_t ws_bytes, int32_t* code, void* stream) {
    if (!ws || !aligned(ws, 256) || ws_bytes < 256) return MOE_ERR_WORKSPACE;
    if (!code) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    MOE_CUDA(cudaMemcpyAsync(code, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    MOE_CUDA(cudaStreamSynchronize(s));
    if (*code & MOE_DEVERR_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
    if (*code & MOE_DEVERR_BOUNDS) return MOE_ERR_DEVICE_BOUNDS;
    return MOE_OK;
}

}  // extern "C"
