// moe_internal.cuh -- device-side declarations shared by the libmoe CUDA sources.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------------------ router tiling

// Router path selection and the rows of its per-block probability sums (an upper bound).
bool router_uses_tensor_cores(const moe_cfg& c);
int64_t router_part_rows(int64_t N);

// ------------------------------------------------------------------ permute tiling

// A grouping block covers 2048 consecutive slots.  A full block gives each of its 8 warps 256
// (8 steps of 32); a short last block spreads its slots evenly over the warps (each warp a
// contiguous run, in warp order), so kPermSlotsPerWarp is the most a warp ever handles.
constexpr int kPermThreads = 256;                    // 8 warps
constexpr int kPermSlotsPerWarp = 256;
constexpr int kPermSlotsPerBlock = kPermSlotsPerWarp * (kPermThreads / 32);
inline int perm_blocks(int64_t slots) {
    return (int)((slots + kPermSlotsPerBlock - 1) / kPermSlotsPerBlock);
}

// ------------------------------------------------------------------ workspace

struct WsLayout {
    size_t err;          // int32 [64]: [0] sticky error word, [8..15] stats counters
    size_t p_part;       // float [router_part_rows(N) * E]
    size_t router_w3;    // bf16 [3, E, d]: exact hi/mid/lo split of W_r (tensor-core router)
    size_t logits;       // float [N, E] (tensor-core router)
    size_t blk_hist;     // int32 [perm_blocks * E]
    size_t blk_base;     // int32 [perm_blocks * E]
    size_t mtile_off;    // int32 [E + 1]: m-tile (or token-chunk) prefix of the routed grouped GEMMs
    size_t stats_f;      // float [2E + 8]: f, P, scalars
    size_t idx, w, gap, lse, P_sum, counts, offsets, kept, kept_offsets, perm, pos;
    size_t rstat;        // double [kRouterStatBlocks + E]: z-loss partials, importance
    size_t row_token, row_weight;
    size_t x_perm, h_perm, y_perm;   // [R, d], [R, F], [R, d]
    size_t h_sh, y_sh;               // [S, N, F_s], [S, N, d]
    size_t total;
};

int64_t grouped_rows(const moe_cfg& c);
int64_t capacity(const moe_cfg& c);  // -1 when unlimited
WsLayout ws_layout(const moe_cfg& c);

// ------------------------------------------------------------------ launches
// All return cudaGetLastError() of their launches.

// lse [N] (nullable): log-sum-exp of each token's logits, for the z-loss; probs [N, E]
// (nullable): the softmax probabilities, for the backward pass.
// w3_ready: the tensor-core router's weight split in w3 is current (moe_router_prepare).
cudaError_t launch_router(const moe_cfg& c, const void* x, const float* W_r, const float* b_r,
                          int32_t* idx, float* w, float* gap, float* lse, float* p_part,
                          float* P_sum, __nv_bfloat16* w3, float* logits, int32_t* err,
                          cudaStream_t s, float* probs = nullptr, bool w3_ready = false);

// Tensor-core router for bf16 x (see router_tc.cu).  w3 holds the exact hi/mid/lo bf16 split of
// W_r [3, E, d] (tc_router_split writes it).  router_tc_split: number of CTA groups that split d
// (1 = none; small N only); router_tc_logits_floats: the floats its unfused logits region needs
// (the logits, plus one [N, E] slice sum per 256 of d when split); router_tc_fused: whether the
// fused kernel (softmax and top-k in the same launch, logits kept on chip) applies;
// router_tc_part_rows: the probability-sum rows the fused kernel writes.
int router_tc_split(int64_t N, int d, int E);
size_t router_tc_logits_floats(int64_t N, int d, int E);
bool router_tc_fused(int64_t N, int d, int E);
int router_tc_part_rows(int64_t N, int E);
cudaError_t tc_router_split(const float* W_r, int E, int d, __nv_bfloat16* w3, cudaStream_t s);
cudaError_t tc_router_logits(const __nv_bfloat16* x, int64_t N, int d, const __nv_bfloat16* w3,
                             int E, float* logits, int32_t* err, cudaStream_t s);
cudaError_t tc_router_fused(const __nv_bfloat16* x, int64_t N, int d, const __nv_bfloat16* w3,
                            int E, const float* b_r, int bias_mode, int k, int renorm,
                            int32_t* idx, float* w, float* gap, float* lse, float* probs,
                            float* p_part, int32_t* err, cudaStream_t s);

cudaError_t launch_permute(const moe_cfg& c, const int32_t* idx, const float* w, const void* x,
                           int32_t* counts, int32_t* offsets, int32_t* kept, int32_t* kept_off,
                           int32_t* perm, int32_t* pos, int32_t* row_token, float* row_weight,
                           void* x_perm, int32_t* blk_hist, int32_t* blk_base, int32_t* err,
                           cudaStream_t s);

// Grouped GEMM problem: G groups; group g owns rows [row0_g, row0_g + rows_g) of A and C.
struct GroupGeom {
    int G;
    const int32_t* rows;       // [G] device, or nullptr for uniform rows
    const int32_t* row_off;    // [G] device (A and C row offsets), or nullptr for uniform
    const int32_t* mtile_off;  // [G+1] device m-tile prefix (non-uniform)
    bool zigzag;               // mtile_off runs over the groups in zigzag_group order
    int uniform_rows;          // rows per group when rows == nullptr
    int64_t a_stride;          // uniform: A row offset of group g = g * a_stride
    int64_t c_stride;          // uniform: C row offset of group g = g * c_stride
    int64_t max_rows;          // upper bound of total rows (grid sizing / tensor extents)
};

// m-tile prefix over groups for the routed experts (from kept); bm = the GEMM's tile height.
// zigzag: the prefix runs over the groups in the order 0, E-1, 1, E-2, ... (zigzag_group), which
// the CTA-pair GEMMs use so that the tiles of heavy and light groups run side by side when a
// skewed router puts the heavy groups at one end.
constexpr int kTcBlockRows = 128;
__host__ __device__ inline int zigzag_group(int i, int E) { return (i & 1) ? E - 1 - (i >> 1) : (i >> 1); }
cudaError_t launch_plan_mtiles(const int32_t* kept, int E, int bm, int32_t* mtile_off,
                               cudaStream_t s, bool zigzag = false);

// bf16 tcgen05 grouped SwiGLU (gate|up) GEMM: H = silu(A Wg^T) * (A Wu^T)
cudaError_t tc_gateup(const GroupGeom& g, const __nv_bfloat16* A, int64_t a_rows, int K,
                      const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int F,
                      __nv_bfloat16* H, int64_t h_rows, int32_t* err, cudaStream_t s);
// bf16 tcgen05 grouped down GEMM: Y = row_scale * (H Wd^T)
cudaError_t tc_down(const GroupGeom& g, const __nv_bfloat16* H, int64_t h_rows, int F,
                    const __nv_bfloat16* Wd, int D, const float* row_scale,
                    __nv_bfloat16* Y, int64_t y_rows, int32_t* err, cudaStream_t s);

// The grouped GEMMs on CTA pairs with the weights as the MMA's M side (grouped_gemm_pair.cu):
// groups are cut into chunks of at most pair_chunk_rows() token rows (GroupGeom.mtile_off then
// holds the chunk prefix); max_group_rows bounds any group's rows (it picks the decode-sized
// variant when <= 64).
int pair_chunk_rows();
cudaError_t pair_gateup(const GroupGeom& g, const __nv_bfloat16* A, int64_t a_rows, int K,
                        const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int F,
                        __nv_bfloat16* H, int64_t h_rows, int32_t* err, int64_t max_group_rows,
                        cudaStream_t s);
cudaError_t pair_down(const GroupGeom& g, const __nv_bfloat16* H, int64_t h_rows, int F,
                      const __nv_bfloat16* Wd, int D, const float* row_scale,
                      __nv_bfloat16* Y, int64_t y_rows, int32_t* err, int64_t max_group_rows,
                      cudaStream_t s);
// Which bf16 grouped GEMM engine the forward uses: the pair kernels unless MOE_GROUPED_GEMM=single.
bool use_pair_gemm();

// fp32 CUDA-core grouped GEMMs (fp32 layers); their m-tiles are simt_block_rows() tall
int simt_block_rows();
cudaError_t simt_gateup_f32(const GroupGeom& g, const float* A, int K, const float* Wg,
                            const float* Wu, int F, float* H, cudaStream_t s);
cudaError_t simt_down_f32(const GroupGeom& g, const float* H, int F, const float* Wd, int D,
                          const float* row_scale, float* Y, cudaStream_t s);

// W4A16 expert FFNs (see w4a16.cu): 4-bit codes + fp32 scale per 128 inputs.
struct W4Mat {
    const uint8_t* q;   // [rows, K/2]
    const float* s;     // [K/128, rows] (group-major)
};
struct W4Group {
    int G;
    const int32_t* rows;      // [G] device, or nullptr for uniform rows
    const int32_t* row_off;   // [G] device, or nullptr
    int uniform_rows;
    int64_t a_stride, c_stride;
};
constexpr int kW4GroupK = 128;
cudaError_t w4_quantize(const __nv_bfloat16* W, int64_t rows, int cols, uint8_t* q, float* s,
                        cudaStream_t st);
// total_rows: rows over all groups (sizes the split of token passes across blocks).
cudaError_t w4_gateup(const W4Group& g, const __nv_bfloat16* A, int K, const W4Mat& Wg,
                      const W4Mat& Wu, int F, __nv_bfloat16* H, int32_t* err, int64_t total_rows,
                      cudaStream_t s);
cudaError_t w4_down(const W4Group& g, const __nv_bfloat16* H, int F, const W4Mat& Wd, int D,
                    const float* row_scale, __nv_bfloat16* Y, int32_t* err, int64_t total_rows,
                    cudaStream_t s);

cudaError_t launch_combine(const moe_cfg& c, const void* y_perm, const int32_t* pos,
                           const void* y_sh, void* out, int32_t* err, cudaStream_t s);

// Router statistics (z-loss partial sums over fixed token blocks, importance per expert
// summed along the expert-sorted permutation), both deterministic, in double.
constexpr int kRouterStatBlocks = 256;
cudaError_t launch_router_stats(int64_t N, int E, int k, const float* lse, const float* w,
                                const int32_t* perm, const int32_t* offsets, double* z_part,
                                double* imp, cudaStream_t s);

cudaError_t launch_stats(const moe_cfg& c, const int32_t* counts, const int32_t* kept,
                         const float* P_sum, const int32_t* pos, const float* gap,
                         int32_t* counters, float* stats_f, cudaStream_t s);

int device_sm_count();

}  // namespace moe
