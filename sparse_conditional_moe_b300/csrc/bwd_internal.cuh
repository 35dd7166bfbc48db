// bwd_internal.cuh -- declarations of the backward pass's GEMMs and helper kernels.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Grouped GEMM geometry of the backward kernels (grouped_gemm_bwd.cu).
enum { TB_ROWS = 0, TB_WEIGHTS = 1 };
enum { TBE_F32 = 0, TBE_DH = 1, TBE_SWIGLU_BWD = 2, TBE_ROWS_F32 = 3 };

struct TbParams {
    int mode;                    // TB_ROWS: M = each group's padded rows; TB_WEIGHTS: K = them
    int G;
    const int32_t* rows;         // [G] real rows of each group
    const int32_t* a_off;        // [G+1] padded row offset of the group in A's row buffer
    const int32_t* c_off;        // [G+1] padded row offset in the output / B's row buffer
    const int32_t* dense_off;    // [G] dense (unpadded) row offset: row weights, forward h
    int64_t max_mtiles;          // bound on c_off[G] / 128 (grid sizing)
    int K;                       // TB_ROWS: reduction length
    int k_split;                 // TB_ROWS, MN-major B: from this k on, B comes from the 2nd map
    int b_rows;                  // TB_ROWS: B rows per group in its map
    int M, N;                    // output dims (TB_WEIGHTS: per group; TB_ROWS: N = columns)
    int m_tiles, n_tiles;
    int split_m;                 // TB_WEIGHTS: rows < split_m go to out_f32, the rest to out_f32b
    float* out_f32;
    float* out_f32b;
    __nv_bfloat16* out_bf16;     // TBE_DH: dh [padded rows, F]; TBE_SWIGLU_BWD: [dG | dU]
    int64_t ld_bf16;
    __nv_bfloat16* out2_bf16;    // TBE_SWIGLU_BWD: w * h [padded rows, F]
    const __nv_bfloat16* aux_bf16;   // TBE_DH: forward h (dense rows); TBE_SWIGLU_BWD: dh (padded)
    int64_t ld_aux;
    const float* row_weight;     // dense rows, nullable (weight 1)
    float* dw_part;              // TBE_DH: [padded rows, n_tiles] partial <dH', h>
    int F;                       // TBE_SWIGLU_BWD: hidden width (dU starts at column F)
    int32_t* err;
};

int tb_dh_tiles(int F);   // column tiles of G1 (dw partials per row)
cudaError_t tb_dh(const TbParams& p, const __nv_bfloat16* dout_pad, int64_t rows_a, int d,
                  const __nv_bfloat16* Wd, int F, cudaStream_t s);
cudaError_t tb_swiglu_bwd(const TbParams& p, const __nv_bfloat16* x_pad, int64_t rows_a, int d,
                          const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int F, cudaStream_t s);
cudaError_t tb_dx(const TbParams& p, const __nv_bfloat16* dgu, int64_t rows_a, int F,
                  const __nv_bfloat16* Wg, const __nv_bfloat16* Wu, int d, cudaStream_t s);
cudaError_t tb_rows_f32(const TbParams& p, const __nv_bfloat16* A, int64_t rows_a, int K,
                        const __nv_bfloat16* B, int N, cudaStream_t s);
cudaError_t tb_wgrad(const TbParams& p, const __nv_bfloat16* A, int64_t rows_a, int M,
                     const __nv_bfloat16* B, int64_t rows_b, int N, cudaStream_t s,
                     int a_cols = 0);
cudaError_t tb_selftest(bool a_mn, bool b_mn, int M, int N, int K, const __nv_bfloat16* A,
                        const __nv_bfloat16* B, float* C, const int32_t* plan, int32_t* err,
                        cudaStream_t s);

// ------------------------------------------------------------------ the backward pass (bwd.cu)

struct BwdLayout {   // byte offsets in the backward workspace (256-byte aligned regions)
    size_t probs, dl, dx_r, dw_row, c_off, s_plan;
    size_t r_plan, dl3, dlT2, w3, x2, db_part;   // router GEMMs on the tensor cores
    size_t dout_pad, x_pad, dh, dgu, hw, dX, dw_part;
    size_t dout_s, x_s, dh_s, dgu_s, hw_s, dX_s, dw_part_s;
    size_t total;
};
BwdLayout bwd_layout(const moe_cfg& c);
int64_t bwd_padded_rows(const moe_cfg& c);   // bound on the routed rows in padded segments
int64_t bwd_shared_rows(const moe_cfg& c);   // N rounded up to 128

struct BwdArgs {
    const moe_cfg* cfg;
    // forward inputs
    const void* x;
    const float* W_r;
    const float* b_r;
    const __nv_bfloat16 *Wg, *Wu, *Wd, *Wsg, *Wsu, *Wsd;
    const __nv_bfloat16* dout;
    double aux_coef, z_coef;
    // outputs (fp32)
    float *dx, *dW_r, *db, *dWg, *dWu, *dWd, *dWsg, *dWsu, *dWsd;
    // the forward's workspace state
    int32_t *idx, *pos, *counts, *kept, *kept_off, *row_token, *err;
    float *w, *gap, *lse, *p_part, *P_sum, *row_weight, *logits;
    __nv_bfloat16* w3;
    const __nv_bfloat16 *h_perm, *h_sh;
    void* bws;
};
cudaError_t run_backward(const BwdArgs& a, cudaStream_t s);

}  // namespace moe
