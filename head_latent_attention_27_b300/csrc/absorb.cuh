// Per-head absorption GEMMs either side of the latent attention
// ("02 · DeepSeek-V2 analysis", section 1.2, the absorption paragraph, and
// section 6.1): W^UK folded into the query, q_nope_h = W^UK_h^T q^C_h, and
// W^UV applied to the aggregated latent, o_h = W^UV_h u_h.  Both are batched
// over heads with a small number of query rows; the kernel computes the
// transposed product (weight rows as the MMA's M, query rows as its N) so the
// 128-row tensor-core tile is filled by the weight side.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

constexpr int kAbsorbBM = 128;   // output columns (weight rows) per CTA
constexpr int kAbsorbBK = 64;    // reduction block

// Query rows per CTA (the MMA's N); the activation tensor map's box is this
// tall.
int absorb_rows_per_cta(bool a_mn_major);

struct AbsorbArgs {
    void* out;          // [n_rows][H][m_total] bf16
    int32_t n_rows;     // query rows (tokens)
    int32_t H;          // heads
    int32_t m_total;    // output width per head (d_c for the query side, d_h for the output side)
    int32_t k_total;    // reduction width per head (d_h for the query side, d_c for the output side)
    int32_t* status;    // nullable device word: MLA_ERR_TIMEOUT if a bounded wait ran out
};

// tm_a: the [H * rows_per_head][d_c] weight matrix; tm_b: the activations
// [n_rows][H][k_total] as a 3-D map.  a_mn_major selects the query side
// (A = W^UK_h^T, contiguous along the output dim).
cudaError_t launch_absorb(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const AbsorbArgs& a, bool a_mn_major,
                          cudaStream_t stream);

}  // namespace mla
