// Absorbed MLA decode for units of at most 16 query rows (Q * H <= 16, e.g.
// 16 heads and one query token), bf16 cache rows of 576 values.
//
// Same function as the two-SM tensor-memory kernel (DeepSeek-V2 analysis
// page, sections 1.2-1.3 and 6.1):
//     S[r,s] = q_nope[r] . c_s + q_rope[r] . k^R_s,  P = softmax_s(S * scale),
//     O[r]   = sum_s P[r,s] c_s
// With 16 rows the fp32 accumulator O is 32 KB, so one SM holds a whole
// unit: no split of the latent dims across a pair and no exchange of
// partial scores.  The contractions are 16 rows wide, below the 64- and
// 128-row shapes of the tensor-memory MMA, so they run as warp-level
// m16n8k16 bf16 MMAs with fp32 accumulation; the cache stream (the bound)
// still goes through TMA into a shared-memory ring.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "decode_plan.cuh"

namespace mla {

constexpr int kShMaxRows = 16;   // query rows of a unit this kernel takes

struct ShArgs {
    const int32_t* page_table;
    const int32_t* seq_lens;
    const void* q_nope;   // bf16 [B*Q*H][512]
    const void* q_rope;   // bf16 [B*Q*H][64]
    void* out;            // bf16 [B*Q*H][512]
    float* lse;           // [B*Q*H] or null
    int32_t num_pages;
    int32_t max_pages_per_seq;
    int32_t Q;
    int32_t H;
    float scale_log2;     // softmax_scale * log2(e)
};

// kv: the bf16 cache pool viewed [pages*64][576], box 64 x 32, 128-byte swizzle.
cudaError_t launch_decode_sh(const CUtensorMap& kv, const ShArgs& a, int32_t num_workers, void* ws,
                             const WsLayout& L, cudaStream_t stream);

}  // namespace mla
