// Expanded (prefill) form of MLA attention ("02 · DeepSeek-V2 analysis",
// sections 1.2-1.3 and 6: prefill may materialise the per-head keys and
// values, decode absorbs them; both compute the same function).
//
// Two kernels:
//   upproj  K^C[t][h][:] = W^UK_h c_t and V[t][h][:] = W^UV_h c_t for the T
//           prompt tokens, a dense bf16 GEMM [T x d_c] x [d_c x H*d_h] per
//           weight (tcgen05, fp32 accumulation in TMEM, bf16 out);
//   attn    causal attention per head with the 192-wide keys
//           [K^C_h || k^R] (k^R shared by all heads, read from the cache)
//           and queries [q^C_h || q^R_h], values V_h, softmax scale
//           1/sqrt(d_h + d_r); out o[t][h][:] (bf16) and lse[t][h] (fp32).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

constexpr int kPrefillDh = 128;   // d_h (per-head key / value width)
constexpr int kPrefillDc = 512;   // d_c (latent width)
constexpr int kPrefillDr = 64;    // d_h^R (RoPE width)

struct UpprojMaps {
    CUtensorMap latent;  // cache pool [pages*64][576], box 64 x 64 (128-byte swizzle)
    CUtensorMap w_uk;    // W^UK viewed [H*d_h][d_c], box 64 x 256
    CUtensorMap w_uv;    // W^UV viewed [H*d_h][d_c], box 64 x 256
};

struct UpprojArgs {
    const int32_t* page_row;  // page-table row of the sequence
    int32_t pages;            // pages holding tokens 0..T-1
    int32_t num_pages;        // pages of the pool
    int32_t T;                // prompt tokens
    int32_t n_per;            // H * d_h (columns of each output)
    void* k_out;              // bf16 [T][H*d_h]
    void* v_out;              // bf16 [T][H*d_h]
    int32_t* status;          // device status word (MLA_ERR_* of device-side checks)
};

struct PrefillAttnMaps {
    CUtensorMap q_c;     // [T][H*d_h], box 64 x 128
    CUtensorMap q_r;     // [T][H*d_r], box 64 x 128
    CUtensorMap k_c;     // [T][H*d_h], box 64 x 128
    CUtensorMap v;       // [T][H*d_h], box 64 x 128
    CUtensorMap k_r;     // cache pool [pages*64][576], box 64 x 64 (the RoPE key at column 512)
};

struct PrefillAttnArgs {
    const int32_t* page_row;
    int32_t pages;
    int32_t num_pages;
    int32_t T;
    int32_t H;
    float scale_log2;    // softmax_scale * log2(e)
    void* out;           // bf16 [T][H][d_h]
    float* lse;          // [T][H] or null
    int32_t* status;
};

cudaError_t launch_upproj(const UpprojMaps& maps, const UpprojArgs& a, int32_t sms, cudaStream_t stream);
cudaError_t launch_prefill_attn(const PrefillAttnMaps& maps, const PrefillAttnArgs& a, int32_t sms,
                                cudaStream_t stream);

}  // namespace mla
