#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// Low-precision cache row: 512 E4M3 latent codes, 4 fp32 group scales (one
// per 128 latent elements), 64 bf16 RoPE values = 656 bytes.
constexpr int kFp8Dc = 512;
constexpr int kFp8Dr = 64;
constexpr int kFp8Group = 128;
constexpr int kFp8RowBytes = kFp8Dc + 4 * (kFp8Dc / kFp8Group) + 2 * kFp8Dr;

struct AppendArgs {
    const int32_t* seq_ids;
    const int32_t* positions;
    const int32_t* page_table;
    const float* gamma;
    int32_t T;
    int32_t num_seqs;
    int32_t num_pages;
    int32_t page_size;
    int32_t max_pages_per_seq;
    int32_t d_c;
    int32_t d_r;
    uint32_t flags;
    float eps;
    // RoPE frequency of pair i (i < d_r/2), in fp64, computed on the host:
    // theta_i = base^(-2i/d_r), adjusted by YaRN when the context is extended.
    double theta[32];
};

cudaError_t launch_append(const AppendArgs& a, const void* ckv, const void* kr, int32_t in_dtype,
                          int32_t cache_dtype, void* cache, cudaStream_t stream);

}  // namespace mla
