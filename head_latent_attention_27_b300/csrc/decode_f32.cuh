#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "decode_plan.cuh"

namespace mla {

struct F32Args {
    const float* cache;
    const int32_t* page_table;
    const int32_t* seq_lens;
    const float* q_nope;
    const float* q_rope;
    float* out;
    float* lse;
    int32_t num_pages;
    int32_t max_pages_per_seq;
    int32_t d_c;
    int32_t d_r;
    int32_t Q;
    int32_t H;
    float scale;
};

cudaError_t launch_decode_f32(const F32Args& a, int32_t num_workers, void* ws, const WsLayout& L,
                              cudaStream_t stream);

}  // namespace mla
