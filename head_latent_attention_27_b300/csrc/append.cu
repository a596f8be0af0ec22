// Cache append: for every new token, RMSNorm the raw latent, rotate the raw
// shared RoPE key at the token's position, and write the row [c_kv || k_R]
// into its page slot.  (DeepSeek-V2 analysis page: RMSNorm after the
// compressed latent, section 1.2; shared k^R with RoPE, cached rotated,
// section 1.3 eq 14-15; RoPE pairs (2i, 2i+1), DeepSeek-V3 model structure
// page, section 2(3).)
//
// One warp per token.  The latent part is fp32 arithmetic with one rounding
// to the cache dtype.  The RoPE frequencies (plain, or YaRN-adjusted for an
// extended context) are computed once on the host in fp64; per pair the angle
// pos * theta_i is formed and reduced modulo 2 pi in fp64 (three operations),
// and sine and cosine are taken in fp32 of the reduced angle, so large
// positions keep full accuracy without fp64 transcendental functions (slow
// on this GPU).
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "append.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

template <typename T>
__device__ __forceinline__ float load_f(const T* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void store_f(T* p, float v);
template <>
__device__ __forceinline__ void store_f<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_f<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename Tin, typename Tc>
__global__ void __launch_bounds__(kWarps * 32)
    append_kernel(AppendArgs a, const Tin* __restrict__ ckv, const Tin* __restrict__ kr, Tc* __restrict__ cache) {
    const int32_t t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int32_t lane = threadIdx.x & 31;
    if (t >= a.T) return;
    const int32_t b = a.seq_ids[t], pos = a.positions[t];
    if (b < 0 || b >= a.num_seqs || pos < 0 || pos >= a.max_pages_per_seq * a.page_size) return;
    const int32_t page = a.page_table[(int64_t)b * a.max_pages_per_seq + pos / a.page_size];
    if (page < 0 || page >= a.num_pages) return;
    const int32_t width = a.d_c + a.d_r;
    Tc* row = cache + ((int64_t)page * a.page_size + pos % a.page_size) * width;
    const Tin* x = ckv + (int64_t)t * a.d_c;

    // latent: optional RMSNorm
    float inv_rms = 1.f;
    if (a.flags & 1u) {
        float ss = 0.f;
        for (int32_t k = lane; k < a.d_c; k += 32) {
            const float v = load_f(x + k);
            ss = fmaf(v, v, ss);
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
        inv_rms = 1.f / sqrtf(ss / (float)a.d_c + a.eps);
    }
    for (int32_t k = lane; k < a.d_c; k += 32) {
        float v = load_f(x + k);
        if (a.flags & 1u) v = v * inv_rms * (a.gamma ? a.gamma[k] : 1.f);
        store_f(row + k, v);
    }

    // shared RoPE key: pair i = (2i, 2i+1)
    const Tin* kx = kr + (int64_t)t * a.d_r;
    for (int32_t i = lane; i < a.d_r / 2; i += 32) {
        const float x0 = load_f(kx + 2 * i), x1 = load_f(kx + 2 * i + 1);
        float y0 = x0, y1 = x1;
        if (a.flags & 2u) {
            constexpr double kTwoPi = 6.283185307179586476925286766559;
            const double ang = (double)pos * a.theta[i];
            const double r = fma(-rint(ang * (1.0 / kTwoPi)), kTwoPi, ang);   // in [-pi, pi]
            float sf, cf;
            sincosf((float)r, &sf, &cf);
            y0 = x0 * cf - x1 * sf;
            y1 = x0 * sf + x1 * cf;
        }
        store_f(row + a.d_c + 2 * i, y0);
        store_f(row + a.d_c + 2 * i + 1, y1);
    }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, const void* ckv, const void* kr, int32_t in_dtype,
                          int32_t cache_dtype, void* cache, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    const dim3 grid((a.T + kWarps - 1) / kWarps);
    const dim3 block(kWarps * 32);
    if (in_dtype == 0 && cache_dtype == 0)
        append_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, block, 0, stream>>>(
            a, static_cast<const __nv_bfloat16*>(ckv), static_cast<const __nv_bfloat16*>(kr),
            static_cast<__nv_bfloat16*>(cache));
    else if (in_dtype == 1 && cache_dtype == 0)
        append_kernel<float, __nv_bfloat16><<<grid, block, 0, stream>>>(
            a, static_cast<const float*>(ckv), static_cast<const float*>(kr), static_cast<__nv_bfloat16*>(cache));
    else if (in_dtype == 0 && cache_dtype == 1)
        append_kernel<__nv_bfloat16, float><<<grid, block, 0, stream>>>(
            a, static_cast<const __nv_bfloat16*>(ckv), static_cast<const __nv_bfloat16*>(kr),
            static_cast<float*>(cache));
    else
        append_kernel<float, float><<<grid, block, 0, stream>>>(
            a, static_cast<const float*>(ckv), static_cast<const float*>(kr), static_cast<float*>(cache));
    return cudaGetLastError();
}

}  // namespace mla
