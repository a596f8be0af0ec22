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
        // sum of squares: lane k sums its contiguous block of d_c/32
        // elements in order (the order of the 576-wide and low-precision
        // kernels), strided when d_c is not a multiple of 32
        float ss = 0.f;
        if (a.d_c % 32 == 0) {
            const int32_t per = a.d_c >> 5;
            for (int32_t i = 0; i < per; ++i) {
                const float v = load_f(x + lane * per + i);
                ss = fmaf(v, v, ss);
            }
        } else {
            for (int32_t k = lane; k < a.d_c; k += 32) {
                const float v = load_f(x + k);
                ss = fmaf(v, v, ss);
            }
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

// RoPE rotation of pair i = (x0, x1) at position pos (flags bit 2), angle
// reduced modulo 2 pi in fp64 as described at the top of the file.
__device__ __forceinline__ void rope_pair(const AppendArgs& a, int32_t pos, int32_t i, float x0, float x1,
                                          float& y0, float& y1) {
    y0 = x0;
    y1 = x1;
    if (a.flags & 2u) {
        constexpr double kTwoPi = 6.283185307179586476925286766559;
        const double ang = (double)pos * a.theta[i];
        const double r = fma(-rint(ang * (1.0 / kTwoPi)), kTwoPi, ang);   // in [-pi, pi]
        float sf, cf;
        sincosf((float)r, &sf, &cf);
        y0 = x0 * cf - x1 * sf;
        y1 = x0 * sf + x1 * cf;
    }
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* v) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// The bf16-input, bf16-cache append at the 576-wide row (d_c = 512,
// d_r = 64): lane k owns latent elements [16k, 16k + 16) (two 16-byte loads
// and stores) and RoPE pair k (one 4-byte load and store).  The token's
// inputs are loaded before its page is looked up, so their latency overlaps
// the index loads.  Sum of squares: each lane's 16 terms in order, then a
// butterfly over the lanes (the low-precision append uses the same order,
// so both form the same bf16 row).
__global__ void __launch_bounds__(kWarps * 32)
    append_bf16_row_kernel(AppendArgs a, const __nv_bfloat16* __restrict__ ckv, const __nv_bfloat16* __restrict__ kr,
                           __nv_bfloat16* __restrict__ cache) {
    const int32_t t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int32_t lane = threadIdx.x & 31;
    if (t >= a.T) return;
    const uint4* xv = reinterpret_cast<const uint4*>(ckv + (int64_t)t * 512) + 2 * lane;
    const uint4 u0 = xv[0], u1 = xv[1];
    const uint32_t kp = reinterpret_cast<const uint32_t*>(kr + (int64_t)t * 64)[lane];
    const int32_t b = a.seq_ids[t], pos = a.positions[t];
    if (b < 0 || b >= a.num_seqs || pos < 0 || pos >= a.max_pages_per_seq * a.page_size) return;
    const int32_t page = a.page_table[(int64_t)b * a.max_pages_per_seq + pos / a.page_size];
    if (page < 0 || page >= a.num_pages) return;
    __nv_bfloat16* row = cache + ((int64_t)page * a.page_size + pos % a.page_size) * 576;

    float v[16];
    unpack_bf16x8(u0, v);
    unpack_bf16x8(u1, v + 8);
    if (a.flags & 1u) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
        const float inv_rms = 1.f / sqrtf(ss / 512.f + a.eps);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = v[i] * inv_rms * (a.gamma ? a.gamma[16 * lane + i] : 1.f);
    }
    uint4* rv = reinterpret_cast<uint4*>(row) + 2 * lane;
    rv[0] = make_uint4(pack_bf16x2_rn(v[0], v[1]), pack_bf16x2_rn(v[2], v[3]), pack_bf16x2_rn(v[4], v[5]),
                       pack_bf16x2_rn(v[6], v[7]));
    rv[1] = make_uint4(pack_bf16x2_rn(v[8], v[9]), pack_bf16x2_rn(v[10], v[11]), pack_bf16x2_rn(v[12], v[13]),
                       pack_bf16x2_rn(v[14], v[15]));
    float y0, y1;
    rope_pair(a, pos, lane, __uint_as_float(kp << 16), __uint_as_float(kp & 0xffff0000u), y0, y1);
    reinterpret_cast<uint32_t*>(row + 512)[lane] = pack_bf16x2_rn(y0, y1);
}

// Low-precision cache row (656 bytes): the 512 latent values as E4M3 codes,
// one fp32 scale per 128-element group, then the RoPE key in bf16.  The row
// is first formed exactly as for the bf16 cache (same arithmetic and
// reduction order, one rounding to bf16), and those bf16 values are
// quantised: s = amax / 448 (fp32 division, s = 1 for an all-zero group),
// code = E4M3(x / s) with the quotient rounded to fp32 first, then to the
// nearest E4M3 value (ties to even, saturating at +-448).  One warp per
// token; lane k owns latent elements [16k, 16k + 16), so a group is 8 lanes.
template <typename Tin>
__global__ void __launch_bounds__(kWarps * 32)
    append_fp8_kernel(AppendArgs a, const Tin* __restrict__ ckv, const Tin* __restrict__ kr, uint8_t* __restrict__ cache) {
    const int32_t t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int32_t lane = threadIdx.x & 31;
    if (t >= a.T) return;
    const int32_t b = a.seq_ids[t], pos = a.positions[t];
    if (b < 0 || b >= a.num_seqs || pos < 0 || pos >= a.max_pages_per_seq * a.page_size) return;
    const int32_t page = a.page_table[(int64_t)b * a.max_pages_per_seq + pos / a.page_size];
    if (page < 0 || page >= a.num_pages) return;
    uint8_t* row = cache + ((int64_t)page * a.page_size + pos % a.page_size) * kFp8RowBytes;
    const Tin* x = ckv + (int64_t)t * kFp8Dc;

    float inv_rms = 1.f;
    if (a.flags & 1u) {   // same summation order as the bf16 row: lane k's 16 elements, then the lanes
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float v = load_f(x + 16 * lane + i);
            ss = fmaf(v, v, ss);
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
        inv_rms = 1.f / sqrtf(ss / (float)kFp8Dc + a.eps);
    }
    float y[16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int32_t k = 16 * lane + i;
        float v = load_f(x + k);
        if (a.flags & 1u) v = v * inv_rms * (a.gamma ? a.gamma[k] : 1.f);
        y[i] = __bfloat162float(__float2bfloat16_rn(v));   // the bf16 row value
        amax = fmaxf(amax, fabsf(y[i]));
    }
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t lo, hi;
        const float q0 = __fdiv_rn(y[4 * j], s), q1 = __fdiv_rn(y[4 * j + 1], s);
        const float q2 = __fdiv_rn(y[4 * j + 2], s), q3 = __fdiv_rn(y[4 * j + 3], s);
        asm("{\n\t.reg .b16 h;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %2, %1;\n\tcvt.u32.u16 %0, h;\n\t}"
            : "=r"(lo) : "f"(q0), "f"(q1));
        asm("{\n\t.reg .b16 h;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %2, %1;\n\tcvt.u32.u16 %0, h;\n\t}"
            : "=r"(hi) : "f"(q2), "f"(q3));
        w[j] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(row + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
    if ((lane & 7) == 0) *reinterpret_cast<float*>(row + kFp8Dc + 4 * (lane >> 3)) = s;

    // shared RoPE key (bf16), as in the bf16 row
    const Tin* kx = kr + (int64_t)t * a.d_r;
    __nv_bfloat16* kr_out = reinterpret_cast<__nv_bfloat16*>(row + kFp8Dc + 16);
    for (int32_t i = lane; i < a.d_r / 2; i += 32) {
        const float x0 = load_f(kx + 2 * i), x1 = load_f(kx + 2 * i + 1);
        float y0 = x0, y1 = x1;
        if (a.flags & 2u) {
            constexpr double kTwoPi = 6.283185307179586476925286766559;
            const double ang = (double)pos * a.theta[i];
            const double r = fma(-rint(ang * (1.0 / kTwoPi)), kTwoPi, ang);
            float sf, cf;
            sincosf((float)r, &sf, &cf);
            y0 = x0 * cf - x1 * sf;
            y1 = x0 * sf + x1 * cf;
        }
        kr_out[2 * i] = __float2bfloat16_rn(y0);
        kr_out[2 * i + 1] = __float2bfloat16_rn(y1);
    }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, const void* ckv, const void* kr, int32_t in_dtype,
                          int32_t cache_dtype, void* cache, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    const dim3 grid((a.T + kWarps - 1) / kWarps);
    const dim3 block(kWarps * 32);
    if (cache_dtype == 2) {   // low-precision (E4M3 latent) rows
        if (in_dtype == 0)
            append_fp8_kernel<__nv_bfloat16><<<grid, block, 0, stream>>>(
                a, static_cast<const __nv_bfloat16*>(ckv), static_cast<const __nv_bfloat16*>(kr),
                static_cast<uint8_t*>(cache));
        else
            append_fp8_kernel<float><<<grid, block, 0, stream>>>(a, static_cast<const float*>(ckv),
                                                                 static_cast<const float*>(kr),
                                                                 static_cast<uint8_t*>(cache));
        return cudaGetLastError();
    }
    const bool aligned = ((reinterpret_cast<uintptr_t>(ckv) | reinterpret_cast<uintptr_t>(cache)) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(kr) & 3u) == 0;
    if (in_dtype == 0 && cache_dtype == 0 && a.d_c == 512 && a.d_r == 64 && aligned)
        append_bf16_row_kernel<<<grid, block, 0, stream>>>(a, static_cast<const __nv_bfloat16*>(ckv),
                                                           static_cast<const __nv_bfloat16*>(kr),
                                                           static_cast<__nv_bfloat16*>(cache));
    else if (in_dtype == 0 && cache_dtype == 0)
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
