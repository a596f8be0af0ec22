// Log-sum-exp merge of the partial rows of units that were split across
// workers (flash-decoding).  For a row with partial results (o_j, lse_j):
//     lse = ln sum_j exp(lse_j),   out = sum_j exp(lse_j - lse) o_j
// Units done by one piece were written by the attention kernel and are
// skipped; units with no visible key get out = 0 and lse = -inf.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_plan.cuh"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 8;

// Four consecutive partial values at element index idx of the partial rows
// (fp16 rows from the tensor-core kernels, fp32 rows from the fp32 path),
// as loaded (Raw) and as floats.
template <bool kF16>
struct PartRaw {
    using T = float4;
};
template <>
struct PartRaw<true> {
    using T = uint2;
};

template <bool kF16>
__device__ __forceinline__ typename PartRaw<kF16>::T load_raw4(const float* o_part, int64_t idx) {
    if constexpr (kF16) {
        return *reinterpret_cast<const uint2*>(reinterpret_cast<const __half*>(o_part) + idx);
    } else {
        return *reinterpret_cast<const float4*>(o_part + idx);
    }
}

template <bool kF16>
__device__ __forceinline__ float4 raw_to_f4(typename PartRaw<kF16>::T u) {
    if constexpr (kF16) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    } else {
        return u;
    }
}

template <bool kF16>
__device__ __forceinline__ float4 load_part4(const float* o_part, int64_t idx) {
    return raw_to_f4<kF16>(load_raw4<kF16>(o_part, idx));
}

// kHeld: pieces whose rows are loaded in the first round trip (8 when the
// grid is small enough that the extra registers cost no residency)
template <bool kF16Part, int kHeld>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    combine_kernel(int32_t Q, int32_t H, int32_t d_c, int32_t out_bf16, void* __restrict__ out,
                   float* __restrict__ lse, void* ws, WsLayout L) {
    // launched as a programmatic dependent of the attention kernel: its
    // launch overlaps the attention's tail; every read of the partials waits
    // here until that grid has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const WsView v = ws_view(ws, L);
    const int32_t u = blockIdx.x;   // the grid has exactly one block column per unit
    const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t QH = Q * H;
    const int32_t RB = units_per_seq(Q, H);
    const int32_t b = u / RB, rb = u % RB;
    const int32_t row = blockIdx.y * kWarpsPerBlock + warp;
    const int32_t rows_valid = min(kRowsPerUnit, QH - rb * kRowsPerUnit);
    if (row >= rows_valid) return;
    const int32_t p0 = v.unit_piece_begin[u], n = v.unit_piece_begin[u + 1] - p0;
    if (n == 1) return;
    const int64_t grow = (int64_t)b * QH + (int64_t)rb * kRowsPerUnit + row;

    // Every piece of the unit wrote finite partial rows, so the loads of the
    // first kHeld pieces' rows are issued together with the lse loads (one
    // memory round trip for a unit of up to kHeld pieces: fp16 rows take 8
    // registers per piece and lane); the weights are applied after.
    const float* lp = v.lse_part + (int64_t)p0 * kRowsPerUnit + row;   // lse of piece k: lp[k * 128]
    const int64_t ob = ((int64_t)p0 * kRowsPerUnit + row) * d_c;   // element index; piece k: + k * 128 * d_c
    const int64_t pstride = (int64_t)kRowsPerUnit * d_c;
    constexpr int kChunks = 4;   // each lane owns up to 4 chunks of 4 columns (d_c <= 512, a multiple of 4)
    constexpr int kCached = 8;   // the lse of the first kCached pieces are loaded together
    float lc[kCached];
#pragma unroll
    for (int k = 0; k < kCached; ++k) lc[k] = k < n ? lp[(int64_t)k * kRowsPerUnit] : -INFINITY;
    static_assert(kHeld == 2 || kHeld == kCached, "held pieces");
    using Raw = typename PartRaw<kF16Part>::T;
    Raw xr[kHeld][kChunks];
#pragma unroll
    for (int k = 0; k < kHeld; ++k) {
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            const int32_t c0 = lane * 4 + 128 * j;
            xr[k][j] = (c0 < d_c && k < n) ? load_raw4<kF16Part>(v.o_part, ob + (int64_t)k * pstride + c0) : Raw{};
        }
    }
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < kCached; ++k) m = fmaxf(m, lc[k]);
    for (int32_t k = kCached; k < n; ++k) m = fmaxf(m, lp[(int64_t)k * kRowsPerUnit]);
    float total_lse = -INFINITY;
    if (m != -INFINITY) {
        float z = 0.f;
#pragma unroll
        for (int k = 0; k < kCached; ++k) z += k < n ? expf(lc[k] - m) : 0.f;
        for (int32_t k = kCached; k < n; ++k) z += expf(lp[(int64_t)k * kRowsPerUnit] - m);
        total_lse = m + logf(z);
    }
    // out = sum_k w_k o_k with w_k = exp(lse_k - lse)
    float wc[kCached];
#pragma unroll
    for (int k = 0; k < kCached; ++k)
        wc[k] = (k < n && total_lse != -INFINITY && lc[k] != -INFINITY) ? expf(lc[k] - total_lse) : 0.f;
    // pieces past n hold zeros and weigh 0
    float4 acc[kChunks];
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
        const float4 x0 = raw_to_f4<kF16Part>(xr[0][j]), x1 = raw_to_f4<kF16Part>(xr[1][j]);
        acc[j].x = wc[0] * x0.x + wc[1] * x1.x;
        acc[j].y = wc[0] * x0.y + wc[1] * x1.y;
        acc[j].z = wc[0] * x0.z + wc[1] * x1.z;
        acc[j].w = wc[0] * x0.w + wc[1] * x1.w;
    }
#pragma unroll
    for (int k = 2; k < kHeld; k += 2) {
        if (k >= n) break;
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            const float4 y0 = raw_to_f4<kF16Part>(xr[k][j]), y1 = raw_to_f4<kF16Part>(xr[k + 1][j]);
            acc[j].x += wc[k] * y0.x + wc[k + 1] * y1.x;
            acc[j].y += wc[k] * y0.y + wc[k + 1] * y1.y;
            acc[j].z += wc[k] * y0.z + wc[k + 1] * y1.z;
            acc[j].w += wc[k] * y0.w + wc[k + 1] * y1.w;
        }
    }
    // acc += w0 o_k0 + w1 o_k1 for the remaining pieces, two at a time
    auto accumulate2 = [&](int32_t k0, float w0, int32_t k1, float w1) {
        float4 y0[kChunks], y1[kChunks];
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            const int32_t c0 = lane * 4 + 128 * j;
            const bool in = c0 < d_c;
            y0[j] = in && w0 != 0.f ? load_part4<kF16Part>(v.o_part, ob + k0 * pstride + c0)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            y1[j] = in && w1 != 0.f ? load_part4<kF16Part>(v.o_part, ob + k1 * pstride + c0)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            acc[j].x += w0 * y0[j].x + w1 * y1[j].x;
            acc[j].y += w0 * y0[j].y + w1 * y1[j].y;
            acc[j].z += w0 * y0[j].z + w1 * y1[j].z;
            acc[j].w += w0 * y0[j].w + w1 * y1[j].w;
        }
    };
#pragma unroll
    for (int k = kHeld; k < kCached; k += 2) {   // compile-time k: the weights stay in registers
        if (k >= n) break;
        accumulate2(k, wc[k], k + 1 < n ? k + 1 : k, k + 1 < n ? wc[k + 1] : 0.f);
    }
    for (int32_t k = kCached; k < n; ++k) {
        const float lk = lp[(int64_t)k * kRowsPerUnit];
        const float w = (total_lse != -INFINITY && lk != -INFINITY) ? expf(lk - total_lse) : 0.f;
        accumulate2(k, w, k, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
        const int32_t c0 = lane * 4 + 128 * j;
        if (c0 >= d_c) continue;
        if (out_bf16) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[j].x, acc[j].y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[j].z, acc[j].w);
            uint2 pk;
            pk.x = *reinterpret_cast<const uint32_t*>(&lo);
            pk.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + grow * d_c + c0) = pk;
        } else {   // fp32 output is only guaranteed 4-byte alignment
            float* dst = static_cast<float*>(out) + grow * d_c + c0;
            dst[0] = acc[j].x; dst[1] = acc[j].y; dst[2] = acc[j].z; dst[3] = acc[j].w;
        }
    }
    if (lse != nullptr && lane == 0) lse[grow] = total_lse;
}

}  // namespace

cudaError_t launch_combine(int32_t B, int32_t Q, int32_t H, int32_t d_c, int32_t out_dtype, bool f16_partials,
                           int32_t num_sms, void* out, float* lse, void* ws, const WsLayout& L,
                           cudaStream_t stream) {
    const int32_t U = B * units_per_seq(Q, H);
    if (U == 0) return cudaSuccess;
    const int32_t rows = min(kRowsPerUnit, Q * H);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(U, (rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int32_t obf = (int32_t)(out_dtype == 0);
    if (!f16_partials) return cudaLaunchKernelEx(&cfg, combine_kernel<false, 2>, Q, H, d_c, obf, out, lse, ws, L);
    // Holding 8 pieces per lane takes ~120 registers (2 blocks per SM): worth
    // it when the whole grid fits in one such wave (units split over many
    // workers, e.g. few sequences or few heads), not on large grids.
    const int64_t blocks = (int64_t)cfg.gridDim.x * cfg.gridDim.y;
    if (blocks <= 2 * (int64_t)num_sms)
        return cudaLaunchKernelEx(&cfg, combine_kernel<true, 8>, Q, H, d_c, obf, out, lse, ws, L);
    return cudaLaunchKernelEx(&cfg, combine_kernel<true, 2>, Q, H, d_c, obf, out, lse, ws, L);
}

}  // namespace mla
