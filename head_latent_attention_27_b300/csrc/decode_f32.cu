// fp32 decode on CUDA cores, for fp32 caches (any d_c <= 512 multiple of 4,
// d_r <= 64).  Same arithmetic as the tensor-core path, kept in fp32
// throughout so that results match an fp64 reference to ~1e-6:
//     x_s = scale (q_nope . c_s + q_rope . k_s),  online softmax,  u = sum a_s c_s
// One warp per query row; the lanes split the latent and RoPE dimensions.
// Each CTA is a worker of the plan and walks its pieces in order.
#include <math.h>
#include <stdint.h>

#include "decode_f32.cuh"
#include "decode_plan.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxDcPerLane = 16;  // 512 / 32
constexpr int kMaxDrPerLane = 2;   // 64 / 32

__global__ void __launch_bounds__(kWarps * 32) decode_f32_kernel(F32Args a, void* ws, WsLayout L) {
    WsView v = ws_view(ws, L);
    const int32_t w = blockIdx.x;
    const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t QH = a.Q * a.H;
    const int32_t RB = units_per_seq(a.Q, a.H);
    const int32_t width = a.d_c + a.d_r;
    const int32_t max_tokens = a.max_pages_per_seq * kTileTokens;
    const int32_t pb = v.worker_begin[w], pe = v.worker_begin[w + 1];
    for (int32_t p = pb; p < pe; ++p) {
        const Piece pc = v.pieces[p];
        const int32_t b = pc.unit / RB, rb = pc.unit % RB;
        const int32_t len = checked_len(a.seq_lens, b, max_tokens, &v.hdr->status);
        const int32_t rows_valid = min(kRowsPerUnit, QH - rb * kRowsPerUnit);
        for (int32_t row = warp; row < rows_valid; row += kWarps) {
            const int32_t qrow = rb * kRowsPerUnit + row;   // row within the sequence
            const int64_t grow = (int64_t)b * QH + qrow;    // row of q/out
            const int32_t vis = visible_len(len, a.Q, a.H, qrow);
            const int32_t s0 = pc.t_begin * kTileTokens;
            const int32_t s1 = min(pc.t_end * kTileTokens, vis);
            float qn[kMaxDcPerLane], qr[kMaxDrPerLane], o[kMaxDcPerLane];
#pragma unroll
            for (int i = 0; i < kMaxDcPerLane; ++i) {
                const int32_t k = lane + 32 * i;
                qn[i] = k < a.d_c ? a.q_nope[grow * a.d_c + k] : 0.f;
                o[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < kMaxDrPerLane; ++i) {
                const int32_t k = lane + 32 * i;
                qr[i] = k < a.d_r ? a.q_rope[grow * a.d_r + k] : 0.f;
            }
            float m = -INFINITY, l = 0.f;
            for (int32_t s = s0; s < s1; ++s) {
                const int32_t page = a.page_table[(int64_t)b * a.max_pages_per_seq + s / kTileTokens];
                if (page < 0 || page >= a.num_pages) {
                    atomicCAS(&v.hdr->status, 0, 1);
                    continue;
                }
                const float* crow = a.cache + ((int64_t)page * kTileTokens + s % kTileTokens) * width;
                float c[kMaxDcPerLane];
                float dot = 0.f;
#pragma unroll
                for (int i = 0; i < kMaxDcPerLane; ++i) {
                    const int32_t k = lane + 32 * i;
                    c[i] = k < a.d_c ? crow[k] : 0.f;
                    dot = fmaf(qn[i], c[i], dot);
                }
#pragma unroll
                for (int i = 0; i < kMaxDrPerLane; ++i) {
                    const int32_t k = lane + 32 * i;
                    if (k < a.d_r) dot = fmaf(qr[i], crow[a.d_c + k], dot);
                }
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, d);
                const float x = dot * a.scale;
                const float m_new = fmaxf(m, x);
                const float corr = expf(m - m_new);  // 0 on the first key
                const float pexp = expf(x - m_new);
                l = l * corr + pexp;
#pragma unroll
                for (int i = 0; i < kMaxDcPerLane; ++i) o[i] = fmaf(pexp, c[i], o[i] * corr);
                m = m_new;
            }
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const float row_lse = l > 0.f ? m + logf(l) : -INFINITY;
            float* dst;
            if (pc.slot < 0) {
                dst = a.out + grow * a.d_c;
                if (a.lse && lane == 0) a.lse[grow] = row_lse;
            } else {
                dst = v.o_part + ((int64_t)pc.slot * kRowsPerUnit + row) * a.d_c;
                if (lane == 0) v.lse_part[(int64_t)pc.slot * kRowsPerUnit + row] = row_lse;
            }
#pragma unroll
            for (int i = 0; i < kMaxDcPerLane; ++i) {
                const int32_t k = lane + 32 * i;
                if (k < a.d_c) dst[k] = o[i] * inv_l;
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode_f32(const F32Args& a, int32_t num_workers, void* ws, const WsLayout& L,
                              cudaStream_t stream) {
    decode_f32_kernel<<<num_workers, kWarps * 32, 0, stream>>>(a, ws, L);
    return cudaGetLastError();
}

}  // namespace mla
