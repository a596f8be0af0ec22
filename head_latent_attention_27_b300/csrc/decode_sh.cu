// Absorbed MLA decode for units of at most 16 query rows (decode_sh.cuh).
//
// One CTA per SM, a worker of the balanced plan (decode_plan.cuh), walks its
// pieces in order.  Per piece it streams the unit's cache tiles through a
// TMA ring of 32-token stages (half a 64-token page: 9 boxes of 64 dims x
// 32 tokens, 128-byte swizzle, 36 KB) and runs, per stage,
//     S   [16 x 32]  = Q [16 x 576] . K^T            (m16n8k16 bf16 MMAs)
//     P              = online softmax of S * scale    (fp32, in registers)
//     O   [16 x 512] += P [16 x 32] . V [32 x 512]    (m16n8k16 bf16 MMAs)
// where K = [c || k^R] and V = c are the same cached rows.
//
// Warps (384 threads, three warpgroups):
//   warps 0-3, 4-7  two consumer groups taking alternate stages; each has
//                   its own running max / sum / O and the two are merged
//                   at the end of a piece (flash-decoding merge inside the
//                   CTA).  In a group, warp w
//                     - scores the stage over dims [144w, 144w + 144): its
//                       query fragments stay in registers for the piece;
//                       the four partial score tiles are summed through
//                       shared memory (one mbarrier wait), every warp
//                       sums them in the same order, so all four hold the
//                       same S, the same max and the same P;
//                     - keeps P as the A operand of the PV MMAs (the
//                       accumulator layout of two adjacent 8-token score
//                       tiles is the A layout of one 16-token k-step);
//                     - accumulates O for dims [128w, 128w + 128).
//   warp 8          TMA producer (one lane); warps 9-11 idle (they only
//                   give their registers to the consumers).
// Every wait is bounded (ptx.cuh: bounded_wait): on a timeout the kernel
// records MLA_ERR_TIMEOUT, waits (time-limited) for its own copies in
// flight and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "decode_sh.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int RM = kShMaxRows;        // 16 rows: one m16 tile
constexpr int ST = 32;                // tokens per stage
constexpr int NSTAGE = 4;
constexpr int kGroups = 2;
constexpr int kGroupWarps = 4;
constexpr int kProducerWarp = kGroups * kGroupWarps;   // warp 8, first of the producer warpgroup
constexpr int kThreads = 32 * (kProducerWarp + 4);     // 384: three warpgroups
// Register split (setmaxnreg): the launch gives every thread the same
// count; the producer warpgroup (one busy lane) hands most of its share to
// the two consumer warpgroups, whose query fragments, scores and O tile
// would not fit the 168 registers of a three-warpgroup launch.  The shares
// add up to the launch's total of 384 x 168; the launcher checks the
// compiled count before every launch.
constexpr int kProducerRegs = 24;
constexpr int kConsumerRegs = 240;
constexpr int kLaunchRegs = 168;
static_assert(4 * kProducerRegs + 8 * kConsumerRegs <= 12 * kLaunchRegs, "register split within the launch");
constexpr int kBoxes = 9;                               // 8 latent boxes + the RoPE box
constexpr int kQkDims = 576 / kGroupWarps;              // 144 dims scored per warp
constexpr int kQkSteps = kQkDims / 16;                  // 9 k-steps
constexpr int kPvDims = 512 / kGroupWarps;              // 128 dims accumulated per warp
constexpr int kPvTiles = kPvDims / 8;                   // 16 n-tiles

constexpr uint32_t BOX_BYTES = ST * 128;                // 32 tokens x 64 bf16
constexpr uint32_t STAGE_BYTES = kBoxes * BOX_BYTES;    // 36864
constexpr uint32_t SP_WARP = RM * ST * 4;               // one warp's partial S (fp32), 2 KB
constexpr uint32_t OFF_KV = 0;
constexpr uint32_t OFF_SP = OFF_KV + NSTAGE * STAGE_BYTES;                  // [group][2][warp]
constexpr uint32_t OFF_MO = OFF_SP + kGroups * 2 * kGroupWarps * SP_WARP;   // group 1's O: [warp][16][lane] float4
constexpr uint32_t MO_BYTES = kGroupWarps * kPvTiles * 32 * 16;
constexpr uint32_t OFF_ML = OFF_MO + MO_BYTES;          // group 1's (m, l) per lane: float4
constexpr uint32_t OFF_BAR = OFF_ML + 32 * 16;
enum : int {
    B_FULL = 0,
    B_EMPTY = NSTAGE,
    B_SPFULL = 2 * NSTAGE,   // [group][buffer] the group's four partial score tiles written
    B_MFULL = B_SPFULL + 2 * kGroups,
    B_MFREE,
    NUM_BARS
};
constexpr uint32_t OFF_ABORT = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t SMEM_USED = OFF_ABORT + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;       // + alignment slack

static_assert(STAGE_BYTES % 1024 == 0 && OFF_SP % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "fits in 227 KB");
static_assert(kQkDims % 16 == 0 && (512 % kQkDims) % 16 == 0, "a k-step never straddles latent and RoPE dims");

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: O and l are rescaled only when the max grows by > 2^8

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// (x, y) += (a, b) and (x*a + c, y*b + d) as packed f32x2 operations, each
// lane rounded to nearest like its scalar form.
__device__ __forceinline__ void add2_to(float& x, float& y, float a, float b) {
    asm("{\n\t.reg .b64 p, q;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %3};\n\t"
        "add.rn.f32x2 p, p, q;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "+f"(x), "+f"(y) : "f"(a), "f"(b));
}
__device__ __forceinline__ float2 fma2(float x, float y, float a, float b, float c, float d) {
    float2 r;
    asm("{\n\t.reg .b64 p, q, w;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\tmov.b64 w, {%6, %7};\n\t"
        "fma.rn.f32x2 p, p, q, w;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "=f"(r.x), "=f"(r.y) : "f"(x), "f"(y), "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// D += A . B, m16n8k16, bf16 operands, fp32 accumulator.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
    const bool ok = bounded_wait<kCluster>(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

// Wait limited by time only: drains copies already in flight before exit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 200000000ull) return;
    }
}

// Byte offset, inside a stage, of the 16-byte chunk `chunk` (8 dims) of
// token `tok` in box `box` (128-byte swizzle: chunk ^ (row & 7)).
__device__ __forceinline__ uint32_t chunk_off(uint32_t box, uint32_t tok, uint32_t chunk) {
    return box * BOX_BYTES + tok * 128u + ((chunk ^ (tok & 7u)) << 4);
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_sh_kernel(const __grid_constant__ CUtensorMap tm_kv, const ShArgs a, void* ws, const WsLayout L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

    WsView v = ws_view(ws, L);
    int* status = &v.hdr->status;
    const int32_t pb = v.worker_begin[blockIdx.x], pe = v.worker_begin[blockIdx.x + 1];
    const int32_t QH = a.Q * a.H;
    const int32_t max_tokens = a.max_pages_per_seq * kTileTokens;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), kGroupWarps);
        }
        for (int i = 0; i < 2 * kGroups; ++i) mbar_init(bar(B_SPFULL + i), kGroupWarps);
        mbar_init(bar(B_MFULL), kGroupWarps);
        mbar_init(bar(B_MFREE), kGroupWarps);
        *abort_flag = 0;
        fence_mbar_init_cluster();
    }
    __syncthreads();

    if (warp >= kProducerWarp) {
        regs_dec<kProducerRegs>();
        if (warp == kProducerWarp && lane == 0) {
            tma_prefetch_desc(&tm_kv);
            const uint64_t pol = l2_policy_evict_first();
            uint32_t cnt = 0;
            bool ok = true;
            for (int32_t p = pb; p < pe && ok; ++p) {
                const Piece pc = v.pieces[p];
                const int32_t b = pc.unit;   // Q*H <= 16: one unit per sequence
                for (int32_t t = pc.t_begin; t < pc.t_end && ok; ++t) {
                    int32_t page = a.page_table[(int64_t)b * a.max_pages_per_seq + t];
                    if (page < 0 || page >= a.num_pages) {
                        atomicCAS(status, 0, 1 /* MLA_ERR_INVALID_ARG */);
                        page = 0;   // keep the stream's protocol; the result is flagged
                    }
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t st = cnt % NSTAGE;
                        ok = bounded_wait(bar(B_EMPTY + st), ((cnt / NSTAGE) & 1u) ^ 1u, abort_flag, status);
                        if (!ok) break;
                        mbar_arrive_expect_tx(bar(B_FULL + st), STAGE_BYTES);
                        const uint32_t dst = sbase + OFF_KV + st * STAGE_BYTES;
                        const int32_t y = page * kTileTokens + hh * ST;
#pragma unroll
                        for (int kb = 0; kb < kBoxes; ++kb)
                            tma_load_2d(dst + kb * BOX_BYTES, &tm_kv, bar(B_FULL + st), 64 * kb, y, pol);
                        ++cnt;
                    }
                }
            }
            // copies in flight land before the CTA exits (immediate on the
            // normal path: the consumers waited for every stage)
            for (uint32_t i = cnt > (uint32_t)NSTAGE ? cnt - NSTAGE : 0u; i < cnt; ++i)
                drain_wait(bar(B_FULL + i % NSTAGE), (i / NSTAGE) & 1u);
        }
    } else {
        regs_inc<kConsumerRegs>();
        const int gi = warp / kGroupWarps, wq = warp % kGroupWarps;
        const int g = lane >> 2, c = lane & 3;
        const float sl2 = a.scale_log2;
        const uint32_t* qn = static_cast<const uint32_t*>(a.q_nope);   // bf16 pairs, 256 per row
        const uint32_t* qr = static_cast<const uint32_t*>(a.q_rope);   // bf16 pairs, 32 per row
        uint32_t cnt = 0, gst = 0, merges = 0;   // gst: stages this group has scored
        bool ok = true;
        for (int32_t p = pb; p < pe && ok; ++p) {
            const Piece pc = v.pieces[p];
            const int32_t b = pc.unit;
            const int32_t len = checked_len(a.seq_lens, b, max_tokens, status);
            const int32_t rows = QH < RM ? QH : RM;
            const int32_t r0 = g, r1 = g + 8;
            const int32_t vis0 = r0 < rows ? visible_len(len, a.Q, a.H, r0) : 0;
            const int32_t vis1 = r1 < rows ? visible_len(len, a.Q, a.H, r1) : 0;
            const int32_t vis_lo = visible_len(len, a.Q, a.H, 0);          // fewest keys of the unit
            const int32_t vis_hi = visible_len(len, a.Q, a.H, rows - 1);   // most keys of the unit

            // query fragments of this warp's 144 dims (A layout of m16n8k16:
            // regs 0/1 rows g / g+8 at k = 2c, regs 2/3 the same at k = 8 + 2c)
            uint32_t qf[kQkSteps][4];
            {
                const int64_t g0 = (int64_t)b * QH + r0, g1 = (int64_t)b * QH + r1;
#pragma unroll
                for (int kk = 0; kk < kQkSteps; ++kk) {
                    const int d = kQkDims * wq + 16 * kk + 2 * c;   // even; d and d + 8 on the same side of 512
                    if (d < 512) {
                        qf[kk][0] = r0 < rows ? qn[g0 * 256 + d / 2] : 0u;
                        qf[kk][1] = r1 < rows ? qn[g1 * 256 + d / 2] : 0u;
                        qf[kk][2] = r0 < rows ? qn[g0 * 256 + (d + 8) / 2] : 0u;
                        qf[kk][3] = r1 < rows ? qn[g1 * 256 + (d + 8) / 2] : 0u;
                    } else {
                        qf[kk][0] = r0 < rows ? qr[g0 * 32 + (d - 512) / 2] : 0u;
                        qf[kk][1] = r1 < rows ? qr[g1 * 32 + (d - 512) / 2] : 0u;
                        qf[kk][2] = r0 < rows ? qr[g0 * 32 + (d + 8 - 512) / 2] : 0u;
                        qf[kk][3] = r1 < rows ? qr[g1 * 32 + (d + 8 - 512) / 2] : 0u;
                    }
                }
            }
            float o[kPvTiles][4];
#pragma unroll
            for (int n = 0; n < kPvTiles; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            float m0 = -INFINITY, m1 = -INFINITY;   // running max (log2 units) of rows r0, r1
            float l0 = 0.f, l1 = 0.f;               // this thread's share of the row sums

            const int32_t nst = 2 * (pc.t_end - pc.t_begin);
            for (int32_t si = 0; si < nst; ++si, ++cnt) {
                if ((int)(cnt % kGroups) != gi) continue;
                const uint32_t st = cnt % NSTAGE;
                ok = warp_wait(bar(B_FULL + st), (cnt / NSTAGE) & 1u, abort_flag, status);
                if (!ok) break;
                const uint32_t sb = sbase + OFF_KV + st * STAGE_BYTES;

                // 1. partial scores over this warp's dims, 4 n-tiles of 8 tokens
                float acc[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < kQkSteps; ++kk) {
                    const int d0 = kQkDims * wq + 16 * kk;
                    const uint32_t box = (uint32_t)d0 >> 6;
                    const uint32_t chunk = (((uint32_t)d0 & 63u) >> 3) + (((uint32_t)lane >> 3) & 1u);
#pragma unroll
                    for (int pr = 0; pr < 2; ++pr) {
                        // matrices: (n-tile 2pr, k lo), (2pr, k hi), (2pr+1, k lo), (2pr+1, k hi)
                        const uint32_t tok = 8u * (2u * pr + ((uint32_t)lane >> 4)) + ((uint32_t)lane & 7u);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(sb + chunk_off(box, tok, chunk), b0, b1, b2, b3);
                        mma16816(acc[2 * pr], qf[kk], b0, b1);
                        mma16816(acc[2 * pr + 1], qf[kk], b2, b3);
                    }
                }
                // 2. sum the group's four partials (same order in every warp)
                //    (double buffer: a warp writes buffer k & 1 of its k-th
                //    stage only after all four passed stage k - 1, i.e.
                //    finished reading stage k - 2's partials)
                const uint32_t spb = gst & 1u;
                float4* sp = reinterpret_cast<float4*>(smem + OFF_SP + (gi * 2 + spb) * kGroupWarps * SP_WARP);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    sp[(wq * 4 + j) * 32 + lane] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_SPFULL + gi * 2 + spb));
                ok = warp_wait(bar(B_SPFULL + gi * 2 + spb), (gst >> 1) & 1u, abort_flag, status);
                if (!ok) break;
                ++gst;
                float s[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 t = sp[j * 32 + lane];
                    s[j][0] = t.x;
                    s[j][1] = t.y;
                    s[j][2] = t.z;
                    s[j][3] = t.w;
#pragma unroll
                    for (int w2 = 1; w2 < kGroupWarps; ++w2) {
                        const float4 u = sp[(w2 * 4 + j) * 32 + lane];
                        add2_to(s[j][0], s[j][1], u.x, u.y);
                        add2_to(s[j][2], s[j][3], u.z, u.w);
                    }
                }
                // 3. mask keys past each row's visible length; tile max per row
                const int32_t tok0 = (2 * pc.t_begin + si) * ST;
                if (tok0 + ST > vis_lo) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int32_t t = tok0 + 8 * j + 2 * c;
                        s[j][0] = t < vis0 ? s[j][0] : -INFINITY;
                        s[j][1] = t + 1 < vis0 ? s[j][1] : -INFINITY;
                        s[j][2] = t < vis1 ? s[j][2] : -INFINITY;
                        s[j][3] = t + 1 < vis1 ? s[j][3] : -INFINITY;
                    }
                }
                float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
                float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
                mx0 = fmaxf(mx0, fmaxf(fmaxf(s[2][0], s[2][1]), fmaxf(s[3][0], s[3][1])));
                mx1 = fmaxf(mx1, fmaxf(fmaxf(s[2][2], s[2][3]), fmaxf(s[3][2], s[3][3])));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                // 4. online softmax with a lazy maximum: the running max m (log2
                //    units) moves, and O and l are rescaled, only when the tile
                //    max exceeds it by more than 2^8; P = 2^(x - m) <= 2^8 then
                //    (bf16 holds it exactly enough; O, l and m stay consistent)
                const float t0 = mx0 * sl2, t1 = mx1 * sl2;
                float f0 = 1.f, f1 = 1.f;
                if (t0 > m0 + kRescaleThreshold) {
                    if (m0 != -INFINITY) f0 = fast_exp2(m0 - t0);
                    m0 = t0;
                }
                if (t1 > m1 + kRescaleThreshold) {
                    if (m1 != -INFINITY) f1 = fast_exp2(m1 - t1);
                    m1 = t1;
                }
                if (__any_sync(0xffffffffu, f0 != 1.f || f1 != 1.f)) {
                    l0 *= f0;
                    l1 *= f1;
#pragma unroll
                    for (int n = 0; n < kPvTiles; ++n) {
                        o[n][0] *= f0;
                        o[n][1] *= f0;
                        o[n][2] *= f1;
                        o[n][3] *= f1;
                    }
                }
                const float neg0 = m0 == -INFINITY ? 0.f : -m0, neg1 = m1 == -INFINITY ? 0.f : -m1;
                uint32_t pa[2][4];
                float ls0 = 0.f, ls0b = 0.f, ls1 = 0.f, ls1b = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x0 = fma2(s[j][0], s[j][1], sl2, sl2, neg0, neg0);
                    const float2 x1 = fma2(s[j][2], s[j][3], sl2, sl2, neg1, neg1);
                    const float p00 = fast_exp2(x0.x), p01 = fast_exp2(x0.y);   // exp2(-inf) = 0
                    const float p10 = fast_exp2(x1.x), p11 = fast_exp2(x1.y);
                    add2_to(ls0, ls0b, p00, p01);
                    add2_to(ls1, ls1b, p10, p11);
                    // n-tile j = tokens 8j..8j+7 -> k-step j/2, k half j&1
                    pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p00, p01);
                    pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p10, p11);
                }
                l0 += ls0 + ls0b;
                l1 += ls1 + ls1b;
                // 5. O += P V over this warp's 128 dims
                if (tok0 + ST <= vis_hi) {
#pragma unroll
                    for (int kk2 = 0; kk2 < 2; ++kk2) {
                        const uint32_t tok = 16u * kk2 + 8u * (((uint32_t)lane >> 3) & 1u) + ((uint32_t)lane & 7u);
#pragma unroll
                        for (int np = 0; np < kPvTiles / 2; ++np) {
                            // matrices: (k lo, n-tile 2np), (k hi, 2np), (k lo, 2np+1), (k hi, 2np+1)
                            const uint32_t nt = 2u * np + ((uint32_t)lane >> 4);
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(sb + chunk_off(2u * wq + (nt >> 3), tok, nt & 7u), b0, b1, b2, b3);
                            mma16816(o[2 * np], pa[kk2], b0, b1);
                            mma16816(o[2 * np + 1], pa[kk2], b2, b3);
                        }
                    }
                } else {
                    // the unit's last stage: rows past its last visible key
                    // are zeroed in the V operand (P is 0 there, but the
                    // slot may hold anything)
#pragma unroll
                    for (int kk2 = 0; kk2 < 2; ++kk2) {
                        const int32_t t = tok0 + 16 * kk2 + 2 * c;
                        const uint32_t mlo = (t < vis_hi ? 0x0000ffffu : 0u) | (t + 1 < vis_hi ? 0xffff0000u : 0u);
                        const uint32_t mhi = (t + 8 < vis_hi ? 0x0000ffffu : 0u) | (t + 9 < vis_hi ? 0xffff0000u : 0u);
                        const uint32_t tok = 16u * kk2 + 8u * (((uint32_t)lane >> 3) & 1u) + ((uint32_t)lane & 7u);
#pragma unroll
                        for (int np = 0; np < kPvTiles / 2; ++np) {
                            const uint32_t nt = 2u * np + ((uint32_t)lane >> 4);
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(sb + chunk_off(2u * wq + (nt >> 3), tok, nt & 7u), b0, b1, b2, b3);
                            mma16816(o[2 * np], pa[kk2], b0 & mlo, b1 & mhi);
                            mma16816(o[2 * np + 1], pa[kk2], b2 & mlo, b3 & mhi);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_EMPTY + st));
            }
            if (!ok) break;

            // row sums over the quad (the four lanes of a row)
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            float4* mo = reinterpret_cast<float4*>(smem + OFF_MO) + wq * kPvTiles * 32;
            float4* ml = reinterpret_cast<float4*>(smem + OFF_ML);
            if (gi == 1) {
                // hand this group's share of the piece to group 0
                ok = warp_wait(bar(B_MFREE), (merges & 1u) ^ 1u, abort_flag, status);
                if (!ok) break;
#pragma unroll
                for (int n = 0; n < kPvTiles; ++n) mo[n * 32 + lane] = make_float4(o[n][0], o[n][1], o[n][2], o[n][3]);
                if (wq == 0) ml[lane] = make_float4(m0, l0, m1, l1);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_MFULL));
                ++merges;
                continue;
            }
            ok = warp_wait(bar(B_MFULL), merges & 1u, abort_flag, status);
            if (!ok) break;
            {
                const float4 o1 = ml[lane];
                const float M0 = fmaxf(m0, o1.x), M1 = fmaxf(m1, o1.z);
                const float fa0 = M0 == -INFINITY ? 0.f : fast_exp2(m0 - M0);
                const float fb0 = M0 == -INFINITY ? 0.f : fast_exp2(o1.x - M0);
                const float fa1 = M1 == -INFINITY ? 0.f : fast_exp2(m1 - M1);
                const float fb1 = M1 == -INFINITY ? 0.f : fast_exp2(o1.z - M1);
                l0 = l0 * fa0 + o1.y * fb0;
                l1 = l1 * fa1 + o1.w * fb1;
                m0 = M0;
                m1 = M1;
#pragma unroll
                for (int n = 0; n < kPvTiles; ++n) {
                    const float4 u = mo[n * 32 + lane];
                    o[n][0] = o[n][0] * fa0 + u.x * fb0;
                    o[n][1] = o[n][1] * fa0 + u.y * fb0;
                    o[n][2] = o[n][2] * fa1 + u.z * fb1;
                    o[n][3] = o[n][3] * fa1 + u.w * fb1;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_MFREE));
            ++merges;

            // epilogue: O / l -> out (bf16) or the piece's fp32 partial slot
            const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
            const float lse0 = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
            const float lse1 = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
            const int64_t grow0 = (int64_t)b * QH + r0, grow1 = (int64_t)b * QH + r1;
            const int32_t dbase = kPvDims * wq + 2 * c;
            if (pc.slot < 0) {
                uint32_t* out = static_cast<uint32_t*>(a.out);   // bf16 pairs, 256 per row
#pragma unroll
                for (int n = 0; n < kPvTiles; ++n) {
                    const int32_t d = dbase + 8 * n;
                    if (r0 < rows) out[grow0 * 256 + d / 2] = pack_bf16x2(o[n][0] * inv0, o[n][1] * inv0);
                    if (r1 < rows) out[grow1 * 256 + d / 2] = pack_bf16x2(o[n][2] * inv1, o[n][3] * inv1);
                }
                if (a.lse && wq == 0 && c == 0) {
                    if (r0 < rows) a.lse[grow0] = lse0;
                    if (r1 < rows) a.lse[grow1] = lse1;
                }
            } else {
                // partial rows of a split unit, normalised, in fp16
                __half* op = reinterpret_cast<__half*>(v.o_part) + (int64_t)pc.slot * kRowsPerUnit * 512;
#pragma unroll
                for (int n = 0; n < kPvTiles; ++n) {
                    const int32_t d = dbase + 8 * n;
                    if (r0 < rows)
                        *reinterpret_cast<__half2*>(op + r0 * 512 + d) = __floats2half2_rn(o[n][0] * inv0, o[n][1] * inv0);
                    if (r1 < rows)
                        *reinterpret_cast<__half2*>(op + r1 * 512 + d) = __floats2half2_rn(o[n][2] * inv1, o[n][3] * inv1);
                }
                if (wq == 0 && c == 0) {
                    float* lp = v.lse_part + (int64_t)pc.slot * kRowsPerUnit;
                    if (r0 < rows) lp[r0] = lse0;
                    if (r1 < rows) lp[r1] = lse1;
                }
            }
        }
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_decode_sh(const CUtensorMap& kv, const ShArgs& a, int32_t num_workers, void* ws,
                             const WsLayout& L, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(decode_sh_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // the register split must fit what the launch allocates, or the
    // consumers' setmaxnreg.inc could never be granted
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, decode_sh_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < 32 * (4 * kProducerRegs + 8 * kConsumerRegs)) return cudaErrorInvalidConfiguration;
    decode_sh_kernel<<<num_workers, kThreads, SMEM_BYTES, stream>>>(kv, a, ws, L);
    return cudaGetLastError();
}

}  // namespace mla
