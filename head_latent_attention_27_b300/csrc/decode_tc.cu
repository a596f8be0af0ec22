// Absorbed MLA decode on tcgen05 tensor cores (sm_103a).
//
// What is computed (DeepSeek-V2 analysis page, sections 1.2-1.3, 6.1): for
// every query row r = (query token j, head h) of a sequence and every
// visible cached token s,
//     S[r,s] = q_nope[r] . c_s + q_rope[r] . k^R_s          (576-long dot)
//     P      = softmax_s(S * scale)                          (online, fp32)
//     O[r]   = sum_s P[r,s] c_s                              (512-wide)
// All heads share one cached row per token, so both products are dense
// contractions over the 128 query rows of a unit: [128 x 576]x[576 x 64]
// and [128 x 64]x[64 x 512] per 64-token tile.
//
// Two SMs per unit.  The fp32 accumulator O (128 rows x 512) is 256 KB,
// exactly one SM's tensor memory, so the two CTAs of a cluster split the
// latent dims: rank r owns c_kv dims [256r, 256r+256) and RoPE dims
// [32r, 32r+32), streams only those columns of every cache tile (the pair
// reads each cached byte once), and keeps the matching query columns
// (q_nope in TMEM as the A operand, q_rope in smem).  Per 64-token tile each
// CTA computes a partial S over its 288 dims; the partials are swapped
// through distributed shared memory in fp16 (16 KB per tile and direction;
// the rounding of the peer's half-sum is far below the bf16 rounding of P)
// and added in fp32, so both CTAs run the same softmax and hold the same P.
// Each accumulates its 256 output columns O += P V with P (bf16) in smem and
// the same cache tile read as an MN-major V operand.
//
// Pipeline (per CTA, 512 threads):
//   warp 0      TMA producer: q_rope per piece, 4-stage ring of cache tiles
//               (low-precision rows: also expands the first half of each
//               tile's codes to fp16)
//   warp 1      QK issuer (owns TMEM): S(g) as soon as tile g has landed and
//               its score buffer is free, up to two tiles ahead of the
//               softmax
//   warps 2-9   softmax, two warpgroups taking alternate tiles (ping-pong):
//               add the peer's half, online softmax with the running max
//               handed between the groups, P -> smem, lazy O rescale,
//               epilogue of a piece's last tile; q_nope -> TMEM
//   warp 10     forwards "peer's scores read" to the peer (a slow remote
//               arrive, kept off the softmax and swap warps); low-precision
//               rows: also expands the second half of each tile's codes
//   warps 11-14 score swap: S(g) from TMEM -> fp16 -> st.async to the peer
//   warp 15     PV issuer: O += P(g) V(g) as soon as P(g) is published, then
//               frees the cache stage.  QK and PV are issued by different
//               threads so that a PV whose P is ready never waits behind a
//               QK whose tile has not landed (with one issuer the stage of
//               tile g stayed occupied ~4,700 cycles after P(g) was ready).
// TMEM: O 256 columns | q_nope 128 | S double buffer 2 x 64.
//
// Every wait is bounded (ptx.cuh: bounded_wait); on a timeout the kernel
// records MLA_ERR_TIMEOUT in the workspace, drains its own copies and MMAs,
// frees TMEM and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "decode_tc.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int BM = 128;          // query rows per unit
constexpr int BN = 64;           // tokens per tile (= page)
constexpr int NSTAGE = 4;        // cache-tile ring depth
constexpr int kSoftmaxWarps = 8;  // two warpgroups
constexpr int kSwapWarps = 4;
constexpr int kForwardWarp = 2 + kSoftmaxWarps;                     // warp 10
constexpr int kPvWarp = kForwardWarp + 1 + kSwapWarps;             // warp 15
constexpr int kThreads = 32 * (4 + kSoftmaxWarps + kSwapWarps);   // 512

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_QR = 0;                               // 32 RoPE dims x 128 rows, 64B swizzle
constexpr uint32_t QR_BYTES = BM * 64;
constexpr uint32_t KN_BLK = BN * 128;                        // 64 dims x 64 tokens, 128B swizzle
constexpr uint32_t KR_BYTES = BN * 64;                       // 32 dims x 64 tokens, 64B swizzle
constexpr uint32_t STAGE_BYTES = 4 * KN_BLK + KR_BYTES;      // 36864
// Low-precision rows: per tile and CTA the 256 latent codes of 64 tokens
// are loaded as two 128-byte-wide boxes into the tile's latent boxes 1 and 3
// and expanded in place to fp16 (boxes 0-1 and 2-3, one half per warp); the
// 4 fp32 group scales of each token go to a small ring of their own.
constexpr uint32_t LP_CODE_BOX = BN * 128;                   // 64 tokens x 128 codes
constexpr uint32_t LP_SCALE_BYTES = BN * 16;                 // 64 tokens x 4 fp32
constexpr uint32_t LP_STAGE_TX = 2 * LP_CODE_BOX + LP_SCALE_BYTES + KR_BYTES;
// Byte offsets of a stage's boxes from the ring's base.
__host__ __device__ constexpr uint32_t nope_box(uint32_t st, uint32_t kb) {   // 64 dims x 64 tokens
    return st * STAGE_BYTES + kb * KN_BLK;
}
__host__ __device__ constexpr uint32_t rope_box(uint32_t st) {                 // 32 dims x 64 tokens
    return st * STAGE_BYTES + 4 * KN_BLK;
}
constexpr uint32_t OFF_KV = OFF_QR + QR_BYTES;
constexpr uint32_t P_BYTES = BM * BN * 2;                    // bf16 P, 128 rows x 128 B, 128B swizzle
constexpr uint32_t OFF_P = OFF_KV + NSTAGE * STAGE_BYTES;
constexpr uint32_t X_BYTES = BM * BN * 2;                    // peer's fp16 partial scores
constexpr uint32_t OFF_X = OFF_P + 2 * P_BYTES;
constexpr uint32_t OFF_BAR = OFF_X + 2 * X_BYTES;
constexpr uint32_t BAR_BYTES = 512;
constexpr uint32_t OFF_M = OFF_BAR + BAR_BYTES;                // [2 slots][128 rows] fp32 running max
constexpr uint32_t OFF_LM = OFF_M + 2 * BM * 4;                // [2][128] float2 (row sum, its max)
constexpr uint32_t OFF_SC = OFF_LM + 2 * BM * 8;                // [NSTAGE] low-precision group scales
constexpr uint32_t SMEM_USED = OFF_SC + NSTAGE * LP_SCALE_BYTES;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;            // + alignment slack

static_assert(OFF_KV % 1024 == 0 && STAGE_BYTES % 1024 == 0 && OFF_P % 1024 == 0 && OFF_X % 1024 == 0,
              "alignment");
static_assert(SMEM_BYTES <= 232448, "fits in 227 KB");

// barriers (slot pairs are indexed by global tile parity)
enum : int {
    B_QRFULL = 0,
    B_QREMPTY,
    B_QNFULL,
    B_KVFULL,
    B_KVEMPTY = B_KVFULL + NSTAGE,
    B_SFULL = B_KVEMPTY + NSTAGE,   // [2]
    B_SEMPTY = B_SFULL + 2,         // [2]
    B_XFULL = B_SEMPTY + 2,         // [2]
    B_PEERFREE = B_XFULL + 2,       // [2]
    B_PFULL = B_PEERFREE + 2,       // [2]
    B_PVDONE = B_PFULL + 2,         // [2]
    B_EXIT = B_PVDONE + 2,
    B_XREAD,                        // [2] this CTA's softmax is done reading the peer's scores
    B_MREADY = B_XREAD + 2,         // [2] running max after tile g published (slot g & 1)
    B_LFULL = B_MREADY + 2,         // [2] a group's row sum of a piece published (piece parity)
    B_LFREE = B_LFULL + 2,          // [2] ... and read
    B_OFREE = B_LFREE + 2,          // epilogue has read O; the next piece may overwrite it
    B_LPFULL,                       // [NSTAGE] low-precision tile landed (codes, scales, RoPE)
    NUM_BARS = B_LPFULL + NSTAGE
};
static_assert(NUM_BARS * 8 <= BAR_BYTES - 16, "barrier area");
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + BAR_BYTES - 16;
constexpr uint32_t OFF_ABORT = OFF_BAR + BAR_BYTES - 12;

// TMEM columns
constexpr uint32_t TM_O = 0, TM_Q = 256, TM_S = 384, TM_COLS = 512;

constexpr uint32_t IDESC_QK = idesc_bf16(128, BN, 0, 0);   // S[128x64] = Q . K^T, K-major operands
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, 0, 1);  // O[128x256] += P . V, V MN-major
// Low-precision cache: the latent operands (q_nope, the dequantised cache
// tile, P) are fp16; the RoPE part stays bf16 (its MMAs keep IDESC_QK/QK2).
constexpr uint32_t IDESC_QK_H = idesc_f16(128, BN, 0, 0);
constexpr uint32_t IDESC_PV_H = idesc_f16(128, 256, 0, 1);

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi);
// bf16 pair -> fp16 pair (each value rounded to nearest fp16).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
    return pack_f16x2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

template <bool kHalf>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi);
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack_p<false>(float lo, float hi) { return pack_bf16x2(lo, hi); }
template <>
__device__ __forceinline__ uint32_t pack_p<true>(float lo, float hi) { return pack_f16x2(lo, hi); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// 2^x on the SFU, flush-to-zero (inputs here are <= 0 or -inf; results
// below 2^-126 only feed the bf16 probabilities and their sum).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (f32x2 add / fma, each lane rounded to nearest like its
// scalar form) and the three-input max: fewer instructions in the per-tile
// softmax, whose issue rate and instruction-cache footprint bound the tile
// period.
// (x, y) += (a, b)
__device__ __forceinline__ void add2_to(float& x, float& y, float a, float b) {
    asm("{\n\t.reg .b64 p, q;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %3};\n\t"
        "add.rn.f32x2 p, p, q;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "+f"(x), "+f"(y) : "f"(a), "f"(b));
}
// (x*a + c, y*b + d)
__device__ __forceinline__ float2 fma2(float x, float y, float a, float b, float c, float d) {
    float2 r;
    asm("{\n\t.reg .b64 p, q, w;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\tmov.b64 w, {%6, %7};\n\t"
        "fma.rn.f32x2 p, p, q, w;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "=f"(r.x), "=f"(r.y) : "f"(x), "f"(y), "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (x, y) += the two fp16 values packed in u (low half to x), each widened
// inside a mixed-precision add (fp16 operand, fp32 accumulator and result):
// no separate conversion instructions.
__device__ __forceinline__ void add_f16x2_to(float& x, float& y, uint32_t u) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
        : "+f"(x), "+f"(y) : "r"(u));
}

// Bounded wait taken by all 32 lanes; the outcome is made warp-uniform so
// that warp-collective tcgen05 instructions stay converged.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
    const bool ok = bounded_wait<kCluster>(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

// Wait limited by time only (ignores the abort flag): used to drain work
// already in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 200000000ull) return;
    }
}

// Walks the (piece, tile) sequence of a worker in order.
struct TileCursor {
    const Piece* pieces;
    int32_t p, p_end, t;
    Piece pc;
    __device__ void init(const Piece* ps, int32_t p0, int32_t p1) {
        pieces = ps;
        p = p0;
        p_end = p1;
        if (p < p_end) {
            pc = pieces[p];
            t = pc.t_begin;
        }
    }
    __device__ bool valid() const { return p < p_end; }
    __device__ bool first() const { return t == pc.t_begin; }
    __device__ bool last() const { return t == pc.t_end - 1; }
    __device__ void next() {
        if (++t >= pc.t_end) {
            ++p;
            if (p < p_end) {
                pc = pieces[p];
                t = pc.t_begin;
            }
        }
    }
};

// One 16-byte chunk of codes (16 latent dims c8*16.. of one token row) ->
// fp16 values in the swizzled K-major layout of boxes box0 and box0+1.
__device__ __forceinline__ void expand16(uint8_t* ring, uint32_t st, uint32_t box0, int row, int c8, uint4 cw,
                                         float sc) {
    const __half2 s2 = __float2half2_rn(sc);
    uint32_t w[8];
    const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t lo, hi;
        asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
            : "=r"(lo), "=r"(hi) : "r"(cws[j]));
        const __half2 l2 = __hmul2(*reinterpret_cast<const __half2*>(&lo), s2);
        const __half2 h2 = __hmul2(*reinterpret_cast<const __half2*>(&hi), s2);
        w[2 * j] = *reinterpret_cast<const uint32_t*>(&l2);
        w[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    // dims 16*c8 .. +16 of the half -> box box0 + (c8 >> 2), 16-byte chunks 2*(c8&3), +1
    uint8_t* rowp = ring + nope_box(st, box0 + (c8 >> 2)) + row * 128;
    const int ch = 2 * (c8 & 3), sw = row & 7;
    *reinterpret_cast<uint4*>(rowp + ((ch ^ sw) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(rowp + (((ch + 1) ^ sw) * 16)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Dequantise half of one tile's low-precision latent codes in place (one
// warp, all 32 lanes).  Half h holds this CTA's latent dims [128h, 128h+128):
// its codes ([64 tokens][128 codes], unswizzled) sit in box 2h+1 and expand,
// value = E4M3(code) * group scale, into fp16 boxes 2h and 2h+1 in the
// 128-byte swizzled K-major layout the MMAs read.  The two halves touch
// disjoint boxes, so two warps expand them concurrently.  Within a half, the
// fp16 values of token row r overwrite only row r's own codes (bytes
// [128r, 128r+128) of box 2h+1), so rows are expanded in batches: a batch's
// codes are all read (and the warp synchronised) before its first store,
// and later batches read other rows.
__device__ __forceinline__ void dequant_half(uint8_t* ring, uint32_t st, const float* scales, uint32_t rank,
                                             int lane, int half) {
    const uint8_t* codes = ring + nope_box(st, 2 * half + 1);
    constexpr int kBatch = 8;   // 8 x 32 chunks of 16 codes = 32 token rows per batch
#pragma unroll 1
    for (int b0 = 0; b0 < 16; b0 += kBatch) {
        uint4 cw[kBatch];
        float sc[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int pidx = (b0 + i) * 32 + lane;   // 512 chunks of 16 codes per half
            const int row = pidx >> 3;
            cw[i] = *reinterpret_cast<const uint4*>(codes + row * 128 + (pidx & 7) * 16);
            sc[i] = scales[row * 4 + 2 * rank + half];
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int pidx = (b0 + i) * 32 + lane;
            expand16(ring, st, 2 * half, pidx >> 3, pidx & 7, cw[i], sc[i]);
        }
        __syncwarp();
    }
}

template <bool kLowp>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_kv_nope, const __grid_constant__ CUtensorMap tm_kv_rope,
                     const __grid_constant__ CUtensorMap tm_q_rope, const __grid_constant__ CUtensorMap tm_kv_scale,
                     const TcArgs a, void* ws, const WsLayout L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int32_t cluster_id = blockIdx.x >> 1;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM_SLOT);

    WsView v = ws_view(ws, L);
    int* status = &v.hdr->status;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_QRFULL), 1);
        mbar_init(bar(B_QREMPTY), 1);
        mbar_init(bar(B_QNFULL), 4);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(bar(B_KVFULL + s), kLowp ? 2 : 1);   // low-precision: the two expander warps
            mbar_init(bar(B_KVEMPTY + s), 1);
            mbar_init(bar(B_LPFULL + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_SFULL + s), 1);
            mbar_init(bar(B_SEMPTY + s), 4 + kSwapWarps);
            mbar_init(bar(B_XFULL + s), 1);
            mbar_init(bar(B_PEERFREE + s), 1);
            mbar_init(bar(B_XREAD + s), 4);
            mbar_init(bar(B_MREADY + s), 4);
            mbar_init(bar(B_LFULL + s), 4);
            mbar_init(bar(B_LFREE + s), 4);
            mbar_init(bar(B_PFULL + s), 4);
            mbar_init(bar(B_PVDONE + s), 1);
        }
        mbar_init(bar(B_EXIT), 2);   // both MMA issuers commit
        mbar_init(bar(B_OFREE), 4);
        *abort_flag = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_kv_nope);
        tma_prefetch_desc(&tm_kv_rope);
        tma_prefetch_desc(&tm_q_rope);
        if constexpr (kLowp) tma_prefetch_desc(&tm_kv_scale);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();  // both CTAs' barriers exist before any remote access
    const uint32_t tmem = *tmem_slot;

    const int32_t p_begin = v.worker_begin[cluster_id];
    const int32_t p_end = v.worker_begin[cluster_id + 1];
    const int32_t QH = a.Q * a.H;
    const int32_t RB = units_per_seq(a.Q, a.H);
    const int32_t max_tokens = a.max_pages_per_seq * kTileTokens;

    if (warp == 0 && kLowp) {
        // ------------------------ TMA producer + in-place dequantiser (half 0)
        // One loop, never blocking on one condition while the other could
        // progress: lane 0 issues the loads of the next tile as soon as its
        // stage is free (and, at a piece's first tile, the previous piece has
        // released q_rope); the whole warp expands the first half of the
        // oldest landed tile and marks it for the MMAs (the forwarder warp
        // expands the second half; the tile is full after both).  Gives up (timeout status) after the
        // same time limit as every other wait when neither can progress.
        const uint64_t pol = a.evict_first ? l2_policy_evict_first() : l2_policy_evict_last();
        uint8_t* ring = smem + OFF_KV;
        uint32_t q_cnt = 0, issued = 0, expanded = 0, total = 0;
        for (int32_t p = p_begin; p < p_end; ++p) total += (uint32_t)(v.pieces[p].t_end - v.pieces[p].t_begin);
        TileCursor ic;
        ic.init(v.pieces, p_begin, p_end);
        bool ok = true;
        uint64_t idle_since = 0;
        while (ok && expanded < total) {
            bool progressed = false;
            // 1. loads of tile `issued`
            if (issued < total) {
                const uint32_t st = issued % NSTAGE, ph = (issued / NSTAGE) & 1u;
                int go = 0;
                if (lane == 0) {
                    const bool new_piece = ic.first();
                    go = mbar_try_wait(bar(B_KVEMPTY + st), ph ^ 1u) &&
                         (!new_piece || mbar_try_wait(bar(B_QREMPTY), (q_cnt & 1u) ^ 1u));
                    if (go) {
                        const int32_t b = ic.pc.unit / RB, rb = ic.pc.unit % RB;
                        if (new_piece) {
                            mbar_arrive_expect_tx(bar(B_QRFULL), QR_BYTES);
                            tma_load_2d(sbase + OFF_QR, &tm_q_rope, bar(B_QRFULL), 32 * rank, b * QH + rb * BM, pol);
                            ++q_cnt;
                        }
                        int32_t page = a.page_table[(int64_t)b * a.max_pages_per_seq + ic.t];
                        if (page < 0 || page >= a.num_pages) {
                            atomicCAS(status, 0, 1);
                            page = 0;
                        }
                        const uint32_t fb = bar(B_LPFULL + st);
                        mbar_arrive_expect_tx(fb, LP_STAGE_TX);
                        const int32_t y0 = page * BN;
                        tma_load_2d(sbase + OFF_KV + nope_box(st, 1), &tm_kv_nope, fb, 256 * rank, y0, pol);
                        tma_load_2d(sbase + OFF_KV + nope_box(st, 3), &tm_kv_nope, fb, 256 * rank + 128, y0, pol);
                        tma_load_2d(sbase + OFF_SC + st * LP_SCALE_BYTES, &tm_kv_scale, fb, 128, y0, pol);
                        tma_load_2d(sbase + OFF_KV + rope_box(st), &tm_kv_rope, fb, 264 + 32 * rank, y0, pol);
                        ic.next();
                    }
                }
                if (__shfl_sync(0xffffffffu, go, 0)) {
                    ++issued;
                    progressed = true;
                }
            }
            // 2. expand tile `expanded` once it has landed
            if (expanded < issued) {
                const uint32_t st = expanded % NSTAGE, ph = (expanded / NSTAGE) & 1u;
                const int landed = lane == 0 ? (mbar_try_wait(bar(B_LPFULL + st), ph) ? 1 : 0) : 0;
                if (__shfl_sync(0xffffffffu, landed, 0)) {
                    dequant_half(ring, st, reinterpret_cast<const float*>(smem + OFF_SC + st * LP_SCALE_BYTES),
                                 rank, lane, 0);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_KVFULL + st));
                    ++expanded;
                    progressed = true;
                }
            }
            if (progressed) {
                idle_since = 0;
            } else {
                __nanosleep(32);   // poll gently: this warp shares its scheduler with softmax warps
                const uint64_t now = global_timer_ns();
                if (idle_since == 0) idle_since = now;
                int stop = 0;
                if (lane == 0 && (*abort_flag || now - idle_since > kWaitLimitNs)) {
                    if (!*abort_flag) {
                        *abort_flag = 1;
                        atomicExch(status, 4 /* MLA_ERR_TIMEOUT */);
                    }
                    stop = 1;
                }
                if (__shfl_sync(0xffffffffu, stop, 0)) ok = false;
            }
        }
        if (lane == 0) {
            // drain this CTA's copies still in flight (abort path)
            for (uint32_t i = expanded; i < issued; ++i)
                drain_wait(bar(B_LPFULL + i % NSTAGE), (i / NSTAGE) & 1u);
            if (q_cnt > 0) drain_wait(bar(B_QRFULL), (q_cnt - 1) & 1u);
        }
    } else if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = a.evict_first ? l2_policy_evict_first() : l2_policy_evict_last();
            uint32_t stage = 0, phase = 0, q_cnt = 0;
            uint32_t issued_mask = 0, last_parity = 0;
            bool ok = true;
            // L2 prefetch `prefetch_tiles` tiles ahead of the loads; rank r
            // prefetches tokens [32r, 32r+32) of a page (one contiguous half),
            // so the pair covers whole pages.
            TileCursor pf;
            pf.init(v.pieces, p_begin, p_end);
            const uint8_t* cache_bytes = static_cast<const uint8_t*>(a.cache);
            auto prefetch_next = [&]() {
                if (!pf.valid()) return;
                const int32_t pb = pf.pc.unit / RB;
                const int32_t page = a.page_table[(int64_t)pb * a.max_pages_per_seq + pf.t];
                if (page >= 0 && page < a.num_pages)
                    bulk_prefetch_l2(cache_bytes + (int64_t)page * (BN * 1152) + rank * (BN * 576), BN * 576);
                pf.next();
            };
            if constexpr (kTcPrefetchTiles > 0)
                for (int32_t i = 0; i < a.prefetch_tiles; ++i) prefetch_next();
            for (int32_t p = p_begin; p < p_end && ok; ++p) {
                const Piece pc = v.pieces[p];
                const int32_t b = pc.unit / RB, rb = pc.unit % RB;
                ok = bounded_wait(bar(B_QREMPTY), (q_cnt & 1u) ^ 1u, abort_flag, status);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(B_QRFULL), QR_BYTES);
                tma_load_2d(sbase + OFF_QR, &tm_q_rope, bar(B_QRFULL), 32 * rank, b * QH + rb * BM, pol);
                ++q_cnt;
                for (int32_t t = pc.t_begin; t < pc.t_end; ++t) {
                    int32_t page = a.page_table[(int64_t)b * a.max_pages_per_seq + t];
                    if (page < 0 || page >= a.num_pages) {
                        atomicCAS(status, 0, 1);
                        page = 0;
                    }
                    if constexpr (kTcPrefetchTiles > 0) prefetch_next();
                    ok = bounded_wait(bar(B_KVEMPTY + stage), phase ^ 1u, abort_flag, status);
                    if (!ok) break;
                    const uint32_t fb = bar(B_KVFULL + stage);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    const uint32_t ring = sbase + OFF_KV;
                    const int32_t y0 = page * BN;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
                        tma_load_2d(ring + nope_box(stage, kb), &tm_kv_nope, fb, 256 * rank + 64 * kb, y0, pol);
                    tma_load_2d(ring + rope_box(stage), &tm_kv_rope, fb, 512 + 32 * rank, y0, pol);
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
#pragma unroll 1
            for (int s = 0; s < NSTAGE; ++s)
                if (issued_mask & (1u << s)) drain_wait(bar(B_KVFULL + s), (last_parity >> s) & 1u);
            if (q_cnt > 0) drain_wait(bar(B_QRFULL), (q_cnt - 1) & 1u);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- QK issuer
        if (lane == 0) {
            const uint32_t tQ = tmem + TM_Q;
            bool ok = true;
            TileCursor qk;
            qk.init(v.pieces, p_begin, p_end);
            uint32_t g_qk = 0, qk_stage = 0, qk_phase = 0, q_cnt = 0;
            const uint64_t bdesc_nope0 = smem_desc(sbase + OFF_KV, 16, 1024, kSwizzle128B);
            const uint64_t bdesc_rope0 = smem_desc(sbase + OFF_KV + 4 * KN_BLK, 16, 512, kSwizzle64B);
            const uint64_t adesc_rope = smem_desc(sbase + OFF_QR, 16, 512, kSwizzle64B);

            auto issue_qk = [&]() -> bool {
                const uint32_t slot = g_qk & 1u;
                if (qk.first()) {
                    if (!bounded_wait(bar(B_QRFULL), q_cnt & 1u, abort_flag, status)) return false;
                    if (!bounded_wait(bar(B_QNFULL), q_cnt & 1u, abort_flag, status)) return false;
                    ++q_cnt;
                }
                if (!bounded_wait(bar(B_KVFULL + qk_stage), qk_phase, abort_flag, status)) return false;
                if (!bounded_wait(bar(B_SEMPTY + slot), ((g_qk >> 1) & 1u) ^ 1u, abort_flag, status)) return false;
                tc_fence_after();
                const uint32_t tS = tmem + TM_S + 64u * slot;
                // Per-MMA descriptors differ from the stage's first one only in
                // the start-address field (address / 16 in the low 14 bits;
                // every shared address here is below 2^18, so the add never
                // carries out of it): one add per MMA.
                const uint64_t stage_off = (uint64_t)(qk_stage * (STAGE_BYTES >> 4));
                const uint64_t bn0 = bdesc_nope0 + stage_off;
                const uint64_t br0 = bdesc_rope0 + stage_off;
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)   // 256 latent dims, A = q_nope from TMEM
                    umma_ts(tS, tQ + kk * 8, bn0 + (uint64_t)((((kk >> 2) * KN_BLK + (kk & 3) * 32)) >> 4),
                            kLowp ? IDESC_QK_H : IDESC_QK, kk != 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)    // 32 RoPE dims, A = q_rope from smem
                    umma_ss(tS, adesc_rope + (uint64_t)(kk * 2), br0 + (uint64_t)(kk * 2), IDESC_QK, 1u);
                umma_commit(bar(B_SFULL + slot));
                if (qk.last()) umma_commit(bar(B_QREMPTY));
                ++g_qk;
                if (++qk_stage == NSTAGE) {
                    qk_stage = 0;
                    qk_phase ^= 1u;
                }
                qk.next();
                return true;
            };
            while (ok && qk.valid()) ok = issue_qk();
            umma_commit(bar(B_EXIT));
            drain_wait(bar(B_EXIT), 0);
        }
    } else if (warp == kPvWarp) {
        // -------------------------------------------------------- PV issuer
        if (lane == 0) {
            const uint32_t tO = tmem + TM_O;
            bool ok = true;
            TileCursor pv;
            pv.init(v.pieces, p_begin, p_end);
            uint32_t g_pv = 0, pv_stage = 0, pv_piece = 0;
            const uint64_t bdesc_v0 = smem_desc(sbase + OFF_KV, KN_BLK, 1024, kSwizzle128B);
            const uint64_t adesc_p0 = smem_desc(sbase + OFF_P, 16, 1024, kSwizzle128B);
            auto issue_pv = [&]() -> bool {
                const uint32_t slot = g_pv & 1u;
                if (pv.first() && pv_piece > 0) {
                    if (!bounded_wait(bar(B_OFREE), (pv_piece - 1) & 1u, abort_flag, status)) return false;
                }
                if (pv.first()) ++pv_piece;
                if (!bounded_wait(bar(B_PFULL + slot), (g_pv >> 1) & 1u, abort_flag, status)) return false;
                tc_fence_after();
                const uint64_t ap0 = adesc_p0 + (uint64_t)(slot * (P_BYTES >> 4));
                const uint64_t bv0 = bdesc_v0 + (uint64_t)(pv_stage * (STAGE_BYTES >> 4));
                const bool first = pv.first();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)   // descriptors: start address + offset / 16
                    umma_ss(tO, ap0 + (uint64_t)(kk * 2), bv0 + (uint64_t)(kk * 128), kLowp ? IDESC_PV_H : IDESC_PV,
                            (first && kk == 0) ? 0u : 1u);
                umma_commit(bar(B_PVDONE + slot));
                umma_commit(bar(B_KVEMPTY + pv_stage));
                ++g_pv;
                if (++pv_stage == NSTAGE) pv_stage = 0;
                pv.next();
                return true;
            };
            while (ok && pv.valid()) ok = issue_pv();
            umma_commit(bar(B_EXIT));
            drain_wait(bar(B_EXIT), 0);
        }
    } else if (warp < 2 + kSoftmaxWarps) {
        // ------------------------------------- softmax / correction / epilogue
        // Two warpgroups take alternate tiles (group g & 1 owns tile g), so
        // the long latency chain of one tile's softmax overlaps the next
        // tile's.  Within a group one thread owns one row.  The running
        // maximum is handed from the owner of tile g-1 to the owner of tile g
        // through shared memory (B_MREADY); each group keeps the row sum of
        // its own tiles relative to the latest maximum it has seen, and the
        // two sums are merged at the end of a piece (B_LFULL / B_LFREE).  The
        // owner of a piece's last tile writes the epilogue and then releases
        // O to the MMA warp (B_OFREE).
        const uint32_t wg = (uint32_t)((warp - 2) >> 2);
        const uint32_t quarter = (uint32_t)(warp & 3);
        const int32_t row = (int32_t)(quarter * 32 + lane);
        const uint32_t lane_off = (quarter * 32u) << 16;
        const uint32_t tO = tmem + TM_O + lane_off, tQ = tmem + TM_Q + lane_off;
        const bool leader = (warp == 2 + 4 * (int)wg) && lane == 0;
        const int32_t gtid = (int32_t)threadIdx.x - 64 - 128 * (int32_t)wg;   // 0..127 within the group
        const int rsw = row & 7;
        float* mrow = reinterpret_cast<float*>(smem + OFF_M);     // [2 slots][128 rows] running max
        float2* lm = reinterpret_cast<float2*>(smem + OFF_LM);    // [2][128] (row sum, its max) of a group
        bool ok = true;

        // q_nope columns of this rank for piece `pp` -> TMEM (A operand of QK)
        auto write_q = [&](int32_t pp) {
            const Piece pc = v.pieces[pp];
            const int32_t qb = pc.unit / RB, qrb = pc.unit % RB;
            const int32_t qrows = min(BM, QH - qrb * BM);
            const int64_t grow = (int64_t)qb * QH + qrb * BM + row;
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_nope) +
                                                              grow * 512 + 256 * rank);
            const bool have = row < qrows;
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t r0[16], r1[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 x = have ? src[c0 / 4 + i] : make_uint4(0, 0, 0, 0);
                    const uint4 y = have ? src[c0 / 4 + 4 + i] : make_uint4(0, 0, 0, 0);
                    r0[4 * i] = x.x; r0[4 * i + 1] = x.y; r0[4 * i + 2] = x.z; r0[4 * i + 3] = x.w;
                    r1[4 * i] = y.x; r1[4 * i + 1] = y.y; r1[4 * i + 2] = y.z; r1[4 * i + 3] = y.w;
                }
                if constexpr (kLowp) {   // the latent MMAs of the low-precision cache take fp16 queries
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        r0[i] = bf16x2_to_f16x2(r0[i]);
                        r1[i] = bf16x2_to_f16x2(r1[i]);
                    }
                }
                tmem_st16(tQ + c0, r0);
                tmem_st16(tQ + c0 + 16, r1);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_QNFULL));
        };

        TileCursor cur;
        cur.init(v.pieces, p_begin, p_end);
        if (wg == 0 && cur.valid()) write_q(cur.p);
        uint32_t g = 0, k = 0;   // tile and piece counters of this worker
        int32_t b = 0, rb = 0, rows_valid = 0, vis = 0, vis_lo = 0, vis_hi = 0, qrow = 0;
        float m_seen = -INFINITY, l = 0.f;
        for (; ok && cur.valid(); ++g, cur.next()) {
            if (cur.first()) {
                b = cur.pc.unit / RB;
                rb = cur.pc.unit % RB;
                const int32_t len = checked_len(a.seq_lens, b, max_tokens, status);
                rows_valid = min(BM, QH - rb * BM);
                qrow = rb * BM + row;
                vis = row < rows_valid ? visible_len(len, a.Q, a.H, qrow) : 0;
                vis_lo = visible_len(len, a.Q, a.H, rb * BM);                    // fewest keys of the unit
                vis_hi = visible_len(len, a.Q, a.H, rb * BM + rows_valid - 1);   // most keys of the unit
                m_seen = -INFINITY;
                l = 0.f;
            }
            if ((g & 1u) != wg) {
                // not ours; after a piece's last tile publish this group's row sum
                if (cur.last()) {
                    ok = warp_wait(bar(B_LFREE + (k & 1u)), ((k >> 1) & 1u) ^ 1u, abort_flag, status);
                    if (!ok) break;
                    lm[(k & 1u) * BM + row] = make_float2(l, m_seen);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_LFULL + (k & 1u)));
                    ++k;
                }
                continue;
            }
            const uint32_t slot = wg, ph = (g >> 1) & 1u;
            // 1. own partial S of tile g (all 64 columns)
            ok = warp_wait(bar(B_SFULL + slot), ph, abort_flag, status);
            if (!ok) break;
            tc_fence_after();
            float s[BN];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + TM_S + 64u * slot + lane_off, r0);
                tmem_ld32(tmem + TM_S + 64u * slot + lane_off + 32, r1);
                tmem_ld_wait64(r0, r1);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    s[i] = __uint_as_float(r0[i]);
                    s[32 + i] = __uint_as_float(r1[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_SEMPTY + slot));
            if (cur.last() && cur.p + 1 < cur.p_end) write_q(cur.p + 1);   // QK of this piece is complete
            // 2. add the peer's fp16 half
            if (leader) mbar_arrive_expect_tx(bar(B_XFULL + slot), X_BYTES);
            ok = warp_wait<true>(bar(B_XFULL + slot), ph, abort_flag, status);
            if (!ok) break;
            {
                const uint4* xb = reinterpret_cast<const uint4*>(smem + OFF_X + slot * X_BYTES) + row * 8;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = xb[c ^ rsw];
                    add_f16x2_to(s[8 * c + 0], s[8 * c + 1], u.x);
                    add_f16x2_to(s[8 * c + 2], s[8 * c + 3], u.y);
                    add_f16x2_to(s[8 * c + 4], s[8 * c + 5], u.z);
                    add_f16x2_to(s[8 * c + 6], s[8 * c + 7], u.w);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_XREAD + slot));   // forwarded to the peer by warp kForwardWarp
            // 3. tile maximum on the raw scores (the scale is positive);
            //    columns past a row's visible length are masked to -inf
            const int32_t tok0 = cur.t * BN;
            if (tok0 + BN > vis_lo) {
#pragma unroll
                for (int c = 0; c < BN; ++c) s[c] = (tok0 + c < vis) ? s[c] : -INFINITY;
            }
            float mx[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) mx[k2] = fmaxf(s[2 * k2], s[2 * k2 + 1]);
#pragma unroll
            for (int c = 8; c < BN; c += 8) {
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) mx[k2] = max3f(mx[k2], s[c + 2 * k2], s[c + 2 * k2 + 1]);
            }
            const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
            // 4. running maximum after tile g-1 (the other group's), lazy
            //    update: O is rescaled only when the max grows by > 2^8
            float m_prev = -INFINITY;
            if (g > 0) {
                ok = warp_wait(bar(B_MREADY + (slot ^ 1u)), ((g - 1) >> 1) & 1u, abort_flag, status);
                if (!ok) break;
                if (!cur.first()) m_prev = mrow[(slot ^ 1u) * BM + row];
            }
            float m_cur = m_prev, factor = 1.f;
            bool rescale = false;
            if (tmax > m_prev + kRescaleThreshold) {
                if (m_prev != -INFINITY) {
                    factor = fast_exp2(m_prev - tmax);
                    rescale = true;
                }
                m_cur = tmax;
            }
            mrow[slot * BM + row] = m_cur;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_MREADY + slot));
            if (m_seen != -INFINITY && m_cur != m_seen) l *= fast_exp2(m_seen - m_cur);
            m_seen = m_cur;
            // 5. P slot free (PV of tile g-2), then P = 2^(x - m) as bf16,
            //    128-byte swizzled K-major rows, 8 columns at a time
            ok = warp_wait(bar(B_PVDONE + slot), ph ^ 1u, abort_flag, status);
            if (!ok) break;
            {
                const float neg_m = (m_cur == -INFINITY) ? 0.f : -m_cur;
                uint8_t* prow = smem + OFF_P + slot * P_BYTES + (row >> 3) * 1024 + (row & 7) * 128;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                const float sl2 = a.scale_log2;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 x = fma2(s[8 * c + 2 * i], s[8 * c + 2 * i + 1], sl2, sl2, neg_m, neg_m);
                        const float p0 = fast_exp2(x.x);   // exp2(-inf) = 0
                        const float p1 = fast_exp2(x.y);
                        add2_to(ls[2 * (i & 1)], ls[2 * (i & 1) + 1], p0, p1);
                        w[i] = pack_p<kLowp>(p0, p1);
                    }
                    *reinterpret_cast<uint4*>(prow + ((c ^ rsw) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            }
            // 6. O rescale (after the PV of tile g-1, before the PV of tile g)
            if (__any_sync(0xffffffffu, rescale)) {
                ok = warp_wait(bar(B_PVDONE + (slot ^ 1u)), ((g - 1) >> 1) & 1u, abort_flag, status);
                if (!ok) break;
                tc_fence_after();
                const float f = rescale ? factor : 1.f;
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tO + c0, r);
                    tmem_ld_wait32(r);
                    uint32_t r0[16], r1[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        r0[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                        r1[i] = __float_as_uint(__uint_as_float(r[16 + i]) * f);
                    }
                    tmem_st16(tO + c0, r0);
                    tmem_st16(tO + c0 + 16, r1);
                }
                tmem_st_wait();
                tc_fence_before();
            }
            // 7. last tile of a ragged unit: clear cache rows past the end so
            //    that P = 0 never meets non-finite garbage in V
            if (tok0 + BN > vis_hi) {
                const int32_t nvalid = max(0, vis_hi - tok0);
                const int32_t nrows = BN - nvalid;
                const uint32_t st = g % NSTAGE;
                const int32_t chunks = nrows * 8 * 4;
                for (int32_t i = gtid; i < chunks; i += 128) {
                    const int32_t kb = i / (nrows * 8);
                    const int32_t rem = i % (nrows * 8);
                    const int32_t rr = nvalid + rem / 8, cc = rem % 8;
                    *reinterpret_cast<uint4*>(smem + OFF_KV + nope_box(st, kb) + rr * 128 + cc * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            // 8. publish P(g)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL + slot));
            // 9. epilogue after the piece's last tile: O / l -> out or partial slot
            if (cur.last()) {
                ok = warp_wait(bar(B_PVDONE + slot), ph, abort_flag, status);
                if (!ok) break;
                ok = warp_wait(bar(B_LFULL + (k & 1u)), (k >> 1) & 1u, abort_flag, status);
                if (!ok) break;
                const float2 other = lm[(k & 1u) * BM + row];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_LFREE + (k & 1u)));
                ++k;
                tc_fence_after();
                // the other group's sum is relative to the max it last saw (<= m_seen)
                const float l_tot = l + (other.y == -INFINITY ? 0.f : other.x * fast_exp2(other.y - m_seen));
                const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
                const float row_lse = l_tot > 0.f ? (m_seen + log2f(l_tot)) * kLn2 : -INFINITY;
                const bool store = row < rows_valid;
                const int64_t grow = (int64_t)b * QH + qrow;
                const int32_t slot_out = cur.pc.slot;
                const int32_t col0 = 256 * (int32_t)rank;
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tO + c0, r);
                    tmem_ld_wait32(r);
                    if (store) {
                        if (slot_out < 0) {
                            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + grow * 512 +
                                                                  col0 + c0);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                dst[q] = make_uint4(
                                    pack_bf16x2(__uint_as_float(r[8 * q + 0]) * inv_l, __uint_as_float(r[8 * q + 1]) * inv_l),
                                    pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv_l, __uint_as_float(r[8 * q + 3]) * inv_l),
                                    pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv_l, __uint_as_float(r[8 * q + 5]) * inv_l),
                                    pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv_l, __uint_as_float(r[8 * q + 7]) * inv_l));
                        } else {
                            // partial row of a split unit, normalised, in fp16 (a convex
                            // combination of cache rows: well inside fp16's range)
                            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(v.o_part) +
                                                                  ((int64_t)slot_out * kRowsPerUnit + row) * 512 +
                                                                  col0 + c0);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                dst[q] = make_uint4(
                                    pack_f16x2(__uint_as_float(r[8 * q + 0]) * inv_l, __uint_as_float(r[8 * q + 1]) * inv_l),
                                    pack_f16x2(__uint_as_float(r[8 * q + 2]) * inv_l, __uint_as_float(r[8 * q + 3]) * inv_l),
                                    pack_f16x2(__uint_as_float(r[8 * q + 4]) * inv_l, __uint_as_float(r[8 * q + 5]) * inv_l),
                                    pack_f16x2(__uint_as_float(r[8 * q + 6]) * inv_l, __uint_as_float(r[8 * q + 7]) * inv_l));
                        }
                    }
                }
                if (store && rank == 0) {
                    if (slot_out < 0) {
                        if (a.lse) a.lse[grow] = row_lse;
                    } else {
                        v.lse_part[(int64_t)slot_out * kRowsPerUnit + row] = row_lse;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_OFREE));   // O may be overwritten by the next piece
            }
        }
    } else if (warp == kForwardWarp && kLowp) {
        // ---------- "scores read" forwarder + in-place dequantiser (half 1)
        // The forwarding below, polled instead of blocking so that the warp
        // also expands the second half of every landed low-precision tile.
        uint8_t* ring = smem + OFF_KV;
        const uint32_t peerfree_remote0 = map_to_cta(bar(B_PEERFREE), peer);
        uint32_t total = 0;
        for (int32_t p = p_begin; p < p_end; ++p) total += (uint32_t)(v.pieces[p].t_end - v.pieces[p].t_begin);
        uint32_t fwd = 0, expanded = 0;
        bool ok = true;
        uint64_t idle_since = 0;
        while (ok && (fwd < total || expanded < total)) {
            bool progressed = false;
            if (fwd < total) {
                int done = 0;
                if (lane == 0 && mbar_try_wait(bar(B_XREAD + (fwd & 1u)), (fwd >> 1) & 1u)) {
                    mbar_arrive_remote(peerfree_remote0 + 8u * (fwd & 1u));
                    done = 1;
                }
                if (__shfl_sync(0xffffffffu, done, 0)) {
                    ++fwd;
                    progressed = true;
                }
            }
            if (expanded < total) {
                const uint32_t st = expanded % NSTAGE, ph = (expanded / NSTAGE) & 1u;
                const int landed = lane == 0 ? (mbar_try_wait(bar(B_LPFULL + st), ph) ? 1 : 0) : 0;
                if (__shfl_sync(0xffffffffu, landed, 0)) {
                    dequant_half(ring, st, reinterpret_cast<const float*>(smem + OFF_SC + st * LP_SCALE_BYTES),
                                 rank, lane, 1);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_KVFULL + st));
                    ++expanded;
                    progressed = true;
                }
            }
            if (progressed) {
                idle_since = 0;
            } else {
                __nanosleep(32);
                const uint64_t now = global_timer_ns();
                if (idle_since == 0) idle_since = now;
                int stop = 0;
                if (lane == 0 && (*abort_flag || now - idle_since > kWaitLimitNs)) {
                    if (!*abort_flag) {
                        *abort_flag = 1;
                        atomicExch(status, 4 /* MLA_ERR_TIMEOUT */);
                    }
                    stop = 1;
                }
                if (__shfl_sync(0xffffffffu, stop, 0)) ok = false;
            }
        }
    } else if (warp == kForwardWarp) {
        // ------------------------------------------- "scores read" forwarder
        // Tells the peer that this CTA's softmax warps have read the scores
        // it sent for tile g, so its swap warps may refill that slot.  A
        // cluster-scope remote arrive takes ~1,000 cycles, so it gets a warp
        // of its own instead of sitting on the softmax or swap critical path.
        if (lane == 0) {
            const uint32_t peerfree_remote0 = map_to_cta(bar(B_PEERFREE), peer);
            TileCursor cur;
            cur.init(v.pieces, p_begin, p_end);
            for (uint32_t g = 0; cur.valid(); ++g, cur.next()) {
                if (!bounded_wait(bar(B_XREAD + (g & 1u)), (g >> 1) & 1u, abort_flag, status)) break;
                mbar_arrive_remote(peerfree_remote0 + 8u * (g & 1u));
            }
        }
    } else {
        // ------------------------------------------------ score swap (fp16)
        const uint32_t quarter = (uint32_t)(warp & 3);
        const int32_t row = (int32_t)(quarter * 32 + lane);
        const uint32_t lane_off = (quarter * 32u) << 16;
        const uint32_t x_remote0 = map_to_cta(sbase + OFF_X, peer);
        const uint32_t xfull_remote0 = map_to_cta(bar(B_XFULL), peer);
        const int rsw = row & 7;
        TileCursor cur;
        cur.init(v.pieces, p_begin, p_end);
        uint32_t g = 0;
        bool ok = true;
        while (ok && cur.valid()) {
            const uint32_t slot = g & 1u, ph = (g >> 1) & 1u;
            ok = warp_wait(bar(B_SFULL + slot), ph, abort_flag, status);
            if (!ok) break;
            tc_fence_after();
            uint32_t h[BN / 2];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + TM_S + 64u * slot + lane_off, r0);
                tmem_ld32(tmem + TM_S + 64u * slot + lane_off + 32, r1);
                tmem_ld_wait64(r0, r1);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    h[i] = pack_f16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                    h[16 + i] = pack_f16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_SEMPTY + slot));
            ok = warp_wait<true>(bar(B_PEERFREE + slot), ph ^ 1u, abort_flag, status);
            if (!ok) break;
            const uint32_t dst = x_remote0 + slot * X_BYTES + (uint32_t)row * 128u;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_async_v4(dst + (uint32_t)((c ^ rsw) * 16), h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3],
                            xfull_remote0 + 8u * slot);
            ++g;
            cur.next();
        }
    }

    // ------------------------------------------------------------ teardown
    // this CTA's work is done: the dependent combine grid may be scheduled
    // (it waits for this grid's completion before reading anything)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer no longer writes into this CTA's smem
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace

size_t decode_tc_smem_bytes() { return SMEM_BYTES; }

cudaError_t decode_tc_max_clusters(int32_t* clusters) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<false>, &cfg);
    if (e != cudaSuccess) return e;
    *clusters = n;
    return cudaSuccess;
}

cudaError_t launch_decode_tc(const TcMaps& maps, const TcArgs& a, int32_t num_clusters, void* ws,
                             const WsLayout& L, cudaStream_t stream, bool lowp) {
    if (lowp)
        decode_tc_kernel<true><<<2 * num_clusters, kThreads, SMEM_BYTES, stream>>>(
            maps.kv_nope, maps.kv_rope, maps.q_rope, maps.kv_scale, a, ws, L);
    else
        decode_tc_kernel<false><<<2 * num_clusters, kThreads, SMEM_BYTES, stream>>>(
            maps.kv_nope, maps.kv_rope, maps.q_rope, maps.kv_scale, a, ws, L);
    return cudaGetLastError();
}

}  // namespace mla
