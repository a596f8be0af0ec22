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
// Why a 2-CTA cluster: the fp32 accumulator O of 128 rows x 512 latent
// columns is 256 KB, exactly one SM's tensor memory.  The two CTAs of a
// cluster therefore split the latent dims: rank r owns c_kv dims
// [256r, 256r+256) and RoPE dims [32r, 32r+32).  Each CTA
//   - streams only its 288 dims of every cache tile by TMA (the pair reads
//     each cached byte once),
//   - computes a partial S over its 288 dims (tcgen05, accumulator in TMEM),
//   - sends its partial S (fp32, 32 KB per tile) to the peer through
//     distributed shared memory (st.async + transaction barrier) and adds
//     the peer's partial: both CTAs then hold the same full S,
//   - runs the same online softmax (identical bits on both CTAs),
//   - accumulates its 256 output columns O += P V, with P (bf16) in TMEM
//     and the same smem tile read as an MN-major V operand.
// TMEM per CTA: O 256 columns, S 64, P 32 (of 512).
//
// Warp roles per CTA (192 threads): warp 0 = TMA producer, warp 1 = MMA
// issuer (and TMEM owner), warps 2-5 = softmax / correction / epilogue, one
// thread per query row (= TMEM lane).
//
// Every wait is bounded (ptx.cuh: bounded_wait); on a timeout the kernel
// records MLA_ERR_TIMEOUT in the workspace, drains its own copies and MMAs,
// frees TMEM and exits.
#include <cuda_bf16.h>
#include <math.h>

#include "decode_tc.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int BM = 128;         // query rows per unit
constexpr int BN = 64;          // tokens per tile (= page)
constexpr int NSTAGE = 3;       // cache-tile ring depth
constexpr int kThreads = 192;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t QN_BLK = BM * 128;                        // 64 dims x 128 rows, 128B swizzle
constexpr uint32_t OFF_QN = 0;
constexpr uint32_t OFF_QR = OFF_QN + 4 * QN_BLK;             // 32 RoPE dims x 128 rows, 64B swizzle
constexpr uint32_t QR_BYTES = BM * 64;
constexpr uint32_t KN_BLK = BN * 128;                        // 64 dims x 64 tokens
constexpr uint32_t KR_BYTES = BN * 64;                       // 32 dims x 64 tokens
constexpr uint32_t STAGE_BYTES = 4 * KN_BLK + KR_BYTES;      // 36864
constexpr uint32_t OFF_KV = OFF_QR + QR_BYTES;
constexpr uint32_t OFF_X = OFF_KV + NSTAGE * STAGE_BYTES;    // peer's partial S
constexpr uint32_t X_BYTES = BM * BN * 4;
constexpr uint32_t OFF_BAR = OFF_X + X_BYTES;
constexpr uint32_t SMEM_USED = OFF_BAR + 256;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;            // + alignment slack
constexpr uint32_t Q_TX = 4 * QN_BLK + QR_BYTES;

static_assert(OFF_QR % 1024 == 0 && OFF_KV % 1024 == 0 && STAGE_BYTES % 1024 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "fits in 227 KB");

// barriers
enum : int {
    B_QFULL = 0,
    B_QEMPTY = 1,
    B_KVFULL = 2,
    B_KVEMPTY = B_KVFULL + NSTAGE,
    B_SFULL = B_KVEMPTY + NSTAGE,
    B_SEMPTY,
    B_XFULL,
    B_PEERFREE,
    B_PFULL,
    B_PVDONE,
    B_EXIT,
    NUM_BARS
};
static_assert(NUM_BARS * 8 <= 128, "barrier area");
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 128;
constexpr uint32_t OFF_ABORT = OFF_BAR + 132;

// TMEM columns
constexpr uint32_t TM_O = 0, TM_S = 256, TM_P = 320, TM_COLS = 512;

constexpr uint32_t IDESC_QK = idesc_bf16(128, BN, 0, 0);   // S[128x64] = Q . K^T, both K-major
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, 0, 1);  // O[128x256] += P . V, V MN-major

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_kv_nope, const __grid_constant__ CUtensorMap tm_kv_rope,
                     const __grid_constant__ CUtensorMap tm_q_nope, const __grid_constant__ CUtensorMap tm_q_rope,
                     const TcArgs a, void* ws, const WsLayout L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
        mbar_init(bar(B_QFULL), 1);
        mbar_init(bar(B_QEMPTY), 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(bar(B_KVFULL + s), 1);
            mbar_init(bar(B_KVEMPTY + s), 1);
        }
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_SEMPTY), 128);
        mbar_init(bar(B_XFULL), 1);
        mbar_init(bar(B_PEERFREE), 128);
        mbar_init(bar(B_PFULL), 128);
        mbar_init(bar(B_PVDONE), 1);
        mbar_init(bar(B_EXIT), 1);
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
        tma_prefetch_desc(&tm_q_nope);
        tma_prefetch_desc(&tm_q_rope);
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

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint64_t pol;
            if (a.evict_first) pol = l2_policy_evict_first();
            else pol = l2_policy_evict_last();
            uint32_t stage = 0, phase = 0, q_cnt = 0;
            uint32_t issued_mask = 0, last_parity = 0;  // per stage: loads in flight for draining
            bool q_issued = false;
            bool ok = true;
            for (int32_t p = p_begin; p < p_end && ok; ++p) {
                const Piece pc = v.pieces[p];
                const int32_t b = pc.unit / RB, rb = pc.unit % RB;
                ok = bounded_wait(bar(B_QEMPTY), (q_cnt & 1u) ^ 1u, abort_flag, status);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(B_QFULL), Q_TX);
                const int32_t y = b * QH + rb * BM;
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)
                    tma_load_2d(sbase + OFF_QN + kb * QN_BLK, &tm_q_nope, bar(B_QFULL), 256 * rank + 64 * kb, y, pol);
                tma_load_2d(sbase + OFF_QR, &tm_q_rope, bar(B_QFULL), 32 * rank, y, pol);
                q_issued = true;
                ++q_cnt;
                for (int32_t t = pc.t_begin; t < pc.t_end; ++t) {
                    int32_t page = a.page_table[(int64_t)b * a.max_pages_per_seq + t];
                    if (page < 0 || page >= a.num_pages) {
                        atomicCAS(status, 0, 1);
                        page = 0;
                    }
                    ok = bounded_wait(bar(B_KVEMPTY + stage), phase ^ 1u, abort_flag, status);
                    if (!ok) break;
                    const uint32_t fb = bar(B_KVFULL + stage);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    const uint32_t dst = sbase + OFF_KV + stage * STAGE_BYTES;
                    const int32_t y0 = page * BN;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
                        tma_load_2d(dst + kb * KN_BLK, &tm_kv_nope, fb, 256 * rank + 64 * kb, y0, pol);
                    tma_load_2d(dst + 4 * KN_BLK, &tm_kv_rope, fb, 512 + 32 * rank, y0, pol);
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // drain: every issued copy must land before the CTA may exit
            for (int s = 0; s < NSTAGE; ++s)
                if (issued_mask & (1u << s)) drain_wait(bar(B_KVFULL + s), (last_parity >> s) & 1u);
            if (q_issued) drain_wait(bar(B_QFULL), (q_cnt - 1) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t tS = tmem + TM_S, tO = tmem + TM_O, tP = tmem + TM_P;
            uint32_t stage = 0, phase = 0, q_cnt = 0;
            uint32_t it = 0;
            bool pend = false, pend_first = false;
            uint32_t pend_stage = 0, pend_it = 0;
            bool ok = true;
            auto issue_pv = [&](uint32_t st, bool first, uint32_t pit) -> bool {
                if (!bounded_wait(bar(B_PFULL), pit & 1u, abort_flag, status)) return false;
                tc_fence_after();
                const uint32_t sk = sbase + OFF_KV + st * STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t bdesc = smem_desc(sk + kk * 2048, KN_BLK, 1024, kSwizzle128B);
                    umma_ts(tO, tP + kk * 8, bdesc, IDESC_PV, (first && kk == 0) ? 0u : 1u);
                }
                umma_commit(bar(B_PVDONE));
                umma_commit(bar(B_KVEMPTY + st));
                return true;
            };
            for (int32_t p = p_begin; p < p_end && ok; ++p) {
                const Piece pc = v.pieces[p];
                ok = bounded_wait(bar(B_QFULL), q_cnt & 1u, abort_flag, status);
                if (!ok) break;
                ++q_cnt;
                for (int32_t t = pc.t_begin; t < pc.t_end; ++t) {
                    ok = bounded_wait(bar(B_KVFULL + stage), phase, abort_flag, status) &&
                         bounded_wait(bar(B_SEMPTY), (it & 1u) ^ 1u, abort_flag, status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sk = sbase + OFF_KV + stage * STAGE_BYTES;
                    const uint32_t sq = sbase + OFF_QN;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = smem_desc(sq + kb * QN_BLK + kk * 32, 16, 1024, kSwizzle128B);
                            const uint64_t bd = smem_desc(sk + kb * KN_BLK + kk * 32, 16, 1024, kSwizzle128B);
                            umma_ss(tS, ad, bd, IDESC_QK, (kb | kk) != 0 ? 1u : 0u);
                        }
                    }
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint64_t ad = smem_desc(sbase + OFF_QR + kk * 32, 16, 512, kSwizzle64B);
                        const uint64_t bd = smem_desc(sk + 4 * KN_BLK + kk * 32, 16, 512, kSwizzle64B);
                        umma_ss(tS, ad, bd, IDESC_QK, 1u);
                    }
                    umma_commit(bar(B_SFULL));
                    if (t == pc.t_end - 1) umma_commit(bar(B_QEMPTY));
                    if (pend) {
                        ok = issue_pv(pend_stage, pend_first, pend_it);
                        if (!ok) break;
                    }
                    pend = true;
                    pend_stage = stage;
                    pend_first = (t == pc.t_begin);
                    pend_it = it;
                    ++it;
                    if (++stage == NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (ok && pend) issue_pv(pend_stage, pend_first, pend_it);
            // drain: all MMAs issued by this thread complete before TMEM is freed
            umma_commit(bar(B_EXIT));
            drain_wait(bar(B_EXIT), 0);
        }
    } else {
        // ------------------------------------- softmax / correction / epilogue
        const uint32_t quarter = (uint32_t)(warp & 3);
        const int32_t row = (int32_t)(quarter * 32 + lane);
        const uint32_t lane_off = (quarter * 32u) << 16;
        const uint32_t tS = tmem + TM_S + lane_off, tO = tmem + TM_O + lane_off, tP = tmem + TM_P + lane_off;
        const uint32_t x_local = sbase + OFF_X;
        const uint32_t x_remote = map_to_cta(x_local, peer);
        const uint32_t xfull_remote = map_to_cta(bar(B_XFULL), peer);
        const uint32_t peerfree_remote = map_to_cta(bar(B_PEERFREE), peer);
        const float4* xbuf = reinterpret_cast<const float4*>(smem + OFF_X);
        const bool leader = (threadIdx.x == 64);
        uint32_t it = 0, stage = 0;
        int64_t pv_waited = -1;
        bool ok = true;
        for (int32_t p = p_begin; p < p_end && ok; ++p) {
            const Piece pc = v.pieces[p];
            const int32_t b = pc.unit / RB, rb = pc.unit % RB;
            const int32_t len = checked_len(a.seq_lens, b, max_tokens, status);
            const int32_t rows_valid = min(BM, QH - rb * BM);
            const int32_t qrow = rb * BM + row;
            const int32_t vis = row < rows_valid ? visible_len(len, a.Q, a.H, qrow) : 0;
            const int32_t vis_max = visible_len(len, a.Q, a.H, rb * BM + rows_valid - 1);
            float m_ref = -INFINITY, l = 0.f;
            for (int32_t t = pc.t_begin; t < pc.t_end; ++t) {
                // 1. partial S of this CTA
                ok = warp_wait(bar(B_SFULL), it & 1u, abort_flag, status);
                if (!ok) break;
                tc_fence_after();
                float s[BN];
                {
                    uint32_t r[16];
#pragma unroll
                    for (int c = 0; c < BN / 16; ++c) {
                        tmem_ld16(tS + 16 * c, r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < 16; ++i) s[16 * c + i] = __uint_as_float(r[i]);
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(B_SEMPTY));
                // 2. swap partials with the peer CTA
                ok = warp_wait<true>(bar(B_PEERFREE), (it & 1u) ^ 1u, abort_flag, status);
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < BN / 4; ++c) {
                    const uint32_t pos = (uint32_t)(c ^ (row & 7));
                    st_async_v4(x_remote + (uint32_t)row * 256u + pos * 16u, __float_as_uint(s[4 * c]),
                                __float_as_uint(s[4 * c + 1]), __float_as_uint(s[4 * c + 2]),
                                __float_as_uint(s[4 * c + 3]), xfull_remote);
                }
                if (leader) mbar_arrive_expect_tx(bar(B_XFULL), X_BYTES);
                ok = warp_wait<true>(bar(B_XFULL), it & 1u, abort_flag, status);
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < BN / 4; ++c) {
                    const float4 o = xbuf[row * 16 + (c ^ (row & 7))];
                    s[4 * c] += o.x;
                    s[4 * c + 1] += o.y;
                    s[4 * c + 2] += o.z;
                    s[4 * c + 3] += o.w;
                }
                mbar_arrive_remote(peerfree_remote);
                // 3. online softmax in base 2 (both CTAs compute identical values)
                const int32_t tok0 = t * BN;
                float tmax = -INFINITY;
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    s[c] = (tok0 + c < vis) ? s[c] * a.scale_log2 : -INFINITY;
                    tmax = fmaxf(tmax, s[c]);
                }
                float factor = 1.f;
                bool rescale = false;
                if (tmax > m_ref + kRescaleThreshold) {
                    if (m_ref != -INFINITY) {
                        factor = exp2f(m_ref - tmax);
                        rescale = true;
                    }
                    l *= factor;
                    m_ref = tmax;
                }
                uint32_t pk[BN / 2];
                float lsum = 0.f;
#pragma unroll
                for (int c = 0; c < BN; c += 2) {
                    const float p0 = (s[c] == -INFINITY) ? 0.f : exp2f(s[c] - m_ref);
                    const float p1 = (s[c + 1] == -INFINITY) ? 0.f : exp2f(s[c + 1] - m_ref);
                    lsum += p0 + p1;
                    pk[c / 2] = pack_bf16x2(p0, p1);
                }
                l += lsum;
                // 4. PV of the previous tile must be done before P and O change
                if (it > 0 && pv_waited < (int64_t)it - 1) {
                    ok = warp_wait(bar(B_PVDONE), (it - 1) & 1u, abort_flag, status);
                    if (!ok) break;
                    pv_waited = (int64_t)it - 1;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
                    const float f = rescale ? factor : 1.f;
#pragma unroll 1
                    for (int c0 = 0; c0 < 256; c0 += 16) {
                        uint32_t r[16];
                        tmem_ld16(tO + c0, r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                        tmem_st16(tO + c0, r);
                    }
                }
                // 5. last tile of a ragged unit: clear cache rows past the end so
                //    that P = 0 never meets non-finite garbage in V
                if (tok0 + BN > vis_max) {
                    const int32_t nvalid = max(0, vis_max - tok0);
                    const int32_t nrows = BN - nvalid;
                    uint8_t* st_base = smem + OFF_KV + stage * STAGE_BYTES;
                    const int32_t chunks = nrows * 8 * 4;  // 16-byte chunks over 4 blocks
                    for (int32_t i = (int32_t)threadIdx.x - 64; i < chunks; i += 128) {
                        const int32_t kb = i / (nrows * 8);
                        const int32_t rem = i % (nrows * 8);
                        const int32_t rr = nvalid + rem / 8, cc = rem % 8;
                        *reinterpret_cast<uint4*>(st_base + kb * KN_BLK + rr * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                {
                    uint32_t r0[16], r1[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        r0[i] = pk[i];
                        r1[i] = pk[16 + i];
                    }
                    tmem_st16(tP, r0);
                    tmem_st16(tP + 16, r1);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(B_PFULL));
                ++it;
                if (++stage == NSTAGE) stage = 0;
            }
            if (!ok) break;
            // epilogue: O / l -> out (whole unit) or the partial slot
            ok = warp_wait(bar(B_PVDONE), (it - 1) & 1u, abort_flag, status);
            if (!ok) break;
            pv_waited = (int64_t)it - 1;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const float row_lse = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
            const bool store = row < rows_valid;
            const int64_t grow = (int64_t)b * QH + qrow;
#pragma unroll 1
            for (int c0 = 0; c0 < 256; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tO + c0, r);
                tmem_ld_wait(r);
                if (store) {
                    if (pc.slot < 0) {
                        uint4 w0, w1;
                        w0.x = pack_bf16x2(__uint_as_float(r[0]) * inv_l, __uint_as_float(r[1]) * inv_l);
                        w0.y = pack_bf16x2(__uint_as_float(r[2]) * inv_l, __uint_as_float(r[3]) * inv_l);
                        w0.z = pack_bf16x2(__uint_as_float(r[4]) * inv_l, __uint_as_float(r[5]) * inv_l);
                        w0.w = pack_bf16x2(__uint_as_float(r[6]) * inv_l, __uint_as_float(r[7]) * inv_l);
                        w1.x = pack_bf16x2(__uint_as_float(r[8]) * inv_l, __uint_as_float(r[9]) * inv_l);
                        w1.y = pack_bf16x2(__uint_as_float(r[10]) * inv_l, __uint_as_float(r[11]) * inv_l);
                        w1.z = pack_bf16x2(__uint_as_float(r[12]) * inv_l, __uint_as_float(r[13]) * inv_l);
                        w1.w = pack_bf16x2(__uint_as_float(r[14]) * inv_l, __uint_as_float(r[15]) * inv_l);
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + grow * 512 +
                                                              256 * rank + c0);
                        dst[0] = w0;
                        dst[1] = w1;
                    } else {
                        float4* dst = reinterpret_cast<float4*>(
                            v.o_part + ((int64_t)pc.slot * kRowsPerUnit + row) * 512 + 256 * rank + c0);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = make_float4(__uint_as_float(r[4 * q]) * inv_l, __uint_as_float(r[4 * q + 1]) * inv_l,
                                                 __uint_as_float(r[4 * q + 2]) * inv_l,
                                                 __uint_as_float(r[4 * q + 3]) * inv_l);
                    }
                }
            }
            if (store && rank == 0) {
                if (pc.slot < 0) {
                    if (a.lse) a.lse[grow] = row_lse;
                } else {
                    v.lse_part[(int64_t)pc.slot * kRowsPerUnit + row] = row_lse;
                }
            }
            tc_fence_before();
        }
    }

    // ------------------------------------------------------------ teardown
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
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
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
    e = cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg);
    if (e != cudaSuccess) return e;
    *clusters = n;
    return cudaSuccess;
}

cudaError_t launch_decode_tc(const TcMaps& maps, const TcArgs& a, int32_t num_clusters, void* ws,
                             const WsLayout& L, cudaStream_t stream) {
    decode_tc_kernel<<<2 * num_clusters, kThreads, SMEM_BYTES, stream>>>(maps.kv_nope, maps.kv_rope, maps.q_nope,
                                                                         maps.q_rope, a, ws, L);
    return cudaGetLastError();
}

}  // namespace mla
