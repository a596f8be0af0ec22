// Expanded (prefill) MLA attention on tcgen05 (see prefill.cuh).
//
// upproj_kernel: persistent GEMM, one 128 (tokens) x 256 (output columns)
// tile at a time.  Warp 0 streams 64-wide reduction blocks of the latent
// rows (two 64-token pages per tile, looked up in the page table) and of
// the weight rows by TMA into a 4-stage ring; warp 1 issues
// tcgen05.mma (M=128, N=256, K=16) into one of two TMEM accumulators;
// warps 2-5 drain the other accumulator (TMEM -> bf16 -> global), so the
// epilogue of tile i overlaps the MMAs of tile i+1.
//
// prefill_attn_kernel: persistent causal flash attention, one (128-query
// tile, head) item at a time, by groups of heads, heaviest items (last
// query tiles) first within a group.
// Warp 0 loads the item's queries [q^C || q^R] (128 x 192) and, per
// 128-key tile, the keys [K^C || k^R] (128 x 192) into a 2-stage key ring;
// warp 2 loads the values (128 x 128) into a 2-stage value ring (a key stage
// is free as soon as its QK completes, a value stage only after its PV);
// warp 1 issues S = Q K^T (12 MMAs, N=128) into one of two TMEM score
// buffers and O += P V (8 MMAs, A = P read from TMEM);
// two softmax warpgroups (warps 4-7 and 8-11, one thread per query row)
// take alternate key tiles and run the online softmax in fp32: causal mask
// on the diagonal tile, running maximum handed from one group to the other
// with a lazy O rescale (only when the maximum grows by more than 2^8), P
// written back as bf16 into the score buffer's first 64 columns; the owner
// of an item's last tile merges both groups' row sums and writes O / l.
// TMEM: S0 128 columns | S1 128 | O 128.
//
// Every wait is bounded (ptx.cuh: bounded_wait); on a timeout the kernel
// records MLA_ERR_TIMEOUT, drains its own copies and MMAs and exits.
#include <cuda_bf16.h>
#include <math.h>

#include "prefill.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 200000000ull) return;
    }
}

template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
    const bool ok = bounded_wait<kCluster>(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Page of token-page index `i` of the sequence, checked against the pool;
// pages past the sequence (ragged last tile) read page 0, whose rows are
// masked or not stored.
__device__ __forceinline__ int32_t page_at(const int32_t* row, int32_t i, int32_t pages, int32_t num_pages,
                                           int* status) {
    if (i >= pages) return 0;
    const int32_t p = row[i];
    if (p < 0 || p >= num_pages) {
        atomicCAS(status, 0, 1 /* MLA_ERR_INVALID_ARG */);
        return 0;
    }
    return p;
}

// ===================================================================== upproj

constexpr int UP_BM = 128, UP_BN = 256, UP_BK = 64, UP_NST = 4, UP_KB = kPrefillDc / UP_BK;
constexpr uint32_t UP_A_BYTES = UP_BM * UP_BK * 2;   // 16 KB: two 64-token page boxes
constexpr uint32_t UP_B_BYTES = UP_BN * UP_BK * 2;   // 32 KB
constexpr uint32_t UP_STAGE = UP_A_BYTES + UP_B_BYTES;
constexpr uint32_t UP_OFF_BAR = UP_NST * UP_STAGE;
constexpr uint32_t UP_SMEM = UP_OFF_BAR + 256 + 1024;
constexpr int UP_THREADS = 192;
enum : int { U_FULL = 0, U_EMPTY = UP_NST, U_AFULL = 2 * UP_NST, U_AEMPTY = U_AFULL + 2, U_EXIT = U_AEMPTY + 2, U_NBARS };
static_assert(U_NBARS * 8 + 16 <= 256, "barrier area");
constexpr uint32_t UP_IDESC = idesc_bf16(128, UP_BN, 0, 0);

__global__ void __launch_bounds__(UP_THREADS, 1)
    upproj_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_wk,
                  const __grid_constant__ CUtensorMap tm_wv, const UpprojArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + UP_OFF_BAR + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + UP_OFF_BAR + 256 - 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + UP_OFF_BAR + 256 - 12);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < UP_NST; ++s) {
            mbar_init(bar(U_FULL + s), 1);
            mbar_init(bar(U_EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(U_AFULL + s), 1);
            mbar_init(bar(U_AEMPTY + s), 4);
        }
        mbar_init(bar(U_EXIT), 1);
        *abort_flag = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_c);
        tma_prefetch_desc(&tm_wk);
        tma_prefetch_desc(&tm_wv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int32_t m_tiles = (a.T + UP_BM - 1) / UP_BM;
    const int32_t n_half = a.n_per / UP_BN;
    const int32_t n_tiles = 2 * n_half;
    const int32_t tiles = m_tiles * n_tiles;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int32_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int32_t mt = t / n_tiles, nt = t % n_tiles;
                const bool is_v = nt >= n_half;
                const int32_t n0 = (nt % n_half) * UP_BN;
                const int32_t p0 = page_at(a.page_row, 2 * mt, a.pages, a.num_pages, a.status);
                const int32_t p1 = page_at(a.page_row, 2 * mt + 1, a.pages, a.num_pages, a.status);
                for (int kb = 0; kb < UP_KB; ++kb) {
                    ok = bounded_wait(bar(U_EMPTY + stage), phase ^ 1u, abort_flag, a.status);
                    if (!ok) break;
                    const uint32_t fb = bar(U_FULL + stage);
                    const uint32_t dst = sbase + stage * UP_STAGE;
                    mbar_arrive_expect_tx(fb, UP_STAGE);
                    tma_load_2d(dst, &tm_c, fb, kb * UP_BK, p0 * 64, pol);
                    tma_load_2d(dst + UP_A_BYTES / 2, &tm_c, fb, kb * UP_BK, p1 * 64, pol);
                    tma_load_2d(dst + UP_A_BYTES, is_v ? &tm_wv : &tm_wk, fb, kb * UP_BK, n0, pol);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == UP_NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < UP_NST; ++s)
                if (issued & (1u << s)) drain_wait(bar(U_FULL + s), (last_par >> s) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, i = 0;
            bool ok = true;
            for (int32_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
                const uint32_t ab = i & 1u;
                ok = bounded_wait(bar(U_AEMPTY + ab), ((i >> 1) & 1u) ^ 1u, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tacc = tmem + ab * UP_BN;
                for (int kb = 0; kb < UP_KB && ok; ++kb) {
                    ok = bounded_wait(bar(U_FULL + stage), phase, abort_flag, a.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sa = sbase + stage * UP_STAGE, sb = sa + UP_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < UP_BK / 16; ++kk)
                        umma_ss(tacc, smem_desc(sa + kk * 32, 16, 1024, kSwizzle128B),
                                smem_desc(sb + kk * 32, 16, 1024, kSwizzle128B), UP_IDESC, (kb | kk) ? 1u : 0u);
                    umma_commit(bar(U_EMPTY + stage));
                    if (++stage == UP_NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit(bar(U_AFULL + ab));
            }
            // every MMA issued by this thread has completed before TMEM is released
            umma_commit(bar(U_EXIT));
            drain_wait(bar(U_EXIT), 0);
        }
    } else {
        // epilogue warps 2..5: TMEM lane quarter = warp % 4
        const uint32_t q = (uint32_t)(warp & 3);
        const int32_t row = (int32_t)(q * 32 + lane);
        uint32_t i = 0;
        bool ok = true;
        for (int32_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
            const uint32_t ab = i & 1u;
            ok = warp_wait(bar(U_AFULL + ab), (i >> 1) & 1u, abort_flag, a.status);
            if (!ok) break;
            tc_fence_after();
            const int32_t mt = t / n_tiles, nt = t % n_tiles;
            const bool is_v = nt >= n_half;
            const int32_t n0 = (nt % n_half) * UP_BN;
            const int32_t tok = mt * UP_BM + row;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_v ? a.v_out : a.k_out) + (int64_t)tok * a.n_per + n0;
            const uint32_t tacc = tmem + ab * UP_BN + ((q * 32u) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < UP_BN; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tacc + c0, r);
                tmem_ld_wait32(r);
                if (tok < a.T) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        d4[k] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * k]), __uint_as_float(r[8 * k + 1])),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 2]), __uint_as_float(r[8 * k + 3])),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 4]), __uint_as_float(r[8 * k + 5])),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 6]), __uint_as_float(r[8 * k + 7])));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(U_AEMPTY + ab));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ================================================================ attention

constexpr int AT_BM = 128, AT_BN = 128;
constexpr uint32_t BOX = 128 * 128;                       // one [128 rows][64 bf16] box, 16 KB
constexpr uint32_t AT_Q_BYTES = 3 * BOX;                  // q^C (2 boxes) || q^R
constexpr uint32_t AT_K_BYTES = 3 * BOX;                  // K^C (2 boxes) || k^R (two 8 KB page boxes)
constexpr uint32_t AT_V_BYTES = 2 * BOX;
constexpr int AT_NST = 2;
constexpr uint32_t AT_OFF_Q = 0;
// Keys and values of a key tile sit in separate rings: a key stage is free
// once its QK has completed, a value stage once its PV has.
constexpr uint32_t AT_OFF_K = AT_Q_BYTES;
constexpr uint32_t AT_OFF_V = AT_OFF_K + AT_NST * AT_K_BYTES;
constexpr uint32_t AT_OFF_BAR = AT_OFF_V + AT_NST * AT_V_BYTES;
constexpr uint32_t AT_OFF_M = AT_OFF_BAR + 256;              // [2 slots][128 rows] running max after a tile
constexpr uint32_t AT_OFF_LM = AT_OFF_M + 2 * 128 * 4;       // [2][128] (row sum, its max) of a group
constexpr uint32_t AT_SMEM = AT_OFF_LM + 2 * 128 * 8 + 1024;
static_assert(AT_SMEM <= 232448, "fits in 227 KB");
// Three warpgroups: warp 0 TMA, warp 1 MMA (warps 2-3 idle), and two
// softmax warpgroups (warps 4-7, 8-11) taking alternate key tiles.  The
// producer warpgroup hands most of its registers to the softmax groups
// (setmaxnreg), whose 128 scores per thread would not fit the 168
// registers of a 384-thread launch; the shares add up to 384 x 168 and the
// launcher checks the compiled count before every launch.
constexpr int AT_THREADS = 384;
constexpr int AT_PRODUCER_REGS = 56;
constexpr int AT_SOFTMAX_REGS = 224;
static_assert(4 * AT_PRODUCER_REGS + 8 * AT_SOFTMAX_REGS <= 12 * 168, "register split within the launch");
enum : int {
    A_QFULL = 0,
    A_QEMPTY,
    A_KFULL,
    A_KEMPTY = A_KFULL + AT_NST,
    A_VFULL = A_KEMPTY + AT_NST,
    A_VEMPTY = A_VFULL + AT_NST,
    A_SFULL = A_VEMPTY + AT_NST,    // [2]
    A_PFULL = A_SFULL + 2,          // [2]
    A_PVDONE = A_PFULL + 2,         // [2] PV of the tile in that slot completed
    A_OFREE = A_PVDONE + 2,         // epilogue read O
    A_EXIT,
    A_MREADY,                       // [2] running max after the tile in that slot published
    A_LFULL = A_MREADY + 2,         // [2] a group's row sum of an item published (item parity)
    A_LFREE = A_LFULL + 2,          // [2] ... and read by the epilogue group
    A_NBARS = A_LFREE + 2
};
static_assert(A_NBARS * 8 + 16 <= 256, "barrier area");
constexpr uint32_t TM_S0 = 0, TM_O = 256;
constexpr uint32_t AT_IDESC_QK = idesc_bf16(128, AT_BN, 0, 0);
constexpr uint32_t AT_IDESC_PV = idesc_bf16(128, kPrefillDh, 0, 1);
constexpr float kRescale = 8.0f;
constexpr float kLn2f = 0.69314718055994530942f;

struct Item {
    int32_t qt, h, ntiles;
};

// Items go head group by head group (8 heads when H allows): within a group
// the heaviest (last) query tiles first, for balance; the ~148 items in
// flight then cover ~8 heads, whose keys and values (2 MB per head at
// T = 4096) stay in L2 across query tiles instead of being fetched from
// DRAM again for every query tile.
__device__ __forceinline__ Item item_of(int32_t w, int32_t m_tiles, int32_t H) {
    const int32_t G = (H % 8 == 0) ? 8 : ((H % 4 == 0) ? 4 : ((H % 2 == 0) ? 2 : 1));
    const int32_t per_group = G * m_tiles;
    const int32_t grp = w / per_group, r = w % per_group;
    Item it;
    it.qt = m_tiles - 1 - r / G;
    it.h = grp * G + r % G;
    it.ntiles = it.qt + 1;
    return it;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tm_qc, const __grid_constant__ CUtensorMap tm_qr,
                        const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_kr, const PrefillAttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + AT_OFF_BAR + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + AT_OFF_BAR + 256 - 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + AT_OFF_BAR + 256 - 12);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(A_QFULL), 1);
        mbar_init(bar(A_QEMPTY), 1);
        for (int s = 0; s < AT_NST; ++s) {
            mbar_init(bar(A_KFULL + s), 1);
            mbar_init(bar(A_KEMPTY + s), 1);
            mbar_init(bar(A_VFULL + s), 1);
            mbar_init(bar(A_VEMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(A_SFULL + s), 1);
            mbar_init(bar(A_PFULL + s), 4);
            mbar_init(bar(A_PVDONE + s), 1);
        }
        mbar_init(bar(A_OFREE), 4);
        mbar_init(bar(A_EXIT), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(A_MREADY + s), 4);
            mbar_init(bar(A_LFULL + s), 4);
            mbar_init(bar(A_LFREE + s), 4);
        }
        *abort_flag = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_qc);
        tma_prefetch_desc(&tm_qr);
        tma_prefetch_desc(&tm_kc);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_kr);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int32_t m_tiles = (a.T + AT_BM - 1) / AT_BM;
    const int32_t items = m_tiles * a.H;

    if (warp < 4) {
    // producer warpgroup: the register budget of the code below is set here
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(AT_PRODUCER_REGS));
    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            uint32_t stage = 0, phase = 0, qn = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int32_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
                const Item it = item_of(w, m_tiles, a.H);
                ok = bounded_wait(bar(A_QEMPTY), (qn & 1u) ^ 1u, abort_flag, a.status);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(A_QFULL), AT_Q_BYTES);
                const int32_t y = it.qt * AT_BM;
                tma_load_2d(sbase + AT_OFF_Q, &tm_qc, bar(A_QFULL), it.h * kPrefillDh, y, pol);
                tma_load_2d(sbase + AT_OFF_Q + BOX, &tm_qc, bar(A_QFULL), it.h * kPrefillDh + 64, y, pol);
                tma_load_2d(sbase + AT_OFF_Q + 2 * BOX, &tm_qr, bar(A_QFULL), it.h * kPrefillDr, y, pol);
                ++qn;
                for (int32_t j = 0; j < it.ntiles; ++j) {
                    ok = bounded_wait(bar(A_KEMPTY + stage), phase ^ 1u, abort_flag, a.status);
                    if (!ok) break;
                    const uint32_t fb = bar(A_KFULL + stage);
                    const uint32_t dst = sbase + AT_OFF_K + stage * AT_K_BYTES;
                    mbar_arrive_expect_tx(fb, AT_K_BYTES);
                    const int32_t yk = j * AT_BN;
                    tma_load_2d(dst, &tm_kc, fb, it.h * kPrefillDh, yk, pol);
                    tma_load_2d(dst + BOX, &tm_kc, fb, it.h * kPrefillDh + 64, yk, pol);
                    const int32_t p0 = page_at(a.page_row, 2 * j, a.pages, a.num_pages, a.status);
                    const int32_t p1 = page_at(a.page_row, 2 * j + 1, a.pages, a.num_pages, a.status);
                    tma_load_2d(dst + 2 * BOX, &tm_kr, fb, kPrefillDc, p0 * 64, pol);
                    tma_load_2d(dst + 2 * BOX + BOX / 2, &tm_kr, fb, kPrefillDc, p1 * 64, pol);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == AT_NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < AT_NST; ++s)
                if (issued & (1u << s)) drain_wait(bar(A_KFULL + s), (last_par >> s) & 1u);
            if (qn > 0) drain_wait(bar(A_QFULL), (qn - 1) & 1u);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------- TMA (values)
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int32_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
                const Item it = item_of(w, m_tiles, a.H);
                for (int32_t j = 0; j < it.ntiles; ++j) {
                    ok = bounded_wait(bar(A_VEMPTY + stage), phase ^ 1u, abort_flag, a.status);
                    if (!ok) break;
                    const uint32_t fb = bar(A_VFULL + stage);
                    const uint32_t dst = sbase + AT_OFF_V + stage * AT_V_BYTES;
                    mbar_arrive_expect_tx(fb, AT_V_BYTES);
                    const int32_t yk = j * AT_BN;
                    tma_load_2d(dst, &tm_v, fb, it.h * kPrefillDh, yk, pol);
                    tma_load_2d(dst + BOX, &tm_v, fb, it.h * kPrefillDh + 64, yk, pol);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == AT_NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < AT_NST; ++s)
                if (issued & (1u << s)) drain_wait(bar(A_VFULL + s), (last_par >> s) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, pv_stage = 0, pv_phase = 0, qn = 0, g = 0, items_done = 0;
            bool ok = true;
            const uint32_t tO = tmem + TM_O;
            auto issue_pv = [&](uint32_t gp, bool first) -> bool {
                const uint32_t slot = gp & 1u;
                if (!bounded_wait(bar(A_PFULL + slot), (gp >> 1) & 1u, abort_flag, a.status)) return false;
                if (!bounded_wait(bar(A_VFULL + pv_stage), pv_phase, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint32_t tP = tmem + TM_S0 + 128u * slot;
                const uint32_t sv = sbase + AT_OFF_V + pv_stage * AT_V_BYTES;
#pragma unroll
                for (int kk = 0; kk < AT_BN / 16; ++kk)
                    umma_ts(tO, tP + kk * 8, smem_desc(sv + kk * 2048, BOX, 1024, kSwizzle128B), AT_IDESC_PV,
                            (first && kk == 0) ? 0u : 1u);
                umma_commit(bar(A_PVDONE + slot));
                umma_commit(bar(A_VEMPTY + pv_stage));
                if (++pv_stage == AT_NST) {
                    pv_stage = 0;
                    pv_phase ^= 1u;
                }
                return true;
            };
            for (int32_t w = blockIdx.x; w < items && ok; w += gridDim.x) {
                const Item it = item_of(w, m_tiles, a.H);
                ok = bounded_wait(bar(A_QFULL), qn & 1u, abort_flag, a.status);
                if (!ok) break;
                ++qn;
                for (int32_t j = 0; j < it.ntiles && ok; ++j, ++g) {
                    const uint32_t slot = g & 1u;
                    ok = bounded_wait(bar(A_KFULL + stage), phase, abort_flag, a.status);
                    if (!ok) break;
                    // the score buffer's previous tile (g - 2): its P was read by PV
                    if (g >= 2) {
                        ok = bounded_wait(bar(A_PVDONE + slot), ((g - 2) >> 1) & 1u, abort_flag, a.status);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint32_t tS = tmem + TM_S0 + 128u * slot;
                    const uint32_t sk = sbase + AT_OFF_K + stage * AT_K_BYTES;
#pragma unroll
                    for (int c = 0; c < 3; ++c)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_ss(tS, smem_desc(sbase + AT_OFF_Q + c * BOX + kk * 32, 16, 1024, kSwizzle128B),
                                    smem_desc(sk + c * BOX + kk * 32, 16, 1024, kSwizzle128B), AT_IDESC_QK,
                                    (c | kk) ? 1u : 0u);
                    umma_commit(bar(A_SFULL + slot));
                    umma_commit(bar(A_KEMPTY + stage));   // the key stage is free once this QK completes
                    if (j == it.ntiles - 1) umma_commit(bar(A_QEMPTY));
                    if (++stage == AT_NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (j >= 1) {
                        if (j == 1 && items_done > 0) {   // O of the previous item read by its epilogue
                            ok = bounded_wait(bar(A_OFREE), (items_done - 1) & 1u, abort_flag, a.status);
                            if (!ok) break;
                        }
                        ok = issue_pv(g - 1, j == 1);
                    }
                }
                if (!ok) break;
                if (it.ntiles == 1 && items_done > 0) {
                    ok = bounded_wait(bar(A_OFREE), (items_done - 1) & 1u, abort_flag, a.status);
                    if (!ok) break;
                }
                ok = issue_pv(g - 1, it.ntiles == 1);
                ++items_done;
            }
            // every MMA issued by this thread has completed before TMEM is released
            umma_commit(bar(A_EXIT));
            drain_wait(bar(A_EXIT), 0);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(AT_SOFTMAX_REGS));
        // ---------------------------------------------------- softmax / epilogue
        // Two warpgroups take alternate key tiles (group g & 1 owns global
        // tile g), so one tile's softmax overlaps the next tile's.  One
        // thread owns one query row.  The running maximum is handed from the
        // owner of tile g-1 to the owner of tile g through shared memory
        // (A_MREADY); each group keeps the row sum of its own tiles relative
        // to the latest maximum it has seen, and the owner of an item's last
        // tile merges the other group's sum (A_LFULL / A_LFREE) and writes
        // the epilogue.
        const uint32_t wg = (uint32_t)((warp - 4) >> 2);
        const uint32_t q = (uint32_t)(warp & 3);
        const int32_t row = (int32_t)(q * 32 + lane);
        const uint32_t lane_off = (q * 32u) << 16;
        const uint32_t tO = tmem + TM_O + lane_off;
        const float sl2 = a.scale_log2;
        float* mrow = reinterpret_cast<float*>(smem + AT_OFF_M);     // [2 slots][128 rows]
        float2* lm = reinterpret_cast<float2*>(smem + AT_OFF_LM);    // [2 items][128 rows]
        uint32_t g = 0, k = 0;   // global tile and item counters of this CTA
        bool ok = true;
        for (int32_t w = blockIdx.x; w < items && ok; w += gridDim.x, ++k) {
            const Item it = item_of(w, m_tiles, a.H);
            const int32_t t = it.qt * AT_BM + row;    // this thread's query position
            float m_seen = -INFINITY, l = 0.f;
            for (int32_t j = 0; j < it.ntiles && ok; ++j, ++g) {
                const uint32_t slot = g & 1u;
                const bool last = j == it.ntiles - 1;
                if (slot != wg) {
                    // not ours; after the item's last tile hand this group's sum over
                    if (last) {
                        ok = warp_wait(bar(A_LFREE + (k & 1u)), ((k >> 1) & 1u) ^ 1u, abort_flag, a.status);
                        if (!ok) break;
                        lm[(k & 1u) * 128 + row] = make_float2(l, m_seen);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(A_LFULL + (k & 1u)));
                    }
                    continue;
                }
                ok = warp_wait(bar(A_SFULL + slot), (g >> 1) & 1u, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tS = tmem + TM_S0 + 128u * slot + lane_off;
                float s[AT_BN];
                {
                    uint32_t r0[32], r1[32];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        tmem_ld32(tS + 64 * h2, r0);
                        tmem_ld32(tS + 64 * h2 + 32, r1);
                        tmem_ld_wait64(r0, r1);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            s[64 * h2 + i] = __uint_as_float(r0[i]);
                            s[64 * h2 + 32 + i] = __uint_as_float(r1[i]);
                        }
                    }
                }
                // causal mask on the diagonal tile (key k visible iff k <= t; also k < T)
                if (j == it.qt) {
                    const int32_t k0 = j * AT_BN;
                    const int32_t lim = min(t, a.T - 1) - k0;   // last visible column
#pragma unroll
                    for (int c = 0; c < AT_BN; ++c) s[c] = (c <= lim) ? s[c] : -INFINITY;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < AT_BN; ++c) mx = fmaxf(mx, s[c]);
                mx *= sl2;
                // running maximum after tile g-1 (the other group's); lazy:
                // it moves, and O is rescaled, only when it grows by > 2^8
                float m_prev = -INFINITY;
                if (g > 0) {
                    ok = warp_wait(bar(A_MREADY + (slot ^ 1u)), ((g - 1) >> 1) & 1u, abort_flag, a.status);
                    if (!ok) break;
                    if (j > 0) m_prev = mrow[(slot ^ 1u) * 128 + row];
                }
                float m_cur = m_prev, factor = 1.f;
                bool rescale = false;
                if (mx > m_prev + kRescale) {
                    if (m_prev != -INFINITY) {
                        factor = fast_exp2(m_prev - mx);
                        rescale = true;
                    }
                    m_cur = mx;
                }
                mrow[slot * 128 + row] = m_cur;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(A_MREADY + slot));
                if (m_seen != -INFINITY && m_cur != m_seen) l *= fast_exp2(m_seen - m_cur);
                m_seen = m_cur;
                const float neg_m = (m_cur == -INFINITY) ? 0.f : -m_cur;
                float ls0 = 0.f, ls1 = 0.f;
                uint32_t pk[AT_BN / 2];
#pragma unroll
                for (int c = 0; c < AT_BN; c += 2) {
                    const float p0 = fast_exp2(fmaf(s[c], sl2, neg_m));
                    const float p1 = fast_exp2(fmaf(s[c + 1], sl2, neg_m));
                    ls0 += p0;
                    ls1 += p1;
                    pk[c / 2] = pack_bf16x2(p0, p1);
                }
                l += ls0 + ls1;
                // O rescale (after the previous tile's PV, before this tile's)
                if (__any_sync(0xffffffffu, rescale) && j > 0) {
                    ok = warp_wait(bar(A_PVDONE + (slot ^ 1u)), ((g - 1) >> 1) & 1u, abort_flag, a.status);
                    if (!ok) break;
                    tc_fence_after();
                    const float f = rescale ? factor : 1.f;
#pragma unroll 1
                    for (int c0 = 0; c0 < kPrefillDh; c0 += 32) {
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
                }
                // P (bf16 pairs along the key axis) into the score buffer's first 64 columns
                {
                    uint32_t* pp = pk;
#pragma unroll
                    for (int c0 = 0; c0 < AT_BN / 2; c0 += 16)
                        tmem_st16(tS + c0, *reinterpret_cast<uint32_t(*)[16]>(pp + c0));
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(A_PFULL + slot));
                if (!last) continue;
                // epilogue after the item's last PV: O / (both groups' sums)
                ok = warp_wait(bar(A_PVDONE + slot), (g >> 1) & 1u, abort_flag, a.status);
                if (!ok) break;
                ok = warp_wait(bar(A_LFULL + (k & 1u)), (k >> 1) & 1u, abort_flag, a.status);
                if (!ok) break;
                const float2 other = lm[(k & 1u) * 128 + row];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(A_LFREE + (k & 1u)));
                tc_fence_after();
                // the other group's sum is relative to the maximum it last saw (<= m_seen)
                const float l_tot = l + (other.y == -INFINITY ? 0.f : other.x * fast_exp2(other.y - m_seen));
                const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
                const bool store = t < a.T;
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)t * a.H + it.h) * kPrefillDh;
#pragma unroll 1
                for (int c0 = 0; c0 < kPrefillDh; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tO + c0, r);
                    tmem_ld_wait32(r);
                    if (store) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            d4[k4] = make_uint4(
                                pack_bf16x2(__uint_as_float(r[8 * k4]) * inv_l, __uint_as_float(r[8 * k4 + 1]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * k4 + 2]) * inv_l, __uint_as_float(r[8 * k4 + 3]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * k4 + 4]) * inv_l, __uint_as_float(r[8 * k4 + 5]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * k4 + 6]) * inv_l, __uint_as_float(r[8 * k4 + 7]) * inv_l));
                    }
                }
                if (store && a.lse)
                    a.lse[(int64_t)t * a.H + it.h] = l_tot > 0.f ? (m_seen + log2f(l_tot)) * kLn2f : -INFINITY;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(A_OFREE));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_upproj(const UpprojMaps& maps, const UpprojArgs& a, int32_t sms, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(upproj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, UP_SMEM);
    if (e != cudaSuccess) return e;
    const int32_t tiles = ((a.T + UP_BM - 1) / UP_BM) * 2 * (a.n_per / UP_BN);
    const int32_t grid = tiles < sms ? tiles : sms;
    if (grid <= 0) return cudaSuccess;
    upproj_kernel<<<grid, UP_THREADS, UP_SMEM, stream>>>(maps.latent, maps.w_uk, maps.w_uv, a);
    return cudaGetLastError();
}

cudaError_t launch_prefill_attn(const PrefillAttnMaps& maps, const PrefillAttnArgs& a, int32_t sms,
                                cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
    if (e != cudaSuccess) return e;
    // the register split must fit what the launch allocates, or the softmax
    // warpgroups' setmaxnreg.inc could never be granted
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, prefill_attn_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * AT_THREADS < 32 * (4 * AT_PRODUCER_REGS + 8 * AT_SOFTMAX_REGS)) return cudaErrorInvalidConfiguration;
    const int32_t items = ((a.T + AT_BM - 1) / AT_BM) * a.H;
    const int32_t grid = items < sms ? items : sms;
    if (grid <= 0) return cudaSuccess;
    prefill_attn_kernel<<<grid, AT_THREADS, AT_SMEM, stream>>>(maps.q_c, maps.q_r, maps.k_c, maps.v, maps.k_r, a);
    return cudaGetLastError();
}

}  // namespace mla
