// Absorption GEMMs (see absorb.cuh).  One CTA computes a 128 x 64 tile of
// the transposed per-head product D[m][n] = sum_k A_h[m][k] * B_h[n][k]:
//   query side:  A_h[m][k] = W^UK[h][k][m]  (MN-major: contiguous along m),
//                B_h[n][k] = q^C[n][h][k],   D -> q_nope[n][h][m];
//   output side: A_h[m][k] = W^UV[h][m][k]  (K-major),
//                B_h[n][k] = u[n][h][k],     D -> o[n][h][m].
// Grid (m_total / 128, H, ceil(n_rows / BN)), BN = 64 query rows per CTA;
// 128 threads: warp 0 lane 0
// streams 64-wide reduction blocks of A and B by TMA into a ring of up to 4
// stages (2 for the query side's 128-deep reduction), warp 1 lane 0 issues
// tcgen05.mma (M=128, N=BN, K=16) into a TMEM accumulator, then all four
// warps read their TMEM lane quarter and store bf16 rows (rows past n_rows
// are zero-filled by TMA and not stored).
// Every wait is bounded; on a timeout the status word (if given) records
// MLA_ERR_TIMEOUT and the CTA drains its copies and MMAs before it exits.
#include <cuda_bf16.h>

#include "absorb.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int NST = 4;                                     // ring depth at most (fewer if K is short)
constexpr uint32_t A_BYTES = kAbsorbBM * kAbsorbBK * 2;   // 16 KB

template <int BN>
struct Tile {
    static constexpr uint32_t B_BYTES = BN * kAbsorbBK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TM_COLS = BN < 32 ? 32 : BN;
    static_assert(STAGE_BYTES % 1024 == 0, "swizzle atoms stay 1024-aligned");
};

// barriers, TMEM slot and abort flag after the ring; + alignment slack
__host__ __device__ constexpr uint32_t smem_bytes(uint32_t stage_bytes, int nst) {
    return (uint32_t)nst * stage_bytes + 128 + 1024;
}

enum : int { B_FULL = 0, B_EMPTY = NST, B_DONE = 2 * NST, NUM_BARS };
static_assert(NUM_BARS * 8 <= 96, "barrier area");

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                            int32_t y, int32_t z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// Wait limited by time only (ignores the abort flag): used to drain copies
// and MMAs already in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 200000000ull) return;
    }
}

template <bool kAMn, int BN>
__global__ void __launch_bounds__(128, 1)
    absorb_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                  const AbsorbArgs a, const int nst) {
    constexpr uint32_t STAGE_BYTES = Tile<BN>::STAGE_BYTES;
    constexpr uint32_t TM_COLS = Tile<BN>::TM_COLS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t mt = blockIdx.x, h = blockIdx.y, nt = blockIdx.z;
    const int32_t kblocks = a.k_total / kAbsorbBK;
    const uint32_t OFF_BAR = (uint32_t)nst * STAGE_BYTES;
    auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 96);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 100);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), 1);
        }
        mbar_init(bar(B_DONE), 1);
        *abort_flag = 0;
        fence_mbar_init_cluster();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        const uint64_t pol_w = l2_policy_evict_first();   // weights: read once
        const uint64_t pol_x = l2_policy_evict_last();    // activations: read by every m tile
        uint32_t issued_mask = 0, last_parity = 0;
        for (int32_t kb = 0; kb < kblocks; ++kb) {
            const uint32_t s = (uint32_t)(kb % nst), ph = (uint32_t)(kb / nst) & 1u;
            if (!bounded_wait(bar(B_EMPTY + s), ph ^ 1u, abort_flag, a.status)) break;
            const uint32_t full = bar(B_FULL + s);
            const uint32_t dst = sbase + s * STAGE_BYTES;
            mbar_arrive_expect_tx(full, STAGE_BYTES);
            if (kAMn) {   // two boxes of 64 (m) x 64 (k rows)
                const int32_t y = h * a.k_total + kb * kAbsorbBK;
                tma_load_2d(dst, &tm_a, full, mt * kAbsorbBM, y, pol_w);
                tma_load_2d(dst + A_BYTES / 2, &tm_a, full, mt * kAbsorbBM + 64, y, pol_w);
            } else {      // one box of 64 (k) x 128 (m rows)
                tma_load_2d(dst, &tm_a, full, kb * kAbsorbBK, h * a.m_total + mt * kAbsorbBM, pol_w);
            }
            tma_load_3d(dst + A_BYTES, &tm_b, full, kb * kAbsorbBK, h, nt * BN, pol_x);
            issued_mask |= 1u << s;
            last_parity = (last_parity & ~(1u << s)) | (ph << s);
        }
        for (int s = 0; s < NST; ++s)   // no copy may land after the CTA is gone
            if (issued_mask & (1u << s)) drain_wait(bar(B_FULL + s), (last_parity >> s) & 1u);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16(kAbsorbBM, BN, kAMn ? 1u : 0u, 0u);
        for (int32_t kb = 0; kb < kblocks; ++kb) {
            const uint32_t s = (uint32_t)(kb % nst), ph = (uint32_t)(kb / nst) & 1u;
            if (!bounded_wait(bar(B_FULL + s), ph, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t sa = sbase + s * STAGE_BYTES, sb = sa + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < kAbsorbBK / 16; ++kk) {
                // MN-major A: 16 k-rows of 128 B per step, the two 64-wide m
                // blocks 8 KB apart; K-major A and B: 32 B per step in the row
                const uint64_t ad = kAMn ? smem_desc(sa + kk * 2048, A_BYTES / 2, 1024, kSwizzle128B)
                                         : smem_desc(sa + kk * 32, 16, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024, kSwizzle128B);
                umma_ss(tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(bar(B_EMPTY + s));
        }
        umma_commit(bar(B_DONE));
        drain_wait(bar(B_DONE), 0);   // TMEM is freed below only after the MMAs are done
    }
    __syncwarp();

    // ------------------------------------------------------------ epilogue
    // (all four warps: warp w owns TMEM lanes 32w..32w+31 = output columns)
    // (the outcome is made warp-uniform: tcgen05.ld is warp-collective)
    if (__all_sync(0xffffffffu, bounded_wait(bar(B_DONE), 0, abort_flag, a.status))) {
        tc_fence_after();
        const uint32_t lane_off = ((uint32_t)(warp & 3) * 32u) << 16;
        const int32_t m = mt * kAbsorbBM + warp * 32 + lane;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
        const int32_t n0 = nt * BN;
        const int64_t row_stride = (int64_t)a.H * a.m_total;
        __nv_bfloat16* col = out + (int64_t)h * a.m_total + m;
        static_assert(BN == 32 || BN == 64, "epilogue reads 32-column groups");
#pragma unroll
        for (int g = 0; g < BN / 32; ++g) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + 32 * g, r);
            tmem_ld_wait32(r);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (n0 + 32 * g + i < a.n_rows)
                    col[(int64_t)(n0 + 32 * g + i) * row_stride] = __float2bfloat16_rn(__uint_as_float(r[i]));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

template <bool kAMn, int BN>
cudaError_t launch_one(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const AbsorbArgs& a, cudaStream_t stream) {
    const int kblocks = a.k_total / kAbsorbBK;
    const int nst = kblocks < NST ? kblocks : NST;
    const uint32_t smem = smem_bytes(Tile<BN>::STAGE_BYTES, nst);
    cudaError_t e = cudaFuncSetAttribute(absorb_kernel<kAMn, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes(Tile<BN>::STAGE_BYTES, NST));
    if (e != cudaSuccess) return e;
    const dim3 grid(a.m_total / kAbsorbBM, a.H, (a.n_rows + BN - 1) / BN);
    absorb_kernel<kAMn, BN><<<grid, 128, smem, stream>>>(tm_a, tm_b, a, nst);
    return cudaGetLastError();
}

}  // namespace

int absorb_rows_per_cta(bool) { return 64; }

cudaError_t launch_absorb(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const AbsorbArgs& a, bool a_mn_major,
                          cudaStream_t stream) {
    // query side: K = d_h is short (2 blocks), so a 2-stage ring and 4 CTAs
    // per SM.  (32 query rows per CTA on the output side, to fill more SMs
    // at a 64-row batch, measured slower: the extra L2 reads of the weights
    // cost more than the added CTAs gain.)
    return a_mn_major ? launch_one<true, 64>(tm_a, tm_b, a, stream) : launch_one<false, 64>(tm_a, tm_b, a, stream);
}

}  // namespace mla
