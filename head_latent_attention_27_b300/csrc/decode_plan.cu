// Device-side planning of a decode: counts every unit's key tiles from
// seq_lens and cuts the tile sequence into pieces for the workers.
//
// Balanced mode (n_split = 0): all units' tiles (plus a fixed per-piece
// overhead) are laid end to end and cut into `num_workers` equal cost
// ranges, so every SM gets the same amount of cache to stream whatever the
// length mix (flash-decoding with a balanced split).
// Uniform mode (n_split >= 1): each unit's tiles are cut into n_split equal
// chunks of whole tiles; chunks are then dealt to workers in order by cost.
#include "decode_plan.cuh"

namespace mla {
namespace {

constexpr int kPlanThreads = 1024;
// The per-unit tile counts and costs and the piece -> worker map are only
// read inside the plan; when they are small enough they stay in shared
// memory (the passes read them back there instead of from global memory,
// and the last pass's binary searches run over shared memory).
constexpr int kSmemUnits = 2048;
constexpr int kSmemPieces = 4096;

// Exclusive scan over the block; returns the exclusive prefix of `v` and
// writes the block total to *total.  All threads must call it.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* total) {
    __shared__ int64_t warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int64_t s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += y;
        }
        if (lane < nw) warp_sums[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const int64_t before = warp > 0 ? warp_sums[warp - 1] : 0;
    *total = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before + x - v;
}

__device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ seq_lens, int32_t B,
                                                           int32_t Q, int32_t H, int32_t n_split,
                                                           int32_t P, int32_t max_tokens, void* ws,
                                                           WsLayout L) {
    WsView v = ws_view(ws, L);
    const int32_t RB = units_per_seq(Q, H);
    const int32_t U = B * RB;
    __shared__ int32_t s_tiles[kSmemUnits], s_cost[kSmemUnits], s_pw[kSmemPieces], s_pb[kSmemUnits + 1];
    // unit_piece_begin is written to the workspace for the other kernels and,
    // when it fits, mirrored here for pass 3 (no global round trip)
    int32_t* unit_tiles = U <= kSmemUnits ? s_tiles : v.unit_tiles;
    int32_t* unit_cost = U <= kSmemUnits ? s_cost : v.unit_cost;
    const int32_t QH = Q * H;
    const int tid = threadIdx.x;
    const bool pb_smem = U <= kSmemUnits;
    if (tid == 0) {
        v.hdr->status = 0;
        v.hdr->num_units = U;
        v.hdr->num_workers = P;
        v.hdr->n_split = n_split;
    }
    __syncthreads();

    // Pass 1: tiles and cost per unit, cost offsets; uniform mode also piece counts.
    int64_t carry_cost = 0, carry_np = 0;
    for (int32_t base = 0; base < U; base += kPlanThreads) {
        const int32_t u = base + tid;
        int64_t tiles = 0, cost = 0, np = 0;
        if (u < U) {
            const int32_t b = u / RB, rb = u % RB;
            const int32_t len = checked_len(seq_lens, b, max_tokens, &v.hdr->status);
            const int32_t last_row = min(QH, (rb + 1) * kRowsPerUnit) - 1;
            const int32_t vis = visible_len(len, Q, H, last_row);
            tiles = ceil_div64(vis, kTileTokens);
            if (n_split > 0) {
                if (tiles > 0) {
                    const int64_t chunk = ceil_div64(tiles, n_split);
                    np = ceil_div64(tiles, chunk);
                }
                cost = tiles + np * kPieceOverheadTiles;
            } else {
                cost = tiles > 0 ? tiles + kPieceOverheadTiles : 0;
            }
        }
        int64_t tot_cost, tot_np;
        const int64_t ex_cost = block_exclusive_scan(cost, &tot_cost);
        const int64_t ex_np = block_exclusive_scan(np, &tot_np);
        if (u < U) {
            unit_tiles[u] = (int32_t)tiles;
            unit_cost[u] = (int32_t)(carry_cost + ex_cost);
            if (n_split > 0) {
                v.unit_piece_begin[u] = (int32_t)(carry_np + ex_np);
                if (pb_smem) s_pb[u] = (int32_t)(carry_np + ex_np);
            }
        }
        carry_cost += tot_cost;
        carry_np += tot_np;
    }
    const int64_t C = carry_cost;
    const int64_t T = C > 0 ? ceil_div64(C, P) : 1;  // cost per worker

    // Pass 2 (balanced): pieces per unit = workers its tiles touch.
    if (n_split == 0) {
        __syncthreads();
        carry_np = 0;
        for (int32_t base = 0; base < U; base += kPlanThreads) {
            const int32_t u = base + tid;
            int64_t np = 0;
            if (u < U) {
                const int64_t tiles = unit_tiles[u];
                if (tiles > 0) {
                    const int64_t a = (int64_t)unit_cost[u] + kPieceOverheadTiles;
                    np = (a + tiles - 1) / T - a / T + 1;
                }
            }
            int64_t tot;
            const int64_t ex = block_exclusive_scan(np, &tot);
            if (u < U) {
                v.unit_piece_begin[u] = (int32_t)(carry_np + ex);
                if (pb_smem) s_pb[u] = (int32_t)(carry_np + ex);
            }
            carry_np += tot;
        }
    }
    const int64_t NP = carry_np;
    int32_t* piece_worker = NP <= kSmemPieces ? s_pw : v.piece_worker;
    if (tid == 0) {
        v.unit_piece_begin[U] = (int32_t)NP;
        if (pb_smem) s_pb[U] = (int32_t)NP;
        v.hdr->num_pieces = (int32_t)NP;
    }
    __syncthreads();

    // Pass 3: write the pieces (one thread per unit).
    for (int32_t u = tid; u < U; u += kPlanThreads) {
        const int32_t tiles = unit_tiles[u];
        if (tiles == 0) continue;
        const int32_t p0 = pb_smem ? s_pb[u] : v.unit_piece_begin[u];
        const int32_t np = (pb_smem ? s_pb[u + 1] : v.unit_piece_begin[u + 1]) - p0;
        const int64_t a = unit_cost[u];
        if (n_split > 0) {
            const int32_t chunk = (int32_t)ceil_div64(tiles, n_split);
            for (int32_t k = 0; k < np; ++k) {
                Piece pc;
                pc.unit = u;
                pc.t_begin = k * chunk;
                pc.t_end = min(tiles, (k + 1) * chunk);
                pc.slot = np > 1 ? p0 + k : -1;
                v.pieces[p0 + k] = pc;
                const int64_t start = a + (int64_t)k * (chunk + kPieceOverheadTiles);
                piece_worker[p0 + k] = (int32_t)(start / T < (int64_t)(P - 1) ? start / T : (int64_t)(P - 1));
            }
        } else {
            const int64_t a0 = a + kPieceOverheadTiles;
            const int64_t c0 = a0 / T;
            for (int32_t k = 0; k < np; ++k) {
                const int64_t c = c0 + k;
                Piece pc;
                pc.unit = u;
                pc.t_begin = (int32_t)(c * T - a0 > 0 ? c * T - a0 : 0);
                pc.t_end = (int32_t)((c + 1) * T - a0 < (int64_t)tiles ? (c + 1) * T - a0 : (int64_t)tiles);
                pc.slot = np > 1 ? p0 + k : -1;
                v.pieces[p0 + k] = pc;
                piece_worker[p0 + k] = (int32_t)c;
            }
        }
    }
    __syncthreads();

    // Pass 4: first piece of every worker (piece_worker is non-decreasing).
    for (int32_t c = tid; c <= P; c += kPlanThreads) {
        int64_t lo = 0, hi = NP;
        while (lo < hi) {
            const int64_t mid = (lo + hi) >> 1;
            if (piece_worker[mid] < c) lo = mid + 1; else hi = mid;
        }
        v.worker_begin[c] = (int32_t)lo;
    }
}

}  // namespace

cudaError_t launch_plan(const int32_t* seq_lens, int32_t B, int32_t Q, int32_t H, int32_t n_split,
                        int32_t num_workers, int32_t max_tokens, void* ws, const WsLayout& L,
                        cudaStream_t stream) {
    plan_kernel<<<1, kPlanThreads, 0, stream>>>(seq_lens, B, Q, H, n_split, num_workers, max_tokens, ws, L);
    return cudaGetLastError();
}

}  // namespace mla
