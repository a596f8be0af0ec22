// Work partition of a decode, kept in the caller's workspace.
//
// A "unit" is one sequence b and one block of up to 128 query rows
// (row = query token j * H + head h; rows of a sequence are contiguous).
// A unit's visible keys are cut into 64-token tiles (= cache pages); a
// "piece" is a contiguous tile range of one unit handled by one worker (a
// 2-CTA cluster on the tensor-core path, one CTA on the fp32 path).  A unit
// done by a single piece is written straight to out/lse; a unit split into
// several pieces writes softmax-normalised fp32 partial rows plus their
// log-sum-exp, merged afterwards (flash-decoding).
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace mla {

constexpr int kRowsPerUnit = 128;
constexpr int kTileTokens = 64;
// Fixed cost of a piece (loading queries, epilogue), in tile units, used
// when balancing work across workers.
constexpr int kPieceOverheadTiles = 2;
constexpr int kMaxSplit = 1024;

struct WsHeader {
    int32_t status;       // mla_status_t recorded by kernels (0 = ok)
    int32_t num_pieces;
    int32_t num_units;
    int32_t num_workers;
    int32_t n_split;      // 0 = balanced partition
    int32_t pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct Piece {
    int32_t unit;
    int32_t t_begin;      // first tile (64-token) of the unit's keys
    int32_t t_end;        // one past the last tile
    int32_t slot;         // partial slot, or -1 when the piece is the whole unit
};

struct WsLayout {
    size_t off_unit_tiles;
    size_t off_unit_cost;
    size_t off_unit_piece_begin;
    size_t off_pieces;
    size_t off_piece_worker;
    size_t off_worker_begin;
    size_t off_lse_part;
    size_t off_o_part;
    size_t total;
    int32_t max_units;
    int32_t max_pieces;
    int32_t max_workers;
    int32_t d_c;
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline int32_t units_per_seq(int32_t Q, int32_t H) {
    return (Q * H + kRowsPerUnit - 1) / kRowsPerUnit;
}

// Layout for a decode with at most `max_workers` workers.  Valid arguments
// are checked by the caller.
__host__ __device__ inline WsLayout ws_layout(int32_t B, int32_t Q, int32_t H, int32_t d_c,
                                              int32_t n_split, int32_t max_workers) {
    WsLayout L{};
    const int64_t U = (int64_t)B * units_per_seq(Q, H);
    const int64_t P = max_workers;
    const int64_t pieces = n_split > 0 ? U * n_split : U + P;
    L.max_units = (int32_t)U;
    L.max_pieces = (int32_t)pieces;
    L.max_workers = (int32_t)P;
    L.d_c = d_c;
    size_t o = ws_align(sizeof(WsHeader));
    L.off_unit_tiles = o;       o = ws_align(o + sizeof(int32_t) * (size_t)U);
    L.off_unit_cost = o;        o = ws_align(o + sizeof(int32_t) * (size_t)U);
    L.off_unit_piece_begin = o; o = ws_align(o + sizeof(int32_t) * (size_t)(U + 1));
    L.off_pieces = o;           o = ws_align(o + sizeof(Piece) * (size_t)pieces);
    L.off_piece_worker = o;     o = ws_align(o + sizeof(int32_t) * (size_t)pieces);
    L.off_worker_begin = o;     o = ws_align(o + sizeof(int32_t) * (size_t)(P + 1));
    L.off_lse_part = o;         o = ws_align(o + sizeof(float) * (size_t)pieces * kRowsPerUnit);
    L.off_o_part = o;           o = ws_align(o + sizeof(float) * (size_t)pieces * kRowsPerUnit * (size_t)d_c);
    L.total = o;
    return L;
}

// Views of the workspace arrays.
struct WsView {
    WsHeader* hdr;
    int32_t* unit_tiles;
    int32_t* unit_cost;
    int32_t* unit_piece_begin;
    Piece* pieces;
    int32_t* piece_worker;
    int32_t* worker_begin;
    float* lse_part;   // [max_pieces][128]
    float* o_part;     // [max_pieces][128][d_c] fp32 (fp32 path) or fp16 in the same space (tensor-core paths)
};

__host__ __device__ inline WsView ws_view(void* ws, const WsLayout& L) {
    uint8_t* p = static_cast<uint8_t*>(ws);
    WsView v;
    v.hdr = reinterpret_cast<WsHeader*>(p);
    v.unit_tiles = reinterpret_cast<int32_t*>(p + L.off_unit_tiles);
    v.unit_cost = reinterpret_cast<int32_t*>(p + L.off_unit_cost);
    v.unit_piece_begin = reinterpret_cast<int32_t*>(p + L.off_unit_piece_begin);
    v.pieces = reinterpret_cast<Piece*>(p + L.off_pieces);
    v.piece_worker = reinterpret_cast<int32_t*>(p + L.off_piece_worker);
    v.worker_begin = reinterpret_cast<int32_t*>(p + L.off_worker_begin);
    v.lse_part = reinterpret_cast<float*>(p + L.off_lse_part);
    v.o_part = reinterpret_cast<float*>(p + L.off_o_part);
    return v;
}

// Visible length of query row `row` (0-based within the sequence, row =
// j*H + h): query j of Q sees positions 0 .. len-Q+j.
__host__ __device__ inline int32_t visible_len(int32_t len, int32_t Q, int32_t H, int32_t row) {
    const int32_t j = row / H;
    const int32_t v = len - Q + 1 + j;
    return v > 0 ? v : 0;
}

// Clamp a device-supplied length to the cache capacity; flags a bad one.
__device__ inline int32_t checked_len(const int32_t* seq_lens, int32_t b, int32_t max_tokens, int32_t* status) {
    int32_t len = seq_lens[b];
    if (len < 0 || len > max_tokens) {
        atomicCAS(status, 0, 1 /* MLA_ERR_INVALID_ARG */);
        len = 0;
    }
    return len;
}

// Launchers (decode_plan.cu, decode_combine.cu).
cudaError_t launch_plan(const int32_t* seq_lens, int32_t B, int32_t Q, int32_t H, int32_t n_split,
                        int32_t num_workers, int32_t max_tokens, void* ws, const WsLayout& L,
                        cudaStream_t stream);
// f16_partials: the partial rows were written in fp16 (the tensor-core
// kernels) rather than fp32 (the fp32 path); num_sms: the device's SM count
// (sizes the per-lane register depth of the merge against the grid).
cudaError_t launch_combine(int32_t B, int32_t Q, int32_t H, int32_t d_c, int32_t out_dtype, bool f16_partials,
                           int32_t num_sms, void* out, float* lse, void* ws, const WsLayout& L,
                           cudaStream_t stream);

}  // namespace mla
