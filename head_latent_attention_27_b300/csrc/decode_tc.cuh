#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "decode_plan.cuh"

namespace mla {

struct TcArgs {
    const int32_t* page_table;
    const int32_t* seq_lens;
    const void* q_nope;  // bf16 [B*Q*H][512]
    const void* cache;   // bf16 [pages][64][576] (L2 prefetch addresses)
    void* out;          // bf16 [B*Q*H][512]
    float* lse;         // [B*Q*H] or null
    int32_t num_pages;
    int32_t max_pages_per_seq;
    int32_t Q;
    int32_t H;
    float scale_log2;   // softmax_scale * log2(e)
    int32_t evict_first;  // stream the cache with an evict-first L2 policy
    int32_t prefetch_tiles;  // L2 prefetch distance of the cache stream, in tiles
    int64_t total_rows;   // B*Q*H
};

struct TcMaps {
    CUtensorMap kv_nope;   // bf16 cache [pages*64][576], box 64 x 64, 128-byte swizzle;
                           // low-precision cache: the rows as bytes [pages*64][656], box 128 x 64
    CUtensorMap kv_rope;   // bf16 RoPE keys, box 32 x 64, 64-byte swizzle (bf16 view of either row format)
    CUtensorMap q_rope;    // [B*Q*H][64], box 32 x 128, 64-byte swizzle
    CUtensorMap kv_scale;  // low-precision cache only: fp32 view [pages*64][164], box 4 x 64 (group scales)
};

// Dynamic shared memory of the kernel (bytes) and its cluster size.
size_t decode_tc_smem_bytes();
constexpr int kTcClusterSize = 2;
// L2 prefetch distance of the cache stream (tiles ahead of the TMA loads of
// a CTA; 0 = off).  Measured on the full-width workload it slowed the kernel
// (the ring is not latency-starved), so it is off by default, and with 0 its
// code is compiled out of the producer loop (a smaller loop measured faster).
#ifndef MLA_TC_PREFETCH_TILES
#define MLA_TC_PREFETCH_TILES 0
#endif
constexpr int kTcPrefetchTiles = MLA_TC_PREFETCH_TILES;

// Maximum number of co-resident 2-CTA clusters on the current device.
cudaError_t decode_tc_max_clusters(int32_t* clusters);

// lowp: the cache holds low-precision rows (E4M3 latent + fp32 group scales +
// bf16 RoPE key, 656 bytes); otherwise bf16 rows.
cudaError_t launch_decode_tc(const TcMaps& maps, const TcArgs& a, int32_t num_clusters, void* ws,
                             const WsLayout& L, cudaStream_t stream, bool lowp);

}  // namespace mla
