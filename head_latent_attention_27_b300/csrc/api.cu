// C ABI of libmla.so (declared in include/mla.h): argument checks, the
// per-device kernel configuration, TMA descriptor encoding and launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "absorb.cuh"
#include "append.cuh"
#include "decode_f32.cuh"
#include "decode_plan.cuh"
#include "decode_sh.cuh"
#include "decode_tc.cuh"
#include "prefill.cuh"
#include "mla.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int32_t sms = 0;
    int32_t tc_clusters = 0;  // co-resident 2-CTA clusters of the tensor-core kernel
    cudaError_t err = cudaSuccess;
};

std::once_flag g_once[kMaxDevices];
DeviceInfo g_info[kMaxDevices];

const DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(g_once[dev], [dev]() {
        DeviceInfo& d = g_info[dev];
        int sms = 0;
        d.err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.err != cudaSuccess) return;
        d.sms = sms;
        int32_t cl = 0;
        d.err = decode_tc_max_clusters(&cl);
        if (d.err != cudaSuccess) return;
        d.tc_clusters = cl < sms / 2 ? cl : sms / 2;
    });
    return &g_info[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 tensor map: rows x cols (row stride `stride_elems`), box
// box_cols x box_rows.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t stride_elems,
               uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {stride_elems * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D tensor map of any element type: rows x cols elements, row stride in
// bytes, box box_cols x box_rows.
bool encode_2d_any(CUtensorMap* m, CUtensorMapDataType t, const void* base, uint64_t rows, uint64_t cols,
                   uint64_t stride_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, t, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor map over a row-major [d2][d1][d0] array, box
// box0 x box1 x box2 (elements along d0 innermost).
bool encode_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1,
               uint32_t box2, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The two absorption GEMMs share one kernel; `query_side` selects
// q_nope = W^UK_h^T q^C_h (reduction over d_h) or o = W^UV_h u_h (over d_c).
mla_status_t run_absorb(const void* w, const void* x, void* y, int32_t n_rows, int32_t H, int32_t d_h, int32_t d_c,
                        int32_t* status, void* stream, bool query_side) {
    if (n_rows < 0 || H < 1 || d_h < 1 || d_c < 1) return MLA_ERR_INVALID_ARG;
    if (d_h % kAbsorbBM != 0 || d_c % kAbsorbBM != 0 || H > 65535) return MLA_ERR_UNSUPPORTED;
    const int32_t rows_per_cta = absorb_rows_per_cta(query_side);
    if (n_rows > 65535 * rows_per_cta || (int64_t)n_rows * H * (d_c > d_h ? d_c : d_h) > ((int64_t)1 << 40))
        return MLA_ERR_UNSUPPORTED;
    if (n_rows == 0) return MLA_OK;
    if (!w || !x || !y) return MLA_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(x) || (reinterpret_cast<uintptr_t>(y) & 1u) != 0) return MLA_ERR_INVALID_ARG;
    const int32_t k_total = query_side ? d_h : d_c;
    const int32_t m_total = query_side ? d_c : d_h;
    CUtensorMap tm_a, tm_b;
    // weights: [H * d_h][d_c] row-major; the query side reads 64 (m) x 64 (k)
    // boxes (A contiguous along m), the output side 64 (k) x 128 (m) boxes
    const bool ok_a = query_side ? encode_2d(&tm_a, w, (uint64_t)H * d_h, d_c, d_c, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)
                                 : encode_2d(&tm_a, w, (uint64_t)H * d_h, d_c, d_c, 64, 128,
                                             CU_TENSOR_MAP_SWIZZLE_128B);
    // activations: [n_rows][H][k_total], 64 rows of one head per box
    const bool ok_b = encode_3d(&tm_b, x, k_total, H, n_rows, 64, 1, rows_per_cta, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok_a || !ok_b) return MLA_ERR_CUDA;
    AbsorbArgs a;
    a.out = y;
    a.n_rows = n_rows;
    a.H = H;
    a.m_total = m_total;
    a.k_total = k_total;
    a.status = status;
    return launch_absorb(tm_a, tm_b, a, query_side, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MLA_OK
                                                                                                      : MLA_ERR_CUDA;
}

mla_status_t check_cache(const mla_cache_t* c) {
    if (!c || !c->data || !c->page_table) return MLA_ERR_INVALID_ARG;
    if (c->dtype != MLA_BF16 && c->dtype != MLA_FP32 && c->dtype != MLA_FP8) return MLA_ERR_INVALID_ARG;
    if (c->num_seqs < 1 || c->num_pages < 1 || c->max_pages_per_seq < 1) return MLA_ERR_INVALID_ARG;
    if (c->num_pages > (1 << 24) || (int64_t)c->max_pages_per_seq * kTileTokens > (1 << 30))
        return MLA_ERR_INVALID_ARG;
    if (c->page_size != kTileTokens) return MLA_ERR_UNSUPPORTED;
    if (c->d_c < 1 || c->d_r < 0 || (c->d_r & 1)) return MLA_ERR_INVALID_ARG;
    if (c->dtype == MLA_BF16 || c->dtype == MLA_FP8) {
        if (c->d_c != 512 || c->d_r != 64) return MLA_ERR_UNSUPPORTED;
        if (!aligned16(c->data)) return MLA_ERR_INVALID_ARG;
    } else {
        if (c->d_c > 512 || (c->d_c & 3) || c->d_r > 64) return MLA_ERR_UNSUPPORTED;
        if ((reinterpret_cast<uintptr_t>(c->data) & 3u) != 0) return MLA_ERR_INVALID_ARG;
    }
    return MLA_OK;
}

struct DecodeShape {
    int32_t B, Q, H, n_split;
};

// bf16 units of at most 16 query rows go to the single-SM kernel
// (decode_sh.cu); larger units to the two-SM tensor-memory kernel.
bool small_rows(const mla_cache_t* c, DecodeShape s) {
    return c->dtype == MLA_BF16 && (int64_t)s.Q * s.H <= kShMaxRows;
}

// Workers of the plan: one CTA per SM on the fp32 and small-unit paths, one
// 2-CTA cluster on the tensor-memory path.
int32_t num_workers(const DeviceInfo* d, const mla_cache_t* c, DecodeShape s) {
    return (c->dtype == MLA_FP32 || small_rows(c, s)) ? d->sms : d->tc_clusters;
}

mla_status_t check_decode(const mla_cache_t* c, const int32_t* seq_lens, DecodeShape s, const void* q_nope,
                          const void* q_rope, const void* out) {
    mla_status_t st = check_cache(c);
    if (st != MLA_OK) return st;
    if (s.B < 0 || s.B > c->num_seqs || s.Q < 1 || s.H < 1) return MLA_ERR_INVALID_ARG;
    if ((int64_t)s.Q * s.H > 4096) return MLA_ERR_UNSUPPORTED;
    if (s.n_split < 0 || s.n_split > kMaxSplit) return MLA_ERR_INVALID_ARG;
    if (s.B > 0 && (!seq_lens || !q_nope || !out || (c->d_r > 0 && !q_rope))) return MLA_ERR_INVALID_ARG;
    if ((int64_t)s.B * s.Q * s.H > (int64_t)1 << 30) return MLA_ERR_UNSUPPORTED;
    if (c->dtype != MLA_FP32 && s.B > 0 && (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(out)))
        return MLA_ERR_INVALID_ARG;
    return MLA_OK;
}

// The softmax scale must be a positive finite number (the kernels take the
// running maximum on unscaled scores).
bool check_scale(float scale) { return scale > 0.f && isfinite(scale); }

mla_status_t check_workspace(void* ws, size_t bytes, const WsLayout& L) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MLA_ERR_WORKSPACE;
    if (bytes < L.total) return MLA_ERR_WORKSPACE;
    return MLA_OK;
}

mla_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

mla_status_t do_plan(const mla_cache_t* c, const int32_t* seq_lens, DecodeShape s, void* ws, size_t ws_bytes,
                     cudaStream_t stream) {
    const DeviceInfo* d = device_info();
    if (!d || d->err != cudaSuccess || d->sms <= 0) return MLA_ERR_CUDA;
    const int32_t P = num_workers(d, c, s);
    if (P <= 0) return MLA_ERR_CUDA;
    const WsLayout L = ws_layout(s.B, s.Q, s.H, c->d_c, s.n_split, P);
    mla_status_t st = check_workspace(ws, ws_bytes, L);
    if (st != MLA_OK) return st;
    return cuda_status(launch_plan(seq_lens, s.B, s.Q, s.H, s.n_split, P, c->max_pages_per_seq * kTileTokens, ws,
                                   L, stream));
}

mla_status_t do_attend(const mla_cache_t* c, const int32_t* seq_lens, DecodeShape s, const void* q_nope,
                       const void* q_rope, float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
    const DeviceInfo* d = device_info();
    if (!d || d->err != cudaSuccess || d->sms <= 0) return MLA_ERR_CUDA;
    const int32_t P = num_workers(d, c, s);
    const WsLayout L = ws_layout(s.B, s.Q, s.H, c->d_c, s.n_split, P);
    mla_status_t st = check_workspace(ws, ws_bytes, L);
    if (st != MLA_OK) return st;
    if (s.B == 0) return MLA_OK;
    if (c->dtype == MLA_FP32) {
        F32Args a;
        a.cache = static_cast<const float*>(c->data);
        a.page_table = c->page_table;
        a.seq_lens = seq_lens;
        a.q_nope = static_cast<const float*>(q_nope);
        a.q_rope = static_cast<const float*>(q_rope);
        a.out = static_cast<float*>(out);
        a.lse = lse;
        a.num_pages = c->num_pages;
        a.max_pages_per_seq = c->max_pages_per_seq;
        a.d_c = c->d_c;
        a.d_r = c->d_r;
        a.Q = s.Q;
        a.H = s.H;
        a.scale = scale;
        return cuda_status(launch_decode_f32(a, P, ws, L, stream));
    }
    const uint64_t cache_rows = (uint64_t)c->num_pages * kTileTokens;
    if (small_rows(c, s)) {
        CUtensorMap kv;
        if (!encode_2d(&kv, c->data, cache_rows, 576, 576, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B)) return MLA_ERR_CUDA;
        ShArgs a;
        a.page_table = c->page_table;
        a.seq_lens = seq_lens;
        a.q_nope = q_nope;
        a.q_rope = q_rope;
        a.out = out;
        a.lse = lse;
        a.num_pages = c->num_pages;
        a.max_pages_per_seq = c->max_pages_per_seq;
        a.Q = s.Q;
        a.H = s.H;
        a.scale_log2 = scale * 1.4426950408889634f;
        return cuda_status(launch_decode_sh(kv, a, P, ws, L, stream));
    }
    TcMaps maps;
    const uint64_t qrows = (uint64_t)s.B * s.Q * s.H;
    const bool lowp = c->dtype == MLA_FP8;
    if (lowp) {
        // 656-byte rows: 512 E4M3 codes | 4 fp32 group scales | 64 bf16 RoPE values
        constexpr uint64_t kRow = kFp8RowBytes;
        if (!encode_2d_any(&maps.kv_nope, CU_TENSOR_MAP_DATA_TYPE_UINT8, c->data, cache_rows, kRow, kRow, 128, 64,
                           CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_2d_any(&maps.kv_scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c->data, cache_rows, kRow / 4, kRow, 4,
                           64, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_2d_any(&maps.kv_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c->data, cache_rows, kRow / 2, kRow, 32,
                           64, CU_TENSOR_MAP_SWIZZLE_64B))
            return MLA_ERR_CUDA;
    } else {
        if (!encode_2d(&maps.kv_nope, c->data, cache_rows, 576, 576, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&maps.kv_rope, c->data, cache_rows, 576, 576, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B))
            return MLA_ERR_CUDA;
        maps.kv_scale = maps.kv_rope;   // unused by the bf16 kernel
    }
    if (!encode_2d(&maps.q_rope, q_rope, qrows, 64, 64, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B)) return MLA_ERR_CUDA;
    TcArgs a;
    a.page_table = c->page_table;
    a.seq_lens = seq_lens;
    a.out = out;
    a.lse = lse;
    a.num_pages = c->num_pages;
    a.max_pages_per_seq = c->max_pages_per_seq;
    a.Q = s.Q;
    a.H = s.H;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.evict_first = units_per_seq(s.Q, s.H) == 1 ? 1 : 0;
    a.q_nope = q_nope;
    a.cache = c->data;
    a.prefetch_tiles = kTcPrefetchTiles;
    a.total_rows = (int64_t)qrows;
    return cuda_status(launch_decode_tc(maps, a, P, ws, L, stream, lowp));
}

mla_status_t do_combine(const mla_cache_t* c, DecodeShape s, void* out, float* lse, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
    const DeviceInfo* d = device_info();
    if (!d || d->err != cudaSuccess || d->sms <= 0) return MLA_ERR_CUDA;
    const int32_t P = num_workers(d, c, s);
    const WsLayout L = ws_layout(s.B, s.Q, s.H, c->d_c, s.n_split, P);
    mla_status_t st = check_workspace(ws, ws_bytes, L);
    if (st != MLA_OK) return st;
    if (s.B == 0) return MLA_OK;
    // the low-precision cache decodes into bf16 output like the bf16 cache
    const int32_t out_dtype = c->dtype == MLA_FP32 ? MLA_FP32 : MLA_BF16;
    return cuda_status(
        launch_combine(s.B, s.Q, s.H, c->d_c, out_dtype, c->dtype != MLA_FP32, d->sms, out, lse, ws, L, stream));
}

mla_status_t run_decode(const mla_cache_t* c, const int32_t* seq_lens, DecodeShape s, const void* q_nope,
                        const void* q_rope, float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
    mla_status_t st = check_decode(c, seq_lens, s, q_nope, q_rope, out);
    if (st != MLA_OK) return st;
    if (!check_scale(scale)) return MLA_ERR_INVALID_ARG;
    if (s.B == 0) return MLA_OK;
    st = do_plan(c, seq_lens, s, ws, ws_bytes, stream);
    if (st != MLA_OK) return st;
    st = do_attend(c, seq_lens, s, q_nope, q_rope, scale, out, lse, ws, ws_bytes, stream);
    if (st != MLA_OK) return st;
    return do_combine(c, s, out, lse, ws, ws_bytes, stream);
}

// RoPE frequencies of the d_r/2 pairs in fp64 (plain RoPE, or YaRN's
// piecewise interpolation when yarn_factor > 1); false for invalid params.
bool rope_frequencies(const mla_rope_t& r, int32_t d_r, double theta[32]) {
    if (!(r.base > 0.f) || !(r.yarn_factor >= 1.f) || !(r.yarn_beta > r.yarn_alpha) || r.original_max_position < 1 ||
        d_r > 64)
        return false;
    const double kTwoPi = 6.283185307179586476925286766559;
    for (int32_t i = 0; i < 32; ++i) {
        if (i >= d_r / 2) {
            theta[i] = 0.0;
            continue;
        }
        const double t = pow((double)r.base, -2.0 * (double)i / (double)d_r);
        if (r.yarn_factor == 1.f) {
            theta[i] = t;
            continue;
        }
        const double turns = (double)r.original_max_position * t / kTwoPi;
        double g = (turns - (double)r.yarn_alpha) / ((double)r.yarn_beta - (double)r.yarn_alpha);
        g = g < 0.0 ? 0.0 : (g > 1.0 ? 1.0 : g);
        theta[i] = t * (g + (1.0 - g) / (double)r.yarn_factor);
    }
    return true;
}

// ------------------------------------------------- bounded-wait self-test --

__global__ void selftest_wait_kernel(int* status, uint32_t timeout_us) {
    __shared__ __align__(8) uint64_t mbar;
    const uint32_t bar = smem_addr(&mbar);
    if (threadIdx.x == 0) mbar_init(bar, 1);  // nothing ever arrives
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        bool done = false;
        while (!(done = mbar_try_wait(bar, 0))) {
            if (global_timer_ns() - t0 > (uint64_t)timeout_us * 1000ull) break;
        }
        if (!done) atomicExch(status, MLA_ERR_TIMEOUT);
    }
}

}  // namespace

// Decode (balanced plan) into a given workspace; used by the fixed-scratch
// entry point in noalloc.cu.  Same checks and launches as mla_decode.
mla_status_t decode_into_workspace(const mla_cache_t* c, const int32_t* seq_lens, int32_t B, const void* q_nope,
                                   const void* q_rope, int32_t Q, int32_t H, float scale, void* out, float* lse,
                                   void* ws, size_t ws_bytes, cudaStream_t stream) {
    return run_decode(c, seq_lens, DecodeShape{B, Q, H, 0}, q_nope, q_rope, scale, out, lse, ws, ws_bytes, stream);
}

}  // namespace mla

using namespace mla;

extern "C" {

mla_status_t mla_cache_append_rope(const mla_cache_t* cache, const void* ckv_raw, const void* kr_raw,
                                   int32_t in_dtype, const float* gamma, float eps, const mla_rope_t* rope,
                                   const int32_t* seq_ids, const int32_t* positions, int32_t T, uint32_t flags,
                                   void* stream) {
    mla_status_t st = check_cache(cache);
    if (st != MLA_OK) return st;
    if (T < 0 || (in_dtype != MLA_BF16 && in_dtype != MLA_FP32)) return MLA_ERR_INVALID_ARG;
    if (flags & ~(MLA_APPEND_RMSNORM | MLA_APPEND_ROPE)) return MLA_ERR_INVALID_ARG;
    if (T == 0) return MLA_OK;
    if (!ckv_raw || (cache->d_r > 0 && !kr_raw) || !seq_ids || !positions) return MLA_ERR_INVALID_ARG;
    if ((flags & MLA_APPEND_RMSNORM) && !(eps >= 0.f)) return MLA_ERR_INVALID_ARG;
    AppendArgs a;
    if (flags & MLA_APPEND_ROPE) {
        if (!rope || !rope_frequencies(*rope, cache->d_r, a.theta)) return MLA_ERR_INVALID_ARG;
    } else {
        for (int i = 0; i < 32; ++i) a.theta[i] = 0.0;
    }
    a.seq_ids = seq_ids;
    a.positions = positions;
    a.page_table = cache->page_table;
    a.gamma = gamma;
    a.T = T;
    a.num_seqs = cache->num_seqs;
    a.num_pages = cache->num_pages;
    a.page_size = cache->page_size;
    a.max_pages_per_seq = cache->max_pages_per_seq;
    a.d_c = cache->d_c;
    a.d_r = cache->d_r;
    a.flags = flags;
    a.eps = eps;
    return cuda_status(launch_append(a, ckv_raw, kr_raw, in_dtype, cache->dtype, cache->data,
                                     static_cast<cudaStream_t>(stream)));
}

mla_status_t mla_cache_append(const mla_cache_t* cache, const void* ckv_raw, const void* kr_raw, int32_t in_dtype,
                              const float* gamma, float eps, float rope_base, const int32_t* seq_ids,
                              const int32_t* positions, int32_t T, uint32_t flags, void* stream) {
    const mla_rope_t rope = {rope_base, 1.f, 1.f, 32.f, 4096};
    return mla_cache_append_rope(cache, ckv_raw, kr_raw, in_dtype, gamma, eps, &rope, seq_ids, positions, T, flags,
                                 stream);
}

float mla_yarn_softmax_scale(float softmax_scale, float yarn_factor, float coef) {
    if (!(yarn_factor > 1.f)) return softmax_scale;
    const double m = (double)coef * log((double)yarn_factor) + 1.0;
    return (float)((double)softmax_scale * m * m);
}

mla_status_t mla_decode(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B, const void* q_nope,
                        const void* q_rope, int32_t Q, int32_t H, float softmax_scale, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return run_decode(cache, seq_lens, DecodeShape{B, Q, H, 0}, q_nope, q_rope, softmax_scale, out, lse, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream));
}

mla_status_t mla_decode_split_combine(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B,
                                      const void* q_nope, const void* q_rope, int32_t Q, int32_t H,
                                      float softmax_scale, int32_t n_split, void* out, float* lse, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    if (n_split < 1 || n_split > kMaxSplit) return MLA_ERR_INVALID_ARG;
    return run_decode(cache, seq_lens, DecodeShape{B, Q, H, n_split}, q_nope, q_rope, softmax_scale, out, lse,
                      workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t mla_decode_workspace_size(int32_t B, int32_t Q, int32_t H, int32_t d_c, int32_t n_split, int32_t num_sms) {
    if (B < 0 || Q < 1 || H < 1 || d_c < 1 || d_c > 512 || n_split < 0 || n_split > kMaxSplit || num_sms < 0)
        return 0;
    if (num_sms == 0) {
        const DeviceInfo* d = device_info();
        if (!d || d->err != cudaSuccess) return 0;
        num_sms = d->sms;
    }
    // fp32 path uses one worker per SM, the tensor path fewer: size for the larger
    return ws_layout(B, Q, H, d_c, n_split, num_sms).total;
}

mla_status_t mla_decode_plan(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B, int32_t Q, int32_t H,
                             int32_t n_split, void* workspace, size_t workspace_bytes, void* stream) {
    mla_status_t st = check_cache(cache);
    if (st != MLA_OK) return st;
    if (B < 0 || B > cache->num_seqs || Q < 1 || H < 1 || n_split < 0 || n_split > kMaxSplit)
        return MLA_ERR_INVALID_ARG;
    if (B > 0 && !seq_lens) return MLA_ERR_INVALID_ARG;
    if (B == 0) return MLA_OK;
    return do_plan(cache, seq_lens, DecodeShape{B, Q, H, n_split}, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream));
}

mla_status_t mla_decode_attend(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B, const void* q_nope,
                               const void* q_rope, int32_t Q, int32_t H, float softmax_scale, int32_t n_split,
                               void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    const DecodeShape s{B, Q, H, n_split};
    mla_status_t st = check_decode(cache, seq_lens, s, q_nope, q_rope, out);
    if (st != MLA_OK) return st;
    if (!check_scale(softmax_scale)) return MLA_ERR_INVALID_ARG;
    return do_attend(cache, seq_lens, s, q_nope, q_rope, softmax_scale, out, lse, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream));
}

mla_status_t mla_decode_combine(const mla_cache_t* cache, int32_t B, int32_t Q, int32_t H, int32_t n_split, void* out,
                                float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    mla_status_t st = check_cache(cache);
    if (st != MLA_OK) return st;
    if (B < 0 || B > cache->num_seqs || Q < 1 || H < 1 || n_split < 0 || n_split > kMaxSplit)
        return MLA_ERR_INVALID_ARG;
    if (B > 0 && !out) return MLA_ERR_INVALID_ARG;
    return do_combine(cache, DecodeShape{B, Q, H, n_split}, out, lse, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream));
}

mla_status_t mla_decode_read_status(void* workspace, size_t workspace_bytes, void* stream, int32_t* status_out) {
    if (!workspace || workspace_bytes < sizeof(WsHeader)) return MLA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t code = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaMemcpy(&code, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
    const int32_t zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) return MLA_ERR_CUDA;
    if (status_out) *status_out = code;
    return static_cast<mla_status_t>(code);
}

mla_status_t mla_selftest_bounded_wait(void* workspace, size_t workspace_bytes, uint32_t timeout_us, void* stream) {
    if (!workspace || workspace_bytes < sizeof(WsHeader)) return MLA_ERR_WORKSPACE;
    if (timeout_us == 0 || timeout_us > 10000000u) return MLA_ERR_INVALID_ARG;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int*>(workspace), timeout_us);
    return cuda_status(cudaGetLastError());
}

mla_status_t mla_absorb_query(const void* w_uk, const void* q_c, void* q_nope, int32_t n_rows, int32_t H,
                              int32_t d_h, int32_t d_c, int32_t* status, void* stream) {
    return run_absorb(w_uk, q_c, q_nope, n_rows, H, d_h, d_c, status, stream, true);
}

mla_status_t mla_absorb_output(const void* w_uv, const void* u, void* o, int32_t n_rows, int32_t H, int32_t d_h,
                               int32_t d_c, int32_t* status, void* stream) {
    return run_absorb(w_uv, u, o, n_rows, H, d_h, d_c, status, stream, false);
}

size_t mla_prefill_workspace_size(int32_t T, int32_t H) {
    if (T < 0 || H < 1 || (int64_t)T * H > ((int64_t)1 << 31)) return 0;
    const size_t kv = ws_align((size_t)T * (size_t)H * kPrefillDh * 2);
    return 256 + 2 * kv;
}

}  // extern "C"

namespace mla {
namespace {

enum PrefillPhase { kPrefillProject = 1, kPrefillAttend = 2, kPrefillBoth = 3 };

mla_status_t run_prefill(const mla_cache_t* cache, int32_t seq, int32_t T, const void* w_uk, const void* w_uv,
                         const void* q_c, const void* q_r, int32_t H, float softmax_scale, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, cudaStream_t s, int phases) {
    mla_status_t st = check_cache(cache);
    if (st != MLA_OK) return st;
    if (cache->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
    if (seq < 0 || seq >= cache->num_seqs || T < 0 || H < 1) return MLA_ERR_INVALID_ARG;
    if (H % 2 != 0 || H > 4096) return MLA_ERR_UNSUPPORTED;
    if ((int64_t)T > (int64_t)cache->max_pages_per_seq * kTileTokens) return MLA_ERR_INVALID_ARG;
    if (!check_scale(softmax_scale)) return MLA_ERR_INVALID_ARG;
    const size_t need = mla_prefill_workspace_size(T, H);
    if (need == 0) return MLA_ERR_UNSUPPORTED;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
        return MLA_ERR_WORKSPACE;
    if (T == 0) return MLA_OK;
    if ((phases & kPrefillProject) && (!w_uk || !w_uv || !aligned16(w_uk) || !aligned16(w_uv)))
        return MLA_ERR_INVALID_ARG;
    if ((phases & kPrefillAttend) &&
        (!q_c || !q_r || !out || !aligned16(q_c) || !aligned16(q_r) || !aligned16(out)))
        return MLA_ERR_INVALID_ARG;
    const DeviceInfo* d = device_info();
    if (!d || d->err != cudaSuccess || d->sms <= 0) return MLA_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t kv = ws_align((size_t)T * (size_t)H * kPrefillDh * 2);
    void* k_c = ws + 256;
    void* v = ws + 256 + kv;
    int32_t* status = reinterpret_cast<int32_t*>(ws);
    const uint64_t pool_rows = (uint64_t)cache->num_pages * kTileTokens;
    const uint64_t n_per = (uint64_t)H * kPrefillDh;
    const int32_t* page_row = cache->page_table + (int64_t)seq * cache->max_pages_per_seq;
    const int32_t pages = (T + kTileTokens - 1) / kTileTokens;
    if (phases & kPrefillProject) {
        // the status word starts each prefill at zero (the projection runs first)
        if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return MLA_ERR_CUDA;
        UpprojMaps um;
        if (!encode_2d(&um.latent, cache->data, pool_rows, 576, 576, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&um.w_uk, w_uk, n_per, kPrefillDc, kPrefillDc, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&um.w_uv, w_uv, n_per, kPrefillDc, kPrefillDc, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B))
            return MLA_ERR_CUDA;
        UpprojArgs ua;
        ua.page_row = page_row;
        ua.pages = pages;
        ua.num_pages = cache->num_pages;
        ua.T = T;
        ua.n_per = (int32_t)n_per;
        ua.k_out = k_c;
        ua.v_out = v;
        ua.status = status;
        if (launch_upproj(um, ua, d->sms, s) != cudaSuccess) return MLA_ERR_CUDA;
    }
    if (phases & kPrefillAttend) {
        PrefillAttnMaps am;
        if (!encode_2d(&am.q_c, q_c, (uint64_t)T, n_per, n_per, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&am.q_r, q_r, (uint64_t)T, (uint64_t)H * kPrefillDr, (uint64_t)H * kPrefillDr, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&am.k_c, k_c, (uint64_t)T, n_per, n_per, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&am.v, v, (uint64_t)T, n_per, n_per, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&am.k_r, cache->data, pool_rows, 576, 576, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
            return MLA_ERR_CUDA;
        PrefillAttnArgs aa;
        aa.page_row = page_row;
        aa.pages = pages;
        aa.num_pages = cache->num_pages;
        aa.T = T;
        aa.H = H;
        aa.scale_log2 = softmax_scale * 1.4426950408889634f;
        aa.out = out;
        aa.lse = lse;
        aa.status = status;
        if (launch_prefill_attn(am, aa, d->sms, s) != cudaSuccess) return MLA_ERR_CUDA;
    }
    return MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" {

mla_status_t mla_prefill_expanded(const mla_cache_t* cache, int32_t seq, int32_t T, const void* w_uk,
                                  const void* w_uv, const void* q_c, const void* q_r, int32_t H, float softmax_scale,
                                  void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    return run_prefill(cache, seq, T, w_uk, w_uv, q_c, q_r, H, softmax_scale, out, lse, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream), kPrefillBoth);
}

mla_status_t mla_prefill_project(const mla_cache_t* cache, int32_t seq, int32_t T, const void* w_uk,
                                 const void* w_uv, int32_t H, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    return run_prefill(cache, seq, T, w_uk, w_uv, nullptr, nullptr, H, 1.f, nullptr, nullptr, workspace,
                       workspace_bytes, static_cast<cudaStream_t>(stream), kPrefillProject);
}

mla_status_t mla_prefill_attend(const mla_cache_t* cache, int32_t seq, int32_t T, const void* q_c, const void* q_r,
                                int32_t H, float softmax_scale, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
    return run_prefill(cache, seq, T, nullptr, nullptr, q_c, q_r, H, softmax_scale, out, lse, workspace,
                       workspace_bytes, static_cast<cudaStream_t>(stream), kPrefillAttend);
}

const char* mla_status_string(mla_status_t s) {
    switch (s) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: invalid argument";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: shape or dtype not supported";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call failed";
        case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded in-kernel wait ran out";
        case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing, misaligned or too small";
        default: return "MLA: unknown status";
    }
}

int32_t mla_version(void) { return 100; }

}  // extern "C"
