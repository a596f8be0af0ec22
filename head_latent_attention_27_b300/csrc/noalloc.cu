// Decode entry point that allocates nothing, not even a caller workspace.
//
// Some callers cannot hand the library any device scratch: a plugin that
// receives only its input and output pointers from a host framework whose
// allocator it cannot reach, or a serving loop that forbids device
// allocation after start-up (cudaMalloc can synchronise the device and
// fragment a fixed memory budget).  For them, mla_decode_noalloc runs the
// same decode as mla_decode (balanced plan, attention kernel, log-sum-exp
// merge) with its scratch in a fixed array of MLA_NOALLOC_SCRATCH_BYTES that
// lives in this library's device image.  Every GPU that loads the library
// keeps that array until the process exits.
//
// The array is shared by every call on a device and keeps the previous
// call's contents.  The planning kernel rewrites everything a decode reads
// (its status word starts each call at zero, plan arrays and partial rows
// are written before they are read), so no clearing is needed between calls;
// calls that overlap on the GPU (different streams, or another thread) race
// on the array and must be serialised by the caller.
//
// Host code cannot pass the array's name to a kernel: in host code it is only
// a stand-in for the symbol.  The device address is looked up once per device
// with cudaGetSymbolAddress, with that device current, on the first call made
// on it; make that first call before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "mla.h"

namespace mla {
mla_status_t decode_into_workspace(const mla_cache_t* c, const int32_t* seq_lens, int32_t B, const void* q_nope,
                                   const void* q_rope, int32_t Q, int32_t H, float scale, void* out, float* lse,
                                   void* ws, size_t ws_bytes, cudaStream_t stream);
}

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[MLA_NOALLOC_SCRATCH_BYTES];

std::once_flag g_setup_once[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_setup_err[kMaxDevices];

// Device address of this device's copy of the scratch array (set-up on the
// first call per device).
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(g_setup_once[dev], [dev]() {
        void* p = nullptr;
        g_setup_err[dev] = cudaGetSymbolAddress(&p, g_decode_scratch);
        g_scratch_ptr[dev] = (g_setup_err[dev] == cudaSuccess) ? p : nullptr;
    });
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" MLA_API mla_status_t mla_decode_noalloc(const mla_cache_t* cache, const int32_t* seq_lens, int32_t B,
                                                   const void* q_nope, const void* q_rope, int32_t Q, int32_t H,
                                                   float softmax_scale, void* out, float* lse, void* stream) {
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return MLA_ERR_CUDA;
    return mla::decode_into_workspace(cache, seq_lens, B, q_nope, q_rope, Q, H, softmax_scale, out, lse, scratch,
                                      (size_t)MLA_NOALLOC_SCRATCH_BYTES, static_cast<cudaStream_t>(stream));
}
