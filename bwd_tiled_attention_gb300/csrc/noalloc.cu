// noalloc.cu -- a backward entry point that needs no memory from the caller
// beyond its inputs and outputs.
//
// Some callers cannot allocate device memory at the point where they run the
// backward pass: for example an inference/training engine plugin whose
// execute step is not allowed to allocate, or a process that reserved all of
// its device memory up front and has no spare workspace to lend.  For them
// fa_bwd_noalloc runs the same preprocess and backward kernels as
// fa_bwd_preprocess + fa_bwd, but keeps D and the backward workspace (dQ
// accumulator, semaphores, schedule, GQA partials) in a fixed-size array that
// the library itself owns.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds kNoAllocScratchBytes for it until the process exits.
// Host code cannot use the array's name as a device address, so the first call
// on each device looks the address up with cudaGetSymbolAddress (with that
// device current) and caches it.  cudaDeviceReset destroys the context that
// address belongs to; the cache is not told, so no call may follow a reset.
//
// Layout of the array: the backward workspace first, so its header -- and the
// device error word at its offset 0 -- sits at the array's base on every
// call, then D.  fa_noalloc_check_device_status reads that word, which is how
// a caller of fa_bwd_noalloc learns of errors found inside the kernels (a
// bounded wait that gave up, a sequence longer than N).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"
#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_bwd_scratch on the current device (looked up once per device).
fa_status scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
            return FA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    fa_dtype o_dtype, const void* dout, const float* lse,
                                    void* dq, void* dk, void* dv, fa_dtype grad_dtype, int B,
                                    int Hq, int Hkv, int N, int total_tokens, int d, float scale,
                                    int causal, const int* cu_seqlens, int deterministic,
                                    fa_stream_t stream) {
    if (d != 64 && d != 96 && d != 128 && d != 192 && d != 256) return FA_ERR_UNSUPPORTED;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || total_tokens < 0) return FA_ERR_INVALID_ARG;
    const long long T = total_tokens > 0 ? (long long)total_tokens : (long long)B * N;
    if (T == 0 || B == 0) return FA_OK;
    const size_t ws_bytes = fa_bwd_workspace_size(B, Hq, Hkv, N, total_tokens, d);
    if (ws_bytes == 0) return FA_ERR_INVALID_ARG;
    const size_t d_bytes = fa::align_up((size_t)Hq * (size_t)T * sizeof(float), fa::kAlign);
    if (d_bytes + ws_bytes > kNoAllocScratchBytes) return FA_ERR_UNSUPPORTED;  // too large
    void* scratch = nullptr;
    fa_status st = scratch_on_current_device(&scratch);
    if (st != FA_OK) return st;
    void* ws = scratch;  // error word at the array's base
    float* D = reinterpret_cast<float*>(static_cast<char*>(scratch) + ws_bytes);
    // fa_bwd_preprocess clears everything in the workspace that must start at
    // zero (dQ accumulator, semaphores, work counter, error word).
    st = fa_bwd_preprocess(o, o_dtype, dout, D, ws, ws_bytes, B, Hq, Hkv, N, total_tokens, d,
                           causal, cu_seqlens, deterministic, stream);
    if (st != FA_OK) return st;
    return fa_bwd(q, k, v, dout, lse, D, dq, dk, dv, grad_dtype, ws, ws_bytes, B, Hq, Hkv, N,
                  total_tokens, d, scale, causal, cu_seqlens, deterministic, stream);
}

extern "C" fa_status fa_noalloc_check_device_status(fa_stream_t stream) {
    void* scratch = nullptr;
    const fa_status st = scratch_on_current_device(&scratch);
    if (st != FA_OK) return st;
    return fa_check_device_status(scratch, stream);
}
