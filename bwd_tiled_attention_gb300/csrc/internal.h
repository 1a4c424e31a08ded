// internal.h -- host-side interfaces between the C ABI layer and the kernel
// launchers (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>

namespace fa {

// Forward kernel arguments (device pointers, tensor maps built on the host).
struct FwdParams {
    CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps over [T, H, d], box {64, 1, 128}
    void* o;
    float* lse;
    const int* cu_seqlens;         // query sequences; null for dense
    void* workspace;               // header + unit list
    size_t units_off;
    int B, Hq, Hkv, N, T, d;       // N, T: query length bound and tokens
    float scale_log2;              // scale * log2(e)
    int causal;
    int o_fp32;
    const int* cu_seqlens_k;       // key/value sequences; null for dense
    int Nk, Tk;                    // key/value length bound and tokens
    int kv;                        // key boundaries differ from the query ones
};

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    CUtensorMap tm_dq_acc;         // fp32 map over the dQ accumulator, box {32, 1, 128}
    const float* lse;
    const float* D;
    void* dk;                      // final dK (MHA) -- bf16 or fp32
    void* dv;
    const int* cu_seqlens;         // query sequences; null for dense
    void* workspace;
    size_t units_off, tile_off_off, sems_off, dq_acc_off, dk_acc_off, dv_acc_off;
    int B, Hq, Hkv, N, T, d;       // N, T: query length bound and tokens
    float scale;                   // softmax scale (dK and dQ factor)
    float scale_log2;              // scale * log2(e)
    int causal;
    int deterministic;
    int grad_fp32;
    int hchunk;                    // query heads one unit walks (bwd_head_run)
    int nchunks;                   // runs of heads per key/value head: (Hq / Hkv) / hchunk
    const int* cu_seqlens_k;       // key/value sequences; null for dense
    int Nk, Tk;                    // key/value length bound and tokens
    int kv;                        // key boundaries differ from the query ones
};

// Writes the unit list over the tiles of `cu_seqlens` / N (T tokens) and,
// when want_tile_off, the per-sequence offsets of the query tiles that
// cu_tiles_seqlens / N_tiles (T_tiles tokens) define (the backward's units
// are key/value tiles, its semaphores query tiles).  Every length is checked
// against its bound and both boundary arrays against their token counts; on a
// mismatch no unit is written and the error word is set.
cudaError_t launch_sched(const int* cu_seqlens, int B, int N, int T, int H, int rows, int order,
                         long long max_units, void* workspace, size_t units_off,
                         size_t tile_off_off, bool want_tile_off, const int* cu_tiles_seqlens,
                         int N_tiles, int T_tiles, cudaStream_t stream);

// Dynamic shared memory the scheduler needs for a packed batch of B sequences
// whose longest spans at most maxnt_bound tiles (one CTA ranks them all).
size_t sched_smem_bytes(int B, int maxnt_bound);

cudaError_t launch_fwd(const FwdParams& p, int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const void* o, int o_fp32, const void* dout, float* D,
                                  float* dq_acc, int* sems, long long n_sems, int T, int Hq,
                                  int d, int num_sms, cudaStream_t stream);

cudaError_t launch_bwd(const BwdParams& p, int num_sms, cudaStream_t stream);

// dk_acc/dv_acc: fp32 partials [Tk, Hkv * nruns, d] to sum per key/value head,
// or null when each unit wrote final dK/dV.
cudaError_t launch_bwd_postprocess(const float* dq_acc, void* dq, const float* dk_acc,
                                   const float* dv_acc, void* dk, void* dv, int Tq, int Tk,
                                   int Hq, int Hkv, int nruns, int d, float scale, int grad_fp32,
                                   int num_sms, cudaStream_t stream);

}  // namespace fa
