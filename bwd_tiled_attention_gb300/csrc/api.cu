// api.cu -- the C ABI declared in include/fa.h: argument validation, TMA
// tensor-map encoding, workspace layout, and the launch sequence of each call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "common.cuh"
#include "internal.h"

using namespace fa;

namespace {

constexpr int kMaxVarlenSeqs = 4096;   // scheduler ranks sequences in one CTA
constexpr int kMaxHeads = 65535;       // head index is packed in 16 bits
constexpr long long kMaxTiles = 65535; // tile index is packed in 16 bits

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Cached SM count per device.
int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n;
    }
    return cache[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// 3-D tensor map over a packed [T, H, d] bf16 array, box {64, 1, 128}, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, int T, int H, int d) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kTile};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D tensor map over the packed [T, H, d] fp32 dQ accumulator, box {32, 1, 128}
// (128-byte rows), 128B swizzle: the target of the backward's bulk reduce-add.
bool make_map_f32(CUtensorMap* m, const void* base, int T, int H, int d) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
    cuuint32_t box[3] = {32, 1, (cuuint32_t)kTile};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct Shape {
    int B, Hq, Hkv, Nq, Tq, Nk, Tk, d;
    bool varlen;
};

// Token count of one side: the dense batch's B * N, or the packed total.
fa_status side_tokens(int B, int N, int total_tokens, bool varlen, int& T) {
    if (N < 0 || total_tokens < 0) return FA_ERR_INVALID_ARG;
    if ((long long)cdiv(N, kTile) > kMaxTiles) return FA_ERR_UNSUPPORTED;
    if (!varlen) {
        const long long t = (long long)B * N;
        if (t > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
        if (total_tokens != 0 && total_tokens != t) return FA_ERR_INVALID_ARG;
        T = (int)t;
    } else {
        T = total_tokens;
    }
    return FA_OK;
}

// Validates the shape arguments shared by every call.  Queries and keys are
// either both dense or both packed.  On success fills `s`.
fa_status check_shape(int B, int Hq, int Hkv, int Nq, int total_q, int Nk, int total_k, int d,
                      const int* cu_q, const int* cu_k, Shape& s) {
    if (B < 0 || Hq <= 0 || Hkv <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (Hq > kMaxHeads) return FA_ERR_UNSUPPORTED;
    if (d != 64 && d != 96 && d != 128 && d != 192 && d != 256) return FA_ERR_UNSUPPORTED;
    if ((cu_q == nullptr) != (cu_k == nullptr)) return FA_ERR_INVALID_ARG;
    s.B = B; s.Hq = Hq; s.Hkv = Hkv; s.Nq = Nq; s.Nk = Nk; s.d = d;
    s.varlen = cu_q != nullptr;
    if (s.varlen) {
        if (B > kMaxVarlenSeqs) return FA_ERR_UNSUPPORTED;
        if (!aligned4(cu_q) || !aligned4(cu_k)) return FA_ERR_INVALID_ARG;
    }
    fa_status st = side_tokens(B, Nq, total_q, s.varlen, s.Tq);
    if (st != FA_OK) return st;
    st = side_tokens(B, Nk, total_k, s.varlen, s.Tk);
    if (st != FA_OK) return st;
    if ((long long)s.Tq * Hq * d > (1LL << 40) || (long long)s.Tk * Hq * d > (1LL << 40))
        return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// A packed batch is ranked by one scheduler CTA, with a prefix entry per tile
// level of the longest sequence: its bound N must fit one CTA's shared memory.
constexpr size_t kSchedSmemMax = 232448;  // 227 KB, the per-block maximum
bool sched_fits(const Shape& s, int N, int rows) {
    return !s.varlen || sched_smem_bytes(s.B, cdiv(N, rows)) <= kSchedSmemMax;
}

// Queries and keys provably have equal lengths (the same boundary array, or a
// dense batch with Nq = Nk): the kernels' square instantiation applies.
bool same_boundaries(const Shape& s, const int* cu_q, const int* cu_k) {
    return cu_q == cu_k && s.Nq == s.Nk && s.Tq == s.Tk;
}

size_t elem_bytes(fa_dtype t) { return t == FA_FP32 ? 4 : 2; }

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype,
                   float* lse, int B, int Hq, int Hkv, int Nq, int total_q, int Nk, int total_k,
                   int d, float scale, int causal, const int* cu_q, const int* cu_k,
                   void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    Shape s;
    fa_status st = check_shape(B, Hq, Hkv, Nq, total_q, Nk, total_k, d, cu_q, cu_k, s);
    if (st != FA_OK) return st;
    if (o_dtype != FA_BF16 && o_dtype != FA_FP32) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_UNSUPPORTED;
    if (s.Tq == 0 || B == 0) return FA_OK;  // nothing to compute
    if (!sched_fits(s, Nq, d > 128 ? kFwdBlockRowsWide : kFwdBlockRows)) return FA_ERR_UNSUPPORTED;
    if (!q || !o || !lse || !workspace || (s.Tk > 0 && (!k || !v))) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
        !aligned16(workspace))
        return FA_ERR_INVALID_ARG;
    const FwdWs lay = fwd_ws_layout(B, Hq, s.Tq);
    if (workspace_bytes < lay.bytes) return FA_ERR_INVALID_ARG;
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    // With no keys at all no unit loads K or V: the query map stands in for them.
    const bool no_keys = s.Tk == 0;
    if (!make_map(&p.tm_q, q, s.Tq, Hq, d) ||
        !make_map(&p.tm_k, no_keys ? q : k, no_keys ? s.Tq : s.Tk, Hkv, d) ||
        !make_map(&p.tm_v, no_keys ? q : v, no_keys ? s.Tq : s.Tk, Hkv, d))
        return FA_ERR_CUDA;
    p.o = o;
    p.lse = lse;
    p.cu_seqlens = cu_q;
    p.cu_seqlens_k = cu_k;
    p.workspace = workspace;
    p.units_off = lay.units;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = Nq; p.T = s.Tq; p.d = d;
    p.Nk = Nk; p.Tk = s.Tk;
    p.kv = same_boundaries(s, cu_q, cu_k) ? 0 : 1;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal ? 1 : 0;
    p.o_fp32 = o_dtype == FA_FP32;
    const int nsm = sm_count();
    if (nsm <= 0) return FA_ERR_CUDA;
    cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_sched(cu_q, B, Nq, s.Tq, Hq, d > 128 ? kFwdBlockRowsWide : kFwdBlockRows,
                                 causal ? kOrderLevelDesc : kOrderSeqDesc, lay.max_units,
                                 workspace, lay.units, 0, false, cu_k, Nk, s.Tk, strm);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    return cuda_status(launch_fwd(p, nsm, strm));
}

size_t bwd_ws_bytes(int B, int Hq, int Hkv, int Nq, int total_q, int Nk, int total_k, int d,
                    bool sems_offset) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || total_q < 0 || Nk < 0 || total_k < 0 ||
        (d != 64 && d != 96 && d != 128 && d != 192 && d != 256))
        return 0;
    const long long Tq = total_q > 0 ? total_q : (long long)B * Nq;
    const long long Tk = total_k > 0 ? total_k : (long long)B * Nk;
    if (Tq > 0x7FFFFFFFLL || Tk > 0x7FFFFFFFLL) return 0;
    const BwdWs lay = bwd_ws_layout(B, Hq, Hkv, (int)Tq, (int)Tk, d);
    return sems_offset ? lay.sems : lay.bytes;
}

fa_status bwd_preprocess_impl(const void* o, fa_dtype o_dtype, const void* dout, float* D,
                              void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                              int Nq, int total_q, int Nk, int total_k, int d, int causal,
                              const int* cu_q, const int* cu_k, int deterministic,
                              fa_stream_t stream) {
    Shape s;
    fa_status st = check_shape(B, Hq, Hkv, Nq, total_q, Nk, total_k, d, cu_q, cu_k, s);
    if (st != FA_OK) return st;
    if (o_dtype != FA_BF16 && o_dtype != FA_FP32) return FA_ERR_INVALID_ARG;
    if (s.Tq == 0 || s.Tk == 0 || B == 0) return FA_OK;  // fa_bwd needs no workspace then
    if (!sched_fits(s, Nk, kTile)) return FA_ERR_UNSUPPORTED;  // units are key/value tiles
    if (!o || !dout || !D || !workspace) return FA_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(dout) || !aligned4(D) || !aligned16(workspace))
        return FA_ERR_INVALID_ARG;
    const BwdWs lay = bwd_ws_layout(B, Hq, Hkv, s.Tq, s.Tk, d);
    if (workspace_bytes < lay.bytes) return FA_ERR_INVALID_ARG;
    const int nsm = sm_count();
    if (nsm <= 0) return FA_ERR_CUDA;
    cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    // deterministic: descending key/value tile, the order of every dQ tile's
    // contributions; atomic: heaviest first
    const int order = deterministic ? kOrderLevelDesc : (causal ? kOrderWorkDesc : kOrderSeqDesc);
    char* ws = static_cast<char*>(workspace);
    // units are key/value tiles; dQ semaphores are numbered by query tile
    // units: (key/value tile, run of query heads), runs innermost
    cudaError_t e = launch_sched(cu_k, B, Nk, s.Tk, Hkv * lay.nruns, kTile, order, lay.max_units,
                                 workspace, lay.units, lay.tile_off, true, cu_q, Nq, s.Tq, strm);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    e = launch_bwd_preprocess(o, o_dtype == FA_FP32, dout, D,
                              reinterpret_cast<float*>(ws + lay.dq_acc),
                              reinterpret_cast<int*>(ws + lay.sems), lay.max_qtiles * Hq, s.Tq,
                              Hq, d, nsm, strm);
    return cuda_status(e);
}

fa_status bwd_impl(const void* q, const void* k, const void* v, const void* dout,
                   const float* lse, const float* D, void* dq, void* dk, void* dv,
                   fa_dtype grad_dtype, void* workspace, size_t workspace_bytes, int B, int Hq,
                   int Hkv, int Nq, int total_q, int Nk, int total_k, int d, float scale,
                   int causal, const int* cu_q, const int* cu_k, int deterministic,
                   fa_stream_t stream) {
    Shape s;
    fa_status st = check_shape(B, Hq, Hkv, Nq, total_q, Nk, total_k, d, cu_q, cu_k, s);
    if (st != FA_OK) return st;
    if (grad_dtype != FA_BF16 && grad_dtype != FA_FP32) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_UNSUPPORTED;
    if (B == 0 || (s.Tq == 0 && s.Tk == 0)) return FA_OK;
    cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    if (s.Tq == 0 || s.Tk == 0) {
        // One side is empty: every gradient of the other side is zero.
        void* out0 = s.Tq == 0 ? dk : dq;
        void* out1 = s.Tq == 0 ? dv : nullptr;
        const size_t n = s.Tq == 0 ? (size_t)s.Tk * Hkv * d : (size_t)s.Tq * Hq * d;
        if (!out0 || (s.Tq == 0 && !out1)) return FA_ERR_INVALID_ARG;
        cudaError_t e = cudaMemsetAsync(out0, 0, n * elem_bytes(grad_dtype), strm);
        if (e == cudaSuccess && out1) e = cudaMemsetAsync(out1, 0, n * elem_bytes(grad_dtype), strm);
        return cuda_status(e);
    }
    if (!sched_fits(s, Nk, kTile)) return FA_ERR_UNSUPPORTED;  // as fa_bwd_preprocess
    if (!q || !k || !v || !dout || !lse || !D || !dq || !dk || !dv || !workspace)
        return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv) || !aligned4(lse) || !aligned4(D) || !aligned16(workspace))
        return FA_ERR_INVALID_ARG;
    const BwdWs lay = bwd_ws_layout(B, Hq, Hkv, s.Tq, s.Tk, d);
    if (workspace_bytes < lay.bytes) return FA_ERR_INVALID_ARG;
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    if (!make_map(&p.tm_q, q, s.Tq, Hq, d) || !make_map(&p.tm_k, k, s.Tk, Hkv, d) ||
        !make_map(&p.tm_v, v, s.Tk, Hkv, d) || !make_map(&p.tm_do, dout, s.Tq, Hq, d) ||
        !make_map_f32(&p.tm_dq_acc, static_cast<char*>(workspace) + lay.dq_acc, s.Tq, Hq, d))
        return FA_ERR_CUDA;
    p.lse = lse;
    p.D = D;
    p.dk = dk;
    p.dv = dv;
    p.cu_seqlens = cu_q;
    p.cu_seqlens_k = cu_k;
    p.workspace = workspace;
    p.units_off = lay.units;
    p.tile_off_off = lay.tile_off;
    p.sems_off = lay.sems;
    p.dq_acc_off = lay.dq_acc;
    p.dk_acc_off = lay.dk_acc;
    p.dv_acc_off = lay.dv_acc;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = Nq; p.T = s.Tq; p.d = d;
    p.Nk = Nk; p.Tk = s.Tk;
    p.kv = same_boundaries(s, cu_q, cu_k) ? 0 : 1;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal ? 1 : 0;
    p.deterministic = deterministic ? 1 : 0;
    p.grad_fp32 = grad_dtype == FA_FP32;
    p.hchunk = lay.hchunk;
    p.nchunks = lay.nruns;
    const int nsm = sm_count();
    if (nsm <= 0) return FA_ERR_CUDA;
    cudaError_t e = launch_bwd(p, nsm, strm);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    const bool partials = lay.nruns > 1;
    e = launch_bwd_postprocess(reinterpret_cast<const float*>(ws + lay.dq_acc), dq,
                               partials ? reinterpret_cast<const float*>(ws + lay.dk_acc) : nullptr,
                               partials ? reinterpret_cast<const float*>(ws + lay.dv_acc) : nullptr,
                               dk, dv, s.Tq, s.Tk, Hq, Hkv, lay.nruns, d, scale, p.grad_fp32, nsm,
                               strm);
    return cuda_status(e);
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

const char* fa_version(void) { return "gb300-tiled-attention sm_103a"; }

size_t fa_fwd_workspace_size(int B, int Hq, int N, int total_tokens) {
    if (B < 0 || Hq <= 0 || N < 0 || total_tokens < 0) return 0;
    const long long T = total_tokens > 0 ? total_tokens : (long long)B * N;
    if (T > 0x7FFFFFFFLL) return 0;
    return fwd_ws_layout(B, Hq, (int)T).bytes;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype,
                 float* lse, int B, int Hq, int Hkv, int N, int total_tokens, int d, float scale,
                 int causal, const int* cu_seqlens, void* workspace, size_t workspace_bytes,
                 fa_stream_t stream) {
    return fwd_impl(q, k, v, o, o_dtype, lse, B, Hq, Hkv, N, total_tokens, N, total_tokens, d,
                    scale, causal, cu_seqlens, cu_seqlens, workspace, workspace_bytes, stream);
}

fa_status fa_fwd_kv(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype,
                    float* lse, int B, int Hq, int Hkv, int Nq, int total_q, int Nk, int total_k,
                    int d, float scale, int causal, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream) {
    return fwd_impl(q, k, v, o, o_dtype, lse, B, Hq, Hkv, Nq, total_q, Nk, total_k, d, scale,
                    causal, cu_seqlens_q, cu_seqlens_k, workspace, workspace_bytes, stream);
}

size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int N, int total_tokens, int d) {
    return bwd_ws_bytes(B, Hq, Hkv, N, total_tokens, N, total_tokens, d, false);
}

size_t fa_bwd_kv_workspace_size(int B, int Hq, int Hkv, int Nq, int total_q, int Nk,
                                int total_k, int d) {
    return bwd_ws_bytes(B, Hq, Hkv, Nq, total_q, Nk, total_k, d, false);
}

size_t fa_bwd_workspace_semaphore_offset(int B, int Hq, int Hkv, int N, int total_tokens, int d) {
    return bwd_ws_bytes(B, Hq, Hkv, N, total_tokens, N, total_tokens, d, true);
}

fa_status fa_bwd_preprocess(const void* o, fa_dtype o_dtype, const void* dout, float* D,
                            void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                            int N, int total_tokens, int d, int causal,
                            const int* cu_seqlens, int deterministic, fa_stream_t stream) {
    return bwd_preprocess_impl(o, o_dtype, dout, D, workspace, workspace_bytes, B, Hq, Hkv, N,
                               total_tokens, N, total_tokens, d, causal, cu_seqlens, cu_seqlens,
                               deterministic, stream);
}

fa_status fa_bwd_kv_preprocess(const void* o, fa_dtype o_dtype, const void* dout, float* D,
                               void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                               int Nq, int total_q, int Nk, int total_k, int d, int causal,
                               const int* cu_seqlens_q, const int* cu_seqlens_k,
                               int deterministic, fa_stream_t stream) {
    return bwd_preprocess_impl(o, o_dtype, dout, D, workspace, workspace_bytes, B, Hq, Hkv, Nq,
                               total_q, Nk, total_k, d, causal, cu_seqlens_q, cu_seqlens_k,
                               deterministic, stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* dout, const float* lse,
                 const float* D, void* dq, void* dk, void* dv, fa_dtype grad_dtype,
                 void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N,
                 int total_tokens, int d, float scale, int causal, const int* cu_seqlens,
                 int deterministic, fa_stream_t stream) {
    return bwd_impl(q, k, v, dout, lse, D, dq, dk, dv, grad_dtype, workspace, workspace_bytes, B,
                    Hq, Hkv, N, total_tokens, N, total_tokens, d, scale, causal, cu_seqlens,
                    cu_seqlens, deterministic, stream);
}

fa_status fa_bwd_kv(const void* q, const void* k, const void* v, const void* dout,
                    const float* lse, const float* D, void* dq, void* dk, void* dv,
                    fa_dtype grad_dtype, void* workspace, size_t workspace_bytes, int B, int Hq,
                    int Hkv, int Nq, int total_q, int Nk, int total_k, int d, float scale,
                    int causal, const int* cu_seqlens_q, const int* cu_seqlens_k,
                    int deterministic, fa_stream_t stream) {
    return bwd_impl(q, k, v, dout, lse, D, dq, dk, dv, grad_dtype, workspace, workspace_bytes, B,
                    Hq, Hkv, Nq, total_q, Nk, total_k, d, scale, causal, cu_seqlens_q,
                    cu_seqlens_k, deterministic, stream);
}

fa_status fa_check_device_status(const void* workspace, fa_stream_t stream) {
    if (!workspace) return FA_ERR_INVALID_ARG;
    cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(strm) != cudaSuccess) return FA_ERR_CUDA;
    int err = 0;
    if (cudaMemcpyAsync(&err, workspace, sizeof(int), cudaMemcpyDeviceToHost, strm) != cudaSuccess)
        return FA_ERR_CUDA;
    if (cudaStreamSynchronize(strm) != cudaSuccess) return FA_ERR_CUDA;
    if (err & kErrTimeout) return FA_ERR_TIMEOUT;
    if (err & kErrSchedule) return FA_ERR_INVALID_ARG;
    if (err) return FA_ERR_CUDA;
    return FA_OK;
}

}  // extern "C"
