/*
 * fa.h -- C ABI of the GB300 (sm_103a) tiled exact-attention library.
 *
 * The library computes exact softmax attention and its gradients without ever
 * forming the N x N score matrix.  Operation definitions follow
 * "FlashAttention-2-ICLR24" (section 问题与动机: standard attention S = QK^T,
 * P = softmax(S), O = PV, reproduced exactly by tiling plus online softmax;
 * section 核心方法 1: deferred normalisation and a stored logsumexp only;
 * section 核心方法 2: forward parallel over query-row blocks, backward parallel
 * over key/value column blocks with dQ merged by atomic adds, causal blocks
 * above the diagonal skipped; section 核心方法 4: MQA/GQA head mapping with
 * dK/dV summed over the query heads sharing a key/value head), and
 * "FlashAttention-4反向传播优化" (section 1.1: the backward is five products
 * S, dP, dV, dK, dQ with P recomputed; section 3.2: deterministic mode
 * serialises the global dQ reduction with semaphores; section 3.3: causal and
 * variable-length tile scheduling).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers marked "device" are CUDA device pointers; the caller allocates
 *   and owns every buffer, including the workspaces.  The library allocates
 *   nothing and keeps no state besides cached device attributes (and the
 *   fixed scratch array that fa_bwd_noalloc uses, described there).
 * - Token-major packed layouts, head dim innermost and contiguous:
 *     q, o, dout, dq : [T, Hq, d]      k, v, dk, dv : [T, Hkv, d]
 *     lse, D         : [Hq, T] fp32
 *   where T = total_tokens.  A dense batch (cu_seqlens == NULL) has T = B*N
 *   and sequence b owns tokens [b*N, (b+1)*N).  A packed variable-length
 *   batch passes cu_seqlens (device int32[B+1], cu_seqlens[0] = 0,
 *   non-decreasing, cu_seqlens[B] = T), T as total_tokens, and N = an upper
 *   bound on every sequence length (a longer sequence is reported as
 *   FA_ERR_INVALID_ARG by fa_check_device_status and produces no output).
 * - q, k, v, dout, dq, dk, dv and o must be 16-byte aligned (TMA).
 * - Query head h uses key/value head floor(h * Hkv / Hq); Hq % Hkv == 0.
 * - d must be 64, 96, 128, 192 or 256.  96 runs on 128-column tiles whose
 *   last 32 columns are zero (at the tensor-core cost of d = 128).  The
 *   forward at 192 and 256 runs one 128-row query tile per work unit.  The
 *   backward at 192 and 256 walks each key/value tile's query tiles twice
 *   (dV, then dK and dQ), streaming Q and dO in 64-column chunks, since S,
 *   dP, dK and dV of a tile would need 256 + 2d of the 512 tensor-memory
 *   columns.  Other head dimensions return FA_ERR_UNSUPPORTED.  Inputs are bf16.
 *   scale multiplies QK^T (usually
 *   1/sqrt(d)) and must be positive.  causal = 1 hides key j from query i
 *   when j > i (positions within the sequence; queries and keys have equal
 *   length).  The *_kv calls take separate query and key/value lengths; their
 *   causal mask is described at fa_fwd_kv.
 * - Size limits (FA_ERR_UNSUPPORTED, nothing launched): Hq <= 65535; every
 *   sequence bound N (Nq, Nk) within 65535 tiles of 128 tokens; a dense
 *   batch's B*N < 2^31; T * Hq * d <= 2^40 on either side.  A packed batch
 *   has B <= 4096 sequences.  One scheduler CTA ranks a packed batch, keeping
 *   8 bytes per tile level of the longest sequence in its shared memory, so
 *   there N must also satisfy 16 * ceil(3B / 4) + 8 * (max(B, ceil(N / R)) + 1)
 *   <= 227 KB. R is the work unit's height: 256 rows for the forward up to
 *   d = 128, 128 rows otherwise, and the backward's key/value units.  That
 *   is N <= ~3.7M tokens, or ~7.4M for the forward up to d = 128.
 * - Every call is asynchronous on `stream` (NULL = the legacy default stream)
 *   and never synchronises, except fa_check_device_status.  The return value
 *   reports argument validation and launch errors only; it never aborts.
 *   Errors found inside a kernel (a bounded wait that gave up) are recorded in
 *   the workspace and reported by fa_check_device_status.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, declared here without the CUDA headers. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, workspace too small */
    FA_ERR_UNSUPPORTED = 2,  /* valid request outside what the kernels implement */
    FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
    FA_ERR_TIMEOUT = 4       /* a bounded wait inside a kernel gave up (device-side) */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP32 = 1 } fa_dtype;

/* Human-readable name of a status code (static string). */
const char* fa_status_string(fa_status s);

/* Library build identifier (static string). */
const char* fa_version(void);

/*
 * Workspace of fa_fwd, in bytes: a small header plus the ordered list of
 * query-block work units that the on-device tile scheduler writes
 * ("FlashAttention-4反向传播优化" section 3.3.2: a preprocessing kernel sorts
 * sequences and writes the virtual-to-actual order the attention kernel walks).
 * total_tokens = 0 means B*N.  Returns 0 for invalid sizes.
 */
size_t fa_fwd_workspace_size(int B, int Hq, int N, int total_tokens);

/*
 * Forward: O = softmax(scale * Q K^T + mask) V and LSE = natural-log
 * logsumexp of the scaled, masked scores of each row ("FlashAttention-2-
 * ICLR24", 核心方法 1: O is normalised once at the end; only LSE is stored).
 *   q [T,Hq,d], k/v [T,Hkv,d]: device bf16, read only.
 *   o [T,Hq,d]: device, written in o_dtype (FA_BF16 or FA_FP32).
 *   lse [Hq,T]: device fp32, written.
 *   workspace: device, >= fa_fwd_workspace_size(B,Hq,N,total_tokens) bytes,
 *   16-byte aligned, contents scratch (rewritten each call).
 * Returns FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED without launching anything
 * when the arguments are wrong, FA_ERR_CUDA if a launch fails, FA_OK (and
 * launches nothing) when there are no tokens.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype,
                 float* lse, int B, int Hq, int Hkv, int N, int total_tokens, int d, float scale,
                 int causal, const int* cu_seqlens, void* workspace, size_t workspace_bytes,
                 fa_stream_t stream);

/*
 * Forward with different query and key/value lengths (new tokens attending
 * to a cache of earlier ones, or cross-attention).  The pages state the
 * causal mask only for equal lengths; here the Lq queries of a sequence are
 * taken to be the LAST Lq positions of its Lk keys, so with causal = 1 query
 * i (0-based within its sequence) sees key j iff j <= i + (Lk - Lq).  For
 * Lq = Lk this is the mask of fa_fwd.  A row that sees no key (causal with
 * i < Lq - Lk, or Lk = 0) gets O = 0 and LSE = -inf.
 *   q, o [Tq,Hq,d], lse [Hq,Tq]; k, v [Tk,Hkv,d].  Other arguments as in fa_fwd.
 *   Dense batch: cu_seqlens_q = cu_seqlens_k = NULL, query sequence b owns
 *   tokens [b*Nq, (b+1)*Nq) and its keys [b*Nk, (b+1)*Nk); Tq = B*Nq and
 *   Tk = B*Nk (total_q / total_k 0 or equal to those).  Packed batch: both
 *   cu_seqlens_q and cu_seqlens_k (device int32[B+1] each) with total_q =
 *   cu_seqlens_q[B], total_k = cu_seqlens_k[B], and Nq, Nk bounds on every
 *   query and key length (a longer one is reported as FA_ERR_INVALID_ARG by
 *   fa_check_device_status and produces no output).  Passing only one of the
 *   two is FA_ERR_INVALID_ARG.
 *   workspace: >= fa_fwd_workspace_size(B, Hq, Nq, total_q) bytes.
 */
fa_status fa_fwd_kv(const void* q, const void* k, const void* v, void* o, fa_dtype o_dtype,
                    float* lse, int B, int Hq, int Hkv, int Nq, int total_q, int Nk, int total_k,
                    int d, float scale, int causal, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream);

/*
 * Workspace of the backward pass (fa_bwd_preprocess + fa_bwd), in bytes: a
 * header (device error word, work counter), the scheduler's ordered unit list
 * and per-sequence tile offsets, one semaphore per (query head, query tile)
 * for deterministic mode, the fp32 dQ accumulator [T,Hq,d], and -- when the
 * query heads of a key/value head take more than one backward unit (a unit
 * walks a run of up to 4 of them, summing their dK/dV on chip) -- fp32 dK/dV
 * partials [T, Hkv * runs, d] each.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int N, int total_tokens, int d);

/*
 * Byte offset of the semaphore array inside the backward workspace (the
 * device error word is the int at offset 0).  Semaphore (h, tile) is the int
 * at index h * n_tiles + tile, where tiles are the 128-row query blocks
 * numbered sequence after sequence and n_tiles is their total count.
 */
size_t fa_bwd_workspace_semaphore_offset(int B, int Hq, int Hkv, int N, int total_tokens, int d);

/*
 * Backward preprocess: D_i = sum_c dO_ic * O_ic for every query row (fp32),
 * and reset of the backward workspace (zeroed dQ accumulator, semaphores,
 * work counter and error word; the tile schedule is rebuilt).  The pages do
 * not spell D out; it is the row term of dS = P * (dP - D) that follows from
 * differentiating the softmax.
 *   o [T,Hq,d]: device, o_dtype as written by fa_fwd.   dout [T,Hq,d]: device bf16.
 *   D [Hq,T]: device fp32, written.
 *   workspace: device, >= fa_bwd_workspace_size(...), 16-byte aligned.
 * causal and deterministic select the unit order the scheduler writes; pass
 * the same values to the fa_bwd call that follows.
 */
fa_status fa_bwd_preprocess(const void* o, fa_dtype o_dtype, const void* dout, float* D,
                            void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                            int N, int total_tokens, int d, int causal,
                            const int* cu_seqlens, int deterministic, fa_stream_t stream);

/*
 * Backward: dQ, dK, dV of L = sum(dO * O) for the forward above, recomputing P
 * from LSE ("FlashAttention-4反向传播优化" section 1.1; "FlashAttention-2-
 * ICLR24" 核心方法 2: parallel over key/value blocks, dQ merged across blocks).
 *   q, k, v, dout: device bf16 as in fa_fwd.  lse, D: device fp32 [Hq,T] from
 *   fa_fwd and fa_bwd_preprocess.
 *   dq [T,Hq,d], dk/dv [T,Hkv,d]: device, written in grad_dtype.
 *   workspace: the one fa_bwd_preprocess just reset, same sizes and flags.
 *   deterministic = 0: dQ partials are added with fp32 atomics (fast, the
 *   summation order varies run to run).  deterministic = 1: each dQ tile's
 *   partials are added in a fixed order serialised by semaphores
 *   ("FlashAttention-4反向传播优化" section 3.2), so repeated runs give
 *   bit-identical dq/dk/dv.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* dout, const float* lse,
                 const float* D, void* dq, void* dk, void* dv, fa_dtype grad_dtype,
                 void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N,
                 int total_tokens, int d, float scale, int causal, const int* cu_seqlens,
                 int deterministic, fa_stream_t stream);

/*
 * Backward with different query and key/value lengths, the gradient of
 * fa_fwd_kv: the same three steps with the query/key geometry of fa_fwd_kv.
 *   fa_bwd_kv_workspace_size: bytes of the workspace (the dQ accumulator and
 *   semaphores cover the Tq query tokens, the unit list and the GQA dK/dV
 *   partials the Tk key tokens).
 *   fa_bwd_kv_preprocess: D [Hq,Tq] and the workspace reset, as
 *   fa_bwd_preprocess; o, dout [Tq,Hq,d].
 *   fa_bwd_kv: dq [Tq,Hq,d], dk/dv [Tk,Hkv,d]; q, dout [Tq,Hq,d], k, v
 *   [Tk,Hkv,d], lse and D [Hq,Tq].  Keys that no query sees get dK = dV = 0;
 *   rows that see no key get dQ = 0.  deterministic = 1 gives bit-identical
 *   results across runs as for fa_bwd.
 * Arguments, errors and ownership otherwise as fa_bwd_preprocess / fa_bwd.
 */
size_t fa_bwd_kv_workspace_size(int B, int Hq, int Hkv, int Nq, int total_q, int Nk,
                                int total_k, int d);

fa_status fa_bwd_kv_preprocess(const void* o, fa_dtype o_dtype, const void* dout, float* D,
                               void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                               int Nq, int total_q, int Nk, int total_k, int d, int causal,
                               const int* cu_seqlens_q, const int* cu_seqlens_k,
                               int deterministic, fa_stream_t stream);

fa_status fa_bwd_kv(const void* q, const void* k, const void* v, const void* dout,
                    const float* lse, const float* D, void* dq, void* dk, void* dv,
                    fa_dtype grad_dtype, void* workspace, size_t workspace_bytes, int B, int Hq,
                    int Hkv, int Nq, int total_q, int Nk, int total_k, int d, float scale,
                    int causal, const int* cu_seqlens_q, const int* cu_seqlens_k,
                    int deterministic, fa_stream_t stream);

/*
 * Backward pass for callers that cannot allocate device memory: same inputs,
 * outputs and results as fa_bwd_preprocess followed by fa_bwd, but D and the
 * backward workspace live in a 64 MiB scratch array owned by the library, so
 * the caller passes no workspace.  The pages have no counterpart of this call;
 * it exists for code that runs where allocation is not allowed (an engine
 * plugin whose execute step must not allocate, a process whose device memory
 * is all reserved up front) and that has no buffer of its own to lend.
 *   Inputs q, k, v, o (o_dtype), dout, lse and outputs dq, dk, dv (grad_dtype)
 *   are as in fa_fwd / fa_bwd; o and lse come from fa_fwd.
 *   Limit: fa_bwd_workspace_size(B,Hq,Hkv,N,total_tokens,d) plus 4*Hq*T bytes
 *   (rounded up to 256) must fit in 64 MiB; larger requests return
 *   FA_ERR_UNSUPPORTED and launch nothing.
 *   Every GPU that loads the library holds the 64 MiB until the process
 *   exits.  The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  The call allocates nothing.
 *   All calls share the one array, which keeps the last call's contents (the
 *   parts that must start at zero are cleared on every call): calls that can
 *   overlap on the GPU -- on different streams, or from different host
 *   threads -- race on it and must be serialised by the caller.
 *   Errors found inside the kernels (a bounded wait that gave up, a sequence
 *   longer than N) are recorded in the array, not returned: read them with
 *   fa_noalloc_check_device_status after the call.  The cached array address
 *   belongs to the device's context: after cudaDeviceReset no call may be made.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         fa_dtype o_dtype, const void* dout, const float* lse, void* dq, void* dk,
                         void* dv, fa_dtype grad_dtype, int B, int Hq, int Hkv, int N,
                         int total_tokens, int d, float scale, int causal, const int* cu_seqlens,
                         int deterministic, fa_stream_t stream);

/*
 * Device status of the last fa_bwd_noalloc call on the current device: as
 * fa_check_device_status, on the error word that the call's kernels keep at
 * the base of the library's scratch array.  Synchronises `stream` (pass the
 * stream of that call).  FA_OK if no fa_bwd_noalloc call has run on the device.
 * The pages have no counterpart of this call: it completes fa_bwd_noalloc,
 * whose caller holds no workspace to pass to fa_check_device_status.
 */
fa_status fa_noalloc_check_device_status(fa_stream_t stream);

/*
 * Synchronises `stream`, then reads the device error word of a backward or
 * forward workspace: FA_OK, FA_ERR_TIMEOUT (a bounded wait gave up),
 * FA_ERR_INVALID_ARG (a sequence longer than N), or FA_ERR_CUDA if
 * synchronisation or the read failed.
 */
fa_status fa_check_device_status(const void* workspace, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
