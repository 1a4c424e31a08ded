// common.cuh -- definitions shared by the host launchers and the kernels:
// tile sizes, workspace layouts, the work-unit encoding written by the tile
// scheduler, and per-sequence geometry.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

namespace fa {

constexpr int kTile = 128;          // rows of one query tile / key-value tile
constexpr int kFwdBlockRows = 256;  // query rows of one forward work unit (two tiles)
constexpr int kFwdBlockRowsWide = 128;  // the same for head dimensions above 128 (one tile)
constexpr size_t kAlign = 256;      // alignment of every workspace segment

// Device error word bits (workspace offset 0).
constexpr int kErrTimeout = 1;      // a bounded wait gave up
constexpr int kErrSmemAlign = 2;    // dynamic shared memory not 1024-byte aligned
constexpr int kErrSchedule = 4;     // scheduler metadata inconsistent (a length > N)

// Header of every workspace (first kAlign bytes).
struct WsHeader {
    int error;          // device error word (kErr* bits)
    int counter;        // dynamic work-unit counter (zeroed by the scheduler kernel)
    int n_units;        // number of valid entries in the unit list
    int n_qtiles;       // query tiles over all sequences (backward)
};

// Unit-list entry: x = sequence index, y = (tile index << 16) | head index.
__host__ __device__ inline int unit_tile(int y) { return (int)((unsigned)y >> 16); }
__host__ __device__ inline int unit_head(int y) { return y & 0xFFFF; }
__host__ __device__ inline int make_unit_y(int tile, int head) { return (tile << 16) | head; }

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation allowed.  It first lets the next kernel in
// the stream be scheduled (pdl_trigger), and waits until the previous kernel
// has completed and its memory is visible (pdl_wait) before it touches any
// global memory; the persistent kernels set up barriers and TMEM in between.
// So no kernel reads its predecessor's output early; what overlaps is the
// next grid's launch and set-up.  Outside such a launch both are no-ops.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
    pdl_trigger();
    pdl_wait();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Upper bound on tiles of `rows` rows over all sequences of a batch:
// sum_b ceil(L_b / rows) <= ceil(T / rows) + B.
__host__ __device__ inline long long max_tiles(int B, int T, int rows) {
    return (long long)cdiv(T, rows) + (long long)B;
}

// Forward workspace: header | unit list (int2).
struct FwdWs {
    size_t units;   // offset of the unit list
    size_t bytes;   // total
    long long max_units;
};

__host__ __device__ inline FwdWs fwd_ws_layout(int B, int Hq, int T) {
    FwdWs w;
    w.max_units = max_tiles(B, T, kFwdBlockRowsWide) * (long long)Hq;  // any head dimension
    w.units = kAlign;
    w.bytes = align_up(w.units + (size_t)w.max_units * 8, kAlign);
    return w;
}

// Backward units walk a run of C query heads of one key/value head ("FlashAttention-
// 4反向传播优化" section 5.2), accumulating dK and dV over them on chip: C is
// the largest divisor of the group size Hq / Hkv up to 4 that still leaves
// kMinBwdUnits units (Hq / C heads' worth of key/value tiles), so that the
// persistent grid stays balanced; 1 for MHA and above d = 128.
constexpr long long kMinBwdUnits = 512;

__host__ __device__ inline int bwd_head_run(int Hq, int Hkv, int Tk, int d) {
    if (d > 128) return 1;  // the wide-head backward walks one query head per unit
    const int grp = Hq / Hkv;
    for (int c = 4; c > 1; --c)
        if (grp % c == 0 && (long long)(Hq / c) * cdiv(Tk, kTile) >= kMinBwdUnits) return c;
    return 1;
}

// Backward workspace: header | unit list (int2) | per-sequence query-tile
// offsets (int[B+1]) | semaphores (int[Hq * max_qtiles]) | dQ accumulator
// fp32 [Tq,Hq,d] | (when a group's heads take several runs) dK and dV
// partials fp32 [Tk, Hkv * runs, d].  Units are key/value tiles (Tk tokens)
// times runs of heads; dQ tiles and semaphores are query tiles (Tq).
struct BwdWs {
    size_t units, tile_off, sems, dq_acc, dk_acc, dv_acc, bytes;
    long long max_units, max_qtiles;
    int hchunk, nruns;  // heads per run, runs per key/value head
};

__host__ __device__ inline BwdWs bwd_ws_layout(int B, int Hq, int Hkv, int Tq, int Tk, int d) {
    BwdWs w;
    w.hchunk = bwd_head_run(Hq, Hkv, Tk, d);
    w.nruns = (Hq / Hkv) / w.hchunk;
    w.max_qtiles = max_tiles(B, Tq, kTile);
    w.max_units = max_tiles(B, Tk, kTile) * (long long)Hkv * w.nruns;
    w.units = kAlign;
    w.tile_off = align_up(w.units + (size_t)w.max_units * 8, kAlign);
    w.sems = align_up(w.tile_off + (size_t)(B + 1) * 4, kAlign);
    w.dq_acc = align_up(w.sems + (size_t)w.max_qtiles * (size_t)Hq * 4, kAlign);
    const size_t acc_q = (size_t)Tq * (size_t)Hq * (size_t)d * 4;
    const size_t acc_k = (size_t)Tk * (size_t)Hkv * (size_t)w.nruns * (size_t)d * 4;
    w.dk_acc = align_up(w.dq_acc + acc_q, kAlign);
    if (w.nruns > 1) {
        w.dv_acc = align_up(w.dk_acc + acc_k, kAlign);
        w.bytes = align_up(w.dv_acc + acc_k, kAlign);
    } else {
        w.dv_acc = w.dk_acc;
        w.bytes = w.dk_acc;
    }
    return w;
}

__host__ __device__ inline BwdWs bwd_ws_layout(int B, int Hq, int Hkv, int T, int d) {
    return bwd_ws_layout(B, Hq, Hkv, T, T, d);
}

// Causal mask with Lq queries and Lk keys: the queries are the last Lq
// positions of the key sequence, so query row r sees key c iff c <= r + off,
// off = Lk - Lq (0 for equal lengths).
__host__ __device__ inline int floor_div(int a, int b) {
    return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// Sequence geometry: start token and length of sequence b.
__device__ __forceinline__ void seq_bounds(const int* cu_seqlens, int N, int b, int& t0, int& L) {
    if (cu_seqlens) {
        t0 = cu_seqlens[b];
        L = cu_seqlens[b + 1] - t0;
    } else {
        t0 = b * N;
        L = N;
    }
}

// Orders the scheduler can write.
enum SchedOrder : int {
    kOrderLevelDesc = 0,   // tile index descending across sequences: causal forward
                           // (heaviest query blocks first) and deterministic backward
                           // (the order of every dQ tile's contributions)
    kOrderWorkDesc = 1,    // causal backward, atomic mode: KV tiles by remaining work,
                           // heaviest first (tile index ascending within a sequence)
    kOrderSeqDesc = 2,     // non-causal: sequences longest first, tiles in order
};

}  // namespace fa
