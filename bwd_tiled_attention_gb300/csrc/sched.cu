// sched.cu -- on-device tile scheduler metadata.
//
// "FlashAttention-4反向传播优化" section 3.3.2: for variable-length batches a
// preprocessing kernel sorts the sequences by their per-tile work, writes a
// virtual-to-actual index mapping, and the attention kernel walks the work in
// that order (longest processing time first).  Section 3.3.1: for the
// deterministic causal backward, key/value blocks are launched in descending
// order (shortest processing time first).  Section 5.2: query heads that share
// a key/value head are walked together.
//
// One CTA reads cu_seqlens (or the dense length N), ranks the sequences by
// tile count (descending, ties by index), and writes the ordered list of work
// units (sequence, tile, head) into the workspace, heads innermost.  The
// attention kernels take units from that list through an atomic counter that
// this kernel resets, so CTAs that finish early pick up the next unit.  The
// backward's units are key/value tiles while its dQ semaphores are per query
// tile, so it also passes the query boundaries, from which this kernel writes
// the per-sequence query-tile offsets; both sides' lengths are checked against
// their bounds.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fa {

constexpr int kSchedThreads = 1024;

struct SchedArgs {
    const int* cu_seqlens;  // device int32[B+1] or null (dense): the unit tiles
    const int* cu_aux;      // the other side's boundaries (null when dense)
    int B, N, H, rows;      // rows per tile
    int T;                  // tokens on the unit side (cu_seqlens[B] must equal it)
    int N_aux, T_aux;       // bound on the other side's lengths, its tokens
    int order;              // SchedOrder
    int max_units;          // capacity of the unit list
    WsHeader* header;
    int2* units;
    int* tile_off;          // int[B+1] offsets of the other side's tiles (may be null)
};

// Number of sequences whose tile count exceeds m, given counts sorted descending.
__device__ __forceinline__ int count_above(const int* nt_sorted, int B, int m) {
    int lo = 0, hi = B;  // first index with nt <= m
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (nt_sorted[mid] > m) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Largest index i in [0, n) with prefix[i] <= u (prefix non-decreasing, prefix[0] = 0).
__device__ __forceinline__ int find_slot(const long long* prefix, int n, long long u) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kSchedThreads) sched_kernel(SchedArgs a) {
    pdl_begin();
    extern __shared__ __align__(16) unsigned char sm[];
    const int tid = threadIdx.x;
    const int B = a.B, H = a.H;
    __shared__ long long s_total;
    __shared__ int s_maxnt, s_bad;

    if (a.cu_seqlens == nullptr) {
        // Dense batch: every sequence has nt tiles; closed-form order.
        const int nt = cdiv(a.N, a.rows);
        const int nt_aux = cdiv(a.N_aux, a.rows);
        const long long per_level = (long long)B * H;
        const long long total = per_level * nt;
        if (tid == 0) {
            a.header->n_units = (int)(total <= a.max_units ? total : 0);
            a.header->counter = 0;
            a.header->error = total <= a.max_units ? 0 : kErrSchedule;
            a.header->n_qtiles = B * nt_aux;
        }
        if (total > a.max_units) return;
        for (long long u = tid; u < total; u += kSchedThreads) {
            int b, tile, h;
            if (a.order == kOrderSeqDesc) {
                b = (int)(u / ((long long)nt * H));
                long long r = u % ((long long)nt * H);
                tile = (int)(r / H);
                h = (int)(r % H);
            } else {
                const int lvl = (int)(u / per_level);
                const long long r = u % per_level;
                b = (int)(r / H);
                h = (int)(r % H);
                tile = (a.order == kOrderLevelDesc) ? nt - 1 - lvl : lvl;
            }
            a.units[u] = make_int2(b, make_unit_y(tile, h));
        }
        if (a.tile_off)
            for (int b = tid; b <= B; b += kSchedThreads) a.tile_off[b] = b * nt_aux;
        return;
    }

    // Variable-length batch.
    int* nt_of = reinterpret_cast<int*>(sm);           // [B] tile count per sequence
    int* sorted = nt_of + B;                           // [B] sequence at rank r
    int* nt_sorted = sorted + B;                       // [B] tile count at rank r
    long long* prefix = reinterpret_cast<long long*>(  // [max(B, maxnt) + 1]
        sm + align_up((size_t)3 * B * sizeof(int), 16));
    if (tid == 0) {
        s_maxnt = 0;
        // the boundaries must span exactly the tokens the buffers hold
        s_bad = a.cu_seqlens[0] != 0 || a.cu_seqlens[B] != a.T ||
                (a.cu_aux && (a.cu_aux[0] != 0 || a.cu_aux[B] != a.T_aux));
    }
    __syncthreads();
    for (int b = tid; b < B; b += kSchedThreads) {
        const int L = a.cu_seqlens[b + 1] - a.cu_seqlens[b];
        if (L < 0 || L > a.N) atomicOr(&s_bad, 1);  // N bounds every length
        if (a.cu_aux) {
            const int La = a.cu_aux[b + 1] - a.cu_aux[b];
            if (La < 0 || La > a.N_aux) atomicOr(&s_bad, 1);
        }
        const int nt = L > 0 ? cdiv(L, a.rows) : 0;
        nt_of[b] = nt;
        atomicMax(&s_maxnt, nt);
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            a.header->n_units = 0;
            a.header->counter = 0;
            a.header->error = kErrSchedule;
            a.header->n_qtiles = 0;
        }
        return;
    }
    // rank by tile count descending, ties by index
    for (int b = tid; b < B; b += kSchedThreads) {
        const int nb = nt_of[b];
        int rank = 0;
        for (int o = 0; o < B; ++o) {
            const int no = nt_of[o];
            rank += (no > nb) || (no == nb && o < b);
        }
        sorted[rank] = b;
        nt_sorted[rank] = nb;
    }
    __syncthreads();
    const int maxnt = s_maxnt;
    int nslots;
    if (a.order == kOrderSeqDesc) {
        nslots = B;
        if (tid == 0) {
            long long acc = 0;
            for (int r = 0; r < B; ++r) { prefix[r] = acc; acc += (long long)nt_sorted[r] * H; }
            prefix[B] = acc;
            s_total = acc;
        }
    } else {
        nslots = maxnt;
        if (tid == 0) {
            long long acc = 0;
            for (int l = 0; l < maxnt; ++l) {
                prefix[l] = acc;
                acc += (long long)count_above(nt_sorted, B, maxnt - 1 - l) * H;
            }
            prefix[maxnt] = acc;
            s_total = acc;
        }
    }
    __syncthreads();
    const long long total = s_total;
    if (tid == 0) {
        a.header->n_units = (int)(total <= a.max_units ? total : 0);
        a.header->counter = 0;
        a.header->error = total <= a.max_units ? 0 : kErrSchedule;
    }
    if (a.tile_off && tid == 0) {
        int acc = 0;
        for (int b = 0; b < B; ++b) {
            a.tile_off[b] = acc;
            acc += cdiv(a.cu_aux[b + 1] - a.cu_aux[b], a.rows);
        }
        a.tile_off[B] = acc;
        a.header->n_qtiles = acc;
    } else if (tid == 0) {
        a.header->n_qtiles = 0;
    }
    if (total > a.max_units || nslots == 0) return;
    for (long long u = tid; u < total; u += kSchedThreads) {
        const int slot = find_slot(prefix, nslots, u);
        const long long r = u - prefix[slot];
        int b, tile;
        const int h = (int)(r % H);
        if (a.order == kOrderSeqDesc) {
            b = sorted[slot];
            tile = (int)(r / H);
        } else {
            const int rank = (int)(r / H);
            b = sorted[rank];
            const int m = maxnt - 1 - slot;   // sequences of this level have nt > m
            tile = (a.order == kOrderLevelDesc) ? m : nt_of[b] - 1 - m;
        }
        a.units[u] = make_int2(b, make_unit_y(tile, h));
    }
}

size_t sched_smem_bytes(int B, int maxnt_bound) {
    const int slots = (B > maxnt_bound ? B : maxnt_bound) + 1;
    return align_up((size_t)3 * B * sizeof(int), 16) + (size_t)slots * sizeof(long long);
}

cudaError_t launch_sched(const int* cu_seqlens, int B, int N, int T, int H, int rows, int order,
                         long long max_units, void* workspace, size_t units_off,
                         size_t tile_off_off, bool want_tile_off, const int* cu_tiles_seqlens,
                         int N_tiles, int T_tiles, cudaStream_t stream) {
    SchedArgs a;
    a.cu_seqlens = cu_seqlens;
    a.cu_aux = cu_tiles_seqlens;
    a.T = T;
    a.N_aux = N_tiles;
    a.T_aux = T_tiles;
    a.B = B;
    a.N = N;
    a.H = H;
    a.rows = rows;
    a.order = order;
    a.max_units = (int)(max_units > 0x7FFFFFFF ? 0x7FFFFFFF : max_units);
    a.header = reinterpret_cast<WsHeader*>(workspace);
    a.units = reinterpret_cast<int2*>(static_cast<char*>(workspace) + units_off);
    a.tile_off = want_tile_off ? reinterpret_cast<int*>(static_cast<char*>(workspace) + tile_off_off)
                               : nullptr;
    size_t smem = 0;
    if (cu_seqlens) {
        smem = sched_smem_bytes(B, cdiv(N, rows));
        cudaError_t e = cudaFuncSetAttribute(sched_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(sched_kernel, dim3(1), dim3(kSchedThreads), smem, stream, a);
}

}  // namespace fa
