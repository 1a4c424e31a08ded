// bwd.cu -- tiled exact-attention backward for sm_103a: preprocess (D and
// workspace reset), the main backward kernel, and the postprocess (dQ
// conversion, GQA dK/dV reduction).
//
// Method: the backward is five products ("FlashAttention-4反向传播优化"
// section 1.1): S = QK^T recomputed, P = exp(S - LSE) from the stored
// logsumexp, dV += P^T dO, dP = dO V^T, dS = P * (dP - D), dK += dS^T Q,
// dQ += dS K.  Work is parallel over key/value tiles ("FlashAttention-2-
// ICLR24" 核心方法 2): a unit owns one key/value tile of one sequence and a
// run of C query heads that share its key/value head, keeps K_j, V_j and the
// dK_j, dV_j accumulators on chip, and walks the query tiles of each of its
// heads in turn, accumulating dK_j and dV_j over all of them ("FlashAttention-
// 4反向传播优化" section 5.2: for MQA/GQA, walk the query heads of a key/value
// head before moving on).  C = 1 for MHA; with C equal to the group the unit
// writes the final dK, dV, otherwise fp32 partials per run of heads that the
// conversion kernel sums in a fixed order.  dQ is a sum over key/value tiles
// and is merged in global memory, either with fp32 atomics or -- deterministic
// mode, section 3.2 of the first page -- in a fixed order enforced by one
// semaphore per dQ tile.
//
// Walk order (section 3.3.1): in deterministic mode the scheduler launches
// units with descending j and every dQ tile takes its contributions in
// descending j, so a unit only ever waits on units taken from the work counter
// before it (no deadlock at any size, whatever CTA holds which unit).  Under
// the causal mask unit j visits query tiles i = j, j+1, ..., so its
// contribution to tile i is the (i - j)-th, unit j+1 wrote the same tile one
// step earlier and no unit waits on its first dQ write.  Without the mask all
// units walk i = 0, 1, ... and unit j's contribution is the (n - 1 - j)-th.
// In atomic mode all units of a (sequence, head) walk the query tiles in one
// common order (for L2 reuse of Q, dO and the dQ accumulator) and are
// launched heaviest-first.
//
// Roles (512 threads):
//   warp 0       producer: K_j, V_j once per unit, then Q_i with LSE_i, D_i
//                (2-stage ring) by TMA / plain loads
//   warp 3       dO producer: dO_i (1 stage) by TMA, as soon as its slot frees
//   warp 1       MMA issuer (tcgen05, one thread).  Per step: dP and dV in the
//                order their inputs arrive, then dQ once dS is in shared memory,
//                S of the NEXT step as soon as dV has released the S columns, and
//                dK last (it only accumulates) -- so the dQ drain starts early and
//                the compute warps find S(i+1) ready when they finish dS(i)
//   warp 2       TMEM allocation
//   warps 4..11  compute, two warpgroups splitting the 128 query columns of a
//                step into halves; one thread per (key row, half): P^T = exp2(S^T*c - LSE2),
//                written bf16 to TMEM (A operand of dV); dS^T = P^T (dP^T - D)
//                written bf16 to shared memory (A operand of dK, K-major, and
//                of dQ, read as MN-major)
//   warps 12..15 dQ drain (one thread per query row): whole tiles are staged
//                through a dedicated 32 KB buffer and merged with bulk tensor
//                reduce-adds,
//                ragged tiles with per-row vector reductions; ordered by the
//                semaphores in deterministic mode.  Then the dK/dV epilogue (one
//                thread per key row)
// TMEM: S^T [0,128), with the bf16 P^T of each 64-column half packed over the
// first 32 columns of that half ([0,32) and [64,96)); dP^T [128,256); dK [256,256+d);
// dV [256+d, 256+2d); dQ reuses dP^T's columns for d = 128 and has its own
// columns [384,448) for d = 64.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kBwdThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kBoxes = D / 64;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 256 + D;
    static constexpr uint32_t kColDQ = D == 128 ? 128 : 384;
    static constexpr bool kDqAliasesDp = D == 128;
};

template <int D>
struct BwdSmem {
    alignas(1024) uint8_t k[BwdCfg<D>::kTileBytes];
    alignas(1024) uint8_t v[BwdCfg<D>::kTileBytes];
    alignas(1024) uint8_t q[2][BwdCfg<D>::kTileBytes];   // Q ring (2 stages)
    alignas(1024) uint8_t dout[BwdCfg<D>::kTileBytes];   // dO (1 stage)
    alignas(1024) uint8_t ds[kTile * kTile * 2];         // dS^T: 128 key rows x 128 query cols
    alignas(1024) uint8_t stage[2][kTile * 128];         // dQ staging: 2 slots of 128 rows x 128 B
    alignas(16) float lse2[2][kTile];                    // -LSE * log2(e) of the Q stage's rows
    alignas(16) float dd[2][kTile];                      // -D of the Q stage's rows
    alignas(8) uint64_t sched_full[2], sched_empty[2];
    uint64_t kv_full, kv_empty;
    uint64_t q_full[2], q_empty[2], do_full, do_empty;
    uint64_t s_full, dp_full, p_ready, ds_ready, s_free, dq_full, dq_free;
    uint64_t dkv_full, dkv_free, drain;
    int2 sched[2];
    uint32_t tmem_base;
    int abort_flag;
    int zero;
};
static_assert(sizeof(BwdSmem<128>) <= 232448, "backward shared memory exceeds 227 KB");

// One work unit: key/value tile j of sequence b, key/value head g, query heads
// h0 .. h0 + C - 1 (run uh of the runs of heads: the unit-list head field).
// t0/L are the query tokens, tk0/Lk the key/value tokens; under the causal
// mask query row r sees key c iff c <= r + off, off = Lk - L.  nt = query
// tiles, ntk = key/value tiles, i0 = first query tile with a row that sees a
// key of tile j, ni = query tiles the unit visits per head, ns = C * ni steps.
struct BUnit {
    int b, j, uh, g, h0, t0, L, tk0, Lk, off, nt, ntk, i0, ni, ns;
};

// KV = false: keys and queries share their boundaries (Lk = L, off = 0), and
// the geometry is the plain square one.  RUNS = false: one query head per
// unit (the unit-list head field is that head); true: runs of p.hchunk > 1.
template <bool KV, bool RUNS>
__device__ __forceinline__ BUnit decode_bunit(int2 u, const BwdParams& p) {
    BUnit x;
    x.b = u.x;
    x.j = unit_tile(u.y);
    x.uh = unit_head(u.y);
    if constexpr (RUNS) {
        x.g = x.uh / p.nchunks;
        x.h0 = x.g * (p.Hq / p.Hkv) + (x.uh - x.g * p.nchunks) * p.hchunk;
    } else {
        x.h0 = x.uh;
        x.g = (int)(((long long)x.uh * p.Hkv) / p.Hq);
    }
    seq_bounds(p.cu_seqlens, p.N, x.b, x.t0, x.L);
    x.nt = cdiv(x.L, kTile);
    if constexpr (KV) {
        seq_bounds(p.cu_seqlens_k, p.Nk, x.b, x.tk0, x.Lk);
        x.off = x.Lk - x.L;
        x.ntk = cdiv(x.Lk, kTile);
        x.i0 = p.causal ? max(0, floor_div(x.j * kTile - x.off, kTile)) : 0;
        x.ni = max(0, x.nt - x.i0);  // 0 only when the sequence has no queries
    } else {
        x.tk0 = x.t0;
        x.Lk = x.L;
        x.off = 0;
        x.ntk = x.nt;
        x.i0 = p.causal ? x.j : 0;
        x.ni = p.causal ? x.nt - x.j : x.nt;
    }
    x.ns = RUNS ? x.ni * p.hchunk : x.ni;
    return x;
}

// Query tile visited at step s of unit x.
//  - deterministic causal: i = i0, i0+1, ... (i0 = j for equal lengths), so
//    unit j+1 reaches every tile one step before unit j;
//  - deterministic non-causal and atomic non-causal: i = 0, 1, ...;
//  - atomic causal: descending from the last tile.
// In atomic mode every unit of a (sequence, head) walks the tiles in the same
// order, so units running side by side load the same Q/dO tile and reduce into
// the same dQ tile while it is resident in L2.
template <bool KV>
__device__ __forceinline__ int walk_tile(const BUnit& x, int s, int deterministic, int causal) {
    if (!causal) return s;
    return deterministic ? (KV ? x.i0 : x.j) + s : x.nt - 1 - s;
}

// Position in a unit's walk: the unit walks the query tiles of head h0, then
// those of h0 + 1, ...; si = step within the current head, hh = head offset.
struct StepPos {
    int hh = 0, si = 0;
    __device__ __forceinline__ void next(int ni) {
        if (++si == ni) {
            si = 0;
            ++hh;
        }
    }
};

// Query head h and query tile i of step s of unit x (w: the walk position of
// step s, used when the unit walks a run of heads).
template <bool KV, bool RUNS>
__device__ __forceinline__ void unit_step(const BUnit& x, int s, const StepPos& w,
                                          const BwdParams& p, int& h, int& i) {
    if constexpr (RUNS) {
        h = x.h0 + w.hh;
        i = walk_tile<KV>(x, w.si, p.deterministic, p.causal);
    } else {
        h = x.h0;
        i = walk_tile<KV>(x, s, p.deterministic, p.causal);
    }
}

// Deterministic mode: how many contributions to dQ tile i precede unit x's.
// Contributions arrive in descending key/value tile: from jmax(i), ..., 0,
// where jmax(i) is the last key/value tile a row of query tile i sees (i for
// equal lengths under the causal mask; ntk - 1 without it).
template <bool KV>
__device__ __forceinline__ int dq_rank(const BUnit& x, int i, int causal) {
    if constexpr (!KV) return causal ? i - x.j : x.nt - 1 - x.j;
    const int jmax = causal ? min(x.ntk - 1, floor_div((i + 1) * kTile + x.off - 1, kTile))
                            : x.ntk - 1;
    return jmax - x.j;
}

__device__ __forceinline__ void raise_abort(volatile int* flag, WsHeader* hdr, int code) {
    *flag = 1;
    atomicOr(&hdr->error, code);
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* flag,
                                              WsHeader* hdr) {
    if (mbar_wait(bar, parity, flag)) return true;
    raise_abort(flag, hdr, kErrTimeout);
    return false;
}

// Whole-warp wait: every lane leaves with the same answer.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* flag,
                                          WsHeader* hdr) {
    return __all_sync(0xffffffffu, wait_or_abort(bar, parity, flag, hdr));
}

// Wait shared by the four warps of the dQ/epilogue warpgroup: they meet on
// named barrier 1 (deterministic mode), so all 128 threads must take the same
// branch after every wait.
__device__ __forceinline__ bool wg_wait(uint32_t bar, uint32_t parity, volatile int* flag,
                                        WsHeader* hdr) {
    return named_bar_and(1, 128, warp_wait(bar, parity, flag, hdr));
}

// Whole-warp wait done by lane 0 only (the producer warp).
__device__ __forceinline__ bool lane0_wait(uint32_t bar, uint32_t parity, volatile int* flag,
                                           WsHeader* hdr) {
    int ok = 1;
    if (lane_id() == 0) ok = wait_or_abort(bar, parity, flag, hdr) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until *sem == target (or some CTA already recorded an error).
// The first polls follow each other back to back (the wait is on the dQ
// chain, where each poll's latency counts); later ones sleep between polls.
__device__ bool sem_wait(const int* sem, int target, const WsHeader* hdr) {
    for (int i = 0; i < 64; ++i)
        if (ld_acquire_gpu(sem) == target) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 16; ++i) {
            __nanosleep(64);
            if (ld_acquire_gpu(sem) == target) return true;
        }
        if (*reinterpret_cast<const volatile int*>(&hdr->error)) return false;
        if (globaltimer() - t0 > kSpinLimitNs) return false;
    }
}

// P^T for one 32-column chunk of a key row: exp2(S^T * c - LSE2) as packed
// bf16 pairs; with MASK, columns outside [lo, hi) are zero.  nl2 holds the
// chunk's LSE2 values negated and cc is c in both halves of an fp32 pair, so
// the scaling is one packed FMA per two columns.
template <bool MASK>
__device__ __forceinline__ void p_chunk(const uint32_t (&sv)[32], const float* nl2, uint64_t cc,
                                           int lo, int hi, int xb, uint32_t (&pk)[16]) {
#pragma unroll
    for (int e4 = 0; e4 < 8; ++e4) {
        const ulonglong2 lv = reinterpret_cast<const ulonglong2*>(nl2)[e4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int e = e4 * 2 + h2;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), cc,
                             h2 ? lv.y : lv.x),
                      x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (MASK) {
                const int y0 = xb + 2 * e, y1 = y0 + 1;
                p0 = (y0 >= lo && y0 < hi) ? p0 : 0.f;
                p1 = (y1 >= lo && y1 < hi) ? p1 : 0.f;
            }
            pk[e] = pack_bf16x2(p0, p1);
        }
    }
}

// D: the tile layout (64 or 128 columns); DR: the head dimension in memory.
// DR = 96 runs on 128-column tiles: the TMA boxes past column 96 read zeros.
// S and dP contract over the first 96 columns only (6 MMAs of K = 16).  dV, dK
// and dQ keep N = 128 (their B operands are read MN-major in 64-column swizzle
// atoms); their last 32 columns are zero and neither stored nor merged.
template <int D, int DR, bool KV, bool RUNS>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ BwdParams p) {
    pdl_trigger();
    using Cfg = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.workspace);
    if (smem_u32(smem_raw) & 1023u) {  // layout relies on a 1024-byte aligned base
        pdl_wait();
        if (threadIdx.x == 0) atomicOr(&hdr->error, kErrSmemAlign);
        return;
    }
    BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
    const char* ws = static_cast<const char*>(p.workspace);
    const int2* units = reinterpret_cast<const int2*>(ws + p.units_off);
    const int* tile_off = reinterpret_cast<const int*>(ws + p.tile_off_off);
    int* sems = reinterpret_cast<int*>(static_cast<char*>(p.workspace) + p.sems_off);
    float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + p.dq_acc_off);
    float* dk_acc = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + p.dk_acc_off);
    float* dv_acc = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + p.dv_acc_off);
    const int warp = warp_id(), lane = lane_id();
    volatile int* abort_flag = &sm.abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.sched_full[i]), 1);
            mbar_init(smem_u32(&sm.sched_empty[i]), 2 + 12);
            mbar_init(smem_u32(&sm.q_full[i]), 1 + 32);
            mbar_init(smem_u32(&sm.q_empty[i]), 1);
        }
        mbar_init(smem_u32(&sm.do_full), 1);
        mbar_init(smem_u32(&sm.do_empty), 1);
        mbar_init(smem_u32(&sm.kv_full), 1);
        mbar_init(smem_u32(&sm.kv_empty), 1);
        mbar_init(smem_u32(&sm.s_full), 1);
        mbar_init(smem_u32(&sm.dp_full), 1);
        mbar_init(smem_u32(&sm.p_ready), 8);
        mbar_init(smem_u32(&sm.ds_ready), 8);
        mbar_init(smem_u32(&sm.s_free), 1);
        mbar_init(smem_u32(&sm.dq_full), 1);
        mbar_init(smem_u32(&sm.dq_free), 4);
        mbar_init(smem_u32(&sm.dkv_full), 1);
        mbar_init(smem_u32(&sm.dkv_free), 4);
        mbar_init(smem_u32(&sm.drain), 1);
        sm.abort_flag = 0;
        sm.zero = 0;
        fence_barrier_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(&sm.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    pdl_wait();  // the unit list, LSE, D and the reset workspace are the previous kernels' output
    const int n_units = hdr->n_units;
    const int n_qtiles = hdr->n_qtiles;
    // Registers: the launch gives every thread 128 (512 x 128 = 65536).  The
    // producer/MMA warpgroup (warps 0..3) gives back to 80 at the top of each
    // role, the two compute warpgroups keep 128 and the dQ drain warpgroup takes
    // 176 (it holds a whole 128-column dQ row): 128*80 + 256*128 + 128*176 = 65536.
    static_assert(128 * 80 + 256 * 128 + 128 * 176 == kBwdThreads * 128,
                  "register split must match the launch");

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        setmaxnreg_dec<80>();
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_do);
        }
        int sched_it = 0, unit_it = 0, c = 0;
        bool ok = true;
        while (ok) {
            const int slot = sched_it & 1;
            if (!(ok = lane0_wait(smem_u32(&sm.sched_empty[slot]), ((sched_it >> 1) & 1) ^ 1,
                                  abort_flag, hdr)))
                break;
            int2 unit = make_int2(-1, 0);
            if (lane == 0) {
                const int u = atomicAdd(&hdr->counter, 1);
                if (u < n_units) unit = units[u];
                sm.sched[slot] = unit;
                mbar_arrive(smem_u32(&sm.sched_full[slot]));
            }
            unit.x = __shfl_sync(0xffffffffu, unit.x, 0);
            unit.y = __shfl_sync(0xffffffffu, unit.y, 0);
            ++sched_it;
            if (unit.x < 0) break;
            const BUnit x = decode_bunit<KV, RUNS>(unit, p);
            if (!(ok = lane0_wait(smem_u32(&sm.kv_empty), (unit_it & 1) ^ 1, abort_flag, hdr)))
                break;
            if (lane == 0) {
                const uint32_t bar = smem_u32(&sm.kv_full);
                mbar_arrive_expect_tx(bar, 2 * Cfg::kTileBytes);
                for (int cb = 0; cb < Cfg::kBoxes; ++cb) {
                    tma_load_3d(smem_u32(sm.k) + cb * 16384, &p.tm_k, bar, cb * 64, x.g,
                                x.tk0 + x.j * kTile);
                    tma_load_3d(smem_u32(sm.v) + cb * 16384, &p.tm_v, bar, cb * 64, x.g,
                                x.tk0 + x.j * kTile);
                }
            }
            ++unit_it;
            StepPos w;
            for (int s = 0; s < x.ns && ok; ++s, ++c, w.next(x.ni)) {
                int h, i;
                unit_step<KV, RUNS>(x, s, w, p, h, i);
                const int st = c & 1;
                // Q_i (with its LSE and D rows) into the 2-stage ring
                if (!(ok = lane0_wait(smem_u32(&sm.q_empty[st]), ((c >> 1) & 1) ^ 1, abort_flag,
                                      hdr)))
                    break;
                const uint32_t qbar = smem_u32(&sm.q_full[st]);
                if (lane == 0) {
                    mbar_arrive_expect_tx(qbar, Cfg::kTileBytes);
                    for (int cb = 0; cb < Cfg::kBoxes; ++cb)
                        tma_load_3d(smem_u32(sm.q[st]) + cb * 16384, &p.tm_q, qbar, cb * 64, h,
                                    x.t0 + i * kTile);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = lane * 4 + e;
                    const int r = i * kTile + rr;
                    float l2 = 0.f, dv = 0.f;
                    if (r < x.L) {
                        const size_t at = (size_t)h * p.T + (size_t)(x.t0 + r);
                        l2 = p.lse[at] * kLog2e;
                        dv = p.D[at];
                    }
                    sm.lse2[st][rr] = -l2;
                    sm.dd[st][rr] = -dv;
                }
                mbar_arrive(qbar);
            }
        }
        if (lane == 0) {
            // never leave a TMA write in flight
            const volatile int* z = &sm.zero;
            for (int e = 0; e < 2 && e < c; ++e) {
                const int it = c - 1 - e;
                mbar_wait(smem_u32(&sm.q_full[it & 1]), (it >> 1) & 1, z);
            }
            if (unit_it > 0) mbar_wait(smem_u32(&sm.kv_full), (unit_it - 1) & 1, z);
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------ dO producer
        // dO_i into its single stage as soon as dP and dV of the previous step
        // have read it, independent of the Q ring's pace
        setmaxnreg_dec<80>();
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_do);
            int sched_it = 0, c = 0;
            bool ok = true;
            while (ok) {
                const int slot = sched_it & 1;
                if (!(ok = wait_or_abort(smem_u32(&sm.sched_full[slot]), (sched_it >> 1) & 1,
                                         abort_flag, hdr)))
                    break;
                const int2 unit = sm.sched[slot];
                mbar_arrive(smem_u32(&sm.sched_empty[slot]));
                ++sched_it;
                if (unit.x < 0) break;
                const BUnit x = decode_bunit<KV, RUNS>(unit, p);
                StepPos w;
                for (int s = 0; s < x.ns; ++s, ++c, w.next(x.ni)) {
                    int h, i;
                    unit_step<KV, RUNS>(x, s, w, p, h, i);
                    if (!(ok = wait_or_abort(smem_u32(&sm.do_empty), (c & 1) ^ 1, abort_flag, hdr)))
                        break;
                    const uint32_t dbar = smem_u32(&sm.do_full);
                    mbar_arrive_expect_tx(dbar, Cfg::kTileBytes);
                    for (int cb = 0; cb < Cfg::kBoxes; ++cb)
                        tma_load_3d(smem_u32(sm.dout) + cb * 16384, &p.tm_do, dbar, cb * 64, h,
                                    x.t0 + i * kTile);
                }
            }
            // never leave a TMA write in flight
            if (c > 0) mbar_wait(smem_u32(&sm.do_full), (c - 1) & 1, &sm.zero);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        setmaxnreg_dec<80>();
        if (lane == 0) {
            constexpr uint32_t idS = make_idesc_bf16(128, 128, false, false);
            constexpr uint32_t idKV = make_idesc_bf16(128, D, false, true);
            constexpr uint32_t idDQ = make_idesc_bf16(128, D, true, true);
            int sched_it = 0, unit_it = 0, cnt = 0;
            bool ok = true;
            const uint32_t kaddr = smem_u32(sm.k), vaddr = smem_u32(sm.v), dsaddr = smem_u32(sm.ds);
            const uint32_t doaddr = smem_u32(sm.dout);
            // S^T(c) = K_j Q_c^T into the S columns: needs Q_c loaded and dV(c-1),
            // the last reader of the previous P^T in those columns, complete.
            auto issue_s = [&](int c) -> bool {
                if (!wait_or_abort(smem_u32(&sm.q_full[c & 1]), (c >> 1) & 1, abort_flag, hdr))
                    return false;
                if (c > 0 && !wait_or_abort(smem_u32(&sm.s_free), (c - 1) & 1, abort_flag, hdr))
                    return false;
                tc_fence_after();
                const uint64_t da = make_sdesc_here(kaddr, 16, 1024);
                const uint64_t db = make_sdesc_here(smem_u32(sm.q[c & 1]), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < DR / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(tmem + Cfg::kColS, sdesc_add(da, off), sdesc_add(db, off), idS, kk > 0);
                }
                mma_commit(smem_u32(&sm.s_full));
                return true;
            };
            while (ok) {
                const int slot = sched_it & 1;
                if (!(ok = wait_or_abort(smem_u32(&sm.sched_full[slot]), (sched_it >> 1) & 1,
                                         abort_flag, hdr)))
                    break;
                const int2 unit = sm.sched[slot];
                mbar_arrive(smem_u32(&sm.sched_empty[slot]));
                ++sched_it;
                if (unit.x < 0) break;
                const BUnit x = decode_bunit<KV, RUNS>(unit, p);
                if (!(ok = wait_or_abort(smem_u32(&sm.kv_full), unit_it & 1, abort_flag, hdr))) break;
                if ((!KV || x.ns > 0) && !(ok = issue_s(cnt))) break;
                for (int s = 0; s < x.ns; ++s, ++cnt) {
                    const int st = cnt & 1;
                    const uint32_t qaddr = smem_u32(sm.q[st]);
                    if (!(ok = wait_or_abort(smem_u32(&sm.do_full), cnt & 1, abort_flag, hdr))) break;
                    // dP^T = V_j dO^T and dV_j += P^T dO in whichever order their inputs
                    // become ready (dP first when both are: it is on the critical path
                    // dQ drain -> dP -> dS -> dK/dQ).  For d = 128, dP reuses the TMEM
                    // columns the previous step's dQ drain reads; dV reads P^T from TMEM
                    // and, on a unit's first step, needs the previous unit's dK/dV
                    // epilogue finished.
                    {
                        bool dp_done = false, dv_done = false;
                        const uint64_t t_start = globaltimer();
                        uint32_t spins = 0;  // the timer and abort flag every 64 polls
                        while (!(dp_done && dv_done)) {
                            if (!dp_done &&
                                (!Cfg::kDqAliasesDp || cnt == 0 ||
                                 mbar_test_wait(smem_u32(&sm.dq_free), (cnt - 1) & 1))) {
                                tc_fence_after();
                                const uint64_t da = make_sdesc_here(vaddr, 16, 1024);
                                const uint64_t db = make_sdesc_here(doaddr, 16, 1024);
#pragma unroll
                                for (int kk = 0; kk < DR / 16; ++kk) {
                                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                                    mma_ss(tmem + Cfg::kColDP, sdesc_add(da, off), sdesc_add(db, off),
                                           idS, kk > 0);
                                }
                                mma_commit(smem_u32(&sm.dp_full));
                                dp_done = true;
                                continue;
                            }
                            if (!dv_done && mbar_test_wait(smem_u32(&sm.p_ready), cnt & 1) &&
                                (s != 0 || unit_it == 0 ||
                                 mbar_test_wait(smem_u32(&sm.dkv_free), (unit_it - 1) & 1))) {
                                tc_fence_after();
                                // P^T of query columns [64h, 64h+64) sits in TMEM
                                // columns [64h, 64h+32)
                                const uint64_t db = make_sdesc_here(doaddr, 16384, 1024);
#pragma unroll
                                for (int kk = 0; kk < kTile / 16; ++kk)
                                    mma_ts(tmem + Cfg::kColDV,
                                           tmem + Cfg::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                                           sdesc_add(db, kk * 2048), idKV, (s > 0 || kk > 0) ? 1u : 0u);
                                mma_commit(smem_u32(&sm.s_free));
                                dv_done = true;
                                continue;
                            }
                            if ((++spins & 63u) == 0 &&
                                (*abort_flag || globaltimer() - t_start > kSpinLimitNs)) {
                                raise_abort(abort_flag, hdr, kErrTimeout);
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                    }
                    mma_commit(smem_u32(&sm.do_empty));  // dO read by dP and dV
                    // Then this step's dQ, the next step's S and this step's dK, in
                    // that priority as their inputs arrive.  dQ is on the critical
                    // loop dQ -> drain -> dP(c+1) -> dS(c+1) -> dQ(c+1); S(c+1) needs
                    // Q(c+1) and dV(c) done with the S columns; dK only accumulates
                    // until the unit ends, so it goes last.
                    {
                        bool s_done = s + 1 >= x.ns, q_done = false, k_done = false;
                        const uint64_t t_start = globaltimer();
                        uint32_t spins = 0;  // the timer and abort flag every 64 polls
                        while (!(s_done && q_done && k_done)) {
                            if (!q_done && mbar_test_wait(smem_u32(&sm.ds_ready), cnt & 1) &&
                                (Cfg::kDqAliasesDp || cnt == 0 ||
                                 mbar_test_wait(smem_u32(&sm.dq_free), (cnt - 1) & 1))) {
                                tc_fence_after();
                                // dQ = dS K_j  (A = dS^T in shared memory read as MN-major)
                                const uint64_t da = make_sdesc_here(dsaddr, 16384, 1024);
                                const uint64_t db = make_sdesc_here(kaddr, 16384, 1024);
#pragma unroll
                                for (int kk = 0; kk < kTile / 16; ++kk)
                                    mma_ss(tmem + Cfg::kColDQ, sdesc_add(da, kk * 2048),
                                           sdesc_add(db, kk * 2048), idDQ, kk > 0);
                                // committed at once: a commit tracks every MMA issued before
                                // it, and the drain must not wait for later ones
                                mma_commit(smem_u32(&sm.dq_full));
                                q_done = true;
                                continue;
                            }
                            if (!s_done &&
                                mbar_test_wait(smem_u32(&sm.q_full[(cnt + 1) & 1]),
                                               ((cnt + 1) >> 1) & 1) &&
                                mbar_test_wait(smem_u32(&sm.s_free), cnt & 1)) {
                                tc_fence_after();
                                const uint64_t da = make_sdesc_here(kaddr, 16, 1024);
                                const uint64_t db = make_sdesc_here(smem_u32(sm.q[(cnt + 1) & 1]), 16, 1024);
#pragma unroll
                                for (int kk = 0; kk < DR / 16; ++kk) {
                                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                                    mma_ss(tmem + Cfg::kColS, sdesc_add(da, off), sdesc_add(db, off),
                                           idS, kk > 0);
                                }
                                mma_commit(smem_u32(&sm.s_full));
                                s_done = true;
                                continue;
                            }
                            if (!k_done && q_done) {
                                // dK_j += dS^T Q  (A = dS^T in shared memory, K-major)
                                const uint64_t da = make_sdesc_here(dsaddr, 16, 1024);
                                const uint64_t db = make_sdesc_here(qaddr, 16384, 1024);
#pragma unroll
                                for (int kk = 0; kk < kTile / 16; ++kk) {
                                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                                    mma_ss(tmem + Cfg::kColDK, sdesc_add(da, off), sdesc_add(db, kk * 2048),
                                           idKV, (s > 0 || kk > 0) ? 1u : 0u);
                                }
                                mma_commit(smem_u32(&sm.q_empty[st]));   // Q(c) read by S(c), dK
                                k_done = true;
                                continue;
                            }
                            if ((++spins & 63u) == 0 &&
                                (*abort_flag || globaltimer() - t_start > kSpinLimitNs)) {
                                raise_abort(abort_flag, hdr, kErrTimeout);
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                    }
                }
                if (!ok) break;
                if constexpr (KV) {
                    // A unit that no query sees issues no dV, whose first one waits
                    // for the previous unit's dK/dV epilogue.  Wait for it here, or
                    // two such units in a row could put dkv_full two phases ahead of
                    // the epilogue warps, which parity cannot tell apart.
                    if (x.ns == 0 && unit_it > 0 &&
                        !(ok = wait_or_abort(smem_u32(&sm.dkv_free), (unit_it - 1) & 1, abort_flag,
                                             hdr)))
                        break;
                }
                mma_commit(smem_u32(&sm.dkv_full));
                mma_commit(smem_u32(&sm.kv_empty));
                ++unit_it;
            }
            mma_commit(smem_u32(&sm.drain));
            mbar_wait(smem_u32(&sm.drain), 0, &sm.zero);
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ compute: P^T and dS^T
        // (keeps the launch's 128 registers)
        const int q4 = warp & 3;
        const int hc = (warp - 4) >> 2;                   // query-column half of this warpgroup
        const int rk = q4 * 32 + lane;                    // key row within the tile (TMEM lane)
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + Cfg::kColS;
        const uint32_t dp_addr = tmem + lane_off + Cfg::kColDP;
        uint8_t* ds_row = sm.ds + hc * 16384 + rk * 128;  // this half's 64-column block
        const int sw = rk & 7;
        const uint64_t cc2 = f2_pack(p.scale_log2, p.scale_log2);
        int sched_it = 0, cnt = 0;
        bool ok = true;
        while (ok) {
            const int slot = sched_it & 1;
            if (!(ok = warp_wait(smem_u32(&sm.sched_full[slot]), (sched_it >> 1) & 1, abort_flag,
                                 hdr)))
                break;
            const int2 unit = sm.sched[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.sched_empty[slot]));
            ++sched_it;
            if (unit.x < 0) break;
            const BUnit x = decode_bunit<KV, RUNS>(unit, p);
            // key position c within its sequence: query column r sees it iff
            // r >= c - off (causal) and r < L; a key past the end sees nothing
            const int c = x.j * kTile + rk;
            const int c_off = c - x.off;
            const int L_vis = c < x.Lk ? x.L : 0;  // (KV only)
            StepPos w;
            for (int s = 0; s < x.ns; ++s, ++cnt, w.next(x.ni)) {
                int h, i;
                unit_step<KV, RUNS>(x, s, w, p, h, i);
                const int st = cnt & 1;
                // visible query columns of this key row: [lo, hi); the warp skips the
                // mask when every row sees every column
                int lo, hi;
                if constexpr (KV) {
                    lo = p.causal ? max(0, c_off - i * kTile) : 0;
                    hi = min(kTile, L_vis - i * kTile);
                } else {
                    lo = p.causal ? max(0, c - i * kTile) : 0;
                    hi = c < x.L ? min(kTile, x.L - i * kTile) : 0;
                }
                const bool full = __all_sync(0xffffffffu, lo == 0 && hi == kTile);
                if (!(ok = warp_wait(smem_u32(&sm.q_full[st]), (cnt >> 1) & 1, abort_flag, hdr)))
                    break;
                if (!(ok = warp_wait(smem_u32(&sm.s_full), cnt & 1, abort_flag, hdr))) break;
                tc_fence_after();
                const float* l2 = sm.lse2[st] + hc * 64;
                uint32_t pk[2][16];
                {
                    uint32_t sv[2][32];  // this half's two 32-column loads, one wait
                    tmem_ld32(s_addr + hc * 64, sv[0]);
                    tmem_ld32(s_addr + hc * 64 + 32, sv[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int xb = hc * 64 + h * 32;  // first query column of the chunk
                        if (full)
                            p_chunk<false>(sv[h], l2 + h * 32, cc2, lo, hi, xb, pk[h]);
                        else
                            p_chunk<true>(sv[h], l2 + h * 32, cc2, lo, hi, xb, pk[h]);
                        // into this half's own S^T columns, which this warp has
                        // already read (the other half's are still being read)
                        tmem_st16(s_addr + hc * 64 + h * 16, pk[h]);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.p_ready));
                // dS^T = P^T * (dP^T - D), bf16, swizzled rows of the dS^T tile
                // dp_full(c) also means dQ(c-1) and dK(c-1), the readers of the
                // last dS^T, are done: the MMA thread issued them before dP(c),
                // and a commit tracks every MMA issued before it
                if (!(ok = warp_wait(smem_u32(&sm.dp_full), cnt & 1, abort_flag, hdr))) break;
                tc_fence_after();
                const float* dd = sm.dd[st] + hc * 64;
                {
                    uint32_t dv[2][32];
                    tmem_ld32(dp_addr + hc * 64, dv[0]);
                    tmem_ld32(dp_addr + hc * 64 + 32, dv[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t out[16];
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const ulonglong2 nd = reinterpret_cast<const ulonglong2*>(dd + h * 32)[e4];
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const int e = e4 * 2 + h2;
                                const uint32_t pp = pk[h][e];
                                const uint64_t pf = f2_pack(__uint_as_float(pp << 16),
                                                            __uint_as_float(pp & 0xffff0000u));
                                const uint64_t t = f2_add(f2_pack(__uint_as_float(dv[h][2 * e]),
                                                                  __uint_as_float(dv[h][2 * e + 1])),
                                                          h2 ? nd.y : nd.x);
                                float d0, d1;
                                f2_unpack(f2_mul(t, pf), d0, d1);
                                out[e] = pack_bf16x2(d0, d1);
                            }
                        }
                        // 32 query columns = 4 chunks of 16 bytes of this half's block
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int ch = h * 4 + e;
                            *reinterpret_cast<uint4*>(ds_row + ((ch ^ sw) << 4)) =
                                make_uint4(out[4 * e], out[4 * e + 1], out[4 * e + 2],
                                           out[4 * e + 3]);
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.ds_ready));
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ dQ drain + dK/dV epilogue
        setmaxnreg_inc<176>();
        const int q4 = warp & 3;
        const int rr = q4 * 32 + lane;  // row within the tile (TMEM lane)
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const bool leader = (warp == 12 && lane == 0);
        const uint32_t stage_base = smem_u32(sm.stage[0]);
        uint8_t* stage_row = sm.stage[0] + rr * 128;  // this thread's row in a staging slot
        const int sw = rr & 7;
        int sched_it = 0, unit_it = 0, cnt = 0, chunk = 0;
        bool ok = true;
        while (ok) {
            const int slot = sched_it & 1;
            if (!(ok = wg_wait(smem_u32(&sm.sched_full[slot]), (sched_it >> 1) & 1, abort_flag,
                               hdr)))
                break;
            const int2 unit = sm.sched[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.sched_empty[slot]));
            ++sched_it;
            if (unit.x < 0) break;
            const BUnit x = decode_bunit<KV, RUNS>(unit, p);
            StepPos w;
            for (int s = 0; s < x.ns; ++s, w.next(x.ni)) {
                int h, i;
                unit_step<KV, RUNS>(x, s, w, p, h, i);
                if (!(ok = wg_wait(smem_u32(&sm.dq_full), cnt & 1, abort_flag, hdr))) break;
                tc_fence_after();
                int* sem = nullptr;
                bool sem_ok = true;
                if (p.deterministic) {
                    sem = sems + (size_t)h * n_qtiles + tile_off[x.b] + i;
                    if (leader) {
                        sem_ok = sem_wait(sem, dq_rank<KV>(x, i, p.causal), hdr);
                        if (!sem_ok) raise_abort(abort_flag, hdr, kErrTimeout);
                    }
                    sem_ok = named_bar_and(1, 128, sem_ok);
                }
                const int row0 = i * kTile;
                // The whole dQ row goes to registers first and its TMEM columns go
                // back at once: the next step's dP MMA waits for them.
                const bool whole = row0 + kTile <= x.L;
                const int qr = row0 + rr;
                uint32_t v[DR / 32][32];
#pragma unroll
                for (int cc = 0; cc < DR / 32; ++cc)
                    tmem_ld32(tmem + lane_off + Cfg::kColDQ + cc * 32, v[cc]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.dq_free));
                if (whole) {
                    // Whole tile: bulk reduce-add, one 32-column chunk at a time,
                    // staged 128B-swizzled through two 16 KB slots.
#pragma unroll
                    for (int cc = 0; cc < DR / 32; ++cc, ++chunk) {
                        const int sl = chunk & 1;
                        // the reduce that last used this slot has read it
                        if (leader) bulk_wait_group_read<1>();
                        named_bar_sync(1, 128);
                        uint8_t* row = stage_row + sl * (kTile * 128);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            *reinterpret_cast<uint4*>(row + ((e ^ sw) << 4)) =
                                make_uint4(v[cc][4 * e], v[cc][4 * e + 1], v[cc][4 * e + 2],
                                           v[cc][4 * e + 3]);
                        fence_proxy_async_smem();
                        named_bar_sync(1, 128);
                        if (leader && sem_ok)
                            tma_reduce_add_3d(&p.tm_dq_acc, stage_base + sl * (kTile * 128), cc * 32,
                                              h, x.t0 + row0);
                        if (leader) bulk_commit_group();
                    }
                } else if (qr < x.L && sem_ok) {
                    // Ragged last tile of a sequence: per-row vector reductions.
                    float* dst = dq_acc + ((size_t)(x.t0 + qr) * p.Hq + h) * DR;
#pragma unroll
                    for (int cc = 0; cc < DR / 32; ++cc)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            red_add_v4(dst + cc * 32 + 4 * e, __uint_as_float(v[cc][4 * e]),
                                       __uint_as_float(v[cc][4 * e + 1]),
                                       __uint_as_float(v[cc][4 * e + 2]),
                                       __uint_as_float(v[cc][4 * e + 3]));
                }
                if (p.deterministic) {
                    // this contribution must be complete before the next one may start:
                    // a whole tile's reduce-adds are the leader's own bulk operations;
                    // a ragged tile's vector reductions are every thread's
                    if (whole) {
                        if (leader) {
                            bulk_wait_group<0>();
                            fence_proxy_async_global();
                            if (sem_ok) red_release_gpu_add(sem, 1);
                        }
                    } else {
                        __threadfence();
                        named_bar_sync(1, 128);
                        if (leader && sem_ok) red_release_gpu_add(sem, 1);
                    }
                }
                ++cnt;
                if (!sem_ok) { ok = false; break; }
            }
            if (!ok) break;
            // dK_j (times scale) and dV_j, summed over the unit's query heads
            if (!(ok = wg_wait(smem_u32(&sm.dkv_full), unit_it & 1, abort_flag, hdr))) break;
            tc_fence_after();
            const int kr = x.j * kTile + rr;
            const bool valid = kr < x.Lk;
            const size_t tok = (size_t)x.tk0 + (size_t)kr;
            const bool none = KV && x.ns == 0;  // no query: dK = dV = 0, TMEM not written
            const bool partial = p.nchunks > 1;  // other units cover the group's other heads
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which == 0 ? Cfg::kColDK : Cfg::kColDV;
                const float mul = which == 0 ? p.scale : 1.f;
#pragma unroll 1
                for (int cc = 0; cc < DR / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + col + cc * 32, v);
                    tmem_ld_wait();
                    if (!valid) continue;
                    if (none) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;
                    }
                    if (partial) {
                        float* acc = (which == 0 ? dk_acc : dv_acc) +
                                     (tok * (size_t)(p.Hkv * p.nchunks) + x.uh) * DR + cc * 32;
                        float4* d4 = reinterpret_cast<float4*>(acc);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            d4[e] = make_float4(__uint_as_float(v[4 * e]) * mul,
                                                __uint_as_float(v[4 * e + 1]) * mul,
                                                __uint_as_float(v[4 * e + 2]) * mul,
                                                __uint_as_float(v[4 * e + 3]) * mul);
                    } else if (p.grad_fp32) {
                        float* out = static_cast<float*>(which == 0 ? p.dk : p.dv) +
                                     (tok * p.Hkv + x.g) * DR + cc * 32;
                        float4* d4 = reinterpret_cast<float4*>(out);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            d4[e] = make_float4(__uint_as_float(v[4 * e]) * mul,
                                                __uint_as_float(v[4 * e + 1]) * mul,
                                                __uint_as_float(v[4 * e + 2]) * mul,
                                                __uint_as_float(v[4 * e + 3]) * mul);
                    } else {
                        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(which == 0 ? p.dk : p.dv) +
                                             (tok * p.Hkv + x.g) * DR + cc * 32;
                        uint4* d4 = reinterpret_cast<uint4*>(out);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            d4[e] = make_uint4(
                                pack_bf16x2(__uint_as_float(v[8 * e]) * mul,
                                            __uint_as_float(v[8 * e + 1]) * mul),
                                pack_bf16x2(__uint_as_float(v[8 * e + 2]) * mul,
                                            __uint_as_float(v[8 * e + 3]) * mul),
                                pack_bf16x2(__uint_as_float(v[8 * e + 4]) * mul,
                                            __uint_as_float(v[8 * e + 5]) * mul),
                                pack_bf16x2(__uint_as_float(v[8 * e + 6]) * mul,
                                            __uint_as_float(v[8 * e + 7]) * mul));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.dkv_free));
            ++unit_it;
        }
        // the staging slots must not be read after the CTA exits
        if (leader) bulk_wait_group<0>();
    } else {
        setmaxnreg_dec<80>();  // warp 2: TMEM allocation only
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- head dimensions 192 and 256
//
// S, dP, dK and dV of one key/value tile need 256 + 2d TMEM columns, more than
// the 512 there are above d = 128, and K, V, Q and dO tiles of 48-64 KB each do
// not fit shared memory together.  So a unit (one key/value tile of one
// sequence and query head) walks its query tiles twice:
//   pass 1: S^T = K Q^T, P^T (bf16, in TMEM over S^T), dV += P^T dO;
//   pass 2: S^T and dP^T = V dO^T, dS^T = P^T (dP^T - D) (bf16, shared memory),
//           dK += dS^T Q, dQ = dS K into the columns S^T and dP^T held.
// dV is stored after pass 1 and dK after pass 2, from the same TMEM columns
// [256, 256 + d).  K and V stay in shared memory for the unit; Q and dO are
// streamed in 64-column chunks through a ring (pass 1 reads Q, dO; pass 2
// reads Q, dO, Q), so pass 2 recomputes S and the MMA work is 1.2 times the
// five products.
//
// A step streams 128 KB (pass 1) or 192 KB (pass 2) of chunks, and a TMA load
// blocks its issuing thread while the SM's TMA unit works through the loads
// before it (about 25 B per cycle per SM), so the loads have a warp of their
// own, as do the MMAs.  Roles (256 threads):
//   warp 0       producer: unit fetch, K and V, the Q/dO chunks in the order
//                the MMAs read them
//   warp 1       MMA issuer (one thread)
//   warp 2       TMEM allocation
//   warps 4..7   compute, one thread per key row (P^T, dS^T, the dK/dV
//                epilogue) or per query row (the dQ merge)
// Pass 1 double-buffers S^T in TMEM columns [0, 128) and [128, 256): the MMA
// issuer computes S^T of the next query tile while the compute warps turn the
// current one into P^T, then dV.  Pass 2 computes S^T and dP^T, waits for dS^T,
// then dK and dQ; the compute warps release dQ's columns in two halves as the
// merge reads them, so the next S^T starts while the merge still runs.
constexpr int kWideThreads = 256;
constexpr int kWideChunkBytes = kTile * 64 * 2;
// Ring of 64-column Q/dO chunks: 4 slots at d = 256 (all the shared memory
// left), 6 at d = 192.
template <int D>
struct WideCfg {
    static constexpr int kSlots = D == 256 ? 4 : 6;
};

template <int D>
struct WideSmem {
    alignas(1024) uint8_t k[kTile * D * 2];
    alignas(1024) uint8_t v[kTile * D * 2];
    alignas(1024) uint8_t ring[WideCfg<D>::kSlots][kWideChunkBytes];
    // dS^T (two 64-column boxes, 128B-swizzled); once dK and dQ have read it,
    // the staging of the dQ merge (two 32-column fp32 slots)
    alignas(1024) uint8_t ds[kTile * kTile * 2];
    alignas(16) float lse2[2][kTile];  // -LSE * log2(e) of the step's query rows
    alignas(16) float dd[2][kTile];    // -D of the step's query rows
    alignas(8) uint64_t sched_full[2], sched_empty[2];
    uint64_t kv_full, kv_empty;
    uint64_t slot_full[WideCfg<D>::kSlots], slot_free[WideCfg<D>::kSlots];
    uint64_t s_full[2], p_ready[2], s_free[2];            // pass 1, per S^T buffer
    uint64_t sdp_full, ds_ready, dq_full, dq_free[2];     // pass 2; dQ columns in halves
    uint64_t dv_full, dk_full;                            // dV / dK done
    uint64_t drain;
    int2 sched[2];
    uint32_t tmem_base;
    int abort_flag;
    int zero;
};
static_assert(sizeof(WideSmem<256>) <= 232448, "wide backward shared memory exceeds 227 KB");
static_assert(sizeof(WideSmem<192>) <= 232448, "wide backward shared memory exceeds 227 KB");

// One write-after-read hand-off of a TMEM region that the MMA issuer still
// has to wait for: the barrier and the parity of the phase.  The issuer waits
// for it before its next write to the region, and before recording another
// one for the same region, so it is never two phases behind a barrier.
struct Pending {
    uint32_t bar = 0, parity = 0;
    bool set = false;
};

template <int D, bool KV>
__global__ void __launch_bounds__(kWideThreads, 1)
    fa_bwd_wide_kernel(const __grid_constant__ BwdParams p) {
    pdl_trigger();
    constexpr int C = D / 64;                       // 64-column chunks of a row
    constexpr int kSlots = WideCfg<D>::kSlots;
    constexpr uint32_t kColDKV = 256;               // dV (pass 1), then dK (pass 2)
    constexpr uint32_t idS = make_idesc_bf16(128, 128, false, false);
    constexpr uint32_t idN = make_idesc_bf16(128, 64, false, true);
    constexpr uint32_t idN2 = make_idesc_bf16(128, 128, false, true);  // two adjacent chunks
    constexpr uint32_t idDQ = make_idesc_bf16(128, D, true, true);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.workspace);
    if (smem_u32(smem_raw) & 1023u) {
        pdl_wait();
        if (threadIdx.x == 0) atomicOr(&hdr->error, kErrSmemAlign);
        return;
    }
    WideSmem<D>& sm = *reinterpret_cast<WideSmem<D>*>(smem_raw);
    const char* ws = static_cast<const char*>(p.workspace);
    const int2* units = reinterpret_cast<const int2*>(ws + p.units_off);
    const int* tile_off = reinterpret_cast<const int*>(ws + p.tile_off_off);
    int* sems = reinterpret_cast<int*>(static_cast<char*>(p.workspace) + p.sems_off);
    float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + p.dq_acc_off);
    float* dk_acc = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + p.dk_acc_off);
    float* dv_acc = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + p.dv_acc_off);
    const int warp = warp_id(), lane = lane_id();
    volatile int* abort_flag = &sm.abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.sched_full[i]), 1);
            mbar_init(smem_u32(&sm.sched_empty[i]), 1 + 4);
            mbar_init(smem_u32(&sm.s_full[i]), 1);
            mbar_init(smem_u32(&sm.p_ready[i]), 4);
            mbar_init(smem_u32(&sm.s_free[i]), 1);
            mbar_init(smem_u32(&sm.dq_free[i]), 4);
        }
        mbar_init(smem_u32(&sm.kv_full), 1);
        mbar_init(smem_u32(&sm.kv_empty), 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(smem_u32(&sm.slot_full[s]), 1);
            mbar_init(smem_u32(&sm.slot_free[s]), 1);
        }
        mbar_init(smem_u32(&sm.sdp_full), 1);
        mbar_init(smem_u32(&sm.ds_ready), 4);
        mbar_init(smem_u32(&sm.dq_full), 1);
        mbar_init(smem_u32(&sm.dv_full), 1);
        mbar_init(smem_u32(&sm.dk_full), 1);
        mbar_init(smem_u32(&sm.drain), 1);
        sm.abort_flag = 0;
        sm.zero = 0;
        fence_barrier_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(&sm.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    pdl_wait();  // the unit list, LSE, D and the reset workspace are the previous kernels' output
    const int n_units = hdr->n_units;
    const int n_qtiles = hdr->n_qtiles;
    const uint32_t kaddr = smem_u32(sm.k), vaddr = smem_u32(sm.v), dsaddr = smem_u32(sm.ds);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_do);
            int sched_it = 0, unit_it = 0, g = 0;  // g: chunks loaded, over all units
            bool ok = true;
            // chunk of query tile i: Q or dO columns [64 cc, +64)
            auto load_chunk = [&](bool is_do, int cc, int h, int row0) -> bool {
                const int slot = g % kSlots, n = g / kSlots;
                if (n > 0 && !wait_or_abort(smem_u32(&sm.slot_free[slot]), (n - 1) & 1, abort_flag, hdr))
                    return false;
                const uint32_t bar = smem_u32(&sm.slot_full[slot]);
                mbar_arrive_expect_tx(bar, kWideChunkBytes);
                tma_load_3d(smem_u32(sm.ring[slot]), is_do ? &p.tm_do : &p.tm_q, bar, cc * 64, h, row0);
                ++g;
                return true;
            };
            while (ok) {
                const int slot = sched_it & 1;
                if (!(ok = wait_or_abort(smem_u32(&sm.sched_empty[slot]), ((sched_it >> 1) & 1) ^ 1,
                                         abort_flag, hdr)))
                    break;
                const int u = atomicAdd(&hdr->counter, 1);
                const int2 unit = u < n_units ? units[u] : make_int2(-1, 0);
                sm.sched[slot] = unit;
                mbar_arrive(smem_u32(&sm.sched_full[slot]));
                ++sched_it;
                if (unit.x < 0) break;
                const BUnit x = decode_bunit<KV, false>(unit, p);
                const int h = x.h0;
                if (unit_it > 0 &&
                    !(ok = wait_or_abort(smem_u32(&sm.kv_empty), (unit_it - 1) & 1, abort_flag, hdr)))
                    break;
                const uint32_t kvbar = smem_u32(&sm.kv_full);
                mbar_arrive_expect_tx(kvbar, 2 * kTile * D * 2);
                for (int cb = 0; cb < C; ++cb) {
                    tma_load_3d(kaddr + cb * 16384, &p.tm_k, kvbar, cb * 64, x.g, x.tk0 + x.j * kTile);
                    tma_load_3d(vaddr + cb * 16384, &p.tm_v, kvbar, cb * 64, x.g, x.tk0 + x.j * kTile);
                }
                ++unit_it;
                auto row0 = [&](int s) {
                    return x.t0 + walk_tile<KV>(x, s, p.deterministic, p.causal) * kTile;
                };
                // pass 1: Q(0), then Q(s), dO(s - 1) for s >= 1, then dO(n - 1)
                for (int s = 0; s <= x.ns && ok; ++s) {
                    for (int cc = 0; cc < C && ok && s < x.ns; ++cc) ok = load_chunk(false, cc, h, row0(s));
                    for (int cc = 0; cc < C && ok && s > 0; ++cc) ok = load_chunk(true, cc, h, row0(s - 1));
                }
                // pass 2: Q(s), dO(s), Q(s)
                for (int s = 0; s < x.ns && ok; ++s) {
                    const int r0 = row0(s);
                    for (int cc = 0; cc < C && ok; ++cc) ok = load_chunk(false, cc, h, r0);
                    for (int cc = 0; cc < C && ok; ++cc) ok = load_chunk(true, cc, h, r0);
                    for (int cc = 0; cc < C && ok; ++cc) ok = load_chunk(false, cc, h, r0);
                }
            }
            // never leave a TMA write in flight
            const volatile int* z = &sm.zero;
            for (int e = 0; e < kSlots && e < g; ++e) {
                const int it = g - 1 - e;
                mbar_wait(smem_u32(&sm.slot_full[it % kSlots]), (it / kSlots) & 1, z);
            }
            if (unit_it > 0) mbar_wait(smem_u32(&sm.kv_full), (unit_it - 1) & 1, z);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int sched_it = 0, unit_it = 0, g = 0;  // g: chunks consumed, over all units
            int c1 = 0, c2 = 0;                    // pass-1 / pass-2 steps, over all units
            // TMEM [0, 128) and [128, 256).  The dK/dV columns need none: the
            // compute warps read dV out before they arrive on ds_ready (pass 2's
            // first dK waits for it) and dK before the next unit's first p_ready.
            Pending pend_s[2];
            bool ok = true;
            auto settle = [&](Pending& pd) -> bool {
                if (!pd.set) return true;
                pd.set = false;
                if (!wait_or_abort(pd.bar, pd.parity, abort_flag, hdr)) return false;
                tc_fence_after();
                return true;
            };
            auto expect = [&](Pending& pd, uint32_t bar, uint32_t parity) -> bool {
                const bool r = settle(pd);
                pd.bar = bar;
                pd.parity = parity;
                pd.set = true;
                return r;
            };
            // next chunk of the ring: its shared-memory address once landed, or 0
            auto acquire = [&](int ahead = 0) -> uint32_t {
                const int ga = g + ahead, slot = ga % kSlots;
                if (!wait_or_abort(smem_u32(&sm.slot_full[slot]), (ga / kSlots) & 1, abort_flag, hdr))
                    return 0u;
                tc_fence_after();
                return smem_u32(sm.ring[slot]);
            };
            auto release = [&]() { mma_commit(smem_u32(&sm.slot_free[g++ % kSlots])); };
            // dV / dK take the chunks' d columns as N: two chunks at once (N = 128)
            // when they sit in adjacent slots (a group of C chunks starts at a
            // multiple of C in the ring, so only a group's last chunk at d = 192
            // goes alone), since N = 64 runs the tensor core at two thirds of its
            // rate.  issue(col, b_addr, n128) issues one chunk or pair into dK/dV
            // columns col; returns the chunks taken (0 on abort).
            auto acc_chunks = [&](int cc, auto&& issue) -> int {
                const uint32_t a = acquire();
                if (!a) return 0;
                if (cc + 1 < C && g % kSlots != kSlots - 1) {
                    const uint32_t a2 = acquire(1);
                    if (!a2) return 0;
                    if (a2 == a + kWideChunkBytes) {
                        issue(kColDKV + cc * 64, a, true);
                        release();
                        release();
                        return 2;
                    }
                }
                issue(kColDKV + cc * 64, a, false);
                release();
                return 1;
            };
            // S^T = K Q^T over C chunks into TMEM column col (accumulating across chunks)
            auto issue_s = [&](uint32_t col, uint32_t abase) -> bool {
                for (int cc = 0; cc < C; ++cc) {
                    const uint32_t a = acquire();
                    if (!a) return false;
                    const uint64_t da = make_sdesc_here(abase + cc * 16384, 16, 1024);
                    const uint64_t db = make_sdesc_here(a, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss(tmem + col, sdesc_add(da, kk * 32), sdesc_add(db, kk * 32), idS,
                               (cc | kk) > 0);
                    release();
                }
                return true;
            };
            while (ok) {
                const int slot = sched_it & 1;
                if (!(ok = wait_or_abort(smem_u32(&sm.sched_full[slot]), (sched_it >> 1) & 1,
                                         abort_flag, hdr)))
                    break;
                const int2 unit = sm.sched[slot];
                mbar_arrive(smem_u32(&sm.sched_empty[slot]));
                ++sched_it;
                if (unit.x < 0) break;
                const BUnit x = decode_bunit<KV, false>(unit, p);
                if (!(ok = wait_or_abort(smem_u32(&sm.kv_full), unit_it & 1, abort_flag, hdr))) break;
                tc_fence_after();
                ++unit_it;
                // ---- pass 1: S(0), then S(s), dV(s - 1), then dV(n - 1)
                for (int s = 0; s <= x.ns && ok; ++s) {
                    if (s < x.ns) {
                        const int c = c1 + s, b = c & 1;
                        if (!(ok = settle(pend_s[b]))) break;
                        if (!(ok = issue_s((uint32_t)b * 128, kaddr))) break;
                        mma_commit(smem_u32(&sm.s_full[b]));
                    }
                    if (s > 0) {
                        const int c = c1 + s - 1, b = c & 1;
                        if (!(ok = wait_or_abort(smem_u32(&sm.p_ready[b]), (c >> 1) & 1, abort_flag, hdr)))
                            break;
                        tc_fence_after();
                        for (int cc = 0; cc < C && ok;) {
                            const int n = acc_chunks(cc, [&](uint32_t col, uint32_t a, bool n128) {
                                const uint64_t db = make_sdesc_here(a, 16384, 1024);
#pragma unroll
                                for (int kk = 0; kk < kTile / 16; ++kk)
                                    mma_ts(tmem + col, tmem + b * 128 + (kk >> 2) * 64 + (kk & 3) * 8,
                                           sdesc_add(db, kk * 2048), n128 ? idN2 : idN,
                                           (s > 1 || kk > 0) ? 1u : 0u);
                            });
                            ok = n > 0;
                            cc += n;
                        }
                        if (!ok) break;
                        mma_commit(smem_u32(&sm.s_free[b]));
                        ok = expect(pend_s[b], smem_u32(&sm.s_free[b]), (c >> 1) & 1);
                    }
                }
                if (!ok) break;
                c1 += x.ns;
                // only units with query tiles signal their accumulators: each such
                // commit follows an arrival of the compute warps on the same unit,
                // so it can never run two phases ahead of their wait
                if (x.ns > 0) mma_commit(smem_u32(&sm.dv_full));
                // ---- pass 2
                for (int s = 0; s < x.ns && ok; ++s) {
                    const int c = c2 + s;
                    if (!(ok = settle(pend_s[0]))) break;
                    if (!(ok = issue_s(0, kaddr))) break;
                    if (!(ok = settle(pend_s[1]))) break;
                    if (!(ok = issue_s(128, vaddr))) break;  // dP^T = V dO^T (the dO chunks)
                    mma_commit(smem_u32(&sm.sdp_full));
                    if (!(ok = wait_or_abort(smem_u32(&sm.ds_ready), c & 1, abort_flag, hdr))) break;
                    tc_fence_after();
                    // dK += dS^T Q_i, 64 columns of Q per chunk (A = dS^T, K-major)
                    for (int cc = 0; cc < C && ok;) {
                        const int n = acc_chunks(cc, [&](uint32_t col, uint32_t a, bool n128) {
                            const uint64_t da = make_sdesc_here(dsaddr, 16, 1024);
                            const uint64_t db = make_sdesc_here(a, 16384, 1024);
#pragma unroll
                            for (int kk = 0; kk < kTile / 16; ++kk)
                                mma_ss(tmem + col, sdesc_add(da, (kk >> 2) * 16384 + (kk & 3) * 32),
                                       sdesc_add(db, kk * 2048), n128 ? idN2 : idN,
                                       (s > 0 || kk > 0) ? 1u : 0u);
                        });
                        ok = n > 0;
                        cc += n;
                    }
                    if (!ok) break;
                    // dQ = dS K_j into [0, D): S^T and dP^T have been read
                    {
                        const uint64_t da = make_sdesc_here(dsaddr, 16384, 1024);
                        const uint64_t db = make_sdesc_here(kaddr, 16384, 1024);
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ss(tmem, sdesc_add(da, kk * 2048), sdesc_add(db, kk * 2048), idDQ,
                                   kk > 0);
                    }
                    mma_commit(smem_u32(&sm.dq_full));
                    if (!(ok = expect(pend_s[0], smem_u32(&sm.dq_free[0]), c & 1))) break;
                    ok = expect(pend_s[1], smem_u32(&sm.dq_free[1]), c & 1);
                }
                if (!ok) break;
                c2 += x.ns;
                if (x.ns > 0) mma_commit(smem_u32(&sm.dk_full));
                mma_commit(smem_u32(&sm.kv_empty));  // K and V read by every MMA issued
            }
            // never leave an MMA in flight
            mma_commit(smem_u32(&sm.drain));
            mbar_wait(smem_u32(&sm.drain), 0, &sm.zero);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ compute
        const int ct = threadIdx.x - 128;  // key row (P, dS, epilogue) / query row (merge)
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const bool leader = ct == 0;
        int sched_it = 0, acc_it = 0, c1 = 0, c2 = 0, rs = 0;  // rs: staged row sets
        // acc_it: units with query tiles (the ones whose dV / dK the MMAs signal)
        bool ok = true;
        while (ok) {
            const int slot = sched_it & 1;
            if (!(ok = wg_wait(smem_u32(&sm.sched_full[slot]), (sched_it >> 1) & 1, abort_flag, hdr)))
                break;
            const int2 unit = sm.sched[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.sched_empty[slot]));
            ++sched_it;
            if (unit.x < 0) break;
            const BUnit x = decode_bunit<KV, false>(unit, p);
            const int h = x.h0;
            const int c = x.j * kTile + ct;  // this thread's key row within its sequence
            const int c_off = c - x.off;
            const int L_vis = c < x.Lk ? x.L : 0;
            auto visible = [&](int i, int& lo, int& hi) {
                if constexpr (KV) {
                    lo = p.causal ? max(0, c_off - i * kTile) : 0;
                    hi = min(kTile, L_vis - i * kTile);
                } else {
                    lo = p.causal ? max(0, c - i * kTile) : 0;
                    hi = c < x.L ? min(kTile, x.L - i * kTile) : 0;
                }
            };
            // LSE (base 2) and D of this thread's query row of tile i
            auto fetch_rows = [&](int i, float& l2, float& dv) {
                const int q = i * kTile + ct;
                l2 = 0.f;
                dv = 0.f;
                if (q < x.L) {
                    const size_t at = (size_t)h * p.T + (size_t)(x.t0 + q);
                    l2 = p.lse[at] * kLog2e;
                    dv = p.D[at];
                }
            };
            // dV (pass 1) or dK times scale (pass 2) of this key row, from TMEM
            auto epilogue = [&](int pass) {
                const bool valid = c < x.Lk;
                const size_t tok = (size_t)x.tk0 + (size_t)c;
                const bool none = x.ns == 0;  // (KV) no query sees the tile: zeros, TMEM not read
                const float mul = pass == 0 ? 1.f : p.scale;
                const bool partial = p.nchunks > 1;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t v[32];
                    if (none) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;
                    } else {
                        tmem_ld32(tmem + lane_off + kColDKV + cc * 32, v);
                        tmem_ld_wait();
                    }
                    if (!valid) continue;
                    if (partial) {
                        float* acc = (pass == 0 ? dv_acc : dk_acc) +
                                     (tok * (size_t)(p.Hkv * p.nchunks) + x.uh) * D + cc * 32;
                        float4* d4 = reinterpret_cast<float4*>(acc);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            d4[e] = make_float4(__uint_as_float(v[4 * e]) * mul,
                                                __uint_as_float(v[4 * e + 1]) * mul,
                                                __uint_as_float(v[4 * e + 2]) * mul,
                                                __uint_as_float(v[4 * e + 3]) * mul);
                    } else if (p.grad_fp32) {
                        float* out = static_cast<float*>(pass == 0 ? p.dv : p.dk) +
                                     (tok * p.Hkv + x.g) * D + cc * 32;
                        float4* d4 = reinterpret_cast<float4*>(out);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            d4[e] = make_float4(__uint_as_float(v[4 * e]) * mul,
                                                __uint_as_float(v[4 * e + 1]) * mul,
                                                __uint_as_float(v[4 * e + 2]) * mul,
                                                __uint_as_float(v[4 * e + 3]) * mul);
                    } else {
                        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(pass == 0 ? p.dv : p.dk) +
                                             (tok * p.Hkv + x.g) * D + cc * 32;
                        uint4* d4 = reinterpret_cast<uint4*>(out);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            d4[e] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * e]) * mul,
                                                           __uint_as_float(v[8 * e + 1]) * mul),
                                               pack_bf16x2(__uint_as_float(v[8 * e + 2]) * mul,
                                                           __uint_as_float(v[8 * e + 3]) * mul),
                                               pack_bf16x2(__uint_as_float(v[8 * e + 4]) * mul,
                                                           __uint_as_float(v[8 * e + 5]) * mul),
                                               pack_bf16x2(__uint_as_float(v[8 * e + 6]) * mul,
                                                           __uint_as_float(v[8 * e + 7]) * mul));
                    }
                }
                tc_fence_before();  // (the next arrival orders these reads before dK / dV)
            };

            const uint64_t cc2 = f2_pack(p.scale_log2, p.scale_log2);
            for (int pass = 0; pass < 2 && ok; ++pass) {
                float nl2 = 0.f, ndd = 0.f;
                if (x.ns > 0) fetch_rows(walk_tile<KV>(x, 0, p.deterministic, p.causal), nl2, ndd);
                for (int s = 0; s < x.ns; ++s) {
                    const int i = walk_tile<KV>(x, s, p.deterministic, p.causal);
                    const int rb = rs++ & 1;  // row buffer: its readers of two steps ago are past
                    sm.lse2[rb][ct] = -nl2;   // the named barrier of the previous step
                    sm.dd[rb][ct] = -ndd;
                    // (the wait's block-wide vote also publishes the rows)
                    const uint32_t full_bar =
                        pass == 0 ? smem_u32(&sm.s_full[(c1 + s) & 1]) : smem_u32(&sm.sdp_full);
                    const uint32_t full_par = pass == 0 ? ((c1 + s) >> 1) & 1 : (c2 + s) & 1;
                    if (!(ok = wg_wait(full_bar, full_par, abort_flag, hdr))) break;
                    tc_fence_after();
                    if (s + 1 < x.ns)
                        fetch_rows(walk_tile<KV>(x, s + 1, p.deterministic, p.causal), nl2, ndd);
                    int lo, hi;
                    visible(i, lo, hi);
                    const bool full = lo == 0 && hi == kTile;
                    if (pass == 0) {
                        // P^T of this key row, bf16, packed over the first 32 columns of
                        // each 64-column half of the S^T buffer (query columns
                        // [64h + 16m, +16) in TMEM columns [64h + 8m, +8)): the A operand of dV
                        const int b = (c1 + s) & 1;
                        const uint32_t sb = tmem + lane_off + (uint32_t)b * 128;
                        uint32_t sv[4][32];
#pragma unroll
                        for (int qc = 0; qc < 4; ++qc) tmem_ld32(sb + qc * 32, sv[qc]);
                        tmem_ld_wait();
#pragma unroll
                        for (int qc = 0; qc < 4; ++qc) {
                            uint32_t pk[16];
                            if (full)
                                p_chunk<false>(sv[qc], sm.lse2[rb] + qc * 32, cc2, lo, hi, qc * 32, pk);
                            else
                                p_chunk<true>(sv[qc], sm.lse2[rb] + qc * 32, cc2, lo, hi, qc * 32, pk);
                            tmem_st16(sb + (qc >> 1) * 64 + (qc & 1) * 16, pk);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&sm.p_ready[b]));
                        continue;
                    }
                    // pass 2: dS^T = P^T (dP^T - D), bf16, swizzled rows of the dS^T tile
                    // (the previous step's dK, dQ and merge staging are done with it)
                    uint8_t* ds_row = sm.ds + ct * 128;
                    const int sw = ct & 7;
#pragma unroll 1
                    for (int qc = 0; qc < 4; ++qc) {
                        uint32_t sv[32], dv[32];
                        tmem_ld32(tmem + lane_off + qc * 32, sv);
                        tmem_ld32(tmem + lane_off + 128 + qc * 32, dv);
                        tmem_ld_wait();
                        uint32_t pk[16];
                        if (full)
                            p_chunk<false>(sv, sm.lse2[rb] + qc * 32, cc2, lo, hi, qc * 32, pk);
                        else
                            p_chunk<true>(sv, sm.lse2[rb] + qc * 32, cc2, lo, hi, qc * 32, pk);
                        uint32_t out[16];
                        const uint64_t* nd = reinterpret_cast<const uint64_t*>(sm.dd[rb] + qc * 32);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const uint64_t pf = f2_pack(__uint_as_float(pk[e] << 16),
                                                        __uint_as_float(pk[e] & 0xffff0000u));
                            const uint64_t t = f2_add(
                                f2_pack(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), nd[e]);
                            float d0, d1;
                            f2_unpack(f2_mul(t, pf), d0, d1);
                            out[e] = pack_bf16x2(d0, d1);
                        }
                        // 32 query columns = 4 chunks of 16 bytes of half (qc >> 1)'s block
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int ch = (qc & 1) * 4 + e;
                            *reinterpret_cast<uint4*>(ds_row + (qc >> 1) * 16384 + ((ch ^ sw) << 4)) =
                                make_uint4(out[4 * e], out[4 * e + 1], out[4 * e + 2], out[4 * e + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sm.ds_ready));
                    // dQ of the step (dK of it issued before)
                    if (!(ok = wg_wait(smem_u32(&sm.dq_full), (c2 + s) & 1, abort_flag, hdr))) break;
                    tc_fence_after();
                    int* sem = nullptr;
                    bool sem_ok = true;
                    if (p.deterministic) {
                        sem = sems + (size_t)h * n_qtiles + tile_off[x.b] + i;
                        if (leader && !sem_wait(sem, dq_rank<KV>(x, i, p.causal), hdr)) {
                            raise_abort(abort_flag, hdr, kErrTimeout);
                            sem_ok = false;
                        }
                    }
                    if (!(ok = named_bar_and(1, 128, sem_ok && *abort_flag == 0))) break;
                    // dQ merge: this thread's query row of tile i.  The columns [0, 128)
                    // are released once read (the next S^T), the rest at the end (dP^T).
                    const int row0 = i * kTile;
                    const int qr = row0 + ct;
                    auto release_half = [&](int cc) {
                        if (cc == 3 || cc == D / 32 - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(smem_u32(&sm.dq_free[cc == 3 ? 0 : 1]));
                        }
                    };
                    if (row0 + kTile <= x.L) {
                        // whole tile: bulk tensor reduce-adds of 32 columns, staged
                        // 128B-swizzled through the dS buffer (dK and dQ have read it)
                        uint8_t* stage_row = sm.ds + ct * 128;
#pragma unroll 1
                        for (int cc = 0; cc < D / 32; ++cc) {
                            const int sl = cc & 1;
                            uint32_t v[32];
                            tmem_ld32(tmem + lane_off + cc * 32, v);
                            tmem_ld_wait();
                            release_half(cc);
                            if (leader && cc >= 2) bulk_wait_group_read<1>();  // the slot's last reduce read it
                            named_bar_sync(1, 128);
                            uint8_t* row = stage_row + sl * (kTile * 128);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                *reinterpret_cast<uint4*>(row + ((e ^ sw) << 4)) =
                                    make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                            fence_proxy_async_smem();
                            named_bar_sync(1, 128);
                            if (leader) {
                                tma_reduce_add_3d(&p.tm_dq_acc, dsaddr + sl * (kTile * 128), cc * 32, h,
                                                  x.t0 + row0);
                                bulk_commit_group();
                            }
                        }
                        // the next step writes dS^T over the staging: its reduces must
                        // have read it (the next step's wait publishes this)
                        if (leader) {
                            if (p.deterministic) {
                                bulk_wait_group<0>();
                                fence_proxy_async_global();
                            } else {
                                bulk_wait_group_read<0>();
                            }
                        }
                    } else {
                        // ragged last tile of a sequence: per-row vector reductions
                        float* dst = dq_acc + ((size_t)(x.t0 + qr) * p.Hq + h) * D;
#pragma unroll 1
                        for (int cc = 0; cc < D / 32; ++cc) {
                            uint32_t v[32];
                            tmem_ld32(tmem + lane_off + cc * 32, v);
                            tmem_ld_wait();
                            release_half(cc);
                            if (qr < x.L) {
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    red_add_v4(dst + cc * 32 + 4 * e, __uint_as_float(v[4 * e]),
                                               __uint_as_float(v[4 * e + 1]), __uint_as_float(v[4 * e + 2]),
                                               __uint_as_float(v[4 * e + 3]));
                            }
                        }
                    }
                    if (p.deterministic) {
                        __threadfence();  // this contribution before the next one
                        named_bar_sync(1, 128);
                        if (leader) red_release_gpu_add(sem, 1);
                    }
                }
                if (!ok) break;
                if (pass == 0) c1 += x.ns; else c2 += x.ns;
                // the pass's accumulator: dV after pass 1, dK after pass 2
                if (x.ns > 0) {
                    if (!(ok = wg_wait(smem_u32(pass == 0 ? &sm.dv_full : &sm.dk_full), acc_it & 1,
                                       abort_flag, hdr)))
                        break;
                    tc_fence_after();
                }
                epilogue(pass);
            }
            if (x.ns > 0) ++acc_it;
        }
        // the staging slots must not be read after the CTA exits
        if (leader) bulk_wait_group<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// D = rowsum(dO * O) per (token, head); zero the dQ accumulator row and the
// semaphores.  Each lane takes 8 elements (16-byte loads), D/8 lanes per row,
// so a warp covers 32/(D/8) rows per grid stride; it takes two strides per
// pass, with the loads of both in flight before either is used (the kernel is
// bound by HBM, and more bytes in flight per SM bring it closer).
template <int D, bool O_FP32>  // D: the head dimension in memory (64, 96 or 128)
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const void* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                          float* __restrict__ Dout, float* __restrict__ dq_acc,
                          int* __restrict__ sems, long long n_sems, int T, int Hq) {
    pdl_begin();
    // lanes per row (a power of two; lanes past the row idle at D = 96 and 192)
    constexpr int LPR = D == 96 ? 16 : (D == 192 ? 32 : D / 8);
    constexpr int RPW = 32 / LPR;  // rows per warp pass
    const long long rows = (long long)T * Hq;
    const long long warp_g = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, l = lane % LPR;
    // two rows per lane and pass, both rows' loads issued before either is used
    for (long long r0 = warp_g * RPW; r0 < rows; r0 += 2 * nwarps * RPW) {
        long long r[2];
        bool valid[2];
        uint4 dv[2], ow[2];
        float4 fa[2], fb[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            r[u] = r0 + (long long)u * nwarps * RPW + sub;
            valid[u] = r[u] < rows && l * 8 < D;
            if (valid[u]) {
                const size_t base = (size_t)r[u] * D + (size_t)l * 8;
                dv[u] = *reinterpret_cast<const uint4*>(dout + base);
                if (O_FP32) {
                    fa[u] = *reinterpret_cast<const float4*>(static_cast<const float*>(o) + base);
                    fb[u] = *reinterpret_cast<const float4*>(static_cast<const float*>(o) + base + 4);
                } else {
                    ow[u] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(o) + base);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float acc = 0.f;
            if (valid[u]) {
                const size_t base = (size_t)r[u] * D + (size_t)l * 8;
                const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv[u]);
                float ov[8];
                if (O_FP32) {
                    ov[0] = fa[u].x; ov[1] = fa[u].y; ov[2] = fa[u].z; ov[3] = fa[u].w;
                    ov[4] = fb[u].x; ov[5] = fb[u].y; ov[6] = fb[u].z; ov[7] = fb[u].w;
                } else {
                    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ow[u]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(o2[e]);
                        ov[2 * e] = f.x;
                        ov[2 * e + 1] = f.y;
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(d2[e]);
                    acc = fmaf(ov[2 * e], f.x, acc);
                    acc = fmaf(ov[2 * e + 1], f.y, acc);
                }
                float4* z = reinterpret_cast<float4*>(dq_acc + base);
                z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (valid[u] && l == 0) Dout[(size_t)(r[u] % Hq) * T + (size_t)(r[u] / Hq)] = acc;
        }
    }
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (long long si = tid; si < n_sems; si += (long long)gridDim.x * blockDim.x) sems[si] = 0;
}

// dq = scale * dq_acc; when the query heads of a key/value head are split over
// several runs, dk/dv[t,g] = sum over the runs (in increasing order) of their
// fp32 partials [t, g * nruns + run].  One flat index space of float4 groups:
// [0, nq) dq, [nq, nq+nkv) dk, [nq+nkv, nq+2nkv) dv.
template <int D, bool F32>
__global__ void __launch_bounds__(256)
    bwd_postprocess_kernel(const float* __restrict__ dq_acc, void* __restrict__ dq,
                           const float* __restrict__ dk_acc, const float* __restrict__ dv_acc,
                           void* __restrict__ dk, void* __restrict__ dv, int Tq, int Tk, int Hq,
                           int Hkv, int nruns, float scale) {
    pdl_begin();
    constexpr int V = D / 4;  // float4 groups per row
    const long long nq = (long long)Tq * Hq * V;
    const long long nkv = dk_acc ? (long long)Tk * Hkv * V : 0;
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    // dQ, four groups per thread and pass, all four loads issued first
    for (; e + 3 * stride < nq; e += 4 * stride) {
        float4 a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = reinterpret_cast<const float4*>(dq_acc)[e + u * stride];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float4 r = make_float4(a[u].x * scale, a[u].y * scale, a[u].z * scale, a[u].w * scale);
            if (F32)
                reinterpret_cast<float4*>(dq)[e + u * stride] = r;
            else
                reinterpret_cast<uint2*>(dq)[e + u * stride] =
                    make_uint2(pack_bf16x2(r.x, r.y), pack_bf16x2(r.z, r.w));
        }
    }
    for (; e < nq + 2 * nkv; e += stride) {
        float4 r;
        void* out;
        long long oi;
        if (e < nq) {
            const float4 a = reinterpret_cast<const float4*>(dq_acc)[e];
            r = make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale);
            out = dq;
            oi = e;
        } else {
            const bool is_v = e >= nq + nkv;
            oi = e - nq - (is_v ? nkv : 0);
            const long long row = oi / V;  // (t, g)
            const int c4 = (int)(oi % V);
            const long long t = row / Hkv;
            const int g = (int)(row % Hkv);
            const float4* src = reinterpret_cast<const float4*>(is_v ? dv_acc : dk_acc);
            r = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int u = 0; u < nruns; ++u) {
                const float4 a = src[(t * ((long long)Hkv * nruns) + (long long)g * nruns + u) * V + c4];
                r.x += a.x; r.y += a.y; r.z += a.z; r.w += a.w;
            }
            out = is_v ? dv : dk;
        }
        if (F32) {
            reinterpret_cast<float4*>(out)[oi] = r;
        } else {
            reinterpret_cast<uint2*>(out)[oi] =
                make_uint2(pack_bf16x2(r.x, r.y), pack_bf16x2(r.z, r.w));
        }
    }
}

int grid_for(long long work, int threads, int num_sms) {
    long long g = (work + threads - 1) / threads;
    const long long cap = (long long)num_sms * 8;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

template <int D>
cudaError_t launch_bwd_wide_t(const BwdParams& p, int num_sms, cudaStream_t stream) {
    auto kern = p.kv ? fa_bwd_wide_kernel<D, true> : fa_bwd_wide_kernel<D, false>;
    const size_t smem = sizeof(WideSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long bound = max_tiles(p.B, p.Tk, kTile) * (long long)p.Hkv * p.nchunks;
    const int grid = (int)(bound < num_sms ? bound : num_sms);
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(kern, dim3(grid), dim3(kWideThreads), smem, stream, p);
}

template <int D, int DR>
cudaError_t launch_bwd_t(const BwdParams& p, int num_sms, cudaStream_t stream) {
    auto kern = p.kv ? (p.hchunk > 1 ? fa_bwd_kernel<D, DR, true, true>
                                     : fa_bwd_kernel<D, DR, true, false>)
                     : (p.hchunk > 1 ? fa_bwd_kernel<D, DR, false, true>
                                     : fa_bwd_kernel<D, DR, false, false>);
    const size_t smem = sizeof(BwdSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // units are (key/value tile, run of query heads)
    const long long bound = max_tiles(p.B, p.Tk, kTile) * (long long)p.Hkv * p.nchunks;
    const int grid = (int)(bound < num_sms ? bound : num_sms);
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(kern, dim3(grid), dim3(kBwdThreads), smem, stream, p);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, int o_fp32, const void* dout, float* D,
                                  float* dq_acc, int* sems, long long n_sems, int T, int Hq,
                                  int d, int num_sms, cudaStream_t stream) {
    const long long rows = (long long)T * Hq;
    const long long threads = rows * (d / 8) > n_sems ? rows * (d / 8) : n_sems;
    const int grid = grid_for(threads, 256, num_sms);
    const __nv_bfloat16* dob = static_cast<const __nv_bfloat16*>(dout);
    cudaError_t e;
#define FA_PRE(DD, FF)                                                                  \
    e = launch_pdl(bwd_preprocess_kernel<DD, FF>, dim3(grid), dim3(256), 0, stream, o, dob, D, \
                   dq_acc, sems, n_sems, T, Hq)
    if (d == 128) {
        if (o_fp32) FA_PRE(128, true); else FA_PRE(128, false);
    } else if (d == 256) {
        if (o_fp32) FA_PRE(256, true); else FA_PRE(256, false);
    } else if (d == 192) {
        if (o_fp32) FA_PRE(192, true); else FA_PRE(192, false);
    } else if (d == 96) {
        if (o_fp32) FA_PRE(96, true); else FA_PRE(96, false);
    } else {
        if (o_fp32) FA_PRE(64, true); else FA_PRE(64, false);
    }
#undef FA_PRE
    return e;
}

cudaError_t launch_bwd(const BwdParams& p, int num_sms, cudaStream_t stream) {
    if (p.d == 256) return launch_bwd_wide_t<256>(p, num_sms, stream);
    if (p.d == 192) return launch_bwd_wide_t<192>(p, num_sms, stream);
    if (p.d == 128) return launch_bwd_t<128, 128>(p, num_sms, stream);
    if (p.d == 96) return launch_bwd_t<128, 96>(p, num_sms, stream);
    return launch_bwd_t<64, 64>(p, num_sms, stream);
}

cudaError_t launch_bwd_postprocess(const float* dq_acc, void* dq, const float* dk_acc,
                                   const float* dv_acc, void* dk, void* dv, int Tq, int Tk,
                                   int Hq, int Hkv, int nruns, int d, float scale, int grad_fp32,
                                   int num_sms, cudaStream_t stream) {
    const long long work = ((long long)Tq * Hq + (dk_acc ? 2LL * Tk * Hkv : 0)) * d / 4;
    const int grid = grid_for(work, 256, num_sms);
    cudaError_t e;
#define FA_POST(DD, FF)                                                                   \
    e = launch_pdl(bwd_postprocess_kernel<DD, FF>, dim3(grid), dim3(256), 0, stream, dq_acc, dq, \
                   dk_acc, dv_acc, dk, dv, Tq, Tk, Hq, Hkv, nruns, scale)
    if (d == 128) {
        if (grad_fp32) FA_POST(128, true); else FA_POST(128, false);
    } else if (d == 256) {
        if (grad_fp32) FA_POST(256, true); else FA_POST(256, false);
    } else if (d == 192) {
        if (grad_fp32) FA_POST(192, true); else FA_POST(192, false);
    } else if (d == 96) {
        if (grad_fp32) FA_POST(96, true); else FA_POST(96, false);
    } else {
        if (grad_fp32) FA_POST(64, true); else FA_POST(64, false);
    }
#undef FA_POST
    return e;
}

}  // namespace fa
