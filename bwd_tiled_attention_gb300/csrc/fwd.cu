// fwd.cu -- tiled exact-attention forward for sm_103a.
//
// Method ("FlashAttention-2-ICLR24", 核心方法 1 and 2): each work unit is a
// block of query rows of one (sequence, head); an inner loop walks the
// key/value tiles, keeping a running row max m and row sum l, an unnormalised
// output O~ that is rescaled when m grows, and one division by l at the end;
// only LSE = m + log l is stored.  Key/value tiles entirely above the causal
// diagonal are never visited; only tiles that straddle it (or the ragged end
// of a sequence) are masked.  Queries and keys may differ in length: the
// queries are then the last positions of the key sequence (query row r sees
// key c iff c <= r + Lk - Lq under the causal mask), and a row that sees no
// key gets O = 0 and LSE = -inf.
//
// Blackwell design ("FlashAttention-4 wird offiziell veröffentlicht", section
// "Neue Hardwaremerkmale von Blackwell": single-thread tcgen05.mma accumulating
// in tensor memory, A operand readable from tensor memory, warp specialisation):
//   warp 0       TMA producer: both query tiles of a unit once, then a ring of
//                key and value tiles (128-byte swizzled, one box per 64 columns)
//   warp 1       MMA issuer: S_t = Q_t K^T into TMEM, then O_t += P_t V with P_t
//                read from TMEM
//   warp 2       TMEM allocation
//   warps 4..7   softmax for query tile 0 (one thread per row)
//   warps 8..11  softmax for query tile 1 (above d = 128: the epilogue)
// A unit covers 256 query rows (two 128-row tiles) so each K/V tile loaded
// feeds two MMAs, and the tensor core works on one tile while the softmax
// warps of the other tile run.  TMEM: S_0 [0,128), S_1 [128,256), O_0
// [256,256+d), O_1 [384,384+d); P_t is written as bf16 over the first 64
// columns of S_t, in two halves (keys [0, 64), then [64, 128)), each handed
// to the MMA issuer on its own, so PV_t starts on the first half while the
// softmax computes the second.  Head dimensions above 128 leave room for one query tile
// (O takes [256,256+d)); its S is then double-buffered over [0,256): S(j+1)
// is issued before O += P(j) V, so the tensor core computes the next scores
// while the softmax warps work on the current ones, and warps 8..11 store O.
// At d = 192, P has the last 64 columns to itself.
//
// Softmax uses exp2 with the scale folded in (s * scale * log2 e), packed
// fp32-pair arithmetic for the scale and the row sum, and 3-input maxima.  All
// exponentials go to the SFU (ex2): the FlashAttention-4 page (section "Die
// Kernidee des kooperativen Designs") moves part of them to a polynomial on the
// FMA units, but on this part that made the forward slower, not faster.  The O~
// rescale is conditional: the reference max is only moved when the row max
// grows by more than 8 (a factor 256 in P), which keeps P in range while
// skipping most rescales; the result is exact because l and O~ always share
// the same reference.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace fa {
namespace {

constexpr int kFwdThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// D = 192 and 256: one query tile per unit, since the S and O columns of two
// tiles (2 x 128 + 2 x D) exceed TMEM's 512, and one K stage, since Q, K and V
// tiles are 48 or 64 KB each.  V has a ring of its own in the room left: V(j)
// is split into chunks of kVChunk columns (PV runs per chunk, N = kVChunk),
// over kVSlots slots -- d = 256: halves of 128 columns in 3 slots of 32 KB;
// d = 192: whole tiles in 2 slots of 48 KB.  Up to 128 the V ring is the K/V
// ring: kStages slots of whole tiles.
template <int D>
struct FwdCfg {
    static constexpr int kStages = D > 128 ? 1 : (D == 128 ? 2 : 4);
    static constexpr int kQTiles = D > 128 ? 1 : 2;    // query tiles per unit
    static constexpr int kUnitRows = kQTiles * kTile;  // query rows per unit
    static constexpr int kTileBytes = kTile * D * 2;   // one 128-row bf16 tile
    static constexpr int kBoxes = D / 64;              // 64-column TMA boxes per tile
    static constexpr int kVChunk = D == 256 ? 128 : D;                   // V columns per chunk
    static constexpr int kVChunks = D / kVChunk;                         // chunks per V tile
    static constexpr int kVSlots = D == 256 ? 3 : (D > 128 ? 2 : kStages);
    static constexpr int kVSlotBytes = kTile * kVChunk * 2;
    // d = 192 leaves 64 TMEM columns past O: P gets them to itself instead of
    // being written over its S buffer, so the next S need not wait for PV.
    static constexpr bool kSepP = D > 128 && 256 + D + 64 <= 512;
    static constexpr int kPCol = 256 + D;  // first column of P when kSepP
    static_assert(kVChunks * kVChunk == D && kVChunk % 64 == 0, "V chunks must tile the row");
    static_assert(!kSepP || kPCol + 64 <= 512, "P past the TMEM columns");
};

template <int D>
struct FwdSmem {
    alignas(1024) uint8_t q[FwdCfg<D>::kQTiles][FwdCfg<D>::kTileBytes];
    alignas(1024) uint8_t k[FwdCfg<D>::kStages][FwdCfg<D>::kTileBytes];
    alignas(1024) uint8_t v[FwdCfg<D>::kVSlots][FwdCfg<D>::kVSlotBytes];
    alignas(8) uint64_t sched_full[2], sched_empty[2];
    uint64_t q_full, q_empty;
    uint64_t k_full[FwdCfg<D>::kStages], v_full[FwdCfg<D>::kVSlots], kv_empty[FwdCfg<D>::kStages];
    // D > 128: K is released box by box (a 64-column box once the S MMAs that
    // read it are done), the V slots one by one
    uint64_t k_empty[D > 128 ? FwdCfg<D>::kBoxes : 1], v_empty[D > 128 ? FwdCfg<D>::kVSlots : 1];
    uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
    // P in two halves, keys [0, 64) (p_full) and [64, 128) (p_hi), so PV's
    // first four MMAs run while the softmax computes the second half
    uint64_t p_hi[2];
    uint64_t drain;
    int2 sched[2];
    uint32_t tmem_base;
    int abort_flag;
    int zero;
    // D > 128: the last unit's row statistics, from the softmax warps to the
    // epilogue warps
    float ep_m[D > 128 ? kTile : 1], ep_l[D > 128 ? kTile : 1];
    uint64_t ep_full;
};

// (the kernel aligns the dynamic shared memory to 1024 bytes itself)
static_assert(sizeof(FwdSmem<64>) + 1024 <= 232448, "forward shared memory exceeds 227 KB");
static_assert(sizeof(FwdSmem<128>) + 1024 <= 232448, "forward shared memory exceeds 227 KB");
static_assert(sizeof(FwdSmem<192>) + 1024 <= 232448, "forward shared memory exceeds 227 KB");
static_assert(sizeof(FwdSmem<256>) + 1024 <= 232448, "forward shared memory exceeds 227 KB");

// One work unit: query rows [Rm, Rm + R) of sequence b, head h (R = 256, or
// 128 when D > 128).  t0/L
// are the query tokens, tk0/Lk the key/value tokens; under the causal mask
// query row r sees key c iff c <= r + Lk - L.  n[t] = key/value tiles query
// tile t visits (0 when the tile is past the end, or sees no key at all).
struct UnitGeom {
    int b, m, h, g, t0, L, tk0, Lk, n[2], nkv;  // nkv >= 1 (see decode_unit)
};

// KV = false: keys and queries share their boundaries (Lk = L, tk0 = t0), and
// the geometry is the plain square one.
template <int D, bool KV>
__device__ __forceinline__ UnitGeom decode_unit(int2 u, const FwdParams& p) {
    UnitGeom x;
    x.b = u.x;
    x.m = unit_tile(u.y);
    x.h = unit_head(u.y);
    x.g = (int)(((long long)x.h * p.Hkv) / p.Hq);
    seq_bounds(p.cu_seqlens, p.N, x.b, x.t0, x.L);
    if constexpr (KV) {
        seq_bounds(p.cu_seqlens_k, p.Nk, x.b, x.tk0, x.Lk);
    } else {
        x.tk0 = x.t0;
        x.Lk = x.L;
    }
    const int r0 = x.m * FwdCfg<D>::kUnitRows;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int rs = r0 + t * kTile;  // first row of tile t
        if (t >= FwdCfg<D>::kQTiles || rs >= x.L) {
            x.n[t] = 0;
        } else if (p.causal) {
            const int re = min(rs + kTile, x.L);  // one past last valid row
            x.n[t] = KV ? cdiv(max(re + x.Lk - x.L, 0), kTile) : cdiv(re, kTile);
        } else {
            x.n[t] = cdiv(x.Lk, kTile);
        }
    }
    // A unit whose rows see no key (KV only) still takes one key/value step
    // with both query tiles masked off (no MMA issued): the producer and MMA
    // thread then keep their usual barrier sequence, and the softmax warps
    // write O = 0.
    x.nkv = KV ? max(max(x.n[0], x.n[1]), 1) : max(x.n[0], x.n[1]);
    return x;
}

// P = 2^(s * c - m) for one 32-column chunk of a row, packed to bf16 pairs, and
// its fp32 row sum accumulated in two packed accumulators.  Masked columns hold
// s = -inf, which ex2 takes to exactly 0.
__device__ __forceinline__ void softmax_chunk(const float* sc, float c, float neg,
                                              uint64_t (&acc)[2], uint32_t (&pk)[16]) {
    const uint64_t c2 = f2_pack(c, c), n2 = f2_pack(neg, neg);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint64_t x = f2_fma(f2_pack(sc[2 * i], sc[2 * i + 1]), c2, n2);
        float x0, x1;
        f2_unpack(x, x0, x1);
        const uint64_t e = f2_pack(ex2_approx(x0), ex2_approx(x1));
        acc[i & 1] = f2_add(acc[i & 1], e);
        float p0, p1;
        f2_unpack(e, p0, p1);
        pk[i] = pack_bf16x2(p0, p1);
    }
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

// A query row that sees no key: O = 0, LSE = -inf.
template <int DR, bool OUT_FP32>
__device__ __forceinline__ void write_keyless_row(const FwdParams& p, int h, size_t tok) {
    p.lse[(size_t)h * p.T + tok] = -INFINITY;
    const size_t base = (tok * p.Hq + h) * DR;
    if (OUT_FP32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + base);
        for (int i = 0; i < DR / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + base);
        for (int i = 0; i < DR / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Epilogue of one row: O = O~ / l and LSE = (m + log2 l) * ln 2, O~ read from
// TMEM columns [o_addr, o_addr + DR).  Only a valid row is stored; every thread
// of the warp takes part in the TMEM loads.
template <int DR, bool OUT_FP32, bool KV>
__device__ __forceinline__ void store_row(const FwdParams& p, uint32_t o_addr, int h, size_t tok,
                                          bool valid, float m_ref, float l) {
    // l = 0 only for a KV row that sees no key
    const float inv_l = KV ? (l > 0.f ? 1.f / l : 0.f) : 1.f / l;
    if (valid) p.lse[(size_t)h * p.T + tok] = (m_ref + __log2f(l)) * 0.69314718055994531f;
#pragma unroll 1
    for (int c = 0; c < DR / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_addr + c * 32, ov);
        tmem_ld_wait();
        if (valid) {
            const size_t base = (tok * p.Hq + h) * DR + c * 32;
            if (OUT_FP32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + base);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_float4(__uint_as_float(ov[4 * i]) * inv_l,
                                         __uint_as_float(ov[4 * i + 1]) * inv_l,
                                         __uint_as_float(ov[4 * i + 2]) * inv_l,
                                         __uint_as_float(ov[4 * i + 3]) * inv_l);
            } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + base);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(pack_bf16x2(__uint_as_float(ov[8 * i]) * inv_l,
                                                    __uint_as_float(ov[8 * i + 1]) * inv_l),
                                        pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv_l,
                                                    __uint_as_float(ov[8 * i + 3]) * inv_l),
                                        pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv_l,
                                                    __uint_as_float(ov[8 * i + 5]) * inv_l),
                                        pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv_l,
                                                    __uint_as_float(ov[8 * i + 7]) * inv_l));
            }
        }
    }
}

// D: the tile layout (64, 128, 192 or 256 columns); DR: the head dimension in
// memory.
// DR = 96 runs on 128-column tiles: the TMA boxes past column 96 read zeros.
// S contracts over the first 96 columns only (6 MMAs of K = 16); PV keeps
// N = 128 (V is read MN-major in 64-column swizzle atoms), and O's last 32
// columns (all zero) are not stored.
template <int D, int DR, bool OUT_FP32, bool KV>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    pdl_trigger();
    using Cfg = FwdCfg<D>;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.workspace);
    const int2* units =
        reinterpret_cast<const int2*>(static_cast<const char*>(p.workspace) + p.units_off);
    const int warp = warp_id(), lane = lane_id();
    volatile int* abort_flag = &sm.abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.sched_full[i]), 1);
            mbar_init(smem_u32(&sm.sched_empty[i]), 1 + 8);
            mbar_init(smem_u32(&sm.s_full[i]), 1);
            mbar_init(smem_u32(&sm.p_full[i]), 4);
            mbar_init(smem_u32(&sm.p_hi[i]), 4);
            mbar_init(smem_u32(&sm.o_done[i]), 1);
            mbar_init(smem_u32(&sm.o_free[i]), 4);
        }
        mbar_init(smem_u32(&sm.q_full), 1);
        mbar_init(smem_u32(&sm.q_empty), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&sm.k_full[s]), 1);
            mbar_init(smem_u32(&sm.kv_empty[s]), 1);
        }
        for (int s = 0; s < Cfg::kVSlots; ++s) mbar_init(smem_u32(&sm.v_full[s]), 1);
        if constexpr (D > 128) {
            for (int c = 0; c < Cfg::kBoxes; ++c) mbar_init(smem_u32(&sm.k_empty[c]), 1);
            for (int s = 0; s < Cfg::kVSlots; ++s) mbar_init(smem_u32(&sm.v_empty[s]), 1);
        }
        mbar_init(smem_u32(&sm.drain), 1);
        if constexpr (D > 128) mbar_init(smem_u32(&sm.ep_full), kTile);
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
    pdl_wait();  // the unit list and inputs are the previous kernels' output
    const int n_units = hdr->n_units;
    // Registers: the launch gives every thread 168 (384 x 168 = 64512).  The
    // producer/MMA warpgroup (warps 0..3) needs few, so each of its warps gives
    // back to 72 at the top of its role, and the two math warpgroups take 216
    // each: 128*72 + 256*216 = 64512 exactly.
    static_assert(128 * 72 + 256 * 216 == 384 * 168, "register split must match the launch");

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        setmaxnreg_dec<72>();
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            int sched_it = 0, kv_it = 0, unit_it = 0;
            int k_it = 0, v_it = 0;  // D > 128: K tiles and V chunks loaded
            bool ok = true;
            while (ok) {
                const int slot = sched_it & 1;
                if (!(ok = wait_or_abort(smem_u32(&sm.sched_empty[slot]),
                                         ((sched_it >> 1) & 1) ^ 1, abort_flag, hdr)))
                    break;
                const int u = atomicAdd(&hdr->counter, 1);
                const int2 unit = u < n_units ? units[u] : make_int2(-1, 0);
                sm.sched[slot] = unit;
                mbar_arrive(smem_u32(&sm.sched_full[slot]));
                ++sched_it;
                if (unit.x < 0) break;
                const UnitGeom x = decode_unit<D, KV>(unit, p);
                const int row0 = x.t0 + x.m * Cfg::kUnitRows;
                if (!(ok = wait_or_abort(smem_u32(&sm.q_empty), (unit_it & 1) ^ 1, abort_flag, hdr)))
                    break;
                // only the query tiles that see a key are loaded (none when no row of
                // the unit sees one: the barrier then completes on the arrival alone;
                // such a unit still loads one key/value tile, which nothing reads)
                const uint32_t qbar = smem_u32(&sm.q_full);
                if constexpr (KV)
                    mbar_arrive_expect_tx(qbar, ((x.n[0] > 0) + (x.n[1] > 0)) * Cfg::kTileBytes);
                else
                    mbar_arrive_expect_tx(qbar, (x.n[1] > 0 ? 2 : 1) * Cfg::kTileBytes);
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (t >= Cfg::kQTiles || x.n[t] == 0) continue;
                    for (int c = 0; c < Cfg::kBoxes; ++c)
                        tma_load_3d(smem_u32(sm.q[t]) + c * 16384, &p.tm_q, qbar, c * 64, x.h,
                                    row0 + t * kTile);
                }
                ++unit_it;
                if constexpr (D > 128) {
                    // K runs one tile ahead of V, in the order the MMA thread
                    // consumes them (S(j+1) is issued before PV(j)): iteration j
                    // loads K(j), each 64-column box as soon as S(j-1)'s MMAs over
                    // it are done (so only the last box's load follows the whole
                    // of S(j-1)), then the chunks of V(j-1), each once its slot's
                    // previous chunk has been read.
                    for (int j = 0; j <= x.nkv && ok; ++j) {
                        if (j < x.nkv) {
                            const uint32_t kb = smem_u32(&sm.k_full[0]);
                            for (int c = 0; c < Cfg::kBoxes && ok; ++c) {
                                if (!(ok = wait_or_abort(smem_u32(&sm.k_empty[c]), (k_it & 1) ^ 1,
                                                         abort_flag, hdr)))
                                    break;
                                // armed once S(j-1) has begun, so K(j-1) has landed and
                                // its phase of k_full is complete
                                if (c == 0) mbar_arrive_expect_tx(kb, Cfg::kTileBytes);
                                tma_load_3d(smem_u32(sm.k[0]) + c * 16384, &p.tm_k, kb, c * 64,
                                            x.g, x.tk0 + j * kTile);
                            }
                            if (!ok) break;
                            ++k_it;
                        }
                        for (int h = 0; j >= 1 && h < Cfg::kVChunks && ok; ++h) {
                            const int slot = v_it % Cfg::kVSlots;
                            if (!(ok = wait_or_abort(smem_u32(&sm.v_empty[slot]),
                                                     ((v_it / Cfg::kVSlots) & 1) ^ 1, abort_flag,
                                                     hdr)))
                                break;
                            const uint32_t vb = smem_u32(&sm.v_full[slot]);
                            mbar_arrive_expect_tx(vb, Cfg::kVSlotBytes);
                            for (int c = 0; c < Cfg::kVChunk / 64; ++c)
                                tma_load_3d(smem_u32(sm.v[slot]) + c * 16384, &p.tm_v, vb,
                                            h * Cfg::kVChunk + c * 64, x.g, x.tk0 + (j - 1) * kTile);
                            ++v_it;
                        }
                    }
                } else {
                    for (int j = 0; j < x.nkv && ok; ++j) {
                        const int st = kv_it % S;
                        if (!(ok = wait_or_abort(smem_u32(&sm.kv_empty[st]), ((kv_it / S) & 1) ^ 1,
                                                 abort_flag, hdr)))
                            break;
                        const uint32_t kb = smem_u32(&sm.k_full[st]), vb = smem_u32(&sm.v_full[st]);
                        mbar_arrive_expect_tx(kb, Cfg::kTileBytes);
                        for (int c = 0; c < Cfg::kBoxes; ++c)
                            tma_load_3d(smem_u32(sm.k[st]) + c * 16384, &p.tm_k, kb, c * 64, x.g,
                                        x.tk0 + j * kTile);
                        mbar_arrive_expect_tx(vb, Cfg::kTileBytes);
                        for (int c = 0; c < Cfg::kBoxes; ++c)
                            tma_load_3d(smem_u32(sm.v[st]) + c * 16384, &p.tm_v, vb, c * 64, x.g,
                                        x.tk0 + j * kTile);
                        ++kv_it;
                    }
                }
            }
            // Never leave a TMA write in flight: wait (bounded) for the last
            // phase armed on every load barrier.
            const volatile int* z = &sm.zero;
            if constexpr (D > 128) {
                if (k_it > 0) mbar_wait(smem_u32(&sm.k_full[0]), (k_it - 1) & 1, z);
                for (int i = 0; i < Cfg::kVSlots && i < v_it; ++i) {
                    const int it = v_it - 1 - i;
                    mbar_wait(smem_u32(&sm.v_full[it % Cfg::kVSlots]), (it / Cfg::kVSlots) & 1, z);
                }
            }
            for (int i = 0; i < S && i < kv_it; ++i) {
                const int it = kv_it - 1 - i, st = it % S, par = (it / S) & 1;
                mbar_wait(smem_u32(&sm.k_full[st]), par, z);
                mbar_wait(smem_u32(&sm.v_full[st]), par, z);
            }
            if (unit_it > 0) mbar_wait(smem_u32(&sm.q_full), (unit_it - 1) & 1, z);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        setmaxnreg_dec<72>();
        if (lane == 0) {
            constexpr uint32_t idS = make_idesc_bf16(128, 128, false, false);
            constexpr uint32_t idPV = make_idesc_bf16(128, Cfg::kVChunk, false, true);
            int sched_it = 0, kv_it = 0, unit_it = 0;
            int it[2] = {0, 0};   // PV MMAs issued per tile (= softmax iterations)
            int ep[2] = {0, 0};   // units whose epilogue must finish before O_t is reused
            int g = 0, k_it = 0, v_it = 0;  // D > 128: S/PV steps, K tiles and V chunks consumed
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
                const UnitGeom x = decode_unit<D, KV>(unit, p);
                if (!(ok = wait_or_abort(smem_u32(&sm.q_full), unit_it & 1, abort_flag, hdr)))
                    break;
                if constexpr (D > 128) {
                    // One query tile, S double-buffered: step g (counted over all
                    // units) computes S into columns [128 (g & 1), +128), and S(j+1)
                    // is issued before PV(j), so the tensor core computes the next
                    // scores while the softmax warps work on the current ones.
                    // Iteration j issues S(j), then PV(j-1).
                    const int n = x.n[0];
                    for (int j = 0; j <= x.nkv && ok; ++j) {
                        if (j < x.nkv) {
                            if (!(ok = wait_or_abort(smem_u32(&sm.k_full[0]), k_it & 1, abort_flag,
                                                     hdr)))
                                break;
                            if (j < n) {
                                const int gj = g + j, b = gj & 1;
                                // The buffer's last scores, S(gj - 2), were read by the
                                // softmax before PV(gj - 2) was issued; with P written
                                // over them it is free once PV(gj - 2) has read P too.
                                if (!Cfg::kSepP && gj >= 2 &&
                                    !(ok = wait_or_abort(smem_u32(&sm.o_done[b]), ((gj - 2) >> 1) & 1,
                                                         abort_flag, hdr)))
                                    break;
                                tc_fence_after();
                                const uint64_t da = make_sdesc_here(smem_u32(sm.q[0]), 16, 1024);
                                const uint64_t db = make_sdesc_here(smem_u32(sm.k[0]), 16, 1024);
#pragma unroll
                                for (int kk = 0; kk < D / 16; ++kk) {
                                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                                    mma_ss(tmem + b * 128, sdesc_add(da, off), sdesc_add(db, off), idS,
                                           kk > 0);
                                    // K's box kk / 4 is read once its four MMAs are done
                                    if ((kk & 3) == 3) mma_commit(smem_u32(&sm.k_empty[kk >> 2]));
                                }
                                mma_commit(smem_u32(&sm.s_full[b]));
                            } else {
#pragma unroll
                                for (int c = 0; c < Cfg::kBoxes; ++c)
                                    mma_commit(smem_u32(&sm.k_empty[c]));
                            }
                            if (j == x.nkv - 1) mma_commit(smem_u32(&sm.q_empty));
                            ++k_it;
                        }
                        if (j >= 1) {
                            // PV(j-1), chunk by chunk of V columns, each V slot
                            // released once its chunk has been read
                            const int jp = j - 1, gj = g + jp, b = gj & 1;
                            if (jp < n) {
                                if (!(ok = wait_or_abort(smem_u32(&sm.p_full[b]), (gj >> 1) & 1,
                                                         abort_flag, hdr)))
                                    break;
                                if (jp == 0 && ep[0] > 0 &&
                                    !(ok = wait_or_abort(smem_u32(&sm.o_free[0]), (ep[0] - 1) & 1,
                                                         abort_flag, hdr)))
                                    break;
                            }
                            for (int h = 0; h < Cfg::kVChunks; ++h) {
                                const int slot = v_it % Cfg::kVSlots;
                                if (!(ok = wait_or_abort(smem_u32(&sm.v_full[slot]),
                                                         (v_it / Cfg::kVSlots) & 1, abort_flag, hdr)))
                                    break;
                                if (jp < n) {
                                    tc_fence_after();
                                    const uint64_t db = make_sdesc_here(smem_u32(sm.v[slot]), 16384, 1024);
                                    // the first chunk starts on keys [0, 64) of P and waits
                                    // for [64, 128) halfway
#pragma unroll
                                    for (int kk = 0; kk < kTile / 16; ++kk) {
                                        if (h == 0 && kk == kTile / 32) {
                                            if (!(ok = wait_or_abort(smem_u32(&sm.p_hi[b]), (gj >> 1) & 1,
                                                                     abort_flag, hdr)))
                                                break;
                                            tc_fence_after();
                                        }
                                        mma_ts(tmem + 256 + h * Cfg::kVChunk,
                                               tmem + (Cfg::kSepP ? Cfg::kPCol : b * 128) + kk * 8,
                                               sdesc_add(db, kk * 2048), idPV,
                                               (jp > 0 || kk > 0) ? 1u : 0u);
                                    }
                                    if (!ok) break;
                                }
                                mma_commit(smem_u32(&sm.v_empty[slot]));
                                ++v_it;
                            }
                            if (!ok) break;
                            if (jp < n) mma_commit(smem_u32(&sm.o_done[b]));
                        }
                    }
                    if (!ok) break;
                    g += n;
                    ++unit_it;
                    ep[0] += n > 0;
                } else {
                    for (int j = 0; j < x.nkv && ok; ++j) {
                        const int st = kv_it % S, par = (kv_it / S) & 1;
                        if (!(ok = wait_or_abort(smem_u32(&sm.k_full[st]), par, abort_flag, hdr))) break;
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            if (!ok) break;
                            if (t >= Cfg::kQTiles || j >= x.n[t]) continue;
                            // S_t / P_t region is free once the previous O_t += P_t V is done
                            if (it[t] > 0 &&
                                !(ok = wait_or_abort(smem_u32(&sm.o_done[t]), (it[t] - 1) & 1,
                                                     abort_flag, hdr)))
                                break;
                            tc_fence_after();
                            const uint32_t qa = smem_u32(sm.q[t]), kb = smem_u32(sm.k[st]);
#pragma unroll
                            for (int kk = 0; kk < DR / 16; ++kk) {  // (columns past DR are zero)
                                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                                mma_ss(tmem + t * 128, make_sdesc(qa + off, 16, 1024),
                                       make_sdesc(kb + off, 16, 1024), idS, kk > 0);
                            }
                            mma_commit(smem_u32(&sm.s_full[t]));
                        }
                        if (!ok) break;
                        // the unit's last S MMAs are issued: Q may be overwritten once they finish
                        if (j == x.nkv - 1) mma_commit(smem_u32(&sm.q_empty));
                        if (!(ok = wait_or_abort(smem_u32(&sm.v_full[st]), par, abort_flag, hdr))) break;
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            if (!ok) break;
                            if (t >= Cfg::kQTiles || j >= x.n[t]) continue;
                            if (!(ok = wait_or_abort(smem_u32(&sm.p_full[t]), it[t] & 1, abort_flag,
                                                     hdr)))
                                break;
                            if (j == 0 && ep[t] > 0 &&
                                !(ok = wait_or_abort(smem_u32(&sm.o_free[t]), (ep[t] - 1) & 1,
                                                     abort_flag, hdr)))
                                break;
                            tc_fence_after();
                            const uint32_t vb = smem_u32(sm.v[st]);
                            const uint32_t o_col = 256 + t * 128, p_col = t * 128;
                            // keys [0, 64) of P_t, then [64, 128) once the softmax has them
#pragma unroll
                            for (int kk = 0; kk < kTile / 16; ++kk) {
                                if (kk == kTile / 32) {
                                    if (!(ok = wait_or_abort(smem_u32(&sm.p_hi[t]), it[t] & 1,
                                                             abort_flag, hdr)))
                                        break;
                                    tc_fence_after();
                                }
                                mma_ts(tmem + o_col, tmem + p_col + kk * 8,
                                       make_sdesc(vb + kk * 2048, 16384, 1024), idPV,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                            }
                            if (!ok) break;
                            mma_commit(smem_u32(&sm.o_done[t]));
                            ++it[t];
                        }
                        mma_commit(smem_u32(&sm.kv_empty[st]));
                        ++kv_it;
                    }
                    if (!ok) break;
                    ++unit_it;
#pragma unroll
                    for (int t = 0; t < 2; ++t) ep[t] += x.n[t] > 0;
                }
            }
            // all issued MMAs complete before TMEM is released
            mma_commit(smem_u32(&sm.drain));
            mbar_wait(smem_u32(&sm.drain), 0, &sm.zero);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax warpgroups
        setmaxnreg_inc<216>();
        const int t = (warp - 4) >> 2;          // query tile of this warpgroup
        const int q4 = warp & 3;                // TMEM lane quarter
        const int row = q4 * 32 + lane;         // row within the tile
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + t * 128;
        // (D > 128: one O, stored by warps 8..11)
        const uint32_t o_addr = tmem + lane_off + 256 + (D > 128 ? 0 : t * 128);
        int sched_it = 0, it = 0;
        int ue = 0;  // D > 128: units handed from the softmax to the epilogue warps
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
            const UnitGeom x = decode_unit<D, KV>(unit, p);
            if constexpr (D > 128) {
                if (t == 1) {
                    // Epilogue warps: store the unit the softmax warps have finished
                    // while those go on with the next one.  it counts the unit's
                    // steps as the softmax warps do, so the last PV is step it - 1.
                    if (x.n[0] == 0) continue;
                    it += x.n[0];
                    if (!(ok = warp_wait(smem_u32(&sm.ep_full), ue & 1, abort_flag, hdr))) break;
                    if (!(ok = warp_wait(smem_u32(&sm.o_done[(it - 1) & 1]), ((it - 1) >> 1) & 1,
                                         abort_flag, hdr)))
                        break;
                    tc_fence_after();
                    ++ue;
                    const int r = x.m * kTile + row;
                    store_row<DR, OUT_FP32, KV>(p, o_addr, x.h, (size_t)x.t0 + (size_t)r, r < x.L,
                                                sm.ep_m[row], sm.ep_l[row]);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sm.o_free[0]));
                    continue;
                }
            }
            const int nt = t == 0 ? x.n[0] : x.n[1];
            if constexpr (!KV) {
                if (nt == 0) continue;  // the tile is past the end
            }
            const int r = x.m * Cfg::kUnitRows + t * kTile + row;  // row within the sequence
            if constexpr (KV) {
                if (nt == 0) {
                    // the tile is past the end, or none of its rows sees a key:
                    // O = 0 and LSE = -inf, nothing on chip.  (With one query tile
                    // per unit, tile 1 is not a tile: its rows are the next unit's.)
                    if (t < Cfg::kQTiles && r < x.L)
                        write_keyless_row<DR, OUT_FP32>(p, x.h, (size_t)x.t0 + (size_t)r);
                    continue;
                }
            }
            // visible keys: col < limit (end-aligned causal mask)
            const int limit = KV ? (p.causal ? min(r + 1 + x.Lk - x.L, x.Lk) : x.Lk)
                                 : (p.causal ? min(r + 1, x.L) : x.L);
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < nt; ++j) {
                // D > 128: S alternates between two buffers, step by step
                const int buf = D > 128 ? (it & 1) : t;
                const uint32_t s_at = D > 128 ? s_addr + (uint32_t)buf * 128 : s_addr;
                if (!(ok = warp_wait(smem_u32(&sm.s_full[buf]), D > 128 ? (it >> 1) & 1 : it & 1,
                                     abort_flag, hdr)))
                    break;
                tc_fence_after();
                float s[128];
                {
                    // all four 32-column loads in flight, one wait
                    uint32_t r0[32], r1[32], r2[32], r3[32];
                    tmem_ld32(s_at, r0);
                    tmem_ld32(s_at + 32, r1);
                    tmem_ld32(s_at + 64, r2);
                    tmem_ld32(s_at + 96, r3);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        s[i] = __uint_as_float(r0[i]);
                        s[32 + i] = __uint_as_float(r1[i]);
                        s[64 + i] = __uint_as_float(r2[i]);
                        s[96 + i] = __uint_as_float(r3[i]);
                    }
                }
                const int thr = limit - j * kTile;
                if (thr < kTile) {
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i >= thr) s[i] = -INFINITY;
                }
                // row max: 8 independent chains of 3-input maxima
                float m8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float m = fmax3(s[k], s[8 + k], s[16 + k]);
#pragma unroll
                    for (int i = 24; i < 120; i += 16) m = fmax3(m, s[i + k], s[i + 8 + k]);
                    m8[k] = fmaxf(m, s[120 + k]);
                }
                float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                                 fmaxf(m8[6], m8[7]));
                mx *= p.scale_log2;
                float alpha = 1.f;
                bool need = false;
                if (j == 0) {
                    m_ref = mx;
                } else if (mx > m_ref + kRescaleThreshold) {
                    need = true;
                    alpha = ex2_approx(m_ref - mx);
                    m_ref = mx;
                    l *= alpha;
                }
                const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
                if constexpr (D <= 128) {
                    // O~ first (stable: S_t(j) was committed after O_t += P_t V of
                    // j - 1), then P in two halves, each handed over as soon as it is
                    // in TMEM: PV_t may start on keys [0, 64) while the exponentials
                    // of [64, 128) run.  (All of S_t is in registers, so P's first
                    // columns may overwrite it.)
                    if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
                        for (int c = 0; c < DR / 32; ++c) {
                            uint32_t ov[32];
                            tmem_ld32(o_addr + c * 32, ov);
                            tmem_ld_wait();
                            uint32_t lo[16], hi[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                lo[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                                hi[i] = __float_as_uint(__uint_as_float(ov[16 + i]) * alpha);
                            }
                            tmem_st16(o_addr + c * 32, lo);
                            tmem_st16(o_addr + c * 32 + 16, hi);
                        }
                    }
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                        for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
                            uint32_t pk[16];
                            softmax_chunk(s + c * 32, p.scale_log2, neg, acc, pk);
                            tmem_st16(s_at + c * 16, pk);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(hf == 0 ? &sm.p_full[buf] : &sm.p_hi[buf]));
                    }
                    float a0, a1, b0, b1;
                    f2_unpack(acc[0], a0, a1);
                    f2_unpack(acc[1], b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                    ++it;
                    continue;
                }
                // One tile (D > 128): S(j) may finish before PV(j-1), so O~ is
                // stable only once PV(j-1) is done (j >= 1 whenever a rescale is
                // needed).  The rescale comes first, then P in two halves as for
                // two tiles; with P in columns of its own (d = 192) each half is
                // computed in registers before it waits for PV(j-1) to have read
                // the previous P.
                bool pv_done = it == 0;
                if (__any_sync(0xffffffffu, need)) {
                    if (!(ok = warp_wait(smem_u32(&sm.o_done[(it - 1) & 1]), ((it - 1) >> 1) & 1,
                                         abort_flag, hdr)))
                        break;
                    tc_fence_after();
                    pv_done = true;
#pragma unroll 1
                    for (int c = 0; c < DR / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(o_addr + c * 32, ov);
                        tmem_ld_wait();
                        uint32_t lo[16], hi[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            lo[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                            hi[i] = __float_as_uint(__uint_as_float(ov[16 + i]) * alpha);
                        }
                        tmem_st16(o_addr + c * 32, lo);
                        tmem_st16(o_addr + c * 32 + 16, hi);
                    }
                }
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    if constexpr (Cfg::kSepP) {
                        uint32_t pk[2][16];
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            softmax_chunk(s + (2 * hf + c) * 32, p.scale_log2, neg, acc, pk[c]);
                        if (!pv_done) {
                            if (!(ok = warp_wait(smem_u32(&sm.o_done[(it - 1) & 1]),
                                                 ((it - 1) >> 1) & 1, abort_flag, hdr)))
                                break;
                            tc_fence_after();
                            pv_done = true;
                        }
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tmem_st16(tmem + lane_off + Cfg::kPCol + (2 * hf + c) * 16, pk[c]);
                    } else {
#pragma unroll
                        for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
                            uint32_t pk[16];
                            softmax_chunk(s + c * 32, p.scale_log2, neg, acc, pk);
                            tmem_st16(s_at + c * 16, pk);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(hf == 0 ? &sm.p_full[buf] : &sm.p_hi[buf]));
                }
                if (!ok) break;
                {
                    float a0, a1, b0, b1;
                    f2_unpack(acc[0], a0, a1);
                    f2_unpack(acc[1], b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                }
                ++it;
            }
            if (!ok) break;
            if constexpr (D > 128) {
                // hand m and l to the epilogue warps, once they have read the
                // previous unit's
                if (ue > 0 &&
                    !(ok = warp_wait(smem_u32(&sm.o_free[0]), (ue - 1) & 1, abort_flag, hdr)))
                    break;
                sm.ep_m[row] = m_ref;
                sm.ep_l[row] = l;
                mbar_arrive(smem_u32(&sm.ep_full));
                ++ue;
                continue;
            }
            // epilogue: O = O~ / l, LSE = (m + log2 l) * ln 2
            if (!(ok = warp_wait(smem_u32(&sm.o_done[t]), (it - 1) & 1, abort_flag, hdr))) break;
            tc_fence_after();
            store_row<DR, OUT_FP32, KV>(p, o_addr, x.h, (size_t)x.t0 + (size_t)r, r < x.L, m_ref, l);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.o_free[t]));
        }
    } else {
        setmaxnreg_dec<72>();  // warps 2 and 3: TMEM allocation only
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, int DR, bool F32, bool KV>
cudaError_t launch_fwd_t(const FwdParams& p, int num_sms, cudaStream_t stream) {
    auto kern = fa_fwd_kernel<D, DR, F32, KV>;
    const size_t smem = sizeof(FwdSmem<D>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long bound = max_tiles(p.B, p.T, FwdCfg<D>::kUnitRows) * p.Hq;
    const int grid = (int)(bound < num_sms ? bound : num_sms);
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(kern, dim3(grid), dim3(kFwdThreads), smem, stream, p);
}

}  // namespace

template <bool KV>
cudaError_t launch_fwd_kv(const FwdParams& p, int num_sms, cudaStream_t stream) {
    if (p.d == 128)
        return p.o_fp32 ? launch_fwd_t<128, 128, true, KV>(p, num_sms, stream)
                        : launch_fwd_t<128, 128, false, KV>(p, num_sms, stream);
    if (p.d == 96)
        return p.o_fp32 ? launch_fwd_t<128, 96, true, KV>(p, num_sms, stream)
                        : launch_fwd_t<128, 96, false, KV>(p, num_sms, stream);
    if (p.d == 256)
        return p.o_fp32 ? launch_fwd_t<256, 256, true, KV>(p, num_sms, stream)
                        : launch_fwd_t<256, 256, false, KV>(p, num_sms, stream);
    if (p.d == 192)
        return p.o_fp32 ? launch_fwd_t<192, 192, true, KV>(p, num_sms, stream)
                        : launch_fwd_t<192, 192, false, KV>(p, num_sms, stream);
    return p.o_fp32 ? launch_fwd_t<64, 64, true, KV>(p, num_sms, stream)
                    : launch_fwd_t<64, 64, false, KV>(p, num_sms, stream);
}

cudaError_t launch_fwd(const FwdParams& p, int num_sms, cudaStream_t stream) {
    return p.kv ? launch_fwd_kv<true>(p, num_sms, stream)
                : launch_fwd_kv<false>(p, num_sms, stream);
}

}  // namespace fa
