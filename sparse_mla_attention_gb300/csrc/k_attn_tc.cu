// k_attn_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of the sparse
// MLA backward core, for one rank chunk [r0, r0 + R).
//
// Definitions (aiter "Sparse MLA training backward", Structure table, dQ and
// dKV-interm phases), token t, head h, rank r (index idx = topk[t, r0 + r]):
//   S  = <q[t,h,:], kv[idx,:]>,  dP = <dO[t,h,:], kv[idx,:]>
//   P  = exp(scale * S - lse[t,h]),  dS = P * (dP - delta[t,h])
//   interm[t, r, :] = sum_h P * dO[t,h,:] + scale * dS * q[t,h,:]
//   dq[t, h, :]    += scale * sum_r dS * kv[idx, :]
//
// sdi_kernel (S, dP, P, dS, interm): persistent, one CTA per SM. A work item
// is (token t, 256 ranks) = two 128-rank tiles.
//  * A stage: per tile, one MMA stream computes S^T and dP^T together:
//    M = 128 ranks, N = 2H (the q rows of token t and its dO rows, in the
//    order the two tensors sit in memory), K = 512, in eight 64-column steps.
//    The kv rows of each step are gathered by two copy warps (16-byte cp.async
//    through L2); q and dO come by TMA, as one box per step when both tensors
//    can be addressed as one paired tensor map, else as two.
//  * Epilogue: each TMEM row (one rank) becomes P and scale*dS, written back
//    into TMEM as bf16 pairs (the A operand of the next GEMM); scale*dS^T is
//    also stashed in global memory for the dq kernel. Results leave TMEM
//    through registers and a per-warp staging tile, by TMA store.
//  * B stage: interm = [P | scale*dS] x [dO ; q] with A from TMEM: M = 128
//    ranks, N = 128 columns of D per step, K = 2H. Each tile has one
//    128-column accumulator; the tiles alternate, and all eight epilogue warps
//    drain each accumulator (TMEM -> bf16 -> staging tile -> TMA store) while
//    the other tile's MMAs run.
//  * Overlap: S^T / dP^T complete per tile; the epilogue warps finish tile 0's
//    P / dS first, and tile 0's B stage runs while they work on tile 1.
// TMEM (512 columns): tile g owns columns [256g, 256g + 256): S^T and dP^T in
// [0, 2H); then, per 16-head chunk k, P^T in [16k, 16k + 8) and scale*dS^T in
// [16k + 8, 16k + 16) (bf16 pairs over chunk k of whichever of S^T / dP^T owns
// [0, H)), and the interm accumulator in [128, 256).
//
// dq_kernel: persistent; item = (token, half of D). dq = (scale*dS) x kv:
// M = 128 (heads, zero-padded), N = 256, K = ranks in 64-rank steps, both
// operands MN-major (scale*dS^T rows by TMA from the stash, kv rows gathered
// by eight copy warps in two teams), accumulated in TMEM (two 256-column
// buffers) and written as bf16 through shared memory by TMA stores (or added
// to an fp32 accumulator between rank chunks).
//
// Every mbarrier wait is bounded (kWaitNs); a timeout sets SMLA_ERR_TIMEOUT in
// the status word, stops the CTA's loops, waits (bounded) for its own copies
// and MMAs in flight and frees its TMEM.
#include "smla_internal.cuh"
#include "sm100.cuh"
#include "tmap.h"

#include <climits>
#include <type_traits>

namespace smla {
using namespace sm100;

namespace {

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

}  // namespace
#ifdef SMLA_TRACE
// Optional phase timestamps (compiled only with -DSMLA_TRACE; the library
// build leaves them out): per kernel, CTA (< 8) and item (< 8), 64 events.
constexpr int kTraceCtas = 8, kTraceItems = 8, kTraceEvents = 256;
__device__ unsigned long long g_smla_trace[2 * kTraceCtas * kTraceItems * kTraceEvents];
// per kernel and CTA (< 1024): start and end time of the CTA's MMA thread
__device__ unsigned long long g_smla_cta_span[2 * 1024 * 3];
__device__ __forceinline__ unsigned smla_smid() {
    unsigned r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}
#define SMLA_TRACE_SPAN(kid, which)                                                         \
    do {                                                                                    \
        if (blockIdx.x < 1024) {                                                            \
            g_smla_cta_span[((kid) * 1024 + blockIdx.x) * 3 + (which)] = globaltimer_ns();  \
            g_smla_cta_span[((kid) * 1024 + blockIdx.x) * 3 + 2] = smla_smid();             \
        }                                                                                   \
    } while (0)
#define SMLA_TRACE_EV(kid, it, ev)                                                          \
    do {                                                                                    \
        if (blockIdx.x < kTraceCtas && (it) < kTraceItems)                                  \
            g_smla_trace[(((kid) * kTraceCtas + blockIdx.x) * kTraceItems + (it)) *         \
                             kTraceEvents + (ev)] = globaltimer_ns();                       \
    } while (0)
#define SMLA_TRACE_VAL(kid, it, ev, val)                                                    \
    do {                                                                                    \
        if (blockIdx.x < kTraceCtas && (it) < kTraceItems)                                  \
            g_smla_trace[(((kid) * kTraceCtas + blockIdx.x) * kTraceItems + (it)) *         \
                             kTraceEvents + (ev)] = (val);                                  \
    } while (0)
#else
#define SMLA_TRACE_EV(kid, it, ev) \
    do {                           \
    } while (0)
#define SMLA_TRACE_VAL(kid, it, ev, val) \
    do {                                 \
    } while (0)
#define SMLA_TRACE_SPAN(kid, which) \
    do {                            \
    } while (0)
#endif
namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, unsigned* status,
                                              uint64_t limit_ns = kWaitNs) {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, limit_ns)) return true;
    *abort_flag = 1;
    flag_status(status, SMLA_ERR_TIMEOUT);
    return false;
}

// For warps that go on to warp-collective tcgen05 loads: every lane waits, and
// the warp goes on only if all of them saw the phase.
__device__ __forceinline__ bool wait_or_abort_warp(uint64_t* bar, uint32_t parity,
                                                   volatile int* abort_flag, unsigned* status) {
    const bool ok = wait_or_abort(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok) != 0;
}

__device__ __forceinline__ void advance(int& slot, uint32_t& phase, int nslots) {
    if (++slot == nslots) { slot = 0; phase ^= 1u; }
}

// Packs 8 fp32 values into one 16-byte piece of bf16.
__device__ __forceinline__ uint4 pack8(const uint32_t* v) {
    return make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                      pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                      pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                      pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
}

// ====================================================================== SDI
struct SdiParams {
    const uint16_t* kv;   // [N, 512]
    const int32_t* topk;
    const float* lse;
    const float* delta;
    uint16_t* interm;     // [T, R, 512]
    uint16_t* dsT;        // scale*dS^T stash [T, ds_rows, Hp]
    int T, K, N, r0, R, Rp, Hp;
    int ds_rows, ds_off;  // stash rank rows per token; this chunk's first row
    int npairs;           // items per token: ceil(R / 256)
    int tiles_last;       // tiles (1 or 2) in a token's last item
    float scale;
    // q / dO loads: 0 = separate [H x 64] boxes of q and dO; 1 = one paired box
    // per load with q first; 2 = paired, dO first (dO sits below q in memory).
    // The tensor that comes first in shared memory owns TMEM columns [0, H) of
    // the S^T | dP^T accumulator and the first half of each B-stage slot.
    int qd_mode;
    int* work_ctr;        // next work item (zeroed before the launch)
    // with cnt set, topk is a compacted table (each token's valid entries
    // first) and cnt[t] their number: a token has ceil(cnt / 128) tiles (at
    // least one), so masked slots cost no tensor work
    const int32_t* cnt;
    // two-token items (heads <= 64, at most 128 ranks per token): item i holds
    // tokens 2i and 2i + 1, one 128-rank tile each
    int tt;
    unsigned* status;
};

// Tiles (0, 1 or 2) of work item `item`: (token, 256-rank pair), or with
// two-token items (tokens 2 item, 2 item + 1).
__device__ __forceinline__ int sdi_ntiles(const SdiParams& p, int item) {
    if (p.tt) return 2 * item + 1 < p.T ? 2 : 1;
    const int t = item / p.npairs, pr = item - t * p.npairs;
    if (p.cnt) {
        int m = __ldg(p.cnt + t);
        if (m < 1) m = 1;              // one all-masked tile: the stash rows dq reads are written
        const int n = ((m + 127) >> 7) - 2 * pr;
        return n < 0 ? 0 : (n > 2 ? 2 : n);
    }
    return pr == p.npairs - 1 ? p.tiles_last : 2;
}

struct SdiShared {
    uint64_t full[8], empty[8];
    // kempty[s]: one phase per use of slot s that is followed (kSlots uses
    // later) by a use the copy warps fill, so the copy warps, who skip the
    // B-stage uses, wait on it for every fill of theirs exactly once, in order
    // (a parity wait on `empty`, which advances on every use, could see the
    // slot two phases on and pass too early)
    uint64_t kempty[8];
    uint64_t s_full[2], p_ready[2], x_full[2], x_empty[2], b_done[2], drain;
    // Work queue: the TMA thread takes items from the global counter and
    // publishes them in order, as item * 4 + its tile count (so that no other
    // role loads the count); every other role reads entry k for its k-th item
    // (the copy warps one item ahead). An item >= the item count ends the
    // CTA's work. CTAs that start late (their SM still busy with another
    // kernel) simply take fewer items.
    int item_q[4];
    uint64_t q_full[4], q_empty[4];
    uint32_t tbase;
    volatile int abort_flag;
};

constexpr int kQueueReaders = 11;   // 2 copy warps + the MMA thread + 8 epilogue warps

// Entry k of the work queue (item * 4 + tiles), read by a whole warp (lane 0
// signals the read).
__device__ __forceinline__ int queue_read_warp(SdiShared& sh, int k, unsigned* status, bool& ok) {
    const int e = k & 3;
    if (!wait_or_abort_warp(&sh.q_full[e], uint32_t(k >> 2) & 1u, &sh.abort_flag, status)) {
        ok = false;
        return INT_MAX;
    }
    const int item = *reinterpret_cast<volatile int*>(&sh.item_q[e]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.q_empty[e]);
    return item;
}

// Entry k of the work queue (item * 4 + tiles), read by one thread.
__device__ __forceinline__ int queue_read_thread(SdiShared& sh, int k, unsigned* status, bool& ok) {
    const int e = k & 3;
    if (!wait_or_abort(&sh.q_full[e], uint32_t(k >> 2) & 1u, &sh.abort_flag, status)) {
        ok = false;
        return INT_MAX;
    }
    const int item = *reinterpret_cast<volatile int*>(&sh.item_q[e]);
    mbar_arrive(&sh.q_empty[e]);
    return item;
}

// Per epilogue warp: a 32-row x 128-byte staging tile that turns one-row-per-
// lane TMEM data into one TMA store; the 16-byte piece j of row r sits at
// piece slot j ^ (r & 7), the 128-byte swizzle of the store's tensor map
// (which also keeps the row-per-lane writes free of bank conflicts). Two
// alternatives measured slower: plain coalesced stores from the staging tile
// (they add the L1 data path to the shared-memory traffic the tensor cores
// need) and 32-byte stores straight from registers, one rank row per lane.
constexpr int kStageBytes = 32 * 128;

// Writes the warp's staged 32 rows x 128 bytes to global memory with plain
// coalesced stores (8 lanes per row, four rows per instruction): row r goes to
// base + r * row_elems (bf16 elements), rows r >= nrows are skipped.
__device__ __forceinline__ void store_staged_rows(const uint8_t* stage, uint16_t* base, int64_t row_elems,
                                                  int nrows, int lane) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int rr = 4 * k + (lane >> 3), piece = lane & 7;
        const uint4 val = reinterpret_cast<const uint4*>(stage + rr * 128)[piece ^ (rr & 7)];
        if (rr < nrows) reinterpret_cast<uint4*>(base + rr * row_elems)[piece] = val;
    }
}

template <int H, bool TT>
struct SdiCfg {
    static_assert(!TT || H <= 64, "two-token items need heads <= 64");
    static constexpr int kTok = TT ? 2 : 1;                 // tokens per item
    static constexpr int kQBytes = H * 128;                 // H rows x 64 columns bf16
    static constexpr int kKvBytes = 128 * 128;              // 128 ranks x 64 columns bf16
    // a slot: the item's q | dO (per token: q block then dO block) then the two
    // kv tiles (A stage), or the item's 128-column q | dO blocks (B stage)
    static constexpr int kKvOff = 2 * kQBytes * kTok;
    static constexpr int kSlotA = kKvOff + 2 * kKvBytes, kSlotB = 4 * kQBytes * kTok;
    static constexpr int kSlotBytes = kSlotA > kSlotB ? kSlotA : kSlotB;
    static constexpr int kSlotsRaw = 196608 / kSlotBytes;
    static constexpr int kSlots = kSlotsRaw > 8 ? 8 : kSlotsRaw;
    static constexpr int kThreads = 384;    // TMA, MMA, 8 epilogue warps, 2 copy warps
    static constexpr int kSmem = int(sizeof(SdiShared)) + 1024 + kSlots * kSlotBytes + 8 * kStageBytes;
    static constexpr uint32_t kIdescA = idesc_bf16(128, 2 * H, false, false);
    static constexpr uint32_t kIdescB = idesc_bf16(128, 128, false, true);
    static constexpr int kUses = 12;        // ring uses per item: 8 A-stage + 4 B-stage
    static_assert(kSlots >= 3, "the copy pipeline needs at least three slots");
    static_assert(kSmem <= 232448, "shared memory of one CTA is at most 227 KB");
};

template <int H, bool TT>
__global__ void __launch_bounds__(384, 1)
sdi_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
           const __grid_constant__ CUtensorMap map_qda, const __grid_constant__ CUtensorMap map_qdb,
           const __grid_constant__ CUtensorMap map_im, const __grid_constant__ CUtensorMap map_ds,
           const SdiParams p) {
    using C = SdiCfg<H, TT>;
    extern __shared__ uint8_t smem_raw[];
    SdiShared& sh = *reinterpret_cast<SdiShared*>(smem_raw);
    uint8_t* slots = align1024(smem_raw + sizeof(SdiShared));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = TT ? (p.T + 1) / 2 : p.T * p.npairs;

    if (threadIdx.x == 0) {
        // full: the TMA thread's arrive (with the q / dO bytes) + 64 copy threads
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(&sh.full[s], 65);
            mbar_init(&sh.empty[s], 1);
            mbar_init(&sh.kempty[s], 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&sh.s_full[g], 1);   // tile g's S^T | dP^T are complete
            mbar_init(&sh.p_ready[g], 8);  // all 8 epilogue warps wrote tile g's P / dS
            mbar_init(&sh.x_full[g], 1);   // tile g's interm accumulator is ready
            mbar_init(&sh.x_empty[g], 8);  // all 8 epilogue warps have read their halves
            mbar_init(&sh.b_done[g], 1);
        }
        mbar_init(&sh.drain, 1);
        for (int e = 0; e < 4; ++e) {
            mbar_init(&sh.q_full[e], 1);
            mbar_init(&sh.q_empty[e], kQueueReaders);
        }
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(&sh.tbase, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sh.tbase;

    if (warp == 0) {
        // ----------------------------------------------- TMA producer (q, dO)
        if (lane == 0) {
            int slot = 0; uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            int pub = 0, last = -1;       // entries published; the last item published
            auto publish = [&]() -> bool {
                const int e = pub & 3;
                if (pub >= 4 &&
                    !wait_or_abort(&sh.q_empty[e], uint32_t((pub >> 2) - 1) & 1u, &sh.abort_flag, p.status))
                    return false;
                int item = atomicAdd(p.work_ctr, 1), nt = 0;
                while (item < nitems && (nt = sdi_ntiles(p, item)) == 0) item = atomicAdd(p.work_ctr, 1);
                if (item > nitems) item = nitems;
                sh.item_q[e] = item * 4 + (item < nitems ? nt : 0);
                mbar_arrive(&sh.q_full[e]);
                last = item;
                ++pub;
                return true;
            };
            ok = publish();
            if (ok && last < nitems) ok = publish();
            for (int it = 0; ok; ++it) {
                const int item = sh.item_q[it & 3] >> 2;
                if (item >= nitems) break;
                // entry it + 2 (the copy warps read entry it + 1 during this item)
                if (last < nitems && !publish()) { ok = false; break; }
                SMLA_TRACE_EV(0, it, 0);
                SMLA_TRACE_VAL(0, it, 45, uint64_t(p.qd_mode));
                const int t = TT ? 2 * item : item / p.npairs;   // the item's first token
                for (int c = 0; c < C::kUses; ++c) {
                    ok = wait_or_abort(&sh.empty[slot], phase ^ 1u, &sh.abort_flag, p.status);
                    if (!ok) break;
                    uint8_t* sb = slots + slot * C::kSlotBytes;
                    SMLA_TRACE_EV(0, it, 48 + c);
                    if (c < 8) {
                        // A stage: q and dO columns [64c, 64c + 64) of the item's token(s)
                        mbar_arrive_expect_tx(&sh.full[slot], C::kKvOff);
                        if (p.qd_mode != 0) {
                            tma_load_5d(sb, &map_qda, 0, 0, c, 0, t, &sh.full[slot]);
                        } else {
#pragma unroll
                            for (int tk = 0; tk < C::kTok; ++tk) {
                                tma_load_2d(sb + tk * 2 * C::kQBytes, &map_q, c * 64, (t + tk) * H, &sh.full[slot]);
                                tma_load_2d(sb + tk * 2 * C::kQBytes + C::kQBytes, &map_do, c * 64, (t + tk) * H,
                                            &sh.full[slot]);
                            }
                        }
                    } else {
                        // B stage: q and dO columns [128b, 128b + 128), two 64-column
                        // blocks each; the copy warps skip these uses, so arrive for them.
                        const int b = c - 8;
                        mbar_arrive_expect_tx(&sh.full[slot], C::kSlotB);
                        if (p.qd_mode != 0) {
                            tma_load_5d(sb, &map_qdb, 0, 0, 2 * b, 0, t, &sh.full[slot]);
                        } else {
#pragma unroll
                            for (int tk = 0; tk < C::kTok; ++tk) {
                                uint8_t* tb = sb + tk * 4 * C::kQBytes;
                                const int row = (t + tk) * H;
                                tma_load_2d(tb, &map_q, b * 128, row, &sh.full[slot]);
                                tma_load_2d(tb + C::kQBytes, &map_q, b * 128 + 64, row, &sh.full[slot]);
                                tma_load_2d(tb + 2 * C::kQBytes, &map_do, b * 128, row, &sh.full[slot]);
                                tma_load_2d(tb + 3 * C::kQBytes, &map_do, b * 128 + 64, row, &sh.full[slot]);
                            }
                        }
                        mbar_arrive_cnt(&sh.full[slot], 64);
                    }
                    ++issued;
                    advance(slot, phase, C::kSlots);
                }
            }
            if (sh.abort_flag) {
                // bounded wait for this thread's own copies still in flight
                int s = slot; uint32_t ph = phase;
                for (int k = 0; k < C::kSlots && k < issued; ++k) {
                    if (--s < 0) { s = C::kSlots - 1; ph ^= 1u; }
                    mbar_wait(&sh.full[s], ph, kWaitNs / 8);
                }
            }
        }
        __syncwarp();
    } else if (warp >= 10) {
        // ------------------------------------------------ kv gather (cp.async)
        // In round i (0..31) copy warp gw copies rows 8i + 4gw .. +3 of the
        // item's 256 ranks; lane l copies the 16-byte piece (l & 7) of row
        // (l >> 3) into the 128-byte-swizzled tile. Lane l keeps the 32 row
        // indices it needs in registers, loaded one item ahead.
        const int gw = warp - 10;
        int slot = 0; uint32_t phase = 0;
        bool ok = true;
        int idx_cur[32], idx_nxt[32];
        auto load_idx = [&](int item, int (&out)[32]) {
            // token and rank of row `row` (0..255, tile row >> 7) of the item
            const int tok0 = TT ? 2 * item : item / p.npairs, tok1 = TT ? 2 * item + 1 : tok0;
            const int rbase = TT ? 0 : (item - tok0 * p.npairs) * 256;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int row = 8 * i + 4 * gw + (lane >> 3);
                const int t = TT && row >= 128 ? tok1 : tok0;
                const int rl = TT ? (row & 127) : rbase + row;
                // masked, invalid, or past the chunk's end: any real row will do
                // (P of that rank is zeroed), but not one fixed row, which every
                // CTA would then read at once: the slot's own rank position
                // spreads them over up to 512 rows (the zero-filling form of
                // cp.async, and a modulo here, both measured slower)
                int j = -1;
                if (rl < p.R && (!TT || t < p.T)) {
                    j = __ldg(p.topk + int64_t(t) * p.K + p.r0 + rl);
                    if (j < -1 || j >= p.N) { flag_status(p.status, SMLA_ERR_INDEX); j = -1; }
                }
                out[i] = j >= 0 ? j : (rl < p.N ? rl : 0);
            }
        };
        int ecur = queue_read_warp(sh, 0, p.status, ok);
        int cur = ecur >> 2;
        if (cur < nitems) load_idx(cur, idx_cur);
#pragma unroll
        for (int i = 0; i < 32; ++i) idx_nxt[i] = 0;
        const char* kvbase = reinterpret_cast<const char*>(p.kv) + (lane & 7) * 16;
        // Slots whose copies are issued but not yet signalled, oldest in the low
        // 4 bits (a packed queue: a runtime-indexed array would live in local
        // memory). At most kSlots - 2 stay pending, so the next slot to fill
        // never waits for one of them.
        uint32_t pend = 0;
        int npend = 0;
        auto flush_one = [&]() {
            fence_proxy_async_smem();
            mbar_arrive(&sh.full[pend & 15u]);
            pend >>= 4;
            --npend;
        };
        int use = 0;              // this CTA's ring use index
        uint32_t kph = 0;         // per slot: parity of its next kempty phase
        for (int k = 0; ok && cur < nitems; ++k) {
            const int ntiles = ecur & 3;
            int enxt = nitems * 4;
            for (int c = 0; c < 8; ++c, ++use) {
                if (use >= C::kSlots) {   // the slot's previous use must be consumed
                    if (lane == 0)
                        ok = wait_or_abort(&sh.kempty[slot], (kph >> slot) & 1u, &sh.abort_flag, p.status);
                    kph ^= 1u << slot;
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                uint8_t* kvb = slots + slot * C::kSlotBytes + C::kKvOff;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int row = 8 * i + 4 * gw + (lane >> 3);   // 0..255 (tile = row >> 7)
                    if ((row >> 7) < ntiles) {
                        const int rr = row & 127;
                        cp_async16(kvb + (row >> 7) * C::kKvBytes + rr * 128 + (((lane & 7) ^ (rr & 7)) << 4),
                                   kvbase + int64_t(idx_cur[i]) * (kD * 2) + c * 128);
                    }
                }
                cp_async_commit();
                pend |= uint32_t(slot) << (4 * npend);
                ++npend;
                if (npend == C::kSlots - 1) { cp_async_wait<C::kSlots - 2>(); flush_one(); }
                if (c == 7) {
                    // signal what is left, then load the next item's indices
                    cp_async_wait<0>();
                    while (npend > 0) flush_one();
                    enxt = queue_read_warp(sh, k + 1, p.status, ok);
                    if ((enxt >> 2) < nitems) load_idx(enxt >> 2, idx_nxt);
                }
                advance(slot, phase, C::kSlots);
            }
            // the B-stage uses of the ring are signalled by the TMA thread
            for (int u = 8; u < C::kUses; ++u, ++use) advance(slot, phase, C::kSlots);
#pragma unroll
            for (int i = 0; i < 32; ++i) idx_cur[i] = idx_nxt[i];
            ecur = enxt;
            cur = ecur >> 2;
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            SMLA_TRACE_SPAN(0, 0);
            int slot = 0; uint32_t phase = 0;
            // Per tile g (scalars, not arrays: a runtime-indexed array would live in
            // local memory, and with shared memory taking most of L1 each access
            // became an L2 round trip on this thread's critical path)
            uint32_t xe_done0 = 0, xe_done1 = 0;   // drains of tile g's accumulator seen
            uint32_t x_uses0 = 0, x_uses1 = 0;     // accumulations of tile g issued
            uint32_t p_seen0 = 0, p_seen1 = 0;     // phases of p_ready[g] waited for
            auto wait_drains = [&](uint32_t& done, uint32_t uses, uint64_t* bar) -> bool {
                while (done < uses) {
                    if (!wait_or_abort(bar, done & 1u, &sh.abort_flag, p.status)) return false;
                    ++done;
                }
                return true;
            };
            // B-stage slot offsets of the dO blocks (P term) and q blocks (dS term)
            const uint32_t do_off = p.qd_mode == 2 ? 0u : 2u * C::kQBytes;
            const uint32_t q_off = p.qd_mode == 2 ? 2u * C::kQBytes : 0u;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int ent = queue_read_thread(sh, it, p.status, ok);
                const int item = ent >> 2;
                if (!ok || item >= nitems) break;
                const int ntiles = ent & 3;
                // A stage may overwrite TMEM only after the previous item's B stage
                // read P / dS ...
                if (it > 0) {
                    ok = ok && wait_or_abort(&sh.b_done[0], (it - 1) & 1, &sh.abort_flag, p.status);
                    ok = ok && wait_or_abort(&sh.b_done[1], (it - 1) & 1, &sh.abort_flag, p.status);
                    SMLA_TRACE_EV(0, it, 1);
                    // ... and after its drains, which follow the dS stash (the stash
                    // reads P^T / dS^T columns that this A stage overwrites)
                    ok = ok && wait_drains(xe_done0, x_uses0, &sh.x_empty[0]);
                    ok = ok && wait_drains(xe_done1, x_uses1, &sh.x_empty[1]);
                    SMLA_TRACE_EV(0, it, 2);
                }
                SMLA_TRACE_EV(0, it, 3);
                for (int c = 0; c < 8 && ok; ++c) {
                    ok = wait_or_abort(&sh.full[slot], phase, &sh.abort_flag, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sb = smem_u32(slots + slot * C::kSlotBytes);
                    for (int g = 0; g < ntiles; ++g) {
                        const uint32_t kvb = sb + C::kKvOff + g * C::kKvBytes;
                        const uint32_t qdb = sb + (TT ? g * 2 * C::kQBytes : 0);   // the tile's token's q | dO
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ss(tbase + g * 256, sdesc_sw128(kvb + k * 32, 16, 1024),
                                   sdesc_sw128(qdb + k * 32, 16, 1024), C::kIdescA, (c | k) != 0);
                        // tile 0's S^T | dP^T are complete one tile-step before tile 1's:
                        // its epilogue starts while tile 1's last MMAs run
                        if (c == 7) mma_commit(&sh.s_full[g]);
                    }
                    mma_commit(&sh.empty[slot]);
                    if ((c + C::kSlots) % C::kUses < 8) mma_commit(&sh.kempty[slot]);
                    advance(slot, phase, C::kSlots);
                }
                if (!ok) break;
                SMLA_TRACE_EV(0, it, 4);
                // B stage: interm columns [128c, 128c + 128), tiles alternating; tile
                // g's first step waits for its P / dS, so tile 0's B stage runs while
                // the epilogue warps work on tile 1.
                for (int c = 0; c < 4 && ok; ++c) {
                    SMLA_TRACE_EV(0, it, 144 + c);
                    ok = wait_or_abort(&sh.full[slot], phase, &sh.abort_flag, p.status);
                    SMLA_TRACE_EV(0, it, 16 + c);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sb = smem_u32(slots + slot * C::kSlotBytes);
                    // one tile-step of the B stage for tile G (a compile-time constant,
                    // so that its counters stay in registers)
                    auto b_step = [&](auto g_tag) -> bool {
                        constexpr int g = decltype(g_tag)::value;
                        uint32_t& p_seen = g ? p_seen1 : p_seen0;
                        uint32_t& xe_done = g ? xe_done1 : xe_done0;
                        uint32_t& x_uses = g ? x_uses1 : x_uses0;
                        if (c == 0) {
                            if (!wait_or_abort(&sh.p_ready[g], p_seen & 1u, &sh.abort_flag, p.status)) return false;
                            ++p_seen;
                            if (g == 0) SMLA_TRACE_EV(0, it, 5);
                        }
                        SMLA_TRACE_EV(0, it, 128 + 2 * c + g);
                        if (!wait_drains(xe_done, x_uses, &sh.x_empty[g])) return false;
                        SMLA_TRACE_EV(0, it, 148 + 2 * c + g);
                        tc_fence_after();
                        SMLA_TRACE_EV(0, it, 24 + 2 * c + g);
                        const uint32_t tile = tbase + g * 256;
#pragma unroll
                        for (int ks = 0; ks < 2 * H / 16; ++ks) {
                            const bool pterm = ks < H / 16;
                            const int kk = pterm ? ks : ks - H / 16;
                            const uint32_t acol = kk * 16 + (pterm ? 0 : 8);
                            // dO (P term) or q (dS term) of the tile's token: two 64-column
                            // blocks of H rows
                            const uint32_t bt = sb + (TT ? g * 4 * C::kQBytes : 0) + (pterm ? do_off : q_off) +
                                                kk * 2048;
                            mma_ts(tile + 128, tile + acol, sdesc_sw128(bt, C::kQBytes, 1024),
                                   C::kIdescB, ks != 0);
                        }
                        SMLA_TRACE_EV(0, it, 136 + 2 * c + g);
                        mma_commit(&sh.x_full[g]);
                        ++x_uses;
                        return true;
                    };
                    ok = b_step(std::integral_constant<int, 0>{});
                    if (ok && ntiles > 1) ok = b_step(std::integral_constant<int, 1>{});
                    if (!ok) break;
                    mma_commit(&sh.empty[slot]);
                    if ((8 + c + C::kSlots) % C::kUses < 8) mma_commit(&sh.kempty[slot]);
                    advance(slot, phase, C::kSlots);
                }
                if (!ok) break;
                mma_commit(&sh.b_done[0]);
                mma_commit(&sh.b_done[1]);
                SMLA_TRACE_EV(0, it, 6);
            }
            // every MMA issued by this thread completes before TMEM is freed
            mma_commit(&sh.drain);
            mbar_wait(&sh.drain, 0, kWaitNs);
            SMLA_TRACE_SPAN(0, 1);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------------- epilogue
        // All eight warps work on every tile. Warp w reads TMEM lane quarter w & 3
        // (ranks 32 (w & 3) .. + 31 of a tile); its group G = (w - 2) >> 2 takes
        // one half of each job: head chunks [0, kSplit) or [kSplit, H / 16) of the
        // P / dS pass, 64-head block G of the dS^T stash, and interm columns
        // [64G, 64G + 64) of each drain. Tile 0 is finished first, so that its B
        // stage starts while the warps work on tile 1.
        const int grp = (warp - 2) >> 2;
        const int quarter = warp & 3;                   // TMEM lane quarter of this warp
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        uint8_t* stage = slots + C::kSlots * C::kSlotBytes + (warp - 2) * kStageBytes;
        // per token of the item (at 2H k for its k-th token): [0, H): -lse*log2(e);
        // [H, 2H): -scale*delta
        float* lsd = reinterpret_cast<float*>(stage);
        static_assert(2 * H * 4 * C::kTok <= kStageBytes, "lse / delta must fit the staging tile");
        constexpr int kChunks = H / 16;                 // 16-head chunks
        constexpr int kSplit = (kChunks + 1) / 2;       // group 0's chunks: [0, kSplit)
        const float c1 = p.scale * kLog2e;
        const float2 c1v = make_float2(c1, c1), scv = make_float2(p.scale, p.scale);
        // TMEM columns of S^T and dP^T (whichever of q / dO came first owns [0, H))
        const uint32_t s_col = p.qd_mode == 2 ? uint32_t(H) : 0u;
        const uint32_t dp_col = p.qd_mode == 2 ? 0u : uint32_t(H);
        constexpr int kHw = (H + 31) / 32;              // head words per lane
        uint32_t s_seen0 = 0, s_seen1 = 0;              // phases of s_full[0 / 1] consumed
        uint32_t p_arr0 = 0, p_arr1 = 0;                // phases of p_ready[0 / 1] arrived on
        uint32_t x_use0 = 0, x_use1 = 0;                // accumulations of tile 0 / 1 consumed
        for (int it = 0;; ++it) {
            if (__any_sync(0xffffffffu, sh.abort_flag != 0)) break;
            bool qok = true;
            const int ent = queue_read_warp(sh, it, p.status, qok);
            const int item = ent >> 2;
            if (!qok || item >= nitems) break;
            const int ntiles = ent & 3;
            // the item's first token and its rank pair (one token per item unless TT)
            const int t = TT ? 2 * item : item / p.npairs, pr = TT ? 0 : item - t * p.npairs;
            auto tok_of = [&](int g) { return TT ? t + g : t; };
            auto rank0_of = [&](int g) { return TT ? 0 : pr * 256 + g * 128; };
            // lane l holds -lse * log2(e) and -scale * delta of heads l, l + 32, ...
            // of each of the item's tokens
            float lse_w[C::kTok][kHw], del_w[C::kTok][kHw];
#pragma unroll
            for (int tk = 0; tk < C::kTok; ++tk) {
                const int tt = t + tk;
#pragma unroll
                for (int k = 0; k < kHw; ++k) {
                    const int h = k * 32 + lane;
                    const bool in = h < H && (!TT || tt < p.T);
                    lse_w[tk][k] = in ? -(__ldg(p.lse + int64_t(tt) * H + h) * kLog2e) : 0.f;
                    del_w[tk][k] = in ? -(p.scale * __ldg(p.delta + int64_t(tt) * H + h)) : 0.f;
                }
            }
            // -lse * log2(e) and -scale * delta of every head go to the head of this
            // warp's staging tile (free once its last TMA store has read it), from
            // where each lane reads them as shared-memory broadcasts
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int tk = 0; tk < C::kTok; ++tk)
#pragma unroll
                for (int k = 0; k < kHw; ++k) {
                    const int h = k * 32 + lane;
                    if (h < H) { lsd[2 * H * tk + h] = lse_w[tk][k]; lsd[2 * H * tk + H + h] = del_w[tk][k]; }
                }
            __syncwarp();
            bool ok = true;
            // ---- P and scale*dS of each tile, written back into TMEM as bf16 pairs
            for (int g2 = 0; g2 < ntiles && ok; ++g2) {
                const int tg = tok_of(g2);
                const int rl = rank0_of(g2) + quarter * 32 + lane;   // this lane's rank
                const float* lsdg = lsd + (TT ? 2 * H * g2 : 0);
                bool valid = false;
                if (rl < p.R) {
                    const int j = __ldg(p.topk + int64_t(tg) * p.K + p.r0 + rl);
                    valid = j >= 0 && j < p.N;
                }
                const uint32_t sphase = (g2 ? s_seen1 : s_seen0) & 1u;
                if (g2) ++s_seen1; else ++s_seen0;
                if (!wait_or_abort_warp(&sh.s_full[g2], sphase, &sh.abort_flag, p.status)) { ok = false; break; }
                if (lane == 0 && warp == 2) SMLA_TRACE_EV(0, it, g2 ? 46 : 7);
                if (lane == 0 && warp == 9 && g2 == 0) SMLA_TRACE_EV(0, it, 44);
                __syncwarp();
                tc_fence_after();
                const uint32_t trow = tbase + lane_off + g2 * 256;
                // P = 2^(S * scale * log2(e) - lse * log2(e)) and
                // scale*dS = P * (scale * dP - scale * delta), two heads per packed
                // fp32x2 operation, over head chunks [K0, K1). Ranks that are masked
                // or past the chunk's end get P = dS = 0 (their bf16 words are
                // cleared); a warp whose 32 ranks are all valid skips that step.
                const uint32_t vmask = valid ? 0xffffffffu : 0u;
                auto pds = [&](auto k0_tag, auto k1_tag, auto masked_tag) {
                    constexpr int K0 = decltype(k0_tag)::value, K1 = decltype(k1_tag)::value;
                    constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
                    for (int c16 = K0; c16 < K1; c16 += 2) {
                        const int nch = (c16 + 1 < K1) ? 2 : 1;
                        uint32_t sv[2][16], dv[2][16];
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            if (u < nch) {
                                tmem_ld16(trow + s_col + (c16 + u) * 16, sv[u]);
                                tmem_ld16(trow + dp_col + (c16 + u) * 16, dv[u]);
                            }
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            if (u >= nch) break;
                            const int k = c16 + u;              // head chunk: heads 16k .. 16k + 15
                            float2 nl[8], nd[8];
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const float4 a = reinterpret_cast<const float4*>(lsdg + k * 16)[v];
                                const float4 b = reinterpret_cast<const float4*>(lsdg + H + k * 16)[v];
                                nl[2 * v] = make_float2(a.x, a.y); nl[2 * v + 1] = make_float2(a.z, a.w);
                                nd[2 * v] = make_float2(b.x, b.y); nd[2 * v + 1] = make_float2(b.z, b.w);
                            }
                            uint32_t pp[8], dd[8];
#pragma unroll
                            for (int j2 = 0; j2 < 8; ++j2) {
                                const float2 sp2 = make_float2(__uint_as_float(sv[u][2 * j2]),
                                                               __uint_as_float(sv[u][2 * j2 + 1]));
                                const float2 dp2 = make_float2(__uint_as_float(dv[u][2 * j2]),
                                                               __uint_as_float(dv[u][2 * j2 + 1]));
                                const float2 arg = __ffma2_rn(sp2, c1v, nl[j2]);
                                const float2 pe = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
                                const float2 ds = __fmul2_rn(pe, __ffma2_rn(dp2, scv, nd[j2]));
                                pp[j2] = pack_bf16x2(pe.x, pe.y);
                                dd[j2] = pack_bf16x2(ds.x, ds.y);
                                if constexpr (kMasked) { pp[j2] &= vmask; dd[j2] &= vmask; }
                            }
                            // P^T and scale*dS^T of chunk k over its columns [16k, 16k + 16)
                            // (chunk k of S^T or of dP^T), already read above
                            tmem_st8(trow + k * 16, pp);
                            tmem_st8(trow + k * 16 + 8, dd);
                        }
                    }
                };
                using Z = std::integral_constant<int, 0>;
                using S = std::integral_constant<int, kSplit>;
                using E = std::integral_constant<int, kChunks>;
                const bool all_valid = __all_sync(0xffffffffu, valid);
                if (grp == 0) {
                    if (all_valid) pds(Z{}, S{}, std::false_type{});
                    else pds(Z{}, S{}, std::true_type{});
                } else {
                    if (all_valid) pds(S{}, E{}, std::false_type{});
                    else pds(S{}, E{}, std::true_type{});
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.p_ready[g2]);
                if (g2) ++p_arr1; else ++p_arr0;
                if (lane == 0 && warp == 2) SMLA_TRACE_EV(0, it, g2 ? 47 : 8);
            }
            if (!ok) break;
            // ---- stash scale * dS^T for the dq kernel: 64-head block `grp` of the
            // warp's 32 rows of tile g2, read back from TMEM (the B-stage MMAs read
            // the same columns; the next item's A stage overwrites them only after
            // this warp's last drain), staged and stored by TMA. Heads >= H are 0;
            // rows past the chunk's end carry dS = 0. A 64-head block may hold
            // chunks the other group wrote, so it is read only once all eight
            // warps have arrived on the tile's p_ready. It runs after the tile's
            // first drain, under the next MMAs rather than before the drains.
            auto stash = [&](int g2) -> bool {
                if (lane == 0) SMLA_TRACE_EV(0, it, 224 + (warp - 2) * 4 + 2 * g2);
                if (grp * 64 >= H) return true;
                const uint32_t pphase = ((g2 ? p_arr1 : p_arr0) - 1u) & 1u;
                if (!wait_or_abort_warp(&sh.p_ready[g2], pphase, &sh.abort_flag, p.status)) return false;
                tc_fence_after();
                const int tg = tok_of(g2);
                const int row0 = rank0_of(g2) + quarter * 32;   // first rank of these rows
                const uint32_t trow = tbase + lane_off + g2 * 256;
                uint32_t dsw[32];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int k = grp * 4 + q4;
                    if (k < kChunks) tmem_ld8(trow + k * 16 + 8, dsw + 8 * q4);
                }
                tmem_wait_ld();
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
                uint4* srow = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const int k = grp * 4 + (v >> 1);
                    srow[v ^ (lane & 7)] = k < kChunks
                        ? make_uint4(dsw[4 * v], dsw[4 * v + 1], dsw[4 * v + 2], dsw[4 * v + 3])
                        : make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&map_ds, grp * 64, tg * p.ds_rows + p.ds_off + row0, stage);
                    bulk_commit();
                }
                __syncwarp();
                if (lane == 0) SMLA_TRACE_EV(0, it, 224 + (warp - 2) * 4 + 2 * g2 + 1);
                return true;
            };
            // ---- drain interm columns [128c, 128c + 128) of every tile, tiles
            // alternating as the MMA issues them; this warp takes columns
            // [64 grp, 64 grp + 64) of its lane quarter
            for (int c = 0; c < 4 && ok; ++c) {
                for (int g2 = 0; g2 < ntiles; ++g2) {
                    const uint32_t xu = g2 ? x_use1 : x_use0;
                    if (!wait_or_abort_warp(&sh.x_full[g2], xu & 1u, &sh.abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    if (g2) ++x_use1; else ++x_use0;
                    if (warp == 2 && lane == 0) SMLA_TRACE_EV(0, it, 32 + 2 * c + g2);
                    if (lane == 0 && (warp == 2 || warp == 9))
                        SMLA_TRACE_EV(0, it, (warp == 2 ? 64 : 96) + 3 * (2 * c + g2));
                    __syncwarp();
                    tc_fence_after();
                    const uint32_t xa = tbase + lane_off + g2 * 256 + 128 + 64 * grp;
                    uint32_t v0[32], v1[32];
                    tmem_ld32(xa, v0);
                    tmem_ld32(xa + 32, v1);
                    tmem_wait_ld();
                    // the accumulator is read: the MMA may reuse it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.x_empty[g2]);
                    if (lane == 0 && (warp == 2 || warp == 9))
                        SMLA_TRACE_EV(0, it, (warp == 2 ? 64 : 96) + 3 * (2 * c + g2) + 1);
                    if (lane == 0) SMLA_TRACE_EV(0, it, 160 + (warp - 2) * 8 + 2 * c + g2);
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    uint4* srow = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll
                    for (int v = 0; v < 4; ++v) srow[v ^ (lane & 7)] = pack8(v0 + 8 * v);
#pragma unroll
                    for (int v = 0; v < 4; ++v) srow[(v + 4) ^ (lane & 7)] = pack8(v1 + 8 * v);
                    const int col = 128 * c + 64 * grp;
                    const int tg = tok_of(g2);
                    const int drow0 = rank0_of(g2) + quarter * 32;   // first rank of these rows
                    if (drow0 + 32 <= p.R) {
                        // the warp's 32 ranks all belong to this chunk: one TMA store
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&map_im, col, tg * p.R + drow0, stage);
                            bulk_commit();
                        }
                    } else {
                        // ragged last rows: plain stores of the rows < R
                        __syncwarp();
                        store_staged_rows(stage, p.interm + (int64_t(tg) * p.R + drow0) * kD + col, kD,
                                          p.R - drow0, lane);
                    }
                    __syncwarp();
                    if (lane == 0 && (warp == 2 || warp == 9))
                        SMLA_TRACE_EV(0, it, (warp == 2 ? 64 : 96) + 3 * (2 * c + g2) + 2);
                    if (c == 0 && !stash(g2)) { ok = false; break; }
                    if (c == 0 && g2 == ntiles - 1 && lane == 0 && warp == 2) SMLA_TRACE_EV(0, it, 14);
                }
                if (warp == 2 && lane == 0) SMLA_TRACE_EV(0, it, 40 + c);
            }
            if (warp == 2 && lane == 0) SMLA_TRACE_EV(0, it, 9);
            if (!ok) break;
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ======================================================================= dq
struct DqParams {
    const uint16_t* kv;   // [N, 512]
    const int32_t* topk;
    float* dq_acc;        // fp32 [T, H, 512] between chunks, or nullptr
    uint16_t* dq_out;     // bf16 [T, H, 512]
    int T, K, N, r0, R, Rp;
    bool first, last;
    const int32_t* cnt;   // compacted table: valid entries per token (see SdiParams), or nullptr
    unsigned* status;
};

// 64-rank chunks of token t: all Rp / 64, or with a compacted table those
// holding its valid entries (at least one: an all-masked token's dq is the
// product of its zero dS rows).
__device__ __forceinline__ int dq_nchunks(const DqParams& p, int t, int nkc) {
    if (!p.cnt) return nkc;
    const int m = __ldg(p.cnt + t);
    return m < 1 ? 1 : (m + 63) >> 6;
}

struct DqShared {
    uint64_t full[4], empty[4];
    uint64_t d_full[2], d_empty[2], drain;
    uint32_t tbase;
    volatile int abort_flag;
};

constexpr int kDqSlots = 4;
// Copy warps: two teams of 4 warps. Chunk n of the CTA's sequence sits in slot
// n % 4; team k fills the chunks n = k, k + 2, ... (16 rows per warp), waits
// for its own copies only and signals the slot. With four 128-byte rows per
// copy instruction, two teams measured faster than four (0.42 vs 0.47 ms at
// T=4096, H=128, topk=512): each copy's latency grows with the copies in flight.
constexpr int kDqTeams = 2;
constexpr int kDqTeamWarps = 4;
constexpr int kDqCopyWarps = kDqTeams * kDqTeamWarps;
static_assert(kDqTeams <= kDqSlots, "parity waits need slots >= teams");
constexpr int kDqThreads = (6 + kDqCopyWarps) * 32;         // TMA, MMA, 4 epilogue, copy warps
constexpr int kDqABytes = 2 * 64 * 128;        // two 64-head blocks x 64 ranks
constexpr int kDqBBytes = 4 * 64 * 128;        // four 64-column blocks x 64 ranks
constexpr int kDqSlotBytes = kDqABytes + kDqBBytes;
// Per epilogue warp, two 32-row x 128-byte staging tiles for the TMA stores of bf16 dq.
constexpr int kDqStageBytes = 4 * 2 * kStageBytes;
constexpr int kDqSmem = int(sizeof(DqShared)) + 1024 + kDqSlots * kDqSlotBytes + kDqStageBytes;
static_assert(kDqSmem <= 232448, "shared memory of one CTA is at most 227 KB");
constexpr uint32_t kDqIdesc = idesc_bf16(128, 256, true, true);

template <int H>
__global__ void __launch_bounds__(kDqThreads, 1)
dq_kernel(const __grid_constant__ CUtensorMap map_ds, const __grid_constant__ CUtensorMap map_dq,
          const DqParams p) {
    extern __shared__ uint8_t smem_raw[];
    DqShared& sh = *reinterpret_cast<DqShared*>(smem_raw);
    uint8_t* slots = align1024(smem_raw + sizeof(DqShared));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = p.T * 2;
    const int nkc = p.Rp / 64;

    if (threadIdx.x == 0) {
        // full: the TMA thread's arrive (with the dS bytes) + the 128 threads of the chunk's team
        for (int s = 0; s < kDqSlots; ++s) {
            mbar_init(&sh.full[s], 1 + 32 * kDqTeamWarps);  // TMA thread + the slot's team
            mbar_init(&sh.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) { mbar_init(&sh.d_full[b], 1); mbar_init(&sh.d_empty[b], 4); }
        mbar_init(&sh.drain, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(&sh.tbase, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sh.tbase;

    if (warp == 0) {
        // -------------------------------------- TMA producer (scale*dS^T tiles)
        if (lane == 0) {
            int slot = 0; uint32_t phase = 0; int issued = 0;
            bool ok = true;
            int it = 0;
            // chunk counts are loaded one item ahead (off this thread's critical path)
            int nk_next = int(blockIdx.x) < nitems ? dq_nchunks(p, int(blockIdx.x) >> 1, nkc) : 0;
            for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++it) {
                const int t = item >> 1;
                const int nk = nk_next;
                const int later = item + int(gridDim.x);
                nk_next = later < nitems ? dq_nchunks(p, later >> 1, nkc) : 0;
                SMLA_TRACE_EV(1, it, 0);
                for (int kc = 0; kc < nk; ++kc) {
                    ok = wait_or_abort(&sh.empty[slot], phase ^ 1u, &sh.abort_flag, p.status);
                    if (!ok) break;
                    uint8_t* sb = slots + slot * kDqSlotBytes;
                    mbar_arrive_expect_tx(&sh.full[slot], kDqABytes);
                    for (int hb = 0; hb < 2; ++hb)
                        tma_load_2d(sb + hb * 8192, &map_ds, hb * 64, t * p.Rp + kc * 64, &sh.full[slot]);
                    ++issued;
                    advance(slot, phase, kDqSlots);
                }
                SMLA_TRACE_EV(1, it, 1);
            }
            if (sh.abort_flag) {
                int s = slot; uint32_t ph = phase;
                for (int k = 0; k < kDqSlots && k < issued; ++k) {
                    if (--s < 0) { s = kDqSlots - 1; ph ^= 1u; }
                    mbar_wait(&sh.full[s], ph, kWaitNs / 8);
                }
            }
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ------------------------------------------------ kv gather (cp.async)
        // Team k (warps 4k .. 4k + 3 of the copy warps) fills the chunks
        // n = k, k + 2, ... of this CTA's chunk sequence (chunk n in slot n % 4); warp w of the team
        // copies rows 16w .. 16w + 15: per round one 64-column block of four rows, lane l
        // copying the 16-byte piece (l & 7) of row 16w + 4q + (l >> 3) (four rows of 128 bytes
        // per instruction measured faster than one row of 512 bytes). Lane i < 16 holds the
        // index of row 16w + i, loaded one chunk of the team ahead.
        const int gw = warp - 6;
        const int team = gw / kDqTeamWarps, wt = gw % kDqTeamWarps;
        const int rq = lane >> 3, piece = lane & 7;
        // The CTA's chunk sequence: its items blockIdx.x, blockIdx.x + gridDim.x,
        // ..., each of dq_nchunks 64-rank chunks; chunk n of the sequence sits in
        // slot n % kDqSlots and is filled by team n % kDqTeams.
        // (nk: the cursor item's chunk count, loaded once per item)
        struct Cursor { int item, kc, nk; };
        auto step = [&](Cursor& c) {
            if (c.item >= nitems) return;
            if (++c.kc == c.nk) {
                c.kc = 0;
                c.item += int(gridDim.x);
                c.nk = c.item < nitems ? dq_nchunks(p, c.item >> 1, nkc) : 0;
            }
        };
        auto load_idx = [&](const Cursor& c) -> int {
            if (c.item >= nitems) return -1;
            const int rl = c.kc * 64 + 16 * wt + (lane & 15);
            int j = -1;
            if (rl < p.R) {
                j = __ldg(p.topk + int64_t(c.item >> 1) * p.K + p.r0 + rl);
                if (j < 0 || j >= p.N) j = -1;     // masked or invalid: its dS is zero
            }
            return j;
        };
        Cursor cur{int(blockIdx.x), 0,
                   int(blockIdx.x) < nitems ? dq_nchunks(p, int(blockIdx.x) >> 1, nkc) : 0};
        for (int k = 0; k < team; ++k) step(cur);
        int idx = load_idx(cur);
        for (int n = team; cur.item < nitems; n += kDqTeams) {
            const int item = cur.item;
            const int slot = n % kDqSlots;
            const uint32_t phase = uint32_t(n / kDqSlots) & 1u;
            uint8_t* sbase = slots + slot * kDqSlotBytes + kDqABytes;
            bool ok = true;
            if (lane == 0) ok = wait_or_abort(&sh.empty[slot], phase ^ 1u, &sh.abort_flag, p.status);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            Cursor nx = cur;
            for (int k = 0; k < kDqTeams; ++k) step(nx);
            const int nxt = load_idx(nx);
            const char* src0 = reinterpret_cast<const char*>(p.kv) + (item & 1) * 512 + piece * 16;
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const int r = 16 * wt + 4 * qd + rq;
                const int j = __shfl_sync(0xffffffffu, idx, 4 * qd + rq);
                const char* src = src0 + int64_t(j < 0 ? 0 : j) * (kD * 2);
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    cp_async16_zfill(sbase + b * 8192 + r * 128 + ((piece ^ (r & 7)) << 4), src + b * 128,
                                     j < 0 ? 0u : 16u);
            }
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(&sh.full[slot]);
            idx = nxt;
            cur = nx;
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            SMLA_TRACE_SPAN(1, 0);
            int slot = 0; uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            int nk_next = int(blockIdx.x) < nitems ? dq_nchunks(p, int(blockIdx.x) >> 1, nkc) : 0;
            for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++it) {
                const int b = it & 1;
                const int nk = nk_next;
                const int later = item + int(gridDim.x);
                nk_next = later < nitems ? dq_nchunks(p, later >> 1, nkc) : 0;
                if (it >= 2) ok = wait_or_abort(&sh.d_empty[b], ((it >> 1) - 1) & 1, &sh.abort_flag, p.status);
                SMLA_TRACE_EV(1, it, 2);
                for (int kc = 0; kc < nk && ok; ++kc) {
                    ok = wait_or_abort(&sh.full[slot], phase, &sh.abort_flag, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sb = smem_u32(slots + slot * kDqSlotBytes);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tbase + 256 * b, sdesc_sw128(sb + ks * 2048, 8192, 1024),
                               sdesc_sw128(sb + kDqABytes + ks * 2048, 8192, 1024), kDqIdesc,
                               (kc | ks) != 0);
                    mma_commit(&sh.empty[slot]);
                    advance(slot, phase, kDqSlots);
                }
                if (!ok) break;
                mma_commit(&sh.d_full[b]);
                SMLA_TRACE_EV(1, it, 3);
            }
            mma_commit(&sh.drain);
            mbar_wait(&sh.drain, 0, kWaitNs);
            SMLA_TRACE_SPAN(1, 1);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        // bf16 dq without an fp32 accumulator, whole 32-head quarters: each warp
        // stages 64 columns of its 32 heads (one row per lane, 128-byte
        // swizzle) and writes them with one TMA store; per-lane 16-byte stores
        // touch 32 rows per instruction instead
        constexpr bool kTmaOut = H % 32 == 0;
        const bool tma_out = kTmaOut && p.dq_acc == nullptr;
        uint8_t* stage = slots + kDqSlots * kDqSlotBytes + (warp - 2) * 2 * kStageBytes;
        int it = 0;
        for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++it) {
            const int t = item >> 1, half = item & 1;
            const int b = it & 1;
            if (!wait_or_abort_warp(&sh.d_full[b], (it >> 1) & 1, &sh.abort_flag, p.status)) break;
            if (warp == 2 && lane == 0) SMLA_TRACE_EV(1, it, 4);
            __syncwarp();                   // tcgen05.ld is warp-collective
            tc_fence_after();
            const int64_t base = (int64_t(t) * H + h) * kD + half * 256;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t v[32];
                tmem_ld32(tbase + lane_off + 256 * b + 32 * c, v);
                tmem_wait_ld();
                if (tma_out) {
                    if (quarter * 32 < H) {
                        uint8_t* st = stage + ((c >> 1) & 1) * kStageBytes;
                        // the staging tile's previous store (two stores ago) has been read
                        if ((c & 1) == 0) {
                            if (lane == 0) bulk_wait_read_1();
                            __syncwarp();
                        }
                        uint4* srow = reinterpret_cast<uint4*>(st + lane * 128);
#pragma unroll
                        for (int k = 0; k < 4; ++k) srow[((c & 1) * 4 + k) ^ (lane & 7)] = pack8(v + 8 * k);
                        if (c & 1) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&map_dq, half * 256 + (c >> 1) * 64, t * H + quarter * 32, st);
                                bulk_commit();
                            }
                        }
                    }
                } else if (h < H) {
                    float f[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) f[k] = __uint_as_float(v[k]);
                    const int64_t off = base + 32 * c;
                    if (p.dq_acc && !p.first) {
                        const float4* acc = reinterpret_cast<const float4*>(p.dq_acc + off);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float4 a = acc[k];
                            f[4 * k] += a.x; f[4 * k + 1] += a.y; f[4 * k + 2] += a.z; f[4 * k + 3] += a.w;
                        }
                    }
                    if (p.dq_acc && !p.last) {
                        float4* acc = reinterpret_cast<float4*>(p.dq_acc + off);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            acc[k] = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
                    } else {
                        uint4* o = reinterpret_cast<uint4*>(p.dq_out + off);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            o[k] = make_uint4(pack_bf16x2(f[8 * k], f[8 * k + 1]),
                                              pack_bf16x2(f[8 * k + 2], f[8 * k + 3]),
                                              pack_bf16x2(f[8 * k + 4], f[8 * k + 5]),
                                              pack_bf16x2(f[8 * k + 6], f[8 * k + 7]));
                    }
                }
                __syncwarp();               // lanes with h >= H rejoin before the next load
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.d_empty[b]);
            if (warp == 2 && lane == 0) SMLA_TRACE_EV(1, it, 5);
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ============================================================ wait self-test
// One CTA of four warps runs the unwind path of the kernels above on purpose:
// warp 0 holds 32 TMEM columns, thread 32 waits (wait_or_abort) on an
// mbarrier that nothing arrives on, with a limit of `limit_ns`; the wait runs
// out, sets SMLA_ERR_TIMEOUT and the abort flag; warps 2-3 stand for the other
// roles and leave their loop when they see the flag (each of their waits is
// bounded too); then TMEM is freed. No copy or MMA is issued, so nothing is in
// flight when the CTA exits.
__global__ void __launch_bounds__(128, 1) wait_selftest_kernel(unsigned* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    __shared__ volatile int abort_flag;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) { tmem_alloc(&tbase, 32); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 32) {
        wait_or_abort(&bar, 0, &abort_flag, status, limit_ns);
    } else if (warp >= 2) {
        // other roles: poll the flag, each poll a bounded wait of its own
        const uint64_t t0 = globaltimer_ns();
        while (!abort_flag && globaltimer_ns() - t0 < 4 * limit_ns) __nanosleep(1000);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, 32);
    }
}

// ================================================================= launchers
int sm_count() {
    static int cached[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) cached[dev] = sms;
    return sms;
}

int set_smem_attrs_once(const void* fn, int smem, bool* done) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 0;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return -1;
        done[dev] = true;
    }
    return 0;
}

template <int H, bool TT>
cudaError_t launch_sdi_hh(const ChunkArgs& a, cudaStream_t s) {
    using C = SdiCfg<H, TT>;
    static bool attr_done[64] = {false};
    if (set_smem_attrs_once(reinterpret_cast<const void*>(sdi_kernel<H, TT>), C::kSmem, attr_done))
        return cudaErrorInvalidValue;
    const int Rp = round_up_ranks(a.R), Hp = pad_heads(H);
    CUtensorMap mq, mdo, mqda, mqdb, mim, mds;
    // q and dO as one paired tensor (one TMA box per ring slot instead of two or
    // four) when their distance is a stride the tensor map can encode
    int qd_mode = 0;
    {
        const uintptr_t uq = reinterpret_cast<uintptr_t>(a.q), ud = reinterpret_cast<uintptr_t>(a.dO);
        const bool q_first = uq < ud;
        const void* lo = q_first ? static_cast<const void*>(a.q) : static_cast<const void*>(a.dO);
        const uint64_t dist = q_first ? uint64_t(ud - uq) : uint64_t(uq - ud);
        if (make_tmap_bf16_pair5d(&mqda, lo, dist, uint64_t(a.T), H, 1, C::kTok) &&
            make_tmap_bf16_pair5d(&mqdb, lo, dist, uint64_t(a.T), H, 2, C::kTok))
            qd_mode = q_first ? 1 : 2;
        else
            mqda = mqdb = CUtensorMap{};
    }
    if (!make_tmap_bf16_2d(&mq, a.q, uint64_t(a.T) * H, kD, kD, H, 64, true) ||
        !make_tmap_bf16_2d(&mdo, a.dO, uint64_t(a.T) * H, kD, kD, H, 64, true) ||
        !make_tmap_bf16_2d(&mim, a.interm, uint64_t(a.T) * a.R, kD, kD, 32, 64, true) ||
        !make_tmap_bf16_2d(&mds, a.dsT, uint64_t(a.T) * a.ds_rows, Hp, Hp, 32, 64, true))
        return cudaErrorInvalidValue;
    SdiParams sp{};
    sp.ds_rows = a.ds_rows; sp.ds_off = a.ds_off;
    sp.kv = a.kv; sp.topk = a.topk; sp.lse = a.lse; sp.delta = a.delta; sp.interm = a.interm;
    sp.dsT = a.dsT;
    sp.T = a.T; sp.K = a.K; sp.N = a.N; sp.r0 = a.r0; sp.R = a.R; sp.Rp = Rp; sp.Hp = Hp;
    sp.npairs = (a.R + 255) / 256;
    sp.tiles_last = (a.R - (sp.npairs - 1) * 256) > 128 ? 2 : 1;
    sp.scale = a.scale; sp.status = a.status;
    sp.qd_mode = qd_mode;
    sp.work_ctr = sdi_work_counter(a.status);
    sp.cnt = a.cnt;
    sp.tt = TT ? 1 : 0;
    const int64_t items = TT ? (int64_t(a.T) + 1) / 2 : int64_t(a.T) * sp.npairs;
    const int sms = sm_count();
    const int grid = int(items < sms ? items : sms);
    cudaError_t e = cudaMemsetAsync(sp.work_ctr, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    sdi_kernel<H, TT><<<grid, C::kThreads, C::kSmem, s>>>(mq, mdo, mqda, mqdb, mim, mds, sp);
    note_launch();
    return cudaGetLastError();
}

// Two-token items when a token has at most one tile (chunks of at most 128
// ranks) and a ring slot holds two tokens' q and dO (heads <= 64): the B
// stage then alternates tiles again, and each TMA box serves two tokens.
template <int H>
cudaError_t launch_sdi_h(const ChunkArgs& a, cudaStream_t s) {
    if constexpr (H <= 64) {
        if (a.R <= 128) return launch_sdi_hh<H, true>(a, s);
    }
    return launch_sdi_hh<H, false>(a, s);
}

template <int H>
cudaError_t launch_dq_h(const ChunkArgs& a, cudaStream_t s) {
    static bool attr_done[64] = {false};
    if (set_smem_attrs_once(reinterpret_cast<const void*>(dq_kernel<H>), kDqSmem, attr_done))
        return cudaErrorInvalidValue;
    const int Rp = round_up_ranks(a.R), Hp = pad_heads(H);
    CUtensorMap mds, mdq = CUtensorMap{};
    if (!make_tmap_bf16_2d(&mds, a.dsT, uint64_t(a.T) * Rp, Hp, Hp, 64, 64, true))
        return cudaErrorInvalidValue;
    // bf16 dq rows in boxes of 32 heads x 64 columns (whole 32-head quarters only)
    if (H % 32 == 0 && !a.dq_acc &&
        !make_tmap_bf16_2d(&mdq, a.dq_out, uint64_t(a.T) * H, kD, kD, 32, 64, true))
        return cudaErrorInvalidValue;
    DqParams dp{};
    dp.kv = a.kv; dp.topk = a.topk; dp.dq_acc = a.dq_acc; dp.dq_out = a.dq_out;
    dp.T = a.T; dp.K = a.K; dp.N = a.N; dp.r0 = a.r0; dp.R = a.R; dp.Rp = Rp;
    dp.first = a.first_chunk; dp.last = a.last_chunk; dp.status = a.status;
    dp.cnt = a.cnt;
    const int64_t items = int64_t(a.T) * 2;
    // dq runs beside the dKV gather (another stream). Each dq CTA's throughput
    // is fixed by its own pipeline, while the gather speeds up with every SM it
    // gets, so dq takes the share of the SMs at which both end together. Beside
    // a whole gather (T=4096, H=128, topk=512): 96 of 152 SMs, 1.809 ms per
    // backward against 1.833 / 1.816 / 1.819 / 1.829 / 1.829 ms with 88 / 104 /
    // 112 / 121 / 136 (dq ends last below 96). Beside the last rank chunk's
    // gather only (rank chunks, dq over all ranks at the end): 4/5 of the SMs.
    const int share = a.dq_beside_part ? (sm_count() * 4) / 5 : (sm_count() * 96) / 152;
    const int sms = share > 0 ? share : 1;
    const int grid = int(items < sms ? items : sms);
    dq_kernel<H><<<grid, kDqThreads, kDqSmem, s>>>(mds, mdq, dp);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

#ifdef SMLA_TRACE
extern "C" int smla_trace_span_copy(unsigned long long* host) {
    return cudaMemcpyFromSymbol(host, g_smla_cta_span, sizeof(g_smla_cta_span)) == cudaSuccess ? 0 : 1;
}
extern "C" int smla_trace_copy(unsigned long long* host, size_t count) {
    const size_t n = sizeof(g_smla_trace) / sizeof(g_smla_trace[0]);
    return cudaMemcpyFromSymbol(host, g_smla_trace,
                                sizeof(unsigned long long) * (count < n ? count : n)) == cudaSuccess
               ? 0 : 1;
}
#endif

#define SMLA_DISPATCH_H(FN, a, s)              \
    switch ((a).H) {                           \
        case 16: return FN<16>(a, s);          \
        case 32: return FN<32>(a, s);          \
        case 48: return FN<48>(a, s);          \
        case 64: return FN<64>(a, s);          \
        case 80: return FN<80>(a, s);          \
        case 96: return FN<96>(a, s);          \
        case 112: return FN<112>(a, s);        \
        case 128: return FN<128>(a, s);        \
        default: return cudaErrorInvalidValue; \
    }

cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 128, 0, s>>>(status, limit_ns);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_attn_sdi(const ChunkArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    SMLA_DISPATCH_H(launch_sdi_h, a, s)
}

cudaError_t launch_attn_dq(const ChunkArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    SMLA_DISPATCH_H(launch_dq_h, a, s)
}

}  // namespace smla
