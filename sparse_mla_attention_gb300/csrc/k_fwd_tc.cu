// k_fwd_tc.cu -- sparse MLA forward on the tensor cores (tcgen05 / TMEM / TMA).
//
// Definition (aiter "Sparse MLA training backward", Contract section and the
// lse paragraph under its usage example): for token t, head h and the valid
// ranks r of topk[t, :] (index idx_r),
//   s_r = scale * <q[t,h,:], kv[idx_r,:]>,
//   m = max(sink_h, max_r s_r),   l = exp(sink_h - m) + sum_r exp(s_r - m),
//   lse = m + ln(l),   O[t,h,:] = sum_r exp(s_r - m) * kv[idx_r,:] / l
// (no sink term without a sink). The last form equals sum_r exp(s_r - lse) kv.
//
// fwd_tc_kernel: persistent, one CTA per SM (TMA warp, MMA warp, 8 epilogue
// warps, 8 copy warps), work item = one token (topk <= 512, H a multiple of 32
// up to 128).
//  * S stage: S = q x kv^T with M = 128 (the heads; lanes >= H unused), N = 256
//    ranks per rank tile, K = 512 in eight 64-column chunks. The chunk loop is
//    outermost, so each 64-column q chunk is loaded once per token (TMA, a ring
//    of three q buffers) and serves every rank tile; kv rows are gathered by the
//    copy teams. S of rank tile j lives in TMEM columns [256j, 256j + 256).
//  * Softmax: two epilogue warps per TMEM lane quarter (one thread per head),
//    each over half of the 32-rank groups: pass 1 takes the max over the valid
//    ranks (the two halves swap theirs; the sink joins), pass 2 forms
//    e = exp(s - m), sums it, and writes bf16(e) pairs over S columns already
//    read: half 0 in ascending group order at column 16gq, half 1 in descending
//    order at column 16ng + 16gq (ng groups in all). Half 1 hands its sum to
//    half 0, which writes lse and drains O.
//  * O stage: O' = P' x kv with A = P' from TMEM, M = 128, N = 128 columns of D
//    per chunk, K = 128 ranks per use (kv rows gathered again, MN-major). The
//    two chunk accumulators lie between the two halves' P' (columns
//    [128, 384) for 512 ranks, [256, 512) for 256) and alternate; the drain
//    scales a row by 1/l, rounds to bf16 and stores it through a staging tile
//    by TMA.
// Shared memory: a ring of five 32 KB kv slots (an S-stage use holds 256 rank
// rows x 64 columns, an O-stage use 128 rank rows x 128 columns as two
// 64-column blocks), three 16 KB q buffers and four 4 KB staging tiles. Uses
// are numbered across the CTA's tokens; copy team k (four warps) fills the
// uses g = k, k + 2, ... in slots of its own (team 0: slots 0-2, team 1: slots
// 3-4; see ft_slot): two teams, because more copies in flight per SM made
// every copy slower (measured with 1 to 5 teams).
// The next token's q is prefetched into L2 while the current one runs.
// Every mbarrier wait is bounded; a timeout sets SMLA_ERR_TIMEOUT, stops the
// CTA's loops, waits (bounded) for its own copies and MMAs and frees TMEM.
#include "smla_internal.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace smla {
using namespace sm100;

namespace {

constexpr uint64_t kFtWaitNs = 2000000000ull;
constexpr float kFtLog2e = 1.4426950408889634f;
constexpr int kFtSlots = 5;
constexpr int kFtSlotBytes = 32768;
constexpr int kFtTeams = 2;

// Kv use g is filled by copy team g % kFtTeams, which owns a fixed set of
// slots and fills them in turn: every slot is filled by one team only, in the
// order the MMA consumes it, so a team waiting for a slot is never more than
// one phase of that slot's empty barrier ahead (a parity wait cannot tell two
// phases apart). With 5 slots, team 0 owns slots 0-2 and team 1 slots 3-4.
__device__ __forceinline__ void ft_slot(int g, int& slot, uint32_t& phase) {
    const int team = g % kFtTeams, i = g / kFtTeams;
    const int base = kFtSlots / kFtTeams, extra = kFtSlots % kFtTeams;
    const int n = base + (team < extra ? 1 : 0);
    const int first = team * base + (team < extra ? team : extra);
    slot = first + i % n;
    phase = uint32_t(i / n) & 1u;
}
constexpr int kFtTeamWarps = 4;
constexpr int kFtEpiWarps = 8;                                     // two per TMEM lane quarter
constexpr int kFtCopyWarp0 = 2 + kFtEpiWarps;
constexpr int kFtThreads = (kFtCopyWarp0 + kFtTeams * kFtTeamWarps) * 32;   // TMA, MMA, 8 epilogue, 8 copy
constexpr int kFtQBufs = 3;
constexpr int kFtQBytes = 128 * 128;                               // up to 128 rows x 64 columns
constexpr int kFtStageBytes = 32 * 128;
constexpr int kFtMaxRanks = 512;

struct FtParams {
    const uint16_t* kv;
    const int32_t* topk;
    const float* sink;     // [H] or nullptr
    float* lse;            // [T, H]
    int T, H, K, N;
    float scale;
    unsigned* status;
};

struct FtShared {
    uint64_t full[kFtSlots], empty[kFtSlots];
    uint64_t q_full[kFtQBufs], q_empty[kFtQBufs];
    uint64_t s_full, p_ready, o_full[2], o_empty[2], drain;
    uint64_t xchg[4], sum_bar[4];          // per lane quarter: the two halves' max / sum hand-over
    uint32_t tbase;
    volatile int abort_flag;
    uint32_t valid[kFtEpiWarps][kFtMaxRanks / 64];   // per epilogue warp: its groups' valid-rank bits
    float red_max[2][128];                 // per half and head: the half's max score
    float red_sum[128];                    // per head: half 1's sum of exp(s - m)
};

constexpr int kFtRing = kFtSlots * kFtSlotBytes;
constexpr int kFtSmem = int(sizeof(FtShared)) + 1024 + kFtRing + kFtQBufs * kFtQBytes + 4 * kFtStageBytes;
static_assert(kFtSmem <= 232448, "shared memory of one CTA is at most 227 KB");
constexpr uint32_t kFtIdescS = idesc_bf16(128, 256, false, false);
constexpr uint32_t kFtIdescO = idesc_bf16(128, 128, false, true);

__device__ __forceinline__ uint8_t* ft_align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool ft_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        unsigned* status) {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, kFtWaitNs)) return true;
    *abort_flag = 1;
    flag_status(status, SMLA_ERR_TIMEOUT);
    return false;
}

// Every lane waits; the warp goes on only if all of them saw the phase (the
// loads that follow are warp-collective).
__device__ __forceinline__ bool ft_wait_warp(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, unsigned* status) {
    const bool ok = ft_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok) != 0;
}

// topk[t, r] as stored (-1 past the last rank). Nothing branches on the value
// here: the copy warps load a use's indices one use ahead and look at them
// only when that use comes up.
__device__ __forceinline__ int ft_raw(const FtParams& p, int t, int r) {
    return r < p.K ? __ldg(p.topk + int64_t(t) * p.K + r) : -1;
}

// Row to copy for a raw index, or -1 for a masked or invalid one (its smem row
// is zero-filled instead: copying one placeholder row for every masked slot
// would send every CTA to the same L2 lines); `bad` collects indices outside
// [-1, N).
__device__ __forceinline__ int ft_row_of(int j, int N, bool& bad) {
    bad |= (j < -1) | (j >= N);
    return (j >= 0 && j < N) ? j : -1;
}

// One 16-byte piece of a kv row into shared memory: `src` is the piece's
// address in row `row`, or in row 0 for a masked slot (row < 0), whose piece
// is zero-filled without reading global memory.
__device__ __forceinline__ void ft_copy_piece(void* dst, const char* src, int row) {
    cp_async16_zfill(dst, src, row < 0 ? 0u : 16u);
}

}  // namespace

__global__ void __launch_bounds__(kFtThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_o,
              const FtParams p) {
    extern __shared__ uint8_t smem_raw[];
    FtShared& sh = *reinterpret_cast<FtShared*>(smem_raw);
    uint8_t* ring = ft_align1024(smem_raw + sizeof(FtShared));
    uint8_t* qbuf = ring + kFtRing;
    uint8_t* stage_base = qbuf + kFtQBufs * kFtQBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt2 = (p.K + 255) / 256;              // 256-rank tiles of the S stage (1..2)
    const int nt = (p.K + 127) / 128;               // 128-rank tiles of the O stage (1..4)
    const int uses = 8 * nt2 + 4 * nt;              // kv uses per token
    const int ng = 8 * nt2;                         // 32-rank groups of S
    // TMEM after the softmax: P' of half 0 in [0, 8ng), of half 1 in [24ng, 32ng); the
    // two O accumulators sit between them (ng = 16) or above S (ng = 8)
    const int acc0 = ng == 16 ? 128 : 256;
    const int ntok = (p.T - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x);
    const int H = p.H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kFtSlots; ++s) {
            mbar_init(&sh.full[s], 32 * kFtTeamWarps);
            mbar_init(&sh.empty[s], 1);
        }
        for (int b = 0; b < kFtQBufs; ++b) {
            mbar_init(&sh.q_full[b], 1);
            mbar_init(&sh.q_empty[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.o_full[b], 1);
            mbar_init(&sh.o_empty[b], 4);
        }
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.p_ready, kFtEpiWarps);
        for (int q = 0; q < 4; ++q) {
            mbar_init(&sh.xchg[q], 2);     // lane 0 of each of the quarter's two warps
            mbar_init(&sh.sum_bar[q], 1);  // lane 0 of the quarter's half-1 warp
        }
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
        // ---------------------------------------------- TMA producer (q chunks)
        if (lane == 0) {
            int qi = 0;
            bool ok = true;
            for (int it = 0; it < ntok && ok; ++it) {
                const int t = int(blockIdx.x) + it * int(gridDim.x);
                if (it + 1 < ntok)      // the next token's q into L2 while this one runs
                    for (int c = 0; c < 8; ++c) tma_prefetch_2d(&map_q, c * 64, (t + int(gridDim.x)) * H);
                for (int c = 0; c < 8; ++c, ++qi) {
                    const int b = qi % kFtQBufs;
                    ok = ft_wait(&sh.q_empty[b], (uint32_t(qi / kFtQBufs) & 1u) ^ 1u, &sh.abort_flag, p.status);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&sh.q_full[b], uint32_t(H) * 128u);
                    tma_load_2d(qbuf + b * kFtQBytes, &map_q, c * 64, t * H, &sh.q_full[b]);
                }
            }
            if (sh.abort_flag)   // the loads already issued land before the CTA exits
                for (int k = 1; k <= kFtQBufs && qi - k >= 0; ++k)
                    mbar_wait(&sh.q_full[(qi - k) % kFtQBufs], uint32_t((qi - k) / kFtQBufs) & 1u, kFtWaitNs / 8);
        }
        __syncwarp();
    } else if (warp >= kFtCopyWarp0) {
        // ------------------------------------------ kv gather (copy teams, cp.async)
        // Team k fills the uses g = k, k + 2, ... An S-stage use (chunk c, rank
        // tile j) is 256 rank rows x 64 columns: warp wt copies rows
        // 64wt .. 64wt + 63. An O-stage use (chunk c, rank tile j) is 128 rank
        // rows x 128 columns: warp wt copies rows 32wt .. 32wt + 31, one
        // 64-column block at a time. Every copy instruction covers four rows of
        // 128 bytes (measured faster than fewer, longer rows).
        // The row indices of the team's next use are loaded during this one.
        const int gw = warp - kFtCopyWarp0;
        const int team = gw / kFtTeamWarps, wt = gw % kFtTeamWarps;
        const int piece = lane & 7;
        const char* kvb = reinterpret_cast<const char*>(p.kv);
        const int total = ntok * uses;
        // lane's raw indices of use g (two for an S-stage use, one for an O-stage use)
        auto load_use = [&](int g, int& r0, int& r1) {
            r0 = -1; r1 = -1;
            if (g >= total) return;
            const int it = g / uses, u = g - it * uses;
            const int t = int(blockIdx.x) + it * int(gridDim.x);
            if (u < 8 * nt2) {
                const int j = u % nt2;
                r0 = ft_raw(p, t, 256 * j + 64 * wt + lane);
                r1 = ft_raw(p, t, 256 * j + 64 * wt + 32 + lane);
            } else {
                const int j = (u - 8 * nt2) % nt;
                r0 = ft_raw(p, t, 128 * j + 32 * wt + lane);
            }
        };
        bool bad = false;
        int raw0, raw1;
        load_use(team, raw0, raw1);
        for (int g = team; g < total; g += kFtTeams) {
            int n0, n1;
            load_use(g + kFtTeams, n0, n1);
            const int c0 = ft_row_of(raw0, p.N, bad), c1 = ft_row_of(raw1, p.N, bad);
            int slot; uint32_t ph;
            ft_slot(g, slot, ph);
            bool ok = true;
            if (lane == 0) ok = ft_wait(&sh.empty[slot], ph ^ 1u, &sh.abort_flag, p.status);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            uint8_t* sb = ring + slot * kFtSlotBytes;
            const int u = g % uses;
            if (u < 8 * nt2) {
                const int c = u / nt2;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int rl = 4 * i + (lane >> 3);              // row within the warp's 64
                    const int row = __shfl_sync(0xffffffffu, i < 8 ? c0 : c1, rl & 31);
                    ft_copy_piece(sb + (64 * wt + rl) * 128 + ((piece ^ (rl & 7)) << 4),
                                  kvb + int64_t(row < 0 ? 0 : row) * (kD * 2) + c * 128 + piece * 16, row);
                }
            } else {
                const int c = (u - 8 * nt2) / nt;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rl = 4 * i + (lane >> 3);              // row within the warp's 32
                    const int row = __shfl_sync(0xffffffffu, c0, rl);
                    const char* src = kvb + int64_t(row < 0 ? 0 : row) * (kD * 2) + c * 256 + piece * 16;
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk)
                        ft_copy_piece(sb + blk * 16384 + (32 * wt + rl) * 128 + ((piece ^ (rl & 7)) << 4),
                                      src + blk * 128, row);
                }
            }
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(&sh.full[slot]);
            raw0 = n0; raw1 = n1;
        }
        cp_async_wait<0>();
        if (bad) flag_status(p.status, SMLA_ERR_INDEX);
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int g = 0, qi = 0;
            uint32_t o_uses[2] = {0, 0}, o_drained[2] = {0, 0};
            bool ok = true;
            for (int it = 0; it < ntok && ok; ++it) {
                // S overwrites TMEM the previous token's O chunks use: wait for their drains
                for (int b = 0; b < 2 && ok; ++b)
                    while (ok && o_drained[b] < o_uses[b]) {
                        ok = ft_wait(&sh.o_empty[b], o_drained[b] & 1u, &sh.abort_flag, p.status);
                        ++o_drained[b];
                    }
                for (int c = 0; c < 8 && ok; ++c, ++qi) {
                    const int b = qi % kFtQBufs;
                    ok = ft_wait(&sh.q_full[b], uint32_t(qi / kFtQBufs) & 1u, &sh.abort_flag, p.status);
                    if (!ok) break;
                    const uint32_t qa = smem_u32(qbuf + b * kFtQBytes);
                    for (int j = 0; j < nt2 && ok; ++j, ++g) {
                        int slot; uint32_t ph;
                        ft_slot(g, slot, ph);
                        ok = ft_wait(&sh.full[slot], ph, &sh.abort_flag, p.status);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t sb = smem_u32(ring + slot * kFtSlotBytes);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ss(tbase + 256 * j, sdesc_sw128(qa + k * 32, 16, 1024),
                                   sdesc_sw128(sb + k * 32, 16, 1024), kFtIdescS, (c | k) != 0);
                        mma_commit(&sh.empty[slot]);
                    }
                    if (ok) mma_commit(&sh.q_empty[b]);
                }
                if (!ok) break;
                mma_commit(&sh.s_full);
                ok = ft_wait(&sh.p_ready, it & 1, &sh.abort_flag, p.status);
                if (!ok) break;
                tc_fence_after();
                for (int c = 0; c < 4 && ok; ++c) {
                    const int b = c & 1;
                    while (ok && o_drained[b] < o_uses[b]) {
                        ok = ft_wait(&sh.o_empty[b], o_drained[b] & 1u, &sh.abort_flag, p.status);
                        ++o_drained[b];
                    }
                    if (!ok) break;
                    tc_fence_after();
                    for (int j = 0; j < nt && ok; ++j, ++g) {
                        int slot; uint32_t ph;
                        ft_slot(g, slot, ph);
                        ok = ft_wait(&sh.full[slot], ph, &sh.abort_flag, p.status);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t sb = smem_u32(ring + slot * kFtSlotBytes);
                        // P' of rank tile j: half 0's groups at 64j, half 1's at 16ng + 64j
                        const uint32_t pa = tbase + (j < nt2 ? 64 * j : 16 * ng + 64 * j);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mma_ts(tbase + acc0 + 128 * b, pa + 8 * k,
                                   sdesc_sw128(sb + k * 2048, 16384, 1024), kFtIdescO, (j | k) != 0);
                        mma_commit(&sh.empty[slot]);
                    }
                    if (!ok) break;
                    mma_commit(&sh.o_full[b]);
                    ++o_uses[b];
                }
            }
            mma_commit(&sh.drain);
            mbar_wait(&sh.drain, 0, kFtWaitNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ softmax + O drain
        // Two warps per TMEM lane quarter: half 0 (warps 2-5) takes the rank groups
        // [0, ng/2), half 1 (warps 6-9) the groups [ng/2, ng). Each writes P' over
        // S columns it has already read: half 0 group gq at 16gq (ascending order),
        // half 1 group gq at 16ng + 16gq (descending order: that column range
        // belongs to S group ng/2 + gq/2 >= gq, read first). The halves swap their
        // maxima, half 1 hands its sum to half 0, and half 0 drains O.
        const int ew = warp - 2;
        const int half = ew >> 2;
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;              // this thread's head (TMEM lane)
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        uint32_t* vmask = sh.valid[ew];
        uint8_t* stage = stage_base + (ew & 3) * kFtStageBytes;
        const bool store_rows = quarter * 32 < H;       // H is a multiple of 32
        const float sink_h = (p.sink && h < H) ? __ldg(p.sink + h) : -INFINITY;
        const float c1 = p.scale * kFtLog2e;
        const int nh = ng / 2;                          // groups per half (4 or 8)
        const int gbeg = half * nh;
        // The TMEM loads below are warp-collective: every lane runs every load,
        // and per-lane conditions only select which loaded values count.
        // Lanes of heads >= H (rows of the q tile left stale) count no rank.
        const uint32_t live = h < H ? 0xffffffffu : 0u;
        uint32_t o_seen[2] = {0, 0};
        for (int it = 0; it < ntok; ++it) {
            const int t = int(blockIdx.x) + it * int(gridDim.x);
            if (__any_sync(0xffffffffu, sh.abort_flag != 0)) break;
            // valid-rank bits of this warp's groups
#pragma unroll
            for (int m = 0; m < kFtMaxRanks / 64; ++m) {
                const int r = 32 * (gbeg + m) + lane;
                bool v = false;
                if (m < nh && r < p.K) {
                    const int j = __ldg(p.topk + int64_t(t) * p.K + r);
                    v = j >= 0 && j < p.N;
                }
                const uint32_t bits = __ballot_sync(0xffffffffu, v);
                if (lane == 0) vmask[m] = bits;
            }
            __syncwarp();
            if (!ft_wait_warp(&sh.s_full, it & 1, &sh.abort_flag, p.status)) break;
            tc_fence_after();
            const uint32_t trow = tbase + lane_off;
            // pass 1: max of the valid scores of this half, then of both halves
            float mx = -INFINITY;
#pragma unroll 1
            for (int m = 0; m < nh; ++m) {
                uint32_t v[32];
                tmem_ld32(trow + 32 * (gbeg + m), v);
                tmem_wait_ld();
                const uint32_t bits = vmask[m] & live;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if ((bits >> e) & 1u) mx = fmaxf(mx, __uint_as_float(v[e]));
            }
            sh.red_max[half][h] = mx;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.xchg[quarter]);
            if (!ft_wait_warp(&sh.xchg[quarter], it & 1, &sh.abort_flag, p.status)) break;
            mx = fmaxf(mx, sh.red_max[half ^ 1][h]);
            // m = max(sink, scale * max s)
            const float m = fmaxf(sink_h, mx * p.scale);
            const bool any = m != -INFINITY;
            const float mb = any ? m * kFtLog2e : 0.f;
            // pass 2: e = exp(s - m) summed, and written as bf16 pairs over columns
            // already read
            float psum = 0.f;
#pragma unroll 1
            for (int mm = 0; mm < nh; ++mm) {
                const int m_i = half == 0 ? mm : nh - 1 - mm;
                const int gq = gbeg + m_i;
                uint32_t v[32];
                tmem_ld32(trow + 32 * gq, v);
                tmem_wait_ld();
                const uint32_t bits = any ? (vmask[m_i] & live) : 0u;
                uint32_t pp[16];
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) {
                    const float a = ((bits >> (2 * e2)) & 1u)
                                        ? ex2_approx(fmaf(__uint_as_float(v[2 * e2]), c1, -mb)) : 0.f;
                    const float b = ((bits >> (2 * e2 + 1)) & 1u)
                                        ? ex2_approx(fmaf(__uint_as_float(v[2 * e2 + 1]), c1, -mb)) : 0.f;
                    psum += a + b;
                    pp[e2] = pack_bf16x2(a, b);
                }
                const uint32_t pcol = half == 0 ? 16 * gq : 16 * ng + 16 * gq;
                tmem_st8(trow + pcol, pp);
                tmem_st8(trow + pcol + 8, pp + 8);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_ready);
            if (half == 1) {
                // hand the sum to half 0 (which drains O); red_sum is rewritten only
                // after half 0 has read it: the next token's S stage waits for the drains
                sh.red_sum[h] = psum;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.sum_bar[quarter]);
                continue;
            }
            if (!ft_wait_warp(&sh.sum_bar[quarter], it & 1, &sh.abort_flag, p.status)) break;
            float sum = (p.sink && any) ? ex2_approx((sink_h - m) * kFtLog2e) : 0.f;
            sum += psum + sh.red_sum[h];
            const float lse = any ? m + logf(sum) : -INFINITY;
            if (h < H) p.lse[int64_t(t) * H + h] = lse;
            const float inv = sum > 0.f ? 1.f / sum : 0.f;
            // drain the four O chunks of 128 columns
            bool ok = true;
            for (int c = 0; c < 4; ++c) {
                const int b = c & 1;
                if (!ft_wait_warp(&sh.o_full[b], o_seen[b] & 1u, &sh.abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                ++o_seen[b];
                tc_fence_after();
                for (int hh = 0; hh < 2; ++hh) {
                    __syncwarp();
                    if (store_rows) {
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
                    }
                    uint4* srow = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll 1
                    for (int gq = 0; gq < 2; ++gq) {
                        uint32_t v[32];
                        tmem_ld32(trow + acc0 + 128 * b + 64 * hh + 32 * gq, v);
                        tmem_wait_ld();
                        if (hh == 1 && gq == 1) {       // the accumulator is read: the MMA may reuse it
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&sh.o_empty[b]);
                        }
                        if (store_rows) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint32_t* a = v + 8 * q;
                                srow[(4 * gq + q) ^ (lane & 7)] = make_uint4(
                                    pack_bf16x2(__uint_as_float(a[0]) * inv, __uint_as_float(a[1]) * inv),
                                    pack_bf16x2(__uint_as_float(a[2]) * inv, __uint_as_float(a[3]) * inv),
                                    pack_bf16x2(__uint_as_float(a[4]) * inv, __uint_as_float(a[5]) * inv),
                                    pack_bf16x2(__uint_as_float(a[6]) * inv, __uint_as_float(a[7]) * inv));
                            }
                        }
                    }
                    if (store_rows) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&map_o, 128 * c + 64 * hh, t * H + quarter * 32, stage);
                            bulk_commit();
                        }
                    }
                }
            }
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

// Tensor-core forward for H a multiple of 32 (32..128) and 1 <= topk <= 512;
// returns cudaErrorNotSupported for other shapes (the caller then uses the
// CUDA-core forward).
cudaError_t launch_fwd_tc(const uint16_t* q, const uint16_t* kv, const int32_t* topk,
                          const float* sink, uint16_t* o, float* lse, int T, int H, int K,
                          int num_kv, float scale, unsigned* status, cudaStream_t s) {
    if (H % 32 != 0 || H < 32 || H > 128 || K < 1 || K > kFtMaxRanks) return cudaErrorNotSupported;
    if (T == 0) return cudaSuccess;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFtSmem) !=
            cudaSuccess)
            return cudaGetLastError();
        attr_done[dev] = true;
    }
    CUtensorMap mq, mo;
    if (!make_tmap_bf16_2d(&mq, q, uint64_t(T) * H, kD, kD, H, 64, true) ||
        !make_tmap_bf16_2d(&mo, o, uint64_t(T) * H, kD, kD, 32, 64, true))
        return cudaErrorInvalidValue;
    FtParams fp{};
    fp.kv = kv; fp.topk = topk; fp.sink = sink; fp.lse = lse;
    fp.T = T; fp.H = H; fp.K = K; fp.N = num_kv; fp.scale = scale; fp.status = status;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = T < sms ? T : sms;
    fwd_tc_kernel<<<grid, kFtThreads, kFtSmem, s>>>(mq, mo, fp);
    note_launch();
    return cudaGetLastError();
}

}  // namespace smla
