// k_fwd_tc.cu -- sparse MLA forward on the tensor cores (tcgen05 / TMEM / TMA).
//
// Definition (aiter "Sparse MLA training backward", Contract section and the
// lse paragraph under its usage example): for token t, head h and the valid
// ranks r of topk[t, :] (index idx_r),
//   s_r = scale * <q[t,h,:], kv[idx_r,:]>,
//   m = max(sink_h, max_r s_r),   lse = m + ln(exp(sink_h - m) + sum_r exp(s_r - m)),
//   O[t,h,:] = sum_r exp(s_r - lse) * kv[idx_r,:]      (no sink term without a sink).
//
// fwd_tc_kernel: persistent, one CTA per SM, work item = one token (topk <= 512,
// H a multiple of 32).
//  * S stage: per 128-rank tile j, S = q x kv^T with M = 128 (the heads, lanes
//    >= H unused), N = 128 ranks, K = 512 in eight 64-column steps; q tiles by
//    TMA, kv rows gathered by the copy teams; S of tile j in TMEM columns
//    [128j, 128j + 128).
//  * Softmax: each epilogue thread owns one head (one TMEM lane): the max and
//    the sum over its valid ranks (and the sink), lse, then P = exp(s - lse) as
//    bf16 pairs written back over the S columns already read: ranks 2m, 2m + 1
//    in column m, so P occupies [0, 64 * tiles).
//  * O stage: O = P x kv with A = P from TMEM, M = 128, N = 128 columns of D
//    per chunk, K = the ranks (kv rows gathered again, MN-major); the chunk
//    accumulators alternate between TMEM columns [256, 384) and [384, 512), and
//    a drained chunk leaves as bf16 through a staging tile and TMA stores.
// Shared memory: a ring of four 32 KB slots. An S-stage slot holds a q tile
// (H rows x 64 columns) and a kv tile (128 rows x 64 columns); an O-stage slot
// holds a kv tile of 128 rows x 128 columns (two 64-column blocks). Copy team k
// (four warps) fills slot k for uses k, k + 4, ...; every token has a multiple
// of four uses, so use u of a token always lands in slot u % 4.
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
constexpr int kFtSlots = 4;
constexpr int kFtSlotBytes = 32768;
constexpr int kFtTeamWarps = 4;
constexpr int kFtThreads = (6 + kFtSlots * kFtTeamWarps) * 32;   // TMA, MMA, 4 epilogue, 16 copy
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
    uint64_t s_full, p_ready, o_full[2], o_empty[2], drain;
    uint32_t tbase;
    volatile int abort_flag;
    uint32_t valid[4][kFtMaxRanks / 32];   // per epilogue warp: valid-rank bits of the token
};

constexpr int kFtSmem = int(sizeof(FtShared)) + 1024 + kFtSlots * kFtSlotBytes + 4 * kFtStageBytes;
static_assert(kFtSmem <= 232448, "shared memory of one CTA is at most 227 KB");
constexpr uint32_t kFtIdescS = idesc_bf16(128, 128, false, false);
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

__device__ __forceinline__ void ft_advance(int& slot, uint32_t& phase) {
    if (++slot == kFtSlots) { slot = 0; phase ^= 1u; }
}

// Row index of rank r of token t (0 for a masked, invalid or out-of-range rank).
__device__ __forceinline__ int ft_row(const FtParams& p, int t, int r) {
    if (r >= p.K) return 0;
    const int j = __ldg(p.topk + int64_t(t) * p.K + r);
    if (j < -1 || j >= p.N) { flag_status(p.status, SMLA_ERR_INDEX); return 0; }
    return j < 0 ? 0 : j;
}

}  // namespace

__global__ void __launch_bounds__(kFtThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_o,
              const FtParams p) {
    extern __shared__ uint8_t smem_raw[];
    FtShared& sh = *reinterpret_cast<FtShared*>(smem_raw);
    uint8_t* slots = ft_align1024(smem_raw + sizeof(FtShared));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = (p.K + 127) / 128;               // rank tiles per token (1..4)
    const int uses = 12 * nt;                       // 8 S-stage and 4 O-stage uses per tile
    const int H = p.H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kFtSlots; ++s) {
            mbar_init(&sh.full[s], 1 + 32 * kFtTeamWarps);   // TMA thread + the slot's team
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.p_ready, 4);
        for (int b = 0; b < 2; ++b) { mbar_init(&sh.o_full[b], 1); mbar_init(&sh.o_empty[b], 4); }
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
        // ---------------------------------------------- TMA producer (q tiles)
        if (lane == 0) {
            int slot = 0; uint32_t phase = 0; int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.T && ok; t += gridDim.x) {
                for (int u = 0; u < uses; ++u) {
                    ok = ft_wait(&sh.empty[slot], phase ^ 1u, &sh.abort_flag, p.status);
                    if (!ok) break;
                    if (u < 8 * nt) {
                        // S stage: q columns [64c, 64c + 64) of the token's H rows
                        const int c = u & 7;
                        mbar_arrive_expect_tx(&sh.full[slot], uint32_t(H) * 128u);
                        tma_load_2d(slots + slot * kFtSlotBytes, &map_q, c * 64, t * H, &sh.full[slot]);
                    } else {
                        mbar_arrive(&sh.full[slot]);        // O stage: the slot holds kv only
                    }
                    ++issued;
                    ft_advance(slot, phase);
                }
            }
            if (sh.abort_flag) {
                int s = slot; uint32_t ph = phase;
                for (int k = 0; k < kFtSlots && k < issued; ++k) {
                    if (--s < 0) { s = kFtSlots - 1; ph ^= 1u; }
                    mbar_wait(&sh.full[s], ph, kFtWaitNs / 8);
                }
            }
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ------------------------------------------ kv gather (copy teams, cp.async)
        // Team k fills slot k for the token's uses k, k + 4, ...; warp wt of the
        // team copies rows 32wt .. 32wt + 31 of the use's 128-row kv tile. Lane i
        // holds the index of row 32wt + i of each rank tile of the token.
        const int gw = warp - 6;
        const int team = gw / kFtTeamWarps, wt = gw % kFtTeamWarps;
        const int piece = lane & 7;
        uint32_t phase = 0;
        bool ok = true;
        uint8_t* sb = slots + team * kFtSlotBytes;
        int cur[4], nxt[4];
        auto load_rows = [&](int t, int (&out)[4]) {
#pragma unroll
            for (int j = 0; j < 4; ++j) out[j] = (t < p.T && j < nt) ? ft_row(p, t, 128 * j + 32 * wt + lane) : 0;
        };
        if (int(blockIdx.x) < p.T) load_rows(blockIdx.x, cur);
        const char* kvb = reinterpret_cast<const char*>(p.kv);
        for (int t = blockIdx.x; t < p.T && ok; t += gridDim.x) {
            load_rows(t + int(gridDim.x), nxt);
            for (int u = team; u < uses; u += kFtSlots) {
                if (lane == 0) ok = ft_wait(&sh.empty[team], phase ^ 1u, &sh.abort_flag, p.status);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                if (u < 8 * nt) {
                    // S stage: tile j, columns [64c, 64c + 64): four rows per round
                    const int j = u >> 3, c = u & 7;
                    const int idx = j == 0 ? cur[0] : j == 1 ? cur[1] : j == 2 ? cur[2] : cur[3];
                    uint8_t* dst = sb + 16384;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rl = 4 * i + (lane >> 3);              // row within the warp's 32
                        const int r = 32 * wt + rl;                      // row of the tile
                        const int row = __shfl_sync(0xffffffffu, idx, rl);
                        cp_async16(dst + r * 128 + ((piece ^ (r & 7)) << 4),
                                   kvb + int64_t(row) * (kD * 2) + c * 128 + piece * 16);
                    }
                } else {
                    // O stage: tile j, columns [128c, 128c + 128) as two 64-column
                    // blocks: two rows per round
                    const int v = u - 8 * nt, c = v / nt, j = v - c * nt;
                    const int idx = j == 0 ? cur[0] : j == 1 ? cur[1] : j == 2 ? cur[2] : cur[3];
                    const int blk = (lane >> 3) & 1;
                    uint8_t* dst = sb + blk * 16384;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int rl = 2 * i + (lane >> 4);
                        const int r = 32 * wt + rl;
                        const int row = __shfl_sync(0xffffffffu, idx, rl);
                        cp_async16(dst + r * 128 + ((piece ^ (r & 7)) << 4),
                                   kvb + int64_t(row) * (kD * 2) + (c * 128 + blk * 64) * 2 + piece * 16);
                    }
                }
                cp_async_commit();
                cp_async_wait<0>();
                fence_proxy_async_smem();
                mbar_arrive(&sh.full[team]);
                phase ^= 1u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
        }
        cp_async_wait<0>();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int slot = 0; uint32_t phase = 0;
            uint32_t o_uses[2] = {0, 0}, o_drained[2] = {0, 0};
            bool ok = true;
            int it = 0;
            for (int t = blockIdx.x; t < p.T && ok; t += gridDim.x, ++it) {
                // S overwrites all of TMEM: the previous token's O chunks must be drained
                for (int b = 0; b < 2 && ok; ++b)
                    while (ok && o_drained[b] < o_uses[b]) {
                        ok = ft_wait(&sh.o_empty[b], o_drained[b] & 1u, &sh.abort_flag, p.status);
                        ++o_drained[b];
                    }
                for (int j = 0; j < nt && ok; ++j)
                    for (int c = 0; c < 8 && ok; ++c) {
                        ok = ft_wait(&sh.full[slot], phase, &sh.abort_flag, p.status);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t sb = smem_u32(slots + slot * kFtSlotBytes);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ss(tbase + 128 * j, sdesc_sw128(sb + k * 32, 16, 1024),
                                   sdesc_sw128(sb + 16384 + k * 32, 16, 1024), kFtIdescS, (c | k) != 0);
                        mma_commit(&sh.empty[slot]);
                        ft_advance(slot, phase);
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
                    for (int j = 0; j < nt && ok; ++j) {
                        ok = ft_wait(&sh.full[slot], phase, &sh.abort_flag, p.status);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t sb = smem_u32(slots + slot * kFtSlotBytes);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mma_ts(tbase + 256 + 128 * b, tbase + 64 * j + 8 * k,
                                   sdesc_sw128(sb + k * 2048, 16384, 1024), kFtIdescO, (j | k) != 0);
                        mma_commit(&sh.empty[slot]);
                        ft_advance(slot, phase);
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
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;              // this thread's head (TMEM lane)
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const int ew = warp - 2;
        uint32_t* vmask = sh.valid[ew];
        uint8_t* stage = slots + kFtSlots * kFtSlotBytes + ew * kFtStageBytes;
        const bool store_rows = quarter * 32 < H;       // H is a multiple of 32
        const float sink_h = (p.sink && h < H) ? __ldg(p.sink + h) : -INFINITY;
        const float c1 = p.scale * kFtLog2e;
        uint32_t o_seen[2] = {0, 0};
        int it = 0;
        for (int t = blockIdx.x; t < p.T; t += gridDim.x, ++it) {
            if (__any_sync(0xffffffffu, sh.abort_flag != 0)) break;
            // valid-rank bits of the token (each warp its own copy)
#pragma unroll
            for (int m = 0; m < kFtMaxRanks / 32; ++m) {
                const int r = 32 * m + lane;
                bool v = false;
                if (r < p.K) {
                    const int j = __ldg(p.topk + int64_t(t) * p.K + r);
                    v = j >= 0 && j < p.N;
                }
                const uint32_t bits = __ballot_sync(0xffffffffu, v);
                if (lane == 0) vmask[m] = bits;
            }
            __syncwarp();
            if (!ft_wait_warp(&sh.s_full, it & 1, &sh.abort_flag, p.status)) break;
            __syncwarp();
            tc_fence_after();
            const uint32_t trow = tbase + lane_off;
            // The TMEM loads below are warp-collective: every lane runs every load,
            // and per-lane conditions only select which loaded values count.
            // Lanes of heads >= H (rows of the q tile left stale) count no rank.
            const uint32_t live = h < H ? 0xffffffffu : 0u;
            // pass 1: max of the valid scores
            float mx = -INFINITY;
            for (int j = 0; j < nt; ++j)
#pragma unroll 1
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t v[32];
                    tmem_ld32(trow + 128 * j + 32 * q4, v);
                    tmem_wait_ld();
                    const uint32_t bits = vmask[4 * j + q4] & live;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if ((bits >> e) & 1u) mx = fmaxf(mx, __uint_as_float(v[e]));
                }
            // m = max(sink, scale * max s); the sum of exp(s - m), plus the sink term
            const float m = fmaxf(sink_h, mx * p.scale);
            const bool any = m != -INFINITY;
            const float mb = any ? m * kFtLog2e : 0.f;
            float sum = (p.sink && any) ? ex2_approx((sink_h - m) * kFtLog2e) : 0.f;
            for (int j = 0; j < nt; ++j)
#pragma unroll 1
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t v[32];
                    tmem_ld32(trow + 128 * j + 32 * q4, v);
                    tmem_wait_ld();
                    const uint32_t bits = any ? (vmask[4 * j + q4] & live) : 0u;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if ((bits >> e) & 1u) sum += ex2_approx(fmaf(__uint_as_float(v[e]), c1, -mb));
                }
            const float lse = m == -INFINITY ? -INFINITY : m + logf(sum);
            if (h < H) p.lse[int64_t(t) * H + h] = lse;
            // pass 3: P = exp(s - lse) as bf16 pairs over the S columns already read
            const float lb = lse * kFtLog2e;
            for (int j = 0; j < nt; ++j)
#pragma unroll 1
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t v[32];
                    tmem_ld32(trow + 128 * j + 32 * q4, v);
                    tmem_wait_ld();
                    const uint32_t bits = lse == -INFINITY ? 0u : (vmask[4 * j + q4] & live);
                    uint32_t pp[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        const float a = ((bits >> (2 * e2)) & 1u)
                                            ? ex2_approx(fmaf(__uint_as_float(v[2 * e2]), c1, -lb)) : 0.f;
                        const float b = ((bits >> (2 * e2 + 1)) & 1u)
                                            ? ex2_approx(fmaf(__uint_as_float(v[2 * e2 + 1]), c1, -lb)) : 0.f;
                        pp[e2] = pack_bf16x2(a, b);
                    }
                    tmem_st8(trow + 64 * j + 16 * q4, pp);
                    tmem_st8(trow + 64 * j + 16 * q4 + 8, pp + 8);
                }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_ready);
            // drain the four O chunks of 128 columns
            bool ok = true;
            for (int c = 0; c < 4; ++c) {
                const int b = c & 1;
                if (!ft_wait_warp(&sh.o_full[b], o_seen[b] & 1u, &sh.abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                ++o_seen[b];
                __syncwarp();
                tc_fence_after();
                for (int hh = 0; hh < 2; ++hh) {
                    __syncwarp();
                    if (store_rows) {
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
                    }
                    uint4* srow = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll 1
                    for (int g = 0; g < 2; ++g) {
                        uint32_t v[32];
                        tmem_ld32(trow + 256 + 128 * b + 64 * hh + 32 * g, v);
                        tmem_wait_ld();
                        if (hh == 1 && g == 1) {        // the accumulator is read: the MMA may reuse it
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&sh.o_empty[b]);
                        }
                        if (store_rows) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint32_t* a = v + 8 * q;
                                srow[(4 * g + q) ^ (lane & 7)] = make_uint4(
                                    pack_bf16x2(__uint_as_float(a[0]), __uint_as_float(a[1])),
                                    pack_bf16x2(__uint_as_float(a[2]), __uint_as_float(a[3])),
                                    pack_bf16x2(__uint_as_float(a[4]), __uint_as_float(a[5])),
                                    pack_bf16x2(__uint_as_float(a[6]), __uint_as_float(a[7])));
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
