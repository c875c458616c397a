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
// is (token t, 256 ranks) = two 128-rank tiles. Per tile, one kv tile gathered
// by TMA (tile::gather4) feeds a single MMA stream that computes S^T and dP^T
// together: M = 128 ranks, N = 2H (the q rows of token t followed by its dO
// rows), K = 512, accumulated in TMEM. Epilogue warps turn each TMEM row
// (one rank) into P and scale*dS, write them back into TMEM as bf16 (the A
// operand of the next GEMM) and stash scale*dS for the dq kernel. Then
// interm = [P | scale*dS] x [dO ; q] runs with A from TMEM (M = 128 ranks,
// N = 64 columns of D per step, K = 2H) and is drained to global memory.
// TMEM (512 columns): tile g owns columns [256g, 256g+256): S^T | dP^T in
// [0, 2H), then P^T (bf16 pairs) in [0, H/2) and scale*dS^T in [H/2, H); the
// interm accumulators double-buffer in [128, 192) and [192, 256).
//
// dq_kernel: persistent; item = (token, half of D). dq = (scale*dS) x kv:
// M = 128 (heads, zero-padded), N = 256, K = ranks, both operands MN-major
// (scale*dS^T rows from the stash, kv rows gathered), accumulated in TMEM
// (two 256-column buffers) and written as bf16 (or added to an fp32
// accumulator between rank chunks).
//
// Every mbarrier wait is bounded (kWaitNs); a timeout sets SMLA_ERR_TIMEOUT in
// the status word, stops the CTA's loops, waits (bounded) for its own copies
// and MMAs in flight and frees its TMEM.
#include "smla_internal.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace smla {
using namespace sm100;

namespace {

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

struct SdiParams {
    const int32_t* topk;
    const float* lse;
    const float* delta;
    uint16_t* interm;     // [T, R, 512]
    uint16_t* dsT;        // [T, Rp, Hp]
    int T, K, N, r0, R, Rp, Hp;
    int npairs;           // items per token: ceil(R / 256)
    int tiles_last;       // tiles (1 or 2) in a token's last item
    float scale;
    unsigned* status;
};

struct SdiShared {
    uint64_t full[8], empty[8];
    uint64_t s_full, p_ready, x_full[2], x_empty[2], b_done[2], drain;
    uint32_t tbase;
    volatile int abort_flag;
    int idx[256];
};

template <int H>
struct SdiCfg {
    static constexpr int kQBytes = H * 128;                 // H rows x 64 columns bf16
    static constexpr int kKvBytes = 128 * 128;              // 128 ranks x 64 columns bf16
    static constexpr int kSlotBytes = 2 * kQBytes + 2 * kKvBytes;
    static constexpr int kSlotsRaw = 196608 / kSlotBytes;
    static constexpr int kSlots = kSlotsRaw > 8 ? 8 : kSlotsRaw;
    static constexpr int kThreads = 320;                    // TMA, MMA, 8 epilogue warps
    static constexpr int kSmem = int(sizeof(SdiShared)) + 1024 + kSlots * kSlotBytes;
    static constexpr uint32_t kIdescA = idesc_bf16(128, 2 * H, false, false);
    static constexpr uint32_t kIdescB = idesc_bf16(128, 64, false, true);
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, unsigned* status) {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, kWaitNs)) return true;
    *abort_flag = 1;
    flag_status(status, SMLA_ERR_TIMEOUT);
    return false;
}

template <int H>
__global__ void __launch_bounds__(320, 1)
sdi_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
           const __grid_constant__ CUtensorMap map_kv, const SdiParams p) {
    using C = SdiCfg<H>;
    extern __shared__ uint8_t smem_raw[];
    SdiShared& sh = *reinterpret_cast<SdiShared*>(smem_raw);
    uint8_t* slots = align1024(smem_raw + sizeof(SdiShared));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = p.T * p.npairs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kSlots; ++s) { mbar_init(&sh.full[s], 1); mbar_init(&sh.empty[s], 1); }
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.p_ready, 8);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.x_full[b], 1);
            mbar_init(&sh.x_empty[b], 8);
            mbar_init(&sh.b_done[b], 1);
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
        // ------------------------------------------------------ TMA producer
        int slot = 0; uint32_t phase = 0;
        int issued = 0;   // slot fills whose completion this warp has not seen
        bool ok = true;
        for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
            const int t = item / p.npairs, pr = item - t * p.npairs;
            const int ntiles = pr == p.npairs - 1 ? p.tiles_last : 2;
            const int rl0 = pr * 256;
            for (int i = lane; i < 256; i += 32) {
                const int rl = rl0 + i;
                int j = 0;
                if (rl < p.R) {
                    j = __ldg(p.topk + int64_t(t) * p.K + p.r0 + rl);
                    if (j < -1 || j >= p.N) { flag_status(p.status, SMLA_ERR_INDEX); j = 0; }
                    if (j < 0) j = 0;            // masked: any real row; its P is zeroed
                }
                sh.idx[i] = j;
            }
            __syncwarp();
            if (lane == 0) {
                for (int c = 0; c < 16 && ok; ++c) {
                    ok = wait_or_abort(&sh.empty[slot], phase ^ 1u, &sh.abort_flag, p.status);
                    if (!ok) break;
                    uint8_t* sb = slots + slot * C::kSlotBytes;
                    const int dc = c & 7;
                    const bool a_stage = c < 8;
                    const uint32_t bytes = 2 * C::kQBytes + (a_stage ? ntiles * C::kKvBytes : 0);
                    mbar_arrive_expect_tx(&sh.full[slot], bytes);
                    tma_load_2d(sb, &map_q, dc * 64, t * H, &sh.full[slot]);
                    tma_load_2d(sb + C::kQBytes, &map_do, dc * 64, t * H, &sh.full[slot]);
                    if (a_stage) {
                        for (int g = 0; g < ntiles; ++g) {
                            uint8_t* kvb = sb + 2 * C::kQBytes + g * C::kKvBytes;
                            const int* ix = sh.idx + g * 128;
                            for (int q4 = 0; q4 < 32; ++q4)
                                tma_gather4(kvb + q4 * 512, &map_kv, dc * 64, ix[4 * q4],
                                            ix[4 * q4 + 1], ix[4 * q4 + 2], ix[4 * q4 + 3],
                                            &sh.full[slot]);
                        }
                    }
                    ++issued;
                    if (++slot == C::kSlots) { slot = 0; phase ^= 1u; }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            __syncwarp();
        }
        if (lane == 0 && sh.abort_flag) {
            // bounded wait for this warp's own copies still in flight
            int s = slot; uint32_t ph = phase;
            for (int k = 0; k < C::kSlots && k < issued; ++k) {
                if (--s < 0) { s = C::kSlots - 1; ph ^= 1u; }
                mbar_wait(&sh.full[s], ph, kWaitNs / 8);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int slot = 0; uint32_t phase = 0;
            uint32_t xe_done[2] = {0, 0};
            bool ok = true;
            int it = 0;
            for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++it) {
                const int t = item / p.npairs, pr = item - t * p.npairs;
                (void)t;
                const int ntiles = pr == p.npairs - 1 ? p.tiles_last : 2;
                // A stage: S^T | dP^T for each tile.
                if (it > 0) {
                    ok = ok && wait_or_abort(&sh.b_done[0], (it - 1) & 1, &sh.abort_flag, p.status);
                    ok = ok && wait_or_abort(&sh.b_done[1], (it - 1) & 1, &sh.abort_flag, p.status);
                    if (2 * H > 128) {   // S^T | dP^T overlaps the interm buffers: wait for the drains
                        for (int b = 0; b < 2 && ok; ++b)
                            while (ok && xe_done[b] < uint32_t(it) * 4u) {
                                ok = wait_or_abort(&sh.x_empty[b], xe_done[b] & 1u, &sh.abort_flag, p.status);
                                ++xe_done[b];
                            }
                    }
                }
                for (int c = 0; c < 8 && ok; ++c) {
                    ok = wait_or_abort(&sh.full[slot], phase, &sh.abort_flag, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sb = smem_u32(slots + slot * C::kSlotBytes);
                    for (int g = 0; g < ntiles; ++g) {
                        const uint32_t kvb = sb + 2 * C::kQBytes + g * C::kKvBytes;
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t ad = sdesc_sw128(kvb + k * 32, 16, 1024);
                            const uint64_t bd = sdesc_sw128(sb + k * 32, 16, 1024);
                            mma_ss(tbase + g * 256, ad, bd, C::kIdescA, (c | k) != 0);
                        }
                    }
                    mma_commit(&sh.empty[slot]);
                    if (++slot == C::kSlots) { slot = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&sh.s_full);
                ok = wait_or_abort(&sh.p_ready, it & 1, &sh.abort_flag, p.status);
                if (!ok) break;
                tc_fence_after();
                // B stage: interm columns [64 dc, 64 dc + 64) for each tile.
                for (int c = 0; c < 8 && ok; ++c) {
                    ok = wait_or_abort(&sh.full[slot], phase, &sh.abort_flag, p.status);
                    const int b = c & 1;
                    const uint32_t need = uint32_t(it) * 4u + uint32_t(c >> 1);
                    while (ok && xe_done[b] < need) {
                        ok = wait_or_abort(&sh.x_empty[b], xe_done[b] & 1u, &sh.abort_flag, p.status);
                        ++xe_done[b];
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sb = smem_u32(slots + slot * C::kSlotBytes);
                    for (int g = 0; g < ntiles; ++g) {
                        const uint32_t tile = tbase + g * 256;
#pragma unroll
                        for (int ks = 0; ks < 2 * H / 16; ++ks) {
                            const bool pterm = ks < H / 16;
                            const int kk = pterm ? ks : ks - H / 16;
                            const uint32_t acol = pterm ? kk * 8 : H / 2 + kk * 8;
                            const uint32_t bt = (pterm ? sb + C::kQBytes : sb) + kk * 2048;
                            mma_ts(tile + 128 + 64 * b, tile + acol, sdesc_sw128(bt, 8192, 1024),
                                   C::kIdescB, ks != 0);
                        }
                    }
                    mma_commit(&sh.empty[slot]);
                    mma_commit(&sh.x_full[b]);
                    if (++slot == C::kSlots) { slot = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&sh.b_done[0]);
                mma_commit(&sh.b_done[1]);
            }
            // all MMAs issued by this thread finish before TMEM is freed
            mma_commit(&sh.drain);
            mbar_wait(&sh.drain, 0, kWaitNs);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- epilogue
        const int g = (warp - 2) >> 2;                  // tile of this warp group
        const int quarter = warp & 3;                   // TMEM lane quarter of this warp
        const int r = quarter * 32 + lane;              // TMEM lane = rank inside the tile
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const float c1 = p.scale * kLog2e;
        int it = 0;
        for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++it) {
            if (sh.abort_flag) break;
            const int t = item / p.npairs, pr = item - t * p.npairs;
            const int ntiles = pr == p.npairs - 1 ? p.tiles_last : 2;
            const bool active = g < ntiles;
            const int rl = pr * 256 + g * 128 + r;
            const float* lse_t = p.lse + int64_t(t) * H;
            const float* delta_t = p.delta + int64_t(t) * H;
            if (!wait_or_abort(&sh.s_full, it & 1, &sh.abort_flag, p.status)) break;
            tc_fence_after();
            if (active) {
                bool valid = false;
                if (rl < p.R) {
                    const int j = __ldg(p.topk + int64_t(t) * p.K + p.r0 + rl);
                    valid = j >= 0 && j < p.N;
                }
                const uint32_t trow = tbase + lane_off + g * 256;
                uint32_t dsp[H / 2];
#pragma unroll
                for (int c16 = 0; c16 < H / 16; ++c16) {
                    uint32_t sv[16], dv[16];
                    tmem_ld16(trow + c16 * 16, sv);
                    tmem_ld16(trow + H + c16 * 16, dv);
                    tmem_wait_ld();
                    uint32_t pp[8];
#pragma unroll
                    for (int j2 = 0; j2 < 8; ++j2) {
                        float pv[2], dsv[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int h = c16 * 16 + 2 * j2 + u;
                            const float s = __uint_as_float(sv[2 * j2 + u]);
                            const float dp = __uint_as_float(dv[2 * j2 + u]);
                            const float pe = valid ? exp2f(fmaf(s, c1, -__ldg(lse_t + h) * kLog2e)) : 0.f;
                            pv[u] = pe;
                            dsv[u] = valid ? p.scale * pe * (dp - __ldg(delta_t + h)) : 0.f;
                        }
                        pp[j2] = pack_bf16x2(pv[0], pv[1]);
                        dsp[c16 * 8 + j2] = pack_bf16x2(dsv[0], dsv[1]);
                    }
                    tmem_st8(trow + c16 * 8, pp);
                }
#pragma unroll
                for (int c16 = 0; c16 < H / 16; ++c16) tmem_st8(trow + H / 2 + c16 * 8, dsp + c16 * 8);
                tmem_wait_st();
                // stash scale * dS^T for the dq kernel (rows up to the padded rank count)
                uint4* dst = reinterpret_cast<uint4*>(p.dsT + (int64_t(t) * p.Rp + rl) * p.Hp);
#pragma unroll
                for (int v = 0; v < H / 8; ++v)
                    dst[v] = make_uint4(dsp[4 * v], dsp[4 * v + 1], dsp[4 * v + 2], dsp[4 * v + 3]);
                for (int v = H / 8; v < p.Hp / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_ready);
            // drain interm columns 64 dc .. 64 dc + 63
            bool ok = true;
            for (int c = 0; c < 8; ++c) {
                const int b = c & 1;
                const uint32_t use = uint32_t(it) * 4u + uint32_t(c >> 1);
                if (!wait_or_abort(&sh.x_full[b], use & 1u, &sh.abort_flag, p.status)) { ok = false; break; }
                tc_fence_after();
                if (active) {
                    const uint32_t xa = tbase + lane_off + g * 256 + 128 + 64 * b;
                    uint32_t v0[32], v1[32];
                    tmem_ld32(xa, v0);
                    tmem_ld32(xa + 32, v1);
                    tmem_wait_ld();
                    if (rl < p.R) {
                        uint4* out = reinterpret_cast<uint4*>(
                            p.interm + (int64_t(t) * p.R + rl) * kD + 64 * c);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            out[v] = make_uint4(
                                pack_bf16x2(__uint_as_float(v0[8 * v]), __uint_as_float(v0[8 * v + 1])),
                                pack_bf16x2(__uint_as_float(v0[8 * v + 2]), __uint_as_float(v0[8 * v + 3])),
                                pack_bf16x2(__uint_as_float(v0[8 * v + 4]), __uint_as_float(v0[8 * v + 5])),
                                pack_bf16x2(__uint_as_float(v0[8 * v + 6]), __uint_as_float(v0[8 * v + 7])));
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            out[4 + v] = make_uint4(
                                pack_bf16x2(__uint_as_float(v1[8 * v]), __uint_as_float(v1[8 * v + 1])),
                                pack_bf16x2(__uint_as_float(v1[8 * v + 2]), __uint_as_float(v1[8 * v + 3])),
                                pack_bf16x2(__uint_as_float(v1[8 * v + 4]), __uint_as_float(v1[8 * v + 5])),
                                pack_bf16x2(__uint_as_float(v1[8 * v + 6]), __uint_as_float(v1[8 * v + 7])));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.x_empty[b]);
            }
            if (!ok) break;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ------------------------------------------------------------------- dq
struct DqParams {
    const int32_t* topk;
    float* dq_acc;        // fp32 [T, H, 512] between chunks, or nullptr
    uint16_t* dq_out;     // bf16 [T, H, 512]
    int T, K, N, r0, R, Rp;
    bool first, last;
    unsigned* status;
};

struct DqShared {
    uint64_t full[4], empty[4];
    uint64_t d_full[2], d_empty[2], drain;
    uint32_t tbase;
    volatile int abort_flag;
    int idx[64];
};

constexpr int kDqSlots = 4;
constexpr int kDqABytes = 2 * 64 * 128;        // two 64-head blocks x 64 ranks
constexpr int kDqBBytes = 4 * 64 * 128;        // four 64-column blocks x 64 ranks
constexpr int kDqSlotBytes = kDqABytes + kDqBBytes;
constexpr int kDqSmem = int(sizeof(DqShared)) + 1024 + kDqSlots * kDqSlotBytes;
constexpr uint32_t kDqIdesc = idesc_bf16(128, 256, true, true);

template <int H>
__global__ void __launch_bounds__(192, 1)
dq_kernel(const __grid_constant__ CUtensorMap map_ds, const __grid_constant__ CUtensorMap map_kv,
          const DqParams p) {
    extern __shared__ uint8_t smem_raw[];
    DqShared& sh = *reinterpret_cast<DqShared*>(smem_raw);
    uint8_t* slots = align1024(smem_raw + sizeof(DqShared));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = p.T * 2;
    const int nkc = p.Rp / 64;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDqSlots; ++s) { mbar_init(&sh.full[s], 1); mbar_init(&sh.empty[s], 1); }
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
        int slot = 0; uint32_t phase = 0; int issued = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
            const int t = item >> 1, half = item & 1;
            for (int kc = 0; kc < nkc && ok; ++kc) {
                for (int i = lane; i < 64; i += 32) {
                    const int rl = kc * 64 + i;
                    int j = 0;
                    if (rl < p.R) {
                        j = __ldg(p.topk + int64_t(t) * p.K + p.r0 + rl);
                        if (j < 0 || j >= p.N) j = 0;     // masked or invalid: its dS is zero
                    }
                    sh.idx[i] = j;
                }
                __syncwarp();
                if (lane == 0) {
                    ok = wait_or_abort(&sh.empty[slot], phase ^ 1u, &sh.abort_flag, p.status);
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (ok && lane == 0) {
                    uint8_t* sb = slots + slot * kDqSlotBytes;
                    mbar_arrive_expect_tx(&sh.full[slot], kDqSlotBytes);
                    for (int hb = 0; hb < 2; ++hb)
                        tma_load_2d(sb + hb * 8192, &map_ds, hb * 64, t * p.Rp + kc * 64, &sh.full[slot]);
                    const int* ix = sh.idx;
                    for (int db = 0; db < 4; ++db)
                        for (int q4 = 0; q4 < 16; ++q4)
                            tma_gather4(sb + kDqABytes + db * 8192 + q4 * 512, &map_kv,
                                        half * 256 + db * 64, ix[4 * q4], ix[4 * q4 + 1],
                                        ix[4 * q4 + 2], ix[4 * q4 + 3], &sh.full[slot]);
                    ++issued;
                }
                if (++slot == kDqSlots) { slot = 0; phase ^= 1u; }
                __syncwarp();
            }
        }
        if (lane == 0 && sh.abort_flag) {
            int s = slot; uint32_t ph = phase;
            for (int k = 0; k < kDqSlots && k < issued; ++k) {
                if (--s < 0) { s = kDqSlots - 1; ph ^= 1u; }
                mbar_wait(&sh.full[s], ph, kWaitNs / 8);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int slot = 0; uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++it) {
                const int b = it & 1;
                if (it >= 2) ok = wait_or_abort(&sh.d_empty[b], ((it >> 1) - 1) & 1, &sh.abort_flag, p.status);
                for (int kc = 0; kc < nkc && ok; ++kc) {
                    ok = wait_or_abort(&sh.full[slot], phase, &sh.abort_flag, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sb = smem_u32(slots + slot * kDqSlotBytes);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ad = sdesc_sw128(sb + ks * 2048, 8192, 1024);
                        const uint64_t bd = sdesc_sw128(sb + kDqABytes + ks * 2048, 8192, 1024);
                        mma_ss(tbase + 256 * b, ad, bd, kDqIdesc, (kc | ks) != 0);
                    }
                    mma_commit(&sh.empty[slot]);
                    if (++slot == kDqSlots) { slot = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&sh.d_full[b]);
            }
            mma_commit(&sh.drain);
            mbar_wait(&sh.drain, 0, kWaitNs);
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        int it = 0;
        for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++it) {
            const int t = item >> 1, half = item & 1;
            const int b = it & 1;
            if (!wait_or_abort(&sh.d_full[b], (it >> 1) & 1, &sh.abort_flag, p.status)) break;
            tc_fence_after();
            const int64_t base = (int64_t(t) * H + h) * kD + half * 256;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t v[32];
                tmem_ld32(tbase + lane_off + 256 * b + 32 * c, v);
                tmem_wait_ld();
                if (h < H) {
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
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.d_empty[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

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

template <int H>
cudaError_t launch_sdi_h(const ChunkArgs& a, cudaStream_t s) {
    using C = SdiCfg<H>;
    static bool attr_done[64] = {false};
    if (set_smem_attrs_once(reinterpret_cast<const void*>(sdi_kernel<H>), C::kSmem, attr_done))
        return cudaErrorInvalidValue;
    CUtensorMap mq, mdo, mkv;
    if (!make_tmap_bf16_2d(&mq, a.q, uint64_t(a.T) * H, kD, kD, H, 64, true) ||
        !make_tmap_bf16_2d(&mdo, a.dO, uint64_t(a.T) * H, kD, kD, H, 64, true) ||
        !make_tmap_bf16_2d(&mkv, a.kv, a.N, kD, kD, 1, 64, true))
        return cudaErrorInvalidValue;
    SdiParams sp{};
    sp.topk = a.topk; sp.lse = a.lse; sp.delta = a.delta; sp.interm = a.interm; sp.dsT = a.dsT;
    sp.T = a.T; sp.K = a.K; sp.N = a.N; sp.r0 = a.r0; sp.R = a.R;
    sp.Rp = round_up_ranks(a.R); sp.Hp = pad_heads(H);
    sp.npairs = (a.R + 255) / 256;
    sp.tiles_last = (a.R - (sp.npairs - 1) * 256) > 128 ? 2 : 1;
    sp.scale = a.scale; sp.status = a.status;
    const int64_t items = int64_t(a.T) * sp.npairs;
    const int sms = sm_count();
    const int grid = int(items < sms ? items : sms);
    sdi_kernel<H><<<grid, C::kThreads, C::kSmem, s>>>(mq, mdo, mkv, sp);
    note_launch();
    return cudaGetLastError();
}

template <int H>
cudaError_t launch_dq_h(const ChunkArgs& a, cudaStream_t s) {
    static bool attr_done[64] = {false};
    if (set_smem_attrs_once(reinterpret_cast<const void*>(dq_kernel<H>), kDqSmem, attr_done))
        return cudaErrorInvalidValue;
    const int Rp = round_up_ranks(a.R);
    const int Hp = pad_heads(H);
    CUtensorMap mds, mkv;
    if (!make_tmap_bf16_2d(&mds, a.dsT, uint64_t(a.T) * Rp, Hp, Hp, 64, 64, true) ||
        !make_tmap_bf16_2d(&mkv, a.kv, a.N, kD, kD, 1, 64, true))
        return cudaErrorInvalidValue;
    DqParams dp{};
    dp.topk = a.topk; dp.dq_acc = a.dq_acc; dp.dq_out = a.dq_out;
    dp.T = a.T; dp.K = a.K; dp.N = a.N; dp.r0 = a.r0; dp.R = a.R; dp.Rp = Rp;
    dp.first = a.first_chunk; dp.last = a.last_chunk; dp.status = a.status;
    const int64_t items = int64_t(a.T) * 2;
    const int sms = sm_count();
    const int grid = int(items < sms ? items : sms);
    dq_kernel<H><<<grid, 192, kDqSmem, s>>>(mds, mkv, dp);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

#define SMLA_DISPATCH_H(FN, a, s)                     \
    switch ((a).H) {                                  \
        case 16: return FN<16>(a, s);                 \
        case 32: return FN<32>(a, s);                 \
        case 48: return FN<48>(a, s);                 \
        case 64: return FN<64>(a, s);                 \
        case 80: return FN<80>(a, s);                 \
        case 96: return FN<96>(a, s);                 \
        case 112: return FN<112>(a, s);               \
        case 128: return FN<128>(a, s);               \
        default: return cudaErrorInvalidValue;        \
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
