// k_fwd.cu -- sparse MLA forward on CUDA cores, for the shapes the tensor-core
// forward (k_fwd_tc.cu) does not take: H not a multiple of 32, or topk > 512.
// launch_fwd tries the tensor-core kernel first. Not a tuned kernel.
//
// Definition (aiter "Sparse MLA training backward", Contract section and the
// lse paragraph under its usage example): for token t, head h and the valid
// ranks r of topk[t, :], s_r = scale * <q[t,h,:], kv[idx_r,:]>; the sink adds
// exp(sink_h) to the softmax denominator only; lse = m + log(sum) with the
// sink folded into the running max m and the sum; O = sum_r exp(s_r - lse) kv.
//
// One block per (token, group of 16 heads): warp w is head h0 + w and keeps an
// online softmax over rank tiles of 32 rows staged in shared memory; lane l
// owns columns [8l, 8l+8) and [256+8l, 256+8l+8) of q and O.
#include "smla_internal.cuh"

namespace smla {

constexpr int kFwdHeads = 16;
constexpr int kFwdTile = 32;

__global__ void __launch_bounds__(kFwdHeads * 32) fwd_kernel(
    const uint4* __restrict__ q, const uint4* __restrict__ kv, const int32_t* __restrict__ topk,
    const float* __restrict__ sink, uint4* __restrict__ o, float* __restrict__ lse, int H, int K,
    int num_kv, float scale, unsigned* status) {
    __shared__ uint4 tile[kFwdTile][kD * 2 / 16];   // 32 rows x 1 KB
    __shared__ int idx[kFwdTile];
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int h = blockIdx.y * kFwdHeads + w;
    const bool head_ok = h < H;
    constexpr int kRowVec = kD * 2 / 16;

    float qf[16];
    if (head_ok) {
        const uint4* qr = q + (int64_t(t) * H + h) * kRowVec;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint4 v = qr[k * 32 + lane];
            const uint32_t* x = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qf[k * 8 + 2 * e] = bf16_lo(x[e]);
                qf[k * 8 + 2 * e + 1] = bf16_hi(x[e]);
            }
        }
    }
    const bool has_sink = sink != nullptr;
    float m = has_sink && head_ok ? sink[h] : -INFINITY;
    float l = has_sink ? 1.f : 0.f;          // exp(sink - m) with m = sink
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;

    for (int r0 = 0; r0 < K; r0 += kFwdTile) {
        __syncthreads();
        if (threadIdx.x < kFwdTile) {
            const int r = r0 + threadIdx.x;
            idx[threadIdx.x] = r < K ? load_index(topk + int64_t(t) * K + r, num_kv, status) : -1;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kFwdTile * kRowVec; i += blockDim.x) {
            const int rr = i / kRowVec, c = i % kRowVec;
            const int j = idx[rr];
            tile[rr][c] = j >= 0 ? __ldg(kv + int64_t(j) * kRowVec + c) : make_uint4(0, 0, 0, 0);
        }
        __syncthreads();
        if (!head_ok) continue;
        // lane r ends up holding the score of rank r0 + r
        float my_s = -INFINITY;
        for (int rr = 0; rr < kFwdTile; ++rr) {
            float part = 0.f;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint4 v = tile[rr][k * 32 + lane];
                const uint32_t* x = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    part = fmaf(qf[k * 8 + 2 * e], bf16_lo(x[e]), part);
                    part = fmaf(qf[k * 8 + 2 * e + 1], bf16_hi(x[e]), part);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if (lane == rr) my_s = part * scale;
        }
        if (idx[lane] < 0) my_s = -INFINITY;
        float tmax = my_s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        const float m_new = fmaxf(m, tmax);
        if (m_new == -INFINITY) continue;            // nothing valid yet and no sink
        const float p = idx[lane] >= 0 ? __expf(my_s - m_new) : 0.f;
        const float corr = __expf(m - m_new);        // m == -inf gives 0
        float psum = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l = l * corr + psum;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] *= corr;
        for (int rr = 0; rr < kFwdTile; ++rr) {
            const float pr = __shfl_sync(0xffffffffu, p, rr);
            if (pr == 0.f) continue;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint4 v = tile[rr][k * 32 + lane];
                const uint32_t* x = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[k * 8 + 2 * e] = fmaf(pr, bf16_lo(x[e]), acc[k * 8 + 2 * e]);
                    acc[k * 8 + 2 * e + 1] = fmaf(pr, bf16_hi(x[e]), acc[k * 8 + 2 * e + 1]);
                }
            }
        }
        m = m_new;
    }
    if (!head_ok) return;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4* orow = o + (int64_t(t) * H + h) * kRowVec;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        uint4 v;
        v.x = pack_bf16x2(acc[k * 8 + 0] * inv, acc[k * 8 + 1] * inv);
        v.y = pack_bf16x2(acc[k * 8 + 2] * inv, acc[k * 8 + 3] * inv);
        v.z = pack_bf16x2(acc[k * 8 + 4] * inv, acc[k * 8 + 5] * inv);
        v.w = pack_bf16x2(acc[k * 8 + 6] * inv, acc[k * 8 + 7] * inv);
        orow[k * 32 + lane] = v;
    }
    if (lane == 0) lse[int64_t(t) * H + h] = l > 0.f ? m + logf(l) : -INFINITY;
}

cudaError_t launch_fwd(const uint16_t* q, const uint16_t* kv, const int32_t* topk,
                       const float* sink, uint16_t* o, float* lse, int T, int H, int K,
                       int num_kv, float scale, unsigned* status, cudaStream_t s) {
    const cudaError_t tc = launch_fwd_tc(q, kv, topk, sink, o, lse, T, H, K, num_kv, scale, status, s);
    if (tc != cudaErrorNotSupported) return tc;
    if (T == 0) return cudaSuccess;
    dim3 grid(T, (H + kFwdHeads - 1) / kFwdHeads);
    fwd_kernel<<<grid, kFwdHeads * 32, 0, s>>>(
        reinterpret_cast<const uint4*>(q), reinterpret_cast<const uint4*>(kv), topk, sink,
        reinterpret_cast<uint4*>(o), lse, H, K, num_kv, scale, status);
    note_launch();
    return cudaGetLastError();
}

}  // namespace smla
