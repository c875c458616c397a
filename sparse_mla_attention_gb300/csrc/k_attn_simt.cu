// k_attn_simt.cu -- CUDA-core version of the per-chunk attention backward
// (S, dP, P, dS, the dKV intermediate and dq). It is the first, simple GPU
// path; the tensor-core kernels replace it for the supported shapes.
//
// Definitions (aiter "Sparse MLA training backward", Structure table, dQ and
// dKV-interm phases), for token t, head h and rank r of the chunk:
//   P  = exp(scale * <q, kv[idx]> - lse[t,h])
//   dS = P * (<dO, kv[idx]> - delta[t,h])
//   interm[t, r, :] = sum_h P * dO[t,h,:] + scale * dS * q[t,h,:]
//   dq[t, h, :]    += scale * sum_r dS * kv[idx_r, :]
#include "smla_internal.cuh"

namespace smla {

constexpr int kSimtTile = 16;     // ranks per block
constexpr int kMaxHeads = 128;

__global__ void __launch_bounds__(256) sdp_simt_kernel(ChunkArgs a) {
    __shared__ uint4 tile[kSimtTile][kD * 2 / 16];
    __shared__ int idx[kSimtTile];
    __shared__ float Ps[kSimtTile][kMaxHeads];
    __shared__ float dSs[kSimtTile][kMaxHeads];
    __shared__ float lse_s[kMaxHeads], delta_s[kMaxHeads];
    constexpr int kRowVec = kD * 2 / 16;
    const int t = blockIdx.y;
    const int rl0 = blockIdx.x * kSimtTile;          // local rank inside the chunk
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int H = a.H;
    if (threadIdx.x < kSimtTile) {
        const int rl = rl0 + threadIdx.x;
        idx[threadIdx.x] = rl < a.R
            ? load_index(a.topk + int64_t(t) * a.K + a.r0 + rl, a.N, a.status) : -1;
    }
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        lse_s[h] = a.lse[int64_t(t) * H + h];
        delta_s[h] = a.delta[int64_t(t) * H + h];
    }
    __syncthreads();
    const uint4* kv = reinterpret_cast<const uint4*>(a.kv);
    for (int i = threadIdx.x; i < kSimtTile * kRowVec; i += blockDim.x) {
        const int rr = i / kRowVec, c = i % kRowVec;
        const int j = idx[rr];
        tile[rr][c] = j >= 0 ? __ldg(kv + int64_t(j) * kRowVec + c) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    const uint4* q = reinterpret_cast<const uint4*>(a.q);
    const uint4* dO = reinterpret_cast<const uint4*>(a.dO);
    for (int h = w; h < H; h += 8) {
        float qf[16], gf[16];
        const int64_t row = (int64_t(t) * H + h) * kRowVec;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint4 vq = q[row + k * 32 + lane], vg = dO[row + k * 32 + lane];
            const uint32_t* x = reinterpret_cast<const uint32_t*>(&vq);
            const uint32_t* y = reinterpret_cast<const uint32_t*>(&vg);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qf[k * 8 + 2 * e] = bf16_lo(x[e]); qf[k * 8 + 2 * e + 1] = bf16_hi(x[e]);
                gf[k * 8 + 2 * e] = bf16_lo(y[e]); gf[k * 8 + 2 * e + 1] = bf16_hi(y[e]);
            }
        }
        float my_s = 0.f, my_dp = 0.f;
        for (int rr = 0; rr < kSimtTile; ++rr) {
            float ps = 0.f, pd = 0.f;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint4 v = tile[rr][k * 32 + lane];
                const uint32_t* x = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float k0 = bf16_lo(x[e]), k1 = bf16_hi(x[e]);
                    ps = fmaf(qf[k * 8 + 2 * e], k0, ps); ps = fmaf(qf[k * 8 + 2 * e + 1], k1, ps);
                    pd = fmaf(gf[k * 8 + 2 * e], k0, pd); pd = fmaf(gf[k * 8 + 2 * e + 1], k1, pd);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                ps += __shfl_xor_sync(0xffffffffu, ps, off);
                pd += __shfl_xor_sync(0xffffffffu, pd, off);
            }
            if (lane == rr) { my_s = ps; my_dp = pd; }
        }
        if (lane < kSimtTile) {
            float p = 0.f, ds = 0.f;
            if (idx[lane] >= 0) {
                p = __expf(my_s * a.scale - lse_s[h]);
                ds = a.scale * p * (my_dp - delta_s[h]);
            }
            Ps[lane][h] = p;
            dSs[lane][h] = ds;
        }
    }
    __syncthreads();

    // dsT[t, rl, h] = scale * dS (bf16) for the dq pass.
    for (int i = threadIdx.x; i < kSimtTile * H; i += blockDim.x) {
        const int rr = i / H, h = i % H;
        const int rl = rl0 + rr;
        if (rl < a.R)
            reinterpret_cast<__nv_bfloat16*>(a.dsT)[(int64_t(t) * a.R + rl) * H + h] =
                __float2bfloat16_rn(dSs[rr][h]);
    }
    // interm rows: thread owns columns 2*tid, 2*tid+1 for all ranks of the tile.
    const int d0 = threadIdx.x * 2;
    float acc[kSimtTile][2];
#pragma unroll
    for (int rr = 0; rr < kSimtTile; ++rr) acc[rr][0] = acc[rr][1] = 0.f;
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q);
    const uint32_t* g32 = reinterpret_cast<const uint32_t*>(a.dO);
    for (int h = 0; h < H; ++h) {
        const int64_t off = ((int64_t(t) * H + h) * kD + d0) / 2;
        const uint32_t qv = q32[off], gv = g32[off];
        const float q0 = bf16_lo(qv), q1 = bf16_hi(qv), g0 = bf16_lo(gv), g1 = bf16_hi(gv);
#pragma unroll
        for (int rr = 0; rr < kSimtTile; ++rr) {
            const float p = Ps[rr][h], ds = dSs[rr][h];
            acc[rr][0] = fmaf(p, g0, fmaf(ds, q0, acc[rr][0]));
            acc[rr][1] = fmaf(p, g1, fmaf(ds, q1, acc[rr][1]));
        }
    }
    uint32_t* out = reinterpret_cast<uint32_t*>(a.interm);
#pragma unroll
    for (int rr = 0; rr < kSimtTile; ++rr) {
        const int rl = rl0 + rr;
        if (rl < a.R) out[((int64_t(t) * a.R + rl) * kD + d0) / 2] = pack_bf16x2(acc[rr][0], acc[rr][1]);
    }
}

// dq[t, h, :] (+)= sum_rl dsT[t, rl, h] * kv[idx_rl, :]; block = (token, 8 heads),
// thread = 2 columns.
__global__ void __launch_bounds__(256) dq_simt_kernel(ChunkArgs a) {
    const int t = blockIdx.y, h0 = blockIdx.x * 8;
    const int d0 = threadIdx.x * 2;
    const int H = a.H;
    float acc[8][2];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = 0.f;
    const uint32_t* kv32 = reinterpret_cast<const uint32_t*>(a.kv);
    const __nv_bfloat16* ds = reinterpret_cast<const __nv_bfloat16*>(a.dsT);
    for (int rl = 0; rl < a.R; ++rl) {
        const int j = load_index(a.topk + int64_t(t) * a.K + a.r0 + rl, a.N, a.status);
        if (j < 0) continue;
        const uint32_t kvv = __ldg(kv32 + (int64_t(j) * kD + d0) / 2);
        const float k0 = bf16_lo(kvv), k1 = bf16_hi(kvv);
        const __nv_bfloat16* dr = ds + (int64_t(t) * a.R + rl) * H + h0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (h0 + i < H) {
                const float c = __bfloat162float(dr[i]);
                acc[i][0] = fmaf(c, k0, acc[i][0]);
                acc[i][1] = fmaf(c, k1, acc[i][1]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int h = h0 + i;
        if (h >= H) break;
        const int64_t off = (int64_t(t) * H + h) * kD + d0;
        float v0 = acc[i][0], v1 = acc[i][1];
        if (a.dq_acc) {
            if (!a.first_chunk) { v0 += a.dq_acc[off]; v1 += a.dq_acc[off + 1]; }
            if (!a.last_chunk) { a.dq_acc[off] = v0; a.dq_acc[off + 1] = v1; continue; }
        }
        reinterpret_cast<uint32_t*>(a.dq_out)[off / 2] = pack_bf16x2(v0, v1);
    }
}

cudaError_t launch_attn_chunk_simt(const ChunkArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    dim3 g1((a.R + kSimtTile - 1) / kSimtTile, a.T);
    sdp_simt_kernel<<<g1, 256, 0, s>>>(a);
    note_launch();
    dim3 g2((a.H + 7) / 8, a.T);
    dq_simt_kernel<<<g2, 256, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace smla
