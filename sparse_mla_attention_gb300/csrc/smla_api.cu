// smla_api.cu -- the C ABI of libsmla.so: argument validation, workspace
// plans and the phase sequence of the sparse MLA backward.
//
// Phase order follows the aiter page "Sparse MLA training backward"
// (Structure table): delta, then per rank chunk (R_CHUNK) the CSR build, the
// dQ / dKV-interm work and the atomic-free dKV gather, then d_sink (which
// needs only delta and lse, and runs on the side stream under the gather). The
// validation rules are the page wrapper's (D == 512, num_kv >= T, shapes),
// plus the review comments on that page (R_CHUNK must divide topk; dtype and
// lse shape checks), plus alignment and overlap checks.
#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include "smla_internal.cuh"

namespace smla {

// ------------------------------------------------------------ phase profiler
namespace prof {
enum Phase { kDelta, kCsr, kSdi, kDq, kGather, kDsink, kFwd, kPhases };
const char* const kNames[kPhases] = {"delta", "csr", "attn_sdi", "attn_dq", "gather", "dsink", "fwd"};
std::atomic<long long> g_launches{0};
bool g_on = false;
struct Pending { int phase; cudaEvent_t a, b; long long launches; };
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_pool;
double g_ms[kPhases];
long long g_calls[kPhases], g_kernels[kPhases];

cudaEvent_t take_event() {
    if (!g_pool.empty()) { cudaEvent_t e = g_pool.back(); g_pool.pop_back(); return e; }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) { cudaGetLastError(); return nullptr; }
    return e;
}

void reset() {
    for (auto& p : g_pending) { g_pool.push_back(p.a); g_pool.push_back(p.b); }
    g_pending.clear();
    for (int i = 0; i < kPhases; ++i) { g_ms[i] = 0; g_calls[i] = 0; g_kernels[i] = 0; }
}

// Brackets one phase with events on the stream while profiling is on.
struct Scope {
    int phase; cudaStream_t s; cudaEvent_t a = nullptr; long long l0;
    Scope(int ph, cudaStream_t st) : phase(ph), s(st), l0(g_launches.load()) {
        if (g_on && (a = take_event())) cudaEventRecord(a, s);
    }
    ~Scope() {
        if (!a) return;
        cudaEvent_t b = take_event();
        if (!b) { g_pool.push_back(a); return; }
        cudaEventRecord(b, s);
        g_pending.push_back({phase, a, b, g_launches.load() - l0});
    }
};
}  // namespace prof

void note_launch(int n) { prof::g_launches += n; }



BwdPlan plan_bwd(const smla_dims& d) {
    BwdPlan p{};
    p.T = d.T; p.H = d.H; p.K = d.topk; p.N = d.num_kv;
    p.R = d.r_chunk > 0 ? d.r_chunk : d.topk;
    p.nchunks = int(p.K / p.R);
    p.csr = plan_csr(p.T, p.R, p.N);
    const int64_t nnz_max = p.T * p.R;
    p.max_segs = (nnz_max + kGatherSeg - 1) / kGatherSeg + p.N;
    size_t off = kStatusBytes;
    auto take = [&](size_t bytes) { size_t o = off; off += align_up(bytes > 0 ? bytes : 1, 256); return o; };
    p.off_delta = take(size_t(p.T * p.H) * 4);
    p.off_rowptr = take(size_t(p.N + 1) * 4);
    p.off_col = take(size_t(nnz_max) * 4);
    p.off_csr = take(p.csr.bytes);
    p.off_segcnt = take(size_t(p.N) * 4);
    p.off_segptr = take(size_t(p.N + 1) * 4);
    p.off_segrow = take(size_t(p.max_segs) * 4);
    p.off_scan_tmp2 = take(scan_tmp_bytes(p.N));
    p.off_partial = take(size_t(p.max_segs) * kD * 4);
    p.off_interm = take(size_t(nnz_max) * kD * 2);
    // With rank chunks of a multiple of 128 ranks the dS^T stash covers all ranks
    // and dq runs once after the last chunk (no fp32 dq accumulator).
    p.full_stash = p.nchunks > 1 && p.R % 128 == 0;
    // Unchunked calls compact each token's valid ranks to the front of its row:
    // masked slots then cost no tensor work, and CSR positions are compacted
    // positions (the interm rows the S/dP/dS kernel writes).
    p.compact = p.nchunks == 1;
    p.off_cidx = take(p.compact ? size_t(p.T * p.K) * 4 : 0);
    p.off_ccnt = take(p.compact ? size_t(p.T) * 4 : 0);
    const int64_t ds_rows = p.full_stash ? p.K : round_up_ranks(int(p.R));
    p.off_dst = take(size_t(p.T) * ds_rows * pad_heads(int(p.H)) * 2);
    p.off_dqacc = take(p.nchunks > 1 && !p.full_stash ? size_t(p.T * p.H) * kD * 4 : 0);
    p.off_dkvacc = take(p.nchunks > 1 ? size_t(p.N) * kD * 4 : 0);
    p.bytes = off;
    return p;
}

namespace {

int check_dims(const smla_dims* d, bool need_bwd_limits) {
    if (!d) return SMLA_ERR_NULL;
    if (d->D != kD) return SMLA_ERR_D512;
    if (d->T < 0 || d->topk < 1 || d->num_kv < 1) return SMLA_ERR_SHAPE;
    if (d->H < 16 || d->H > 128 || d->H % 16 != 0) return SMLA_ERR_SHAPE;
    if (d->num_kv < d->T) return SMLA_ERR_NUM_KV_LT_T;
    if (int64_t(d->T) * d->topk > int64_t(INT32_MAX)) return SMLA_ERR_SHAPE;
    if (!std::isfinite(d->scale) || d->scale < 0.f) return SMLA_ERR_ARG;
    if (need_bwd_limits) {
        if (d->r_chunk < 0 || d->r_chunk > d->topk) return SMLA_ERR_RCHUNK;
        if (d->r_chunk > 0 && d->topk % d->r_chunk != 0) return SMLA_ERR_RCHUNK;
    }
    return SMLA_OK;
}

float eff_scale(const smla_dims& d) {
    return d.scale > 0.f ? d.scale : 1.0f / std::sqrt(float(d.D));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span { const void* p; size_t n; };

bool overlaps(const Span& a, const Span& b) {
    if (!a.p || !b.p || a.n == 0 || b.n == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Each output must be disjoint from every other span (inputs, outputs, workspace).
int check_overlap(const Span* outs, int nout, const Span* ins, int nin) {
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlaps(outs[i], ins[j])) return SMLA_ERR_OVERLAP;
        for (int j = i + 1; j < nout; ++j)
            if (overlaps(outs[i], outs[j])) return SMLA_ERR_OVERLAP;
    }
    return SMLA_OK;
}

int check_arch() {
    static int cached[64];          // 0 unknown, 1 ok, 2 wrong arch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SMLA_ERR_CUDA; }
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev] == 1 ? SMLA_OK : SMLA_ERR_ARCH;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return SMLA_ERR_CUDA;
    }
    const bool ok = major == 10 && minor == 3;
    if (dev >= 0 && dev < 64) cached[dev] = ok ? 1 : 2;
    return ok ? SMLA_OK : SMLA_ERR_ARCH;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA; }

}  // namespace

// Every non-NULL pointer must be device memory of the current device (or
// managed memory): a host pointer handed to a kernel faults the GPU, so it is
// refused here, before anything is enqueued. Needs a CUDA context, so it runs
// after the arch check.
int check_device_ptrs(const void* const* ptrs, int n) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SMLA_ERR_CUDA; }
    for (int i = 0; i < n; ++i) {
        if (!ptrs[i]) continue;
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, ptrs[i]) != cudaSuccess) {
            cudaGetLastError();
            return SMLA_ERR_DEVICE;
        }
        if (a.type == cudaMemoryTypeManaged) continue;
        if (a.type != cudaMemoryTypeDevice || a.device != dev) return SMLA_ERR_DEVICE;
    }
    return SMLA_OK;
}

namespace {

// A side stream (and its events) per host thread and device, created on first
// use. The CSR build of a rank chunk (a chain of small kernels that needs only
// topk) runs on it, forked from the caller's stream at the start of the chunk
// and joined back before the chunk's gather, so that it overlaps the delta and
// attention phases. The dq kernel runs on it too, after the chunk's S/dP/dS
// kernel, while the dKV gather runs on the caller's stream: dq is bound by the
// latency of its kv copies and the gather by HBM bandwidth, so the two share
// the SMs (dq is dispatched first, from the higher-priority stream, and the
// gather's blocks fill the room beside it). The caller sees all work ordered
// on its own stream.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, sdi_done = nullptr, dq_done = nullptr;
};

SideStream* side_stream() {
    thread_local SideStream per_dev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) { cudaGetLastError(); return nullptr; }
    SideStream& ss = per_dev[dev];
    if (!ss.stream) {
        // greatest priority: the CSR blocks, overlapped with delta, then leave the
        // SMs to the attention kernels sooner (measured 2.12 -> 2.10 ms per call)
        int lo = 0, hi = 0;
        cudaDeviceGetStreamPriorityRange(&lo, &hi);
        if (cudaStreamCreateWithPriority(&ss.stream, cudaStreamNonBlocking, hi) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.sdi_done, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.dq_done, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            ss = SideStream{};
            return nullptr;
        }
    }
    return &ss;
}


// Device pointers of one backward call.
struct BwdArgs {
    const uint16_t* q; const uint16_t* kv; const uint16_t* dO; const uint16_t* o;
    const float* lse; const int32_t* topk; const float* sink;
    uint16_t* dq; uint16_t* dkv; float* d_sink;
    float* dkv_f32;   // when set, dkv is written here in fp32, unrounded (dkv unused)
};

// Optional token pipelining of a call whose inputs arrive in token chunks:
// before its first use of tokens [t[i], t[i+1]) the compute stream waits for
// in_ready[i]; after their final dq it records dq_ready[i].
struct TokenFeed {
    int n;
    const int* t;
    cudaEvent_t* in_ready;
    cudaEvent_t* dq_ready;
};

// Enqueues the whole backward on stream s (validation done by the caller).
int enqueue_bwd(const BwdArgs& A, const smla_dims& d, const BwdPlan& plan, char* ws,
                cudaStream_t s, const TokenFeed* feed) {
    int rc = SMLA_OK;
    unsigned* status = reinterpret_cast<unsigned*>(ws);
    if ((rc = cuda_rc(cudaMemsetAsync(status, 0, sizeof(unsigned), s)))) return rc;
    if (d.T == 0) {
        if (A.dkv_f32) {
            if ((rc = cuda_rc(cudaMemsetAsync(A.dkv_f32, 0, size_t(d.num_kv) * kD * 4, s)))) return rc;
        } else if ((rc = cuda_rc(cudaMemsetAsync(A.dkv, 0, size_t(d.num_kv) * kD * 2, s)))) {
            return rc;
        }
        if (A.d_sink) return cuda_rc(cudaMemsetAsync(A.d_sink, 0, size_t(d.H) * 4, s));
        return SMLA_OK;
    }
    float* delta = reinterpret_cast<float*>(ws + plan.off_delta);
    int32_t* row_ptr = reinterpret_cast<int32_t*>(ws + plan.off_rowptr);
    int32_t* col = reinterpret_cast<int32_t*>(ws + plan.off_col);
    uint16_t* interm = reinterpret_cast<uint16_t*>(ws + plan.off_interm);
    uint16_t* dsT = reinterpret_cast<uint16_t*>(ws + plan.off_dst);
    float* dq_acc = plan.nchunks > 1 && !plan.full_stash
                        ? reinterpret_cast<float*>(ws + plan.off_dqacc) : nullptr;
    // fp32 dkv accumulator across rank chunks; with an fp32 output it is the output
    float* dkv_acc = A.dkv_f32 ? A.dkv_f32
                     : plan.nchunks > 1 ? reinterpret_cast<float*>(ws + plan.off_dkvacc) : nullptr;
    const int64_t Hp = pad_heads(d.H);
    const int64_t ds_rows = plan.full_stash ? plan.K : round_up_ranks(int(plan.R));
    const int whole[2] = {0, d.T};
    const int nt = feed ? feed->n : 1;
    const int* tb = feed ? feed->t : whole;

    SideStream* side = side_stream();
    if (!side) return SMLA_ERR_CUDA;
    const float scale = eff_scale(d);
    int32_t* cidx = plan.compact ? reinterpret_cast<int32_t*>(ws + plan.off_cidx) : nullptr;
    int32_t* ccnt = plan.compact ? reinterpret_cast<int32_t*>(ws + plan.off_ccnt) : nullptr;
    for (int c = 0; c < plan.nchunks; ++c) {
        const int r0 = int(c * plan.R);
        const bool first = c == 0, last = c == plan.nchunks - 1;
        // the compacted table, on this stream before delta: the S/dP/dS and dq
        // kernels and the CSR read it (on the side stream it waited for delta's
        // blocks, which fill the SMs)
        if (plan.compact) {
            prof::Scope ph(prof::kCsr, s);
            rc = cuda_rc(launch_compact_ranks(A.topk, d.T, d.topk, d.num_kv, cidx, ccnt, status, s));
            if (rc) return rc;
        }
        // CSR of this chunk on the side stream (after the previous chunk's gather,
        // which read the CSR buffers); joined back before this chunk's gather
        if ((rc = cuda_rc(cudaEventRecord(side->fork, s)))) return rc;
        if ((rc = cuda_rc(cudaStreamWaitEvent(side->stream, side->fork, 0)))) return rc;
        {
            prof::Scope ph(prof::kCsr, side->stream);
            rc = cuda_rc(launch_csr(plan.compact ? cidx : A.topk, d.T, d.topk, r0, int(plan.R), d.num_kv,
                                    row_ptr, col, ws + plan.off_csr, plan.csr, status, side->stream));
            if (rc) return rc;
        }
        if ((rc = cuda_rc(cudaEventRecord(side->join, side->stream)))) return rc;
        for (int i = 0; i < nt; ++i) {
            const int t0 = tb[i], t1 = tb[i + 1];
            if (t1 <= t0) continue;
            const int64_t th = int64_t(t0) * d.H;
            if (first && feed && (rc = cuda_rc(cudaStreamWaitEvent(s, feed->in_ready[i], 0)))) return rc;
            if (first) {
                prof::Scope ph(prof::kDelta, s);
                if ((rc = cuda_rc(launch_delta(A.o + th * kD, A.dO + th * kD, delta + th,
                                               int64_t(t1 - t0) * d.H, s)))) return rc;
            }
            ChunkArgs a{};
            a.q = A.q + th * kD; a.kv = A.kv; a.dO = A.dO + th * kD; a.lse = A.lse + th;
            a.delta = delta + th;
            a.topk = (plan.compact ? cidx : A.topk) + int64_t(t0) * d.topk;
            a.cnt = plan.compact ? ccnt + t0 : nullptr;
            a.T = t1 - t0; a.H = d.H; a.K = d.topk; a.N = d.num_kv; a.r0 = r0; a.R = int(plan.R);
            a.scale = scale;
            a.interm = interm + int64_t(t0) * plan.R * kD;
            a.dsT = dsT + int64_t(t0) * ds_rows * Hp;
            a.ds_rows = int(ds_rows); a.ds_off = plan.full_stash ? r0 : 0;
            a.dq_acc = dq_acc ? dq_acc + th * kD : nullptr;
            a.dq_out = A.dq + th * kD;
            a.first_chunk = first; a.last_chunk = last; a.status = status;
            {
                prof::Scope ph(prof::kSdi, s);
                if ((rc = cuda_rc(launch_attn_sdi(a, s)))) return rc;
            }
            // dq on the side stream, after this SDI (dq of earlier token or rank
            // chunks precede it on that stream, so the dq accumulator keeps its order)
            if (!plan.full_stash || last) {
                ChunkArgs b = a;
                b.dq_beside_part = plan.nchunks > 1;
                if (plan.full_stash) {
                    // dq over all ranks from the full stash, once
                    b.r0 = 0; b.R = int(plan.K); b.ds_off = 0;
                    b.first_chunk = b.last_chunk = true; b.dq_acc = nullptr;
                }
                if ((rc = cuda_rc(cudaEventRecord(side->sdi_done, s)))) return rc;
                if ((rc = cuda_rc(cudaStreamWaitEvent(side->stream, side->sdi_done, 0)))) return rc;
                {
                    prof::Scope ph(prof::kDq, side->stream);
                    if ((rc = cuda_rc(launch_attn_dq(b, side->stream)))) return rc;
                }
                if (last && feed &&
                    (rc = cuda_rc(cudaEventRecord(feed->dq_ready[i], side->stream)))) return rc;
            }
        }
        if ((rc = cuda_rc(cudaStreamWaitEvent(s, side->join, 0)))) return rc;
        prof::Scope ph(prof::kGather, s);
        rc = cuda_rc(launch_gather(row_ptr, col, interm, d.num_kv, plan.max_segs,
                                   reinterpret_cast<int32_t*>(ws + plan.off_segcnt),
                                   reinterpret_cast<int32_t*>(ws + plan.off_segptr),
                                   reinterpret_cast<int32_t*>(ws + plan.off_segrow),
                                   ws + plan.off_scan_tmp2,
                                   reinterpret_cast<float*>(ws + plan.off_partial), dkv_acc, A.dkv,
                                   first, last && !A.dkv_f32, s));
        if (rc) return rc;
        // the next chunk's SDI rewrites the per-chunk dS^T stash that this dq reads
        if (!last && !plan.full_stash) {
            if ((rc = cuda_rc(cudaEventRecord(side->dq_done, side->stream)))) return rc;
            if ((rc = cuda_rc(cudaStreamWaitEvent(s, side->dq_done, 0)))) return rc;
        }
    }
    // d_sink needs only delta and lse: on the side stream after the last dq
    // (delta precedes every S/dP/dS launch whose completion the side stream
    // waited for), so that it runs under the gather's tail instead of after it;
    // the caller's stream then waits for both
    if (A.sink) {
        prof::Scope ph(prof::kDsink, side->stream);
        if ((rc = cuda_rc(launch_dsink(delta, A.lse, A.sink, A.d_sink, d.T, d.H, side->stream)))) return rc;
    }
    if ((rc = cuda_rc(cudaEventRecord(side->dq_done, side->stream)))) return rc;
    if ((rc = cuda_rc(cudaStreamWaitEvent(s, side->dq_done, 0)))) return rc;
    return SMLA_OK;
}

// Copy streams of the host-buffer entry point (per host thread and device):
// host-to-device and device-to-host copies each get a stream of their own so
// that they overlap each other and the compute stream.
constexpr int kMaxTokenChunks = 32;
struct HostStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t fork = nullptr, small_in = nullptr, done = nullptr, out_done = nullptr;
    cudaEvent_t in_ready[kMaxTokenChunks] = {}, dq_ready[kMaxTokenChunks] = {};
};

HostStreams* host_streams() {
    thread_local HostStreams per_dev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) { cudaGetLastError(); return nullptr; }
    HostStreams& h = per_dev[dev];
    if (!h.in) {
        bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess;
        cudaEvent_t* evs[] = {&h.fork, &h.small_in, &h.done, &h.out_done};
        for (cudaEvent_t* e : evs)
            ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; i < kMaxTokenChunks; ++i)
            ok = ok && cudaEventCreateWithFlags(&h.in_ready[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.dq_ready[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) { cudaGetLastError(); h = HostStreams{}; return nullptr; }
    }
    return &h;
}

// Device copies of the inputs and outputs of the host-buffer entry point,
// placed after the backward's own workspace.
struct HostPlan {
    size_t off_q, off_kv, off_dO, off_o, off_lse, off_topk, off_sink, off_dq, off_dkv, off_dsink, bytes;
};

HostPlan plan_host(const smla_dims& d, const BwdPlan& bp) {
    HostPlan h{};
    size_t off = align_up(bp.bytes, 256);
    auto take = [&](size_t bytes) { size_t o = off; off += align_up(bytes > 0 ? bytes : 1, 256); return o; };
    const size_t thd = size_t(d.T) * d.H * kD * 2, th4 = size_t(d.T) * d.H * 4;
    h.off_q = take(thd); h.off_kv = take(size_t(d.num_kv) * kD * 2); h.off_dO = take(thd);
    h.off_o = take(thd); h.off_lse = take(th4); h.off_topk = take(size_t(d.T) * d.topk * 4);
    h.off_sink = take(size_t(d.H) * 4); h.off_dq = take(thd);
    h.off_dkv = take(size_t(d.num_kv) * kD * 2); h.off_dsink = take(size_t(d.H) * 4);
    h.bytes = off;
    return h;
}
}  // namespace
}  // namespace smla

namespace smla {
namespace {

// Validation and launch shared by smla_bwd (bf16 dkv) and smla_bwd_partial
// (fp32 dkv, A.dkv_f32). Pointers to zero-size tensors (T == 0) may be NULL.
int validate_and_enqueue_bwd(const BwdArgs& A, const smla_dims* dims, void* workspace,
                             size_t workspace_bytes, void* stream) {
    int rc = check_dims(dims, true);
    if (rc) return rc;
    const smla_dims& d = *dims;
    const bool has_tokens = d.T > 0;
    const void* dkv_out = A.dkv_f32 ? static_cast<const void*>(A.dkv_f32) : A.dkv;
    const size_t dkv_bytes = size_t(d.num_kv) * kD * (A.dkv_f32 ? 4 : 2);
    if (!A.kv || !dkv_out || !workspace) return SMLA_ERR_NULL;
    if (has_tokens && (!A.q || !A.dO || !A.o || !A.lse || !A.topk || !A.dq)) return SMLA_ERR_NULL;
    if ((A.sink == nullptr) != (A.d_sink == nullptr)) return SMLA_ERR_SINK;
    const void* ptrs[] = {A.q, A.kv, A.dO, A.o, A.lse, A.topk, A.sink, A.dq, dkv_out, A.d_sink, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SMLA_ERR_ALIGN;
    const BwdPlan plan = plan_bwd(d);
    if (workspace_bytes < plan.bytes) return SMLA_ERR_WORKSPACE;
    const size_t thd = size_t(d.T) * d.H * kD * 2, th4 = size_t(d.T) * d.H * 4;
    const Span ins[] = {{A.q, thd}, {A.kv, size_t(d.num_kv) * kD * 2}, {A.dO, thd}, {A.o, thd},
                        {A.lse, th4}, {A.topk, size_t(d.T) * d.topk * 4},
                        {A.sink, A.sink ? size_t(d.H) * 4 : 0}};
    const Span outs[] = {{A.dq, thd}, {dkv_out, dkv_bytes},
                         {A.d_sink, A.d_sink ? size_t(d.H) * 4 : 0}, {workspace, workspace_bytes}};
    if ((rc = check_overlap(outs, 4, ins, 7))) return rc;
    if ((rc = check_arch())) return rc;
    if ((rc = check_device_ptrs(ptrs, 11))) return rc;
    return enqueue_bwd(A, d, plan, static_cast<char*>(workspace), static_cast<cudaStream_t>(stream),
                       nullptr);
}

}  // namespace
}  // namespace smla

using namespace smla;

extern "C" {

int smla_version(void) { return 100; }

const char* smla_status_string(int code) {
    switch (code) {
        case SMLA_OK: return "ok";
        case SMLA_ERR_NULL: return "a required pointer is NULL";
        case SMLA_ERR_SHAPE: return "unsupported shape (H must be a multiple of 16 in 16..128; T >= 0; topk, num_kv >= 1; T*topk < 2^31)";
        case SMLA_ERR_D512: return "D must be 512";
        case SMLA_ERR_NUM_KV_LT_T: return "num_kv must be >= T";
        case SMLA_ERR_RCHUNK: return "r_chunk must be 0 or a divisor of topk";
        case SMLA_ERR_ALIGN: return "every device pointer must be 16-byte aligned";
        case SMLA_ERR_OVERLAP: return "an output overlaps an input, another output or the workspace";
        case SMLA_ERR_WORKSPACE: return "workspace missing or smaller than smla_workspace_size()";
        case SMLA_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103)";
        case SMLA_ERR_CUDA: return "a CUDA runtime call failed";
        case SMLA_ERR_INDEX: return "a topk index outside [-1, num_kv) was seen (treated as masked)";
        case SMLA_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
        case SMLA_ERR_SINK: return "d_sink must be given exactly when sink is given";
        case SMLA_ERR_ARG: return "invalid argument (scale must be finite and >= 0)";
        case SMLA_ERR_DEVICE: return "a pointer that must be device memory is not device memory of the current device";
        default: return "unknown status code";
    }
}

int smla_workspace_size(int op, const smla_dims* dims, size_t* bytes) {
    if (!bytes) return SMLA_ERR_NULL;
    if (!dims) return SMLA_ERR_NULL;
    if (op == SMLA_OP_CSR) {
        const int64_t R = dims->r_chunk > 0 ? dims->r_chunk : dims->topk;
        if (dims->T < 0 || dims->topk < 1 || dims->num_kv < 1 || R < 1 || R > dims->topk)
            return SMLA_ERR_SHAPE;
        *bytes = kStatusBytes + plan_csr(dims->T, R, dims->num_kv).bytes;
        return SMLA_OK;
    }
    const int rc = check_dims(dims, op == SMLA_OP_BWD);
    if (rc) return rc;
    if (op == SMLA_OP_FWD) { *bytes = kStatusBytes; return SMLA_OK; }
    if (op == SMLA_OP_BWD) { *bytes = plan_bwd(*dims).bytes; return SMLA_OK; }
    if (op == SMLA_OP_BWD_HOST) { *bytes = plan_host(*dims, plan_bwd(*dims)).bytes; return SMLA_OK; }
    return SMLA_ERR_ARG;
}

int smla_fwd(const uint16_t* q, const uint16_t* kv, const int32_t* topk, const float* sink,
             uint16_t* o, float* lse, const smla_dims* dims, void* workspace,
             size_t workspace_bytes, void* stream) {
    int rc = check_dims(dims, false);
    if (rc) return rc;
    const smla_dims& d = *dims;
    if (!kv || !workspace) return SMLA_ERR_NULL;
    if (d.T > 0 && (!q || !topk || !o || !lse)) return SMLA_ERR_NULL;   // NULL allowed when T == 0
    const void* fptrs[] = {q, kv, topk, sink, o, lse, workspace};
    for (const void* p : fptrs)
        if (p && !aligned16(p)) return SMLA_ERR_ALIGN;
    if (workspace_bytes < kStatusBytes) return SMLA_ERR_WORKSPACE;
    const size_t thd = size_t(d.T) * d.H * kD * 2;
    const Span ins[] = {{q, thd}, {kv, size_t(d.num_kv) * kD * 2}, {topk, size_t(d.T) * d.topk * 4},
                        {sink, sink ? size_t(d.H) * 4 : 0}, {workspace, workspace_bytes}};
    const Span outs[] = {{o, thd}, {lse, size_t(d.T) * d.H * 4}};
    if ((rc = check_overlap(outs, 2, ins, 5))) return rc;
    if (overlaps(Span{workspace, workspace_bytes}, ins[0]) ||
        overlaps(Span{workspace, workspace_bytes}, ins[1]))
        return SMLA_ERR_OVERLAP;
    if ((rc = check_arch())) return rc;
    if ((rc = check_device_ptrs(fptrs, 7))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* status = static_cast<unsigned*>(workspace);
    if ((rc = cuda_rc(cudaMemsetAsync(status, 0, sizeof(unsigned), s)))) return rc;
    prof::Scope ph(prof::kFwd, s);
    return cuda_rc(launch_fwd(q, kv, topk, sink, o, lse, d.T, d.H, d.topk, d.num_kv, eff_scale(d),
                              status, s));
}

int smla_bwd(const uint16_t* q, const uint16_t* kv, const uint16_t* dO, const uint16_t* o,
             const float* lse, const int32_t* topk, const float* sink, uint16_t* dq,
             uint16_t* dkv, float* d_sink, const smla_dims* dims, void* workspace,
             size_t workspace_bytes, void* stream) {
    const BwdArgs A{q, kv, dO, o, lse, topk, sink, dq, dkv, d_sink, nullptr};
    return validate_and_enqueue_bwd(A, dims, workspace, workspace_bytes, stream);
}

int smla_bwd_partial(const uint16_t* q, const uint16_t* kv, const uint16_t* dO, const uint16_t* o,
                     const float* lse, const int32_t* topk, const float* sink, uint16_t* dq,
                     float* dkv_partial, float* d_sink_partial, const smla_dims* dims,
                     void* workspace, size_t workspace_bytes, void* stream) {
    const BwdArgs A{q, kv, dO, o, lse, topk, sink, dq, nullptr, d_sink_partial, dkv_partial};
    return validate_and_enqueue_bwd(A, dims, workspace, workspace_bytes, stream);
}

int smla_reduce_partials(const float* partials, int32_t n_parts, int64_t n, uint16_t* out_bf16,
                         float* out_f32, void* stream) {
    if (!partials && n > 0) return SMLA_ERR_NULL;
    if (!out_bf16 && !out_f32) return SMLA_ERR_NULL;
    if (n_parts < 1 || n < 0 || n % 4 != 0) return SMLA_ERR_SHAPE;
    const void* ptrs[] = {partials, out_bf16, out_f32};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SMLA_ERR_ALIGN;
    const Span ins[] = {{partials, size_t(n_parts) * size_t(n) * 4}};
    const Span outs[] = {{out_bf16, out_bf16 ? size_t(n) * 2 : 0}, {out_f32, out_f32 ? size_t(n) * 4 : 0}};
    int rc = check_overlap(outs, 2, ins, 1);
    if (rc) return rc;
    if ((rc = check_arch())) return rc;
    if ((rc = check_device_ptrs(ptrs, 3))) return rc;
    if (n == 0) return SMLA_OK;
    return cuda_rc(launch_reduce_partials(partials, n_parts, n, out_bf16, out_f32,
                                          static_cast<cudaStream_t>(stream)));
}

int smla_bwd_host(const uint16_t* q, const uint16_t* kv, const uint16_t* dO, const uint16_t* o,
                  const float* lse, const int32_t* topk, const float* sink, uint16_t* dq,
                  uint16_t* dkv, float* d_sink, const smla_dims* dims, void* workspace,
                  size_t workspace_bytes, void* stream) {
    int rc = check_dims(dims, true);
    if (rc) return rc;
    const smla_dims& d = *dims;
    const bool has_tokens = d.T > 0;
    if (!kv || !dkv || !workspace) return SMLA_ERR_NULL;
    if (has_tokens && (!q || !dO || !o || !lse || !topk || !dq)) return SMLA_ERR_NULL;
    if ((sink == nullptr) != (d_sink == nullptr)) return SMLA_ERR_SINK;
    if (!aligned16(workspace)) return SMLA_ERR_ALIGN;
    const BwdPlan plan = plan_bwd(d);
    const HostPlan hp = plan_host(d, plan);
    if (workspace_bytes < hp.bytes) return SMLA_ERR_WORKSPACE;
    const size_t thd = size_t(d.T) * d.H * kD * 2, th4 = size_t(d.T) * d.H * 4;
    const size_t kvb = size_t(d.num_kv) * kD * 2, tkb = size_t(d.T) * d.topk * 4;
    const size_t hb = sink ? size_t(d.H) * 4 : 0;
    const Span ins[] = {{q, thd}, {kv, kvb}, {dO, thd}, {o, thd}, {lse, th4}, {topk, tkb}, {sink, hb}};
    const Span outs[] = {{dq, thd}, {dkv, kvb}, {d_sink, hb}};
    if ((rc = check_overlap(outs, 3, ins, 7))) return rc;
    if ((rc = check_arch())) return rc;
    const void* wsp[] = {workspace};
    if ((rc = check_device_ptrs(wsp, 1))) return rc;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    HostStreams* H = host_streams();
    if (!H) return SMLA_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    BwdArgs A{};
    A.q = reinterpret_cast<uint16_t*>(ws + hp.off_q);
    A.kv = reinterpret_cast<uint16_t*>(ws + hp.off_kv);
    A.dO = reinterpret_cast<uint16_t*>(ws + hp.off_dO);
    A.o = reinterpret_cast<uint16_t*>(ws + hp.off_o);
    A.lse = reinterpret_cast<float*>(ws + hp.off_lse);
    A.topk = reinterpret_cast<int32_t*>(ws + hp.off_topk);
    A.sink = sink ? reinterpret_cast<float*>(ws + hp.off_sink) : nullptr;
    A.dq = reinterpret_cast<uint16_t*>(ws + hp.off_dq);
    A.dkv = reinterpret_cast<uint16_t*>(ws + hp.off_dkv);
    A.d_sink = sink ? reinterpret_cast<float*>(ws + hp.off_dsink) : nullptr;
    auto h2d = [&](const void* dst, const void* src, size_t n) {
        return n ? cudaMemcpyAsync(const_cast<void*>(dst), src, n, cudaMemcpyHostToDevice, H->in)
                 : cudaSuccess;
    };
    auto d2h = [&](void* dst, const void* src, size_t n) {
        return n ? cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, H->out) : cudaSuccess;
    };
    // the copy streams start after everything already queued on the caller's
    // stream (earlier calls may still use this workspace)
    if ((rc = cuda_rc(cudaEventRecord(H->fork, s)))) return rc;
    if ((rc = cuda_rc(cudaStreamWaitEvent(H->in, H->fork, 0)))) return rc;
    if ((rc = cuda_rc(cudaStreamWaitEvent(H->out, H->fork, 0)))) return rc;
    // small inputs first: the CSR build needs only topk
    if ((rc = cuda_rc(h2d(A.topk, topk, tkb)))) return rc;
    if ((rc = cuda_rc(h2d(A.kv, kv, kvb)))) return rc;
    if ((rc = cuda_rc(h2d(A.lse, lse, th4)))) return rc;
    if ((rc = cuda_rc(h2d(A.sink, sink, hb)))) return rc;
    if ((rc = cuda_rc(cudaEventRecord(H->small_in, H->in)))) return rc;
    // then o, dO and q in token chunks of about 512 tokens
    int nt = (d.T + 511) / 512;
    if (nt < 1) nt = 1;
    if (nt > kMaxTokenChunks) nt = kMaxTokenChunks;
    int tb[kMaxTokenChunks + 1];
    for (int i = 0; i <= nt; ++i) tb[i] = int(int64_t(d.T) * i / nt);
    for (int i = 0; i < nt; ++i) {
        const size_t b0 = size_t(tb[i]) * d.H * kD * 2, nb = size_t(tb[i + 1] - tb[i]) * d.H * kD * 2;
        const char* ob = reinterpret_cast<const char*>(o);
        const char* db = reinterpret_cast<const char*>(dO);
        const char* qb = reinterpret_cast<const char*>(q);
        if ((rc = cuda_rc(h2d(reinterpret_cast<const char*>(A.o) + b0, ob + b0, nb)))) return rc;
        if ((rc = cuda_rc(h2d(reinterpret_cast<const char*>(A.dO) + b0, db + b0, nb)))) return rc;
        if ((rc = cuda_rc(h2d(reinterpret_cast<const char*>(A.q) + b0, qb + b0, nb)))) return rc;
        if ((rc = cuda_rc(cudaEventRecord(H->in_ready[i], H->in)))) return rc;
    }
    if ((rc = cuda_rc(cudaStreamWaitEvent(s, H->small_in, 0)))) return rc;
    const TokenFeed feed{nt, tb, H->in_ready, H->dq_ready};
    if ((rc = enqueue_bwd(A, d, plan, ws, s, &feed))) return rc;
    // results: dq per token chunk as soon as it is final, then dkv and d_sink
    if (has_tokens) {
        for (int i = 0; i < nt; ++i) {
            if (tb[i + 1] <= tb[i]) continue;
            const size_t b0 = size_t(tb[i]) * d.H * kD * 2, nb = size_t(tb[i + 1] - tb[i]) * d.H * kD * 2;
            if ((rc = cuda_rc(cudaStreamWaitEvent(H->out, H->dq_ready[i], 0)))) return rc;
            if ((rc = cuda_rc(d2h(reinterpret_cast<char*>(dq) + b0,
                                  reinterpret_cast<const char*>(A.dq) + b0, nb)))) return rc;
        }
    } else {
        // T == 0: wait for the input copies before the caller's stream goes on
        if ((rc = cuda_rc(cudaStreamWaitEvent(s, H->in_ready[0], 0)))) return rc;
    }
    if ((rc = cuda_rc(cudaEventRecord(H->done, s)))) return rc;
    if ((rc = cuda_rc(cudaStreamWaitEvent(H->out, H->done, 0)))) return rc;
    if ((rc = cuda_rc(d2h(dkv, A.dkv, kvb)))) return rc;
    if ((rc = cuda_rc(d2h(d_sink, A.d_sink, hb)))) return rc;
    // the caller's stream waits for the copies out, so that synchronizing it
    // (or an event recorded on it) covers the whole call
    if ((rc = cuda_rc(cudaEventRecord(H->out_done, H->out)))) return rc;
    return cuda_rc(cudaStreamWaitEvent(s, H->out_done, 0));
}

int smla_csr_build(const int32_t* topk, int32_t T, int32_t topk_w, int32_t r0, int32_t r_len,
                   int32_t num_kv, int32_t* row_ptr, int32_t* col, void* workspace,
                   size_t workspace_bytes, void* stream) {
    if (!row_ptr || !workspace) return SMLA_ERR_NULL;
    if (T > 0 && (!topk || !col)) return SMLA_ERR_NULL;        // NULL allowed when T == 0
    if (T < 0 || topk_w < 1 || num_kv < 1 || r0 < 0 || r_len < 1 ||
        int64_t(r0) + r_len > topk_w || int64_t(T) * topk_w > int64_t(INT32_MAX))
        return SMLA_ERR_SHAPE;
    if ((topk && !aligned16(topk)) || !aligned16(row_ptr) || (col && !aligned16(col)) ||
        !aligned16(workspace))
        return SMLA_ERR_ALIGN;
    const CsrPlan plan = plan_csr(T, r_len, num_kv);
    if (workspace_bytes < kStatusBytes + plan.bytes) return SMLA_ERR_WORKSPACE;
    const Span ins[] = {{topk, size_t(T) * topk_w * 4}};
    const Span outs[] = {{row_ptr, size_t(num_kv + 1) * 4}, {col, size_t(T) * r_len * 4},
                         {workspace, workspace_bytes}};
    int rc = check_overlap(outs, 3, ins, 1);
    if (rc) return rc;
    if ((rc = check_arch())) return rc;
    const void* cptrs[] = {topk, row_ptr, col, workspace};
    if ((rc = check_device_ptrs(cptrs, 4))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    unsigned* status = reinterpret_cast<unsigned*>(ws);
    if ((rc = cuda_rc(cudaMemsetAsync(status, 0, sizeof(unsigned), s)))) return rc;
    return cuda_rc(launch_csr(topk, T, topk_w, r0, r_len, num_kv, row_ptr, col, ws + kStatusBytes,
                              plan, status, s));
}

int smla_selftest_wait_timeout(void* workspace, size_t workspace_bytes, uint32_t limit_us,
                               void* stream) {
    if (!workspace) return SMLA_ERR_NULL;
    if (!aligned16(workspace)) return SMLA_ERR_ALIGN;
    if (workspace_bytes < kStatusBytes) return SMLA_ERR_WORKSPACE;
    if (limit_us < 1 || limit_us > 1000000) return SMLA_ERR_ARG;
    int rc = check_arch();
    if (rc) return rc;
    const void* wsp[] = {workspace};
    if ((rc = check_device_ptrs(wsp, 1))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* status = static_cast<unsigned*>(workspace);
    if ((rc = cuda_rc(cudaMemsetAsync(status, 0, sizeof(unsigned), s)))) return rc;
    return cuda_rc(launch_wait_selftest(status, uint64_t(limit_us) * 1000u, s));
}

int smla_profiling(int enable) {
    prof::reset();
    prof::g_on = enable != 0;
    return SMLA_OK;
}

int smla_profile_read(smla_phase_stat* out, int max, int* n) {
    if (!n) return SMLA_ERR_NULL;
    int rc = SMLA_OK;
    for (auto& p : prof::g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) {
            cudaGetLastError();
            rc = SMLA_ERR_CUDA;
        }
        prof::g_ms[p.phase] += ms;
        prof::g_calls[p.phase] += 1;
        prof::g_kernels[p.phase] += p.launches;
        prof::g_pool.push_back(p.a);
        prof::g_pool.push_back(p.b);
    }
    prof::g_pending.clear();
    int k = 0;
    for (int i = 0; i < prof::kPhases; ++i) {
        if (prof::g_calls[i] == 0) continue;
        if (out && k < max)
            out[k] = smla_phase_stat{prof::kNames[i], prof::g_ms[i], prof::g_calls[i], prof::g_kernels[i]};
        ++k;
    }
    *n = k;
    return rc;
}

int smla_get_device_status(const void* workspace, void* stream, int* status) {
    if (!workspace || !status) return SMLA_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) { cudaGetLastError(); return SMLA_ERR_CUDA; }
    unsigned bits = 0;
    if (cudaMemcpy(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return SMLA_ERR_CUDA;
    }
    *status = SMLA_OK;
    if (bits & (1u << SMLA_ERR_INDEX)) *status = SMLA_ERR_INDEX;
    else if (bits & (1u << SMLA_ERR_TIMEOUT)) *status = SMLA_ERR_TIMEOUT;
    else if (bits) *status = SMLA_ERR_CUDA;
    return SMLA_OK;
}

}  // extern "C"
