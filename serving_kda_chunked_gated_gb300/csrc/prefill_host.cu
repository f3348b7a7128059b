// The host-buffer prefill (include/kda.h, kda_prefill_from_host): one sequence
// from page-locked host memory through slab-sized device staging, results back
// to host memory.  Slab i's kda_prefill resumes from the state slab i - 1 left
// (S0 and S_T both point at the carried state).  Host-to-device copies run one
// slab ahead on one stream, device-to-host copies one slab behind on another,
// through two staging buffers of each kind; the compute runs on the caller's
// stream.  Events are kept by buffer parity: a buffer is refilled once the slab
// two back has finished with it.  Allocates no device memory (the caller passes
// the staging); creates two streams and seven events per call and releases them
// before returning (their pending work completes on its own).
#include <string.h>

#include "kda_common.cuh"

namespace {

constexpr size_t ALIGN = 256;
size_t up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

// staging layout for slabs of L tokens
struct Plan {
    int L, esz;
    bool gate;
    size_t q, k, v, z, beta, g, in_bytes;   // offsets inside one input buffer
    size_t in[2], o[2], y[2], state, A, w, cu, ws, ws_bytes, total;
};

kda_prefill_args slab_args(const kda_prefill_args& a, int n, const int32_t* cu_host) {
    kda_prefill_args s = a;
    s.num_seqs = 1;
    s.T_total = n;
    s.cu_seqlens_host = cu_host;
    s.S_snap = nullptr;
    s.snap_interval = 0;
    return s;
}

Plan plan(const kda_prefill_args& a, int slab) {
    Plan p;
    p.L = a.T_total < slab ? (a.T_total > 0 ? a.T_total : 64) : slab;
    p.esz = a.qkv_dtype == KDA_BF16 ? 2 : 4;
    p.gate = a.g_in != nullptr;
    const size_t L = (size_t)p.L, H = (size_t)a.H, dk = (size_t)a.dk, dv = (size_t)a.dv;
    size_t off = 0;
    p.q = off; off = up(off + L * H * dk * p.esz);
    p.k = off; off = up(off + L * H * dk * p.esz);
    p.v = off; off = up(off + L * H * dv * p.esz);
    p.z = off; off = up(off + L * H * dk * 4);
    p.beta = off; off = up(off + L * H * 4);
    p.g = off; off = up(off + (p.gate ? L * H * dv * 2 : 0));
    p.in_bytes = off;
    size_t t = 0;
    for (int b = 0; b < 2; ++b) { p.in[b] = t; t += p.in_bytes; }
    for (int b = 0; b < 2; ++b) { p.o[b] = t; t = up(t + L * H * dv * p.esz); }
    for (int b = 0; b < 2; ++b) { p.y[b] = t; t = up(t + (p.gate ? L * H * dv * 2 : 0)); }
    p.state = t; t = up(t + H * dk * dv * 4);
    p.A = t; t = up(t + H * 4);
    p.w = t; t = up(t + dv * 4);
    p.cu = t; t = up(t + 8 * sizeof(int32_t));   // {0, L} and {0, last}, 16 bytes apart
    // the slab call's workspace: its size from the slab's shapes (the device
    // pointers it will get are aligned staging; stand-ins here, never read)
    const int32_t cu_h[2] = {0, p.L};
    kda_prefill_args s = slab_args(a, p.L, cu_h);
    const void* dev = reinterpret_cast<const void*>(uintptr_t(ALIGN));
    s.q = s.k = s.v = dev;
    s.z = s.beta = s.A = reinterpret_cast<const float*>(dev);
    s.o = const_cast<void*>(dev);
    s.S0 = s.S_T = nullptr;
    s.norm_w = nullptr;
    s.g_in = p.gate ? dev : nullptr;
    s.y = p.gate ? const_cast<void*>(dev) : nullptr;
    s.cu_seqlens = reinterpret_cast<const int32_t*>(dev);
    p.ws_bytes = kda_prefill_workspace_size(&s);
    p.ws = t; t = up(t + p.ws_bytes);
    p.total = t;
    return p;
}

}  // namespace

extern "C" {

size_t kda_prefill_from_host_staging_size(const kda_prefill_args* a, int slab) {
    if (!a || slab <= 0 || slab % 64 || a->num_seqs != 1 || a->T_total < 0 || a->H <= 0) return 0;
    return plan(*a, slab).total;
}

kda_status kda_prefill_from_host(const kda_prefill_args* a, int slab, void* staging, size_t staging_bytes,
                                 void* stream) {
    if (!a) return KDA_ERR_NULL;
    if (slab <= 0 || slab % 64 || a->num_seqs != 1 || a->T_total < 0 || a->H <= 0 || a->dk <= 0 || a->dv <= 0)
        return KDA_ERR_SHAPE;
    if (a->S_snap) return KDA_ERR_UNSUPPORTED;
    if (!a->A || !a->S_T) return KDA_ERR_NULL;
    if (a->T_total > 0 && (!a->q || !a->k || !a->v || !a->z || !a->beta || !a->o)) return KDA_ERR_NULL;
    if (a->g_in && !a->y) return KDA_ERR_NULL;
    if (!staging) return KDA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(staging) & 15u) return KDA_ERR_ALIGN;
    const Plan p = plan(*a, slab);
    if (staging_bytes < p.total) return KDA_ERR_WORKSPACE;

    uint8_t* st = static_cast<uint8_t*>(staging);
    cudaStream_t s_cmp = reinterpret_cast<cudaStream_t>(stream);
    const int T = a->T_total, L = p.L;
    const size_t H = (size_t)a->H, dk = (size_t)a->dk, dv = (size_t)a->dv;
    const int n_slabs = (T + L - 1) / L;
    const int last = T - (n_slabs > 0 ? (n_slabs - 1) * L : 0);

    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_in[2] = {}, ev_cmp[2] = {}, ev_out[2] = {};
    cudaError_t e = cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
        e = cudaEventCreateWithFlags(&ev_in[b], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_cmp[b], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_out[b], cudaEventDisableTiming);
    }
    kda_status status = KDA_OK;
    auto h2d = [&](void* dst, const void* src, size_t n, cudaStream_t s) {
        if (e == cudaSuccess && n) e = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s);
    };
    auto d2h = [&](void* dst, const void* src, size_t n, cudaStream_t s) {
        if (e == cudaSuccess && n) e = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, s);
    };
    // the copies start after the caller's earlier work on `stream`
    if (e == cudaSuccess) e = cudaEventRecord(ev_start, s_cmp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_start, 0);

    // per-call constants and the carried state, ahead of slab 0's inputs on s_in
    float* state = reinterpret_cast<float*>(st + p.state);
    const int32_t cu_vals[8] = {0, L, 0, 0, 0, last, 0, 0};   // copied out before cudaMemcpyAsync returns
    h2d(st + p.A, a->A, H * 4, s_in);
    if (a->norm_w) h2d(st + p.w, a->norm_w, dv * 4, s_in);
    h2d(st + p.cu, cu_vals, sizeof(cu_vals), s_in);
    if (a->S0) h2d(state, a->S0, H * dk * dv * 4, s_in);
    else if (e == cudaSuccess) e = cudaMemsetAsync(state, 0, H * dk * dv * 4, s_in);

    auto in_ptr = [&](int b, size_t off) { return st + p.in[b] + off; };
    auto upload = [&](int i) {   // slab i's inputs into buffer i & 1, on s_in
        const int b = i & 1;
        const size_t t0 = (size_t)i * L, n = (size_t)(i + 1 < n_slabs ? L : last);
        if (i >= 2 && e == cudaSuccess) e = cudaStreamWaitEvent(s_in, ev_cmp[b], 0);   // slab i - 2 is done with it
        const uint8_t* q = static_cast<const uint8_t*>(a->q);
        const uint8_t* k = static_cast<const uint8_t*>(a->k);
        const uint8_t* v = static_cast<const uint8_t*>(a->v);
        h2d(in_ptr(b, p.q), q + t0 * H * dk * p.esz, n * H * dk * p.esz, s_in);
        h2d(in_ptr(b, p.k), k + t0 * H * dk * p.esz, n * H * dk * p.esz, s_in);
        h2d(in_ptr(b, p.v), v + t0 * H * dv * p.esz, n * H * dv * p.esz, s_in);
        h2d(in_ptr(b, p.z), a->z + t0 * H * dk, n * H * dk * 4, s_in);
        h2d(in_ptr(b, p.beta), a->beta + t0 * H, n * H * 4, s_in);
        if (p.gate)
            h2d(in_ptr(b, p.g), static_cast<const uint8_t*>(a->g_in) + t0 * H * dv * 2, n * H * dv * 2, s_in);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in[b], s_in);
    };

    if (n_slabs > 0) upload(0);
    for (int i = 0; i < n_slabs && e == cudaSuccess && status == KDA_OK; ++i) {
        if (i + 1 < n_slabs) upload(i + 1);
        const int b = i & 1;
        const size_t t0 = (size_t)i * L;
        const int n = i + 1 < n_slabs ? L : last;
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_cmp, ev_in[b], 0);
        if (i >= 2 && e == cudaSuccess) e = cudaStreamWaitEvent(s_cmp, ev_out[b], 0);   // outputs of slab i - 2 copied
        if (e != cudaSuccess) break;
        const int32_t cu_h[2] = {0, n};
        kda_prefill_args sa = slab_args(*a, n, cu_h);
        sa.cu_seqlens = reinterpret_cast<const int32_t*>(st + p.cu) + (i + 1 < n_slabs ? 0 : 4);
        sa.q = in_ptr(b, p.q);
        sa.k = in_ptr(b, p.k);
        sa.v = in_ptr(b, p.v);
        sa.z = reinterpret_cast<const float*>(in_ptr(b, p.z));
        sa.beta = reinterpret_cast<const float*>(in_ptr(b, p.beta));
        sa.g_in = p.gate ? in_ptr(b, p.g) : nullptr;
        sa.A = reinterpret_cast<const float*>(st + p.A);
        sa.norm_w = a->norm_w ? reinterpret_cast<const float*>(st + p.w) : nullptr;
        sa.S0 = state;
        sa.S_T = state;
        sa.o = st + p.o[b];
        sa.y = p.gate ? st + p.y[b] : nullptr;
        sa.workspace = st + p.ws;
        sa.workspace_bytes = p.ws_bytes;
        status = kda_prefill(&sa, s_cmp);
        if (status != KDA_OK) break;
        if (e == cudaSuccess) e = cudaEventRecord(ev_cmp[b], s_cmp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_cmp[b], 0);
        d2h(static_cast<uint8_t*>(a->o) + t0 * H * dv * p.esz, st + p.o[b], (size_t)n * H * dv * p.esz, s_out);
        if (p.gate) d2h(static_cast<uint8_t*>(a->y) + t0 * H * dv * 2, st + p.y[b], (size_t)n * H * dv * 2, s_out);
        if (e == cudaSuccess) e = cudaEventRecord(ev_out[b], s_out);
    }
    if (status == KDA_OK && e == cudaSuccess) {
        // the final state, after the last slab (or S0 itself for an empty sequence)
        if (n_slabs > 0) e = cudaStreamWaitEvent(s_out, ev_cmp[(n_slabs - 1) & 1], 0);
        else e = cudaStreamWaitEvent(s_out, ev_start, 0);
        if (n_slabs == 0 && e == cudaSuccess) {   // the state upload ran on s_in
            e = cudaEventRecord(ev_in[0], s_in);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_in[0], 0);
        }
        d2h(a->S_T, state, H * dk * dv * 4, s_out);
        if (e == cudaSuccess) e = cudaEventRecord(ev_out[0], s_out);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_cmp, ev_out[0], 0);   // everything precedes later work
    }
    // streams and events are released once their pending work has completed
    for (int b = 0; b < 2; ++b) {
        if (ev_in[b]) cudaEventDestroy(ev_in[b]);
        if (ev_cmp[b]) cudaEventDestroy(ev_cmp[b]);
        if (ev_out[b]) cudaEventDestroy(ev_out[b]);
    }
    if (ev_start) cudaEventDestroy(ev_start);
    if (s_in) cudaStreamDestroy(s_in);
    if (s_out) cudaStreamDestroy(s_out);
    if (status != KDA_OK) return status;
    return e == cudaSuccess ? KDA_OK : kda::cuda_failure(e);
}

}  // extern "C"
