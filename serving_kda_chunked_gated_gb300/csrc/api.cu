// Host side of the C ABI declared in include/kda.h: argument validation and
// kernel dispatch.  No device memory is allocated here; every launch goes on
// the caller's stream.
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "kda_common.cuh"
#include "tcgen05.cuh"

namespace kda {
cudaError_t launch_decode_step(const kda_decode_args& a, cudaStream_t stream);
cudaError_t launch_gate_norm(const void* o, const void* g, const float* w, float eps, void* y,
                             long rows, int dv, bool bf16, cudaStream_t s);
cudaError_t launch_prefill_recurrent(const kda_prefill_args& a, cudaStream_t s);
bool prefill_tc_supported(const kda_prefill_args& a);
size_t prefill_noalloc_scratch_needed(const kda_prefill_args& a);
cudaError_t launch_prefill_tc_noalloc(const kda_prefill_args& a, cudaStream_t s);
size_t prefill_tc_workspace_size(const kda_prefill_args& a);
cudaError_t launch_prefill_tc(const kda_prefill_args& a, cudaStream_t s);
size_t prefill_split_workspace_size(const kda_prefill_args& a);
bool prefill_split_supported(const kda_prefill_args& a);
cudaError_t launch_prefill_split(const kda_prefill_args& a, cudaStream_t s);
cudaError_t launch_prefill_split_parts(const kda_prefill_args& a, int parts, int scan_flags, cudaStream_t s);
cudaError_t launch_short_conv(const kda_short_conv_args& a, cudaStream_t s);
cudaError_t launch_kcp_apply(const float* M, float* X, const float* Add, int H, int d, int n, cudaStream_t s);
cudaError_t launch_short_conv_step(const kda_short_conv_step_args& a, cudaStream_t s);
cudaError_t noalloc_scratch_address(void** out);
}  // namespace kda

static thread_local char g_last_error[256] = "no error";
static thread_local uint64_t g_launches = 0;
static std::atomic<uint32_t> g_wait_limit{KDA_WAIT_LIMIT_DEFAULT};   // kda_debug_set_wait_limit

namespace kda {
// called by every launch wrapper once per kernel enqueued
void count_launches(int n) { g_launches += (uint64_t)n; }
// a failed CUDA runtime call outside this file: its status and the error string
kda_status cuda_failure(cudaError_t e) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return KDA_ERR_CUDA;
}
// poll bound of the prefill kernels' waits on local copies and MMAs
uint32_t wait_limit() {
    const uint32_t v = g_wait_limit.load(std::memory_order_relaxed);
    return v == KDA_WAIT_LIMIT_DEFAULT ? tc::WAIT_POLLS : v;
}
}  // namespace kda

static kda_status cuda_fail(cudaError_t e) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return KDA_ERR_CUDA;
}

static bool misaligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u); }

extern "C" {

const char* kda_status_str(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_NULL: return "required pointer is NULL";
        case KDA_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case KDA_ERR_DTYPE: return "unsupported dtype";
        case KDA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case KDA_ERR_SEQLENS: return "invalid cu_seqlens";
        case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up (outputs invalid)";
    }
    return "unknown status";
}

const char* kda_last_error_string(void) { return g_last_error; }

kda_status kda_get_last_device_error(void* workspace, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void* word = workspace;
    cudaError_t e = cudaSuccess;
    if (!word && (e = kda::noalloc_scratch_address(&word)) != cudaSuccess) return cuda_fail(e);
    if (misaligned(word)) return KDA_ERR_ALIGN;
    int32_t h = 0;
    if ((e = cudaMemcpyAsync(&h, word, sizeof(h), cudaMemcpyDeviceToHost, s)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemsetAsync(word, 0, sizeof(h), s)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
    return h ? KDA_ERR_TIMEOUT : KDA_OK;
}

uint32_t kda_debug_set_wait_limit(uint32_t polls) { return g_wait_limit.exchange(polls); }

uint64_t kda_launch_count(void) { return g_launches; }

const char* kda_version(void) { return "kda-gb300 0.1 (sm_103a; tcgen05 tf32 chunked prefill)"; }

// ---------------------------------------------------------------------------
// prefill
// ---------------------------------------------------------------------------

static kda_status validate_prefill(const kda_prefill_args* a) {
    if (!a) return KDA_ERR_NULL;
    if (a->num_seqs < 0 || a->T_total < 0 || a->H <= 0) return KDA_ERR_SHAPE;
    if (a->dk != a->dv) return KDA_ERR_SHAPE;
    if (a->qkv_dtype != KDA_BF16 && a->qkv_dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (!(a->dk == 32 || a->dk == 64 || a->dk == 128)) return KDA_ERR_SHAPE;
    if (!a->cu_seqlens || !a->cu_seqlens_host) return KDA_ERR_NULL;
    if (a->T_total > 0 && (!a->q || !a->k || !a->v || !a->z || !a->beta)) return KDA_ERR_NULL;
    if (!a->A) return KDA_ERR_NULL;
    if (a->g_in && !a->y) return KDA_ERR_NULL;
    if (a->g_in && a->qkv_dtype != KDA_BF16) return KDA_ERR_DTYPE;
    const void* ptrs[] = {a->q, a->k, a->v, a->z, a->beta, a->A, a->S0, a->o, a->S_T,
                          a->g_in, a->norm_w, a->y, a->cu_seqlens};
    for (const void* p : ptrs)
        if (misaligned(p)) return KDA_ERR_ALIGN;
    const int32_t* cu = a->cu_seqlens_host;
    if (cu[0] != 0) return KDA_ERR_SEQLENS;
    for (int n = 0; n < a->num_seqs; ++n)
        if (cu[n + 1] < cu[n]) return KDA_ERR_SEQLENS;
    if (cu[a->num_seqs] != a->T_total) return KDA_ERR_SEQLENS;
    if (a->gate_mode != KDA_GATE_BOUNDED && a->gate_mode != KDA_GATE_SOFTPLUS) return KDA_ERR_UNSUPPORTED;
    if (a->S_snap) {
        if (a->snap_interval <= 0 || a->snap_interval % 64 != 0) return KDA_ERR_SHAPE;
        if (misaligned(a->S_snap)) return KDA_ERR_ALIGN;
    }
    return KDA_OK;
}

long kda_prefill_snapshot_count(const kda_prefill_args* a) {
    if (validate_prefill(a) != KDA_OK || !a->S_snap) return 0;
    long rows = 0;
    for (int n = 0; n < a->num_seqs; ++n)
        rows += (a->cu_seqlens_host[n + 1] - a->cu_seqlens_host[n]) / a->snap_interval;
    return rows;
}

size_t kda_prefill_workspace_size(const kda_prefill_args* a) {
    if (validate_prefill(a) != KDA_OK) return 0;
    if (kda::prefill_split_supported(*a)) return kda::prefill_split_workspace_size(*a);
    return 0;
}

kda_status kda_prefill(const kda_prefill_args* a, void* stream) {
    kda_status st = validate_prefill(a);
    if (st != KDA_OK) return st;
    if (a->num_seqs == 0) return KDA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (kda::prefill_tc_supported(*a)) {          // bf16, d = 128: the workspace picks the schedule
        if (!a->workspace || a->workspace_bytes < KDA_PREFILL_MIN_WORKSPACE) return KDA_ERR_WORKSPACE;
        if (misaligned(a->workspace)) return KDA_ERR_ALIGN;
        if (a->workspace_bytes >= kda::prefill_split_workspace_size(*a))
            e = kda::launch_prefill_split(*a, s);
        else if (a->gate_mode != KDA_GATE_BOUNDED)
            return KDA_ERR_UNSUPPORTED;   // the single-pass schedule relies on the bounded gate
        else
            e = kda::launch_prefill_tc(*a, s);
    } else if (kda::prefill_split_supported(*a) && a->workspace &&
               a->workspace_bytes >= kda::prefill_split_workspace_size(*a)) {
        // float32, d = 32 or 64, with the chunk-parallel workspace: the chunked form
        if (misaligned(a->workspace)) return KDA_ERR_ALIGN;
        e = kda::launch_prefill_split(*a, s);
    } else {
        e = kda::launch_prefill_recurrent(*a, s);   // the per-token recurrence on CUDA cores
    }
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

// the chunk-parallel schedule's halves: parts 1 = records, 2 = scan
static kda_status prefill_split_part(const kda_prefill_args* a, int parts, int flags, void* stream) {
    kda_status st = validate_prefill(a);
    if (st != KDA_OK) return st;
    if (flags & ~KDA_SCAN_ZERO_V) return KDA_ERR_SHAPE;
    if (!kda::prefill_split_supported(*a)) return KDA_ERR_UNSUPPORTED;
    if (a->num_seqs == 0) return KDA_OK;
    if (!a->workspace || a->workspace_bytes < kda::prefill_split_workspace_size(*a)) return KDA_ERR_WORKSPACE;
    if (misaligned(a->workspace)) return KDA_ERR_ALIGN;
    const cudaError_t e = kda::launch_prefill_split_parts(*a, parts, flags, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

kda_status kda_prefill_records(const kda_prefill_args* a, void* stream) {
    return prefill_split_part(a, 1, 0, stream);
}

kda_status kda_prefill_scan(const kda_prefill_args* a, int flags, void* stream) {
    return prefill_split_part(a, 2, flags, stream);
}

kda_status kda_prefill_noalloc(const kda_prefill_args* a, void* stream) {
    kda_status st = validate_prefill(a);
    if (st != KDA_OK) return st;
    const size_t need = kda::prefill_noalloc_scratch_needed(*a);
    if (need > KDA_NOALLOC_SCRATCH_BYTES) {
        snprintf(g_last_error, sizeof(g_last_error),
                 "kda_prefill_noalloc: this call needs %zu bytes of scratch, the fixed array holds %d",
                 need, KDA_NOALLOC_SCRATCH_BYTES);
        return KDA_ERR_WORKSPACE;
    }
    if (kda::prefill_tc_supported(*a) && a->gate_mode != KDA_GATE_BOUNDED) return KDA_ERR_UNSUPPORTED;
    if (a->num_seqs == 0) return KDA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = kda::prefill_tc_supported(*a) ? kda::launch_prefill_tc_noalloc(*a, s)
                                                  : kda::launch_prefill_recurrent(*a, s);
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

kda_status kda_prefill_recurrent(const kda_prefill_args* a, void* stream) {
    kda_status st = validate_prefill(a);
    if (st != KDA_OK) return st;
    if (a->num_seqs == 0) return KDA_OK;
    cudaError_t e = kda::launch_prefill_recurrent(*a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

// ---------------------------------------------------------------------------
// ShortConv + Swish prologue
// ---------------------------------------------------------------------------

kda_status kda_short_conv(const kda_short_conv_args* a, void* stream) {
    if (!a) return KDA_ERR_NULL;
    if (a->num_seqs < 0 || a->T_total < 0 || a->channels <= 0 || a->channels % 8 != 0) return KDA_ERR_SHAPE;
    if (a->width < 1 || a->width > 8) return KDA_ERR_SHAPE;
    if (a->dtype != KDA_BF16 && a->dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (!a->cu_seqlens || !a->cu_seqlens_host) return KDA_ERR_NULL;
    if (a->T_total > 0 && (!a->x || !a->y || !a->weight)) return KDA_ERR_NULL;
    if (a->x && a->x == a->y) return KDA_ERR_SHAPE;
    if (a->state_in && a->state_in == a->state_out) return KDA_ERR_SHAPE;
    const void* ptrs[] = {a->x, a->y, a->weight, a->bias, a->state_in, a->state_out, a->cu_seqlens};
    for (const void* p : ptrs)
        if (misaligned(p)) return KDA_ERR_ALIGN;
    const int32_t* cu = a->cu_seqlens_host;
    if (cu[0] != 0) return KDA_ERR_SEQLENS;
    for (int n = 0; n < a->num_seqs; ++n)
        if (cu[n + 1] < cu[n]) return KDA_ERR_SEQLENS;
    if (cu[a->num_seqs] != a->T_total) return KDA_ERR_SEQLENS;
    if (a->num_seqs == 0) return KDA_OK;
    cudaError_t e = kda::launch_short_conv(*a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

kda_status kda_short_conv_step(const kda_short_conv_step_args* a, void* stream) {
    if (!a) return KDA_ERR_NULL;
    if (a->N < 0 || a->num_slots < 0 || a->channels <= 0 || a->channels % 8 != 0) return KDA_ERR_SHAPE;
    if (a->width < 1 || a->width > 8) return KDA_ERR_SHAPE;
    if (a->dtype != KDA_BF16 && a->dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (!a->slots && a->num_slots < a->N) return KDA_ERR_SHAPE;
    if (a->N > 0 && (!a->x || !a->y || !a->weight || (a->width > 1 && !a->state))) return KDA_ERR_NULL;
    const void* ptrs[] = {a->x, a->y, a->weight, a->bias, a->state, a->slots};
    for (const void* p : ptrs)
        if (misaligned(p)) return KDA_ERR_ALIGN;
    cudaError_t e = kda::launch_short_conv_step(*a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

// ---------------------------------------------------------------------------
// context parallelism: apply a segment's transition pair
// ---------------------------------------------------------------------------

kda_status kda_kcp_apply(const float* M, float* X, const float* add, int H, int d, int n, void* stream) {
    if (H < 0 || d < 1 || d > 256 || n < 1) return KDA_ERR_SHAPE;
    if (H > 0 && (!M || !X)) return KDA_ERR_NULL;
    if (misaligned(M) || misaligned(X) || misaligned(add)) return KDA_ERR_ALIGN;
    if (X == M || (add && X == add)) return KDA_ERR_SHAPE;
    cudaError_t e = kda::launch_kcp_apply(M, X, add, H, d, n, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------

kda_status kda_decode_step(const kda_decode_args* a, void* stream) {
    if (!a) return KDA_ERR_NULL;
    if (a->N < 0 || a->H <= 0 || a->num_slots < 0) return KDA_ERR_SHAPE;
    if (a->dk != 128 || a->dv != 128) return KDA_ERR_SHAPE;
    if (!a->slots && a->num_slots < a->N) return KDA_ERR_SHAPE;
    if (a->N > 0 && (!a->q || !a->k || !a->v || !a->z || !a->beta || !a->A || !a->state))
        return KDA_ERR_NULL;
    if (!a->o && !a->y) return KDA_ERR_NULL;
    if (a->g_in && !a->y) return KDA_ERR_NULL;
    if (a->y && !a->g_in) return KDA_ERR_NULL;
    if (a->gate_mode != KDA_GATE_BOUNDED && a->gate_mode != KDA_GATE_SOFTPLUS) return KDA_ERR_UNSUPPORTED;
    const void* ptrs[] = {a->q, a->k, a->v, a->z, a->beta, a->A, a->state, a->slots, a->o,
                          a->g_in, a->norm_w, a->y};
    for (const void* p : ptrs)
        if (misaligned(p)) return KDA_ERR_ALIGN;
    cudaError_t e = kda::launch_decode_step(*a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

// ---------------------------------------------------------------------------
// gate-norm
// ---------------------------------------------------------------------------

kda_status kda_gate_norm(const void* o, const void* g_in, const float* norm_w, float eps, void* y,
                         long rows, int dv, kda_dtype dtype, void* stream) {
    if (rows < 0) return KDA_ERR_SHAPE;
    if (!(dv == 32 || dv == 64 || dv == 128 || dv == 256)) return KDA_ERR_SHAPE;
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (rows > 0 && (!o || !g_in || !y)) return KDA_ERR_NULL;
    if (misaligned(o) || misaligned(g_in) || misaligned(y) || misaligned(norm_w)) return KDA_ERR_ALIGN;
    cudaError_t e = kda::launch_gate_norm(o, g_in, norm_w, eps, y, rows, dv, dtype == KDA_BF16,
                                          reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : cuda_fail(e);
}

}  // extern "C"
