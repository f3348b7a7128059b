/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention operator library.
 *
 * The operator ("Kimi K3: KDA, attention residuals and Stable LatentMoE",
 * hs-black.github.io, Sec. 2.1-2.3), per sequence and head, dk = dv = d:
 *
 *   alpha_t = exp(g_t),  g_t = g_min * Sigmoid(exp(A_h) * z_t)        (Sec. 2.2)
 *   S_t     = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t     = scale * S_t^T q_t                                        (Sec. 2.1)
 *   y_t     = Sigmoid(g_in_t) (.) w (.) o_t / sqrt(mean(o_t^2) + eps)  (Sec. 2.3)
 *
 * with q, k optionally L2-normalised per token: x / sqrt(sum x^2 + 1e-6).
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is DEVICE memory owned by the caller, unless the
 *    comment says otherwise.  The library never allocates device memory and
 *    keeps no state between calls.
 *  - All work is enqueued on the caller's `stream` (cudaStream_t passed as
 *    void*; NULL = legacy default stream).  Calls return as soon as the work
 *    is enqueued; arguments are validated on the host before anything is
 *    enqueued, and nothing is enqueued when validation fails.
 *  - Tensors are dense, row-major, last index fastest, with the layouts below;
 *    every pointer must be 16-byte aligned.
 *  - No call throws.  Errors are reported through kda_status; a failed launch
 *    returns KDA_ERR_CUDA (the CUDA error string is available from
 *    kda_last_error_string()).
 *  - Calls on distinct streams may run concurrently; the library is
 *    thread-safe.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,        /* a required pointer is NULL                        */
    KDA_ERR_SHAPE = 2,       /* unsupported or inconsistent sizes                 */
    KDA_ERR_DTYPE = 3,       /* unsupported dtype combination                     */
    KDA_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned                  */
    KDA_ERR_SEQLENS = 5,     /* cu_seqlens not monotone / not ending at tokens    */
    KDA_ERR_UNSUPPORTED = 6, /* valid request the library does not implement      */
    KDA_ERR_CUDA = 7,        /* a CUDA runtime call or a launch failed            */
    KDA_ERR_WORKSPACE = 8,   /* workspace missing or smaller than required        */
    KDA_ERR_TIMEOUT = 9      /* a bounded wait inside a kernel gave up (read by
                                kda_get_last_device_error; see there)            */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

/*
 * Decay gate (Sec. 2.2).  KDA_GATE_BOUNDED is K3's g = g_min * Sigmoid(exp(A_h) z),
 * g in (g_min, 0) -- the operator of this library.  KDA_GATE_SOFTPLUS is the gate
 * it replaces, Kimi Linear's g = -exp(A_h) * Softplus(z) (g_min unused), unbounded
 * below: a 16-token sub-chunk can then span more than the bf16/fp32 range, so the
 * chunked prefill forms the diagonal Gram sub-blocks pair by pair on CUDA cores
 * (supported by the chunk-parallel schedule and the CUDA-core paths; the
 * single-pass schedule and kda_prefill_noalloc return KDA_ERR_UNSUPPORTED).
 */
typedef enum { KDA_GATE_BOUNDED = 0, KDA_GATE_SOFTPLUS = 1 } kda_gate;

/*
 * Chunked prefill over packed sequences (Sec. 2.1 chunked form, Sec. 2.2
 * 16-token sub-chunks; chunk length 64), with optional prefix-cache state
 * snapshots at chunk-aligned intervals (Sec. 13.1: a cached prefix is only
 * reusable where the recurrent state can be restored at the same boundary;
 * "Kimi-K3 深度技术分析" (liuhc.cn), Sec. 5.2 KDA Prefill Cache: the state is
 * cached per contiguous block, and a new request resumes its prefill from the
 * nearest cached block boundary).
 *
 * Token layout: the T_total tokens of num_seqs sequences are packed; sequence n
 * owns tokens [cu_seqlens[n], cu_seqlens[n+1]).  cu_seqlens is a DEVICE int32
 * array of num_seqs+1 entries and a HOST copy (cu_seqlens_host) of the same
 * values is required too: the host copy sizes the launch and is validated
 * (cu_seqlens_host[0] == 0, non-decreasing, last == T_total); the device copy
 * must hold identical values.
 *
 *   q, k  [T_total, H, dk]   dtype qkv_dtype
 *   v     [T_total, H, dv]   dtype qkv_dtype
 *   z     [T_total, H, dk]   float32  decay logits (bias included)
 *   beta  [T_total, H]       float32  write strengths in (0, 1)
 *   A     [H]                float32  per-head log scale
 *   S0    [num_seqs, H, dk, dv] float32 initial states, or NULL (zero state)
 *   o     [T_total, H, dv]   dtype qkv_dtype (output), or NULL when only the
 *         final states are wanted (e.g. the KCP transition pairs below)
 *   S_T   [num_seqs, H, dk, dv] float32 final states (output), or NULL;
 *         S_T may equal S0 (in-place state update).
 *   g_in  [T_total, H, dv]   bf16 gate pre-activations, or NULL (no fused gate)
 *   norm_w [dv] float32 RMSNorm weight, or NULL (ones); used with g_in
 *   y     [T_total, H, dv]   bf16 fused output gate result (required iff g_in)
 *
 * Supported: dk = dv = 128 with bf16 q/k/v, and dk = dv in {32, 64, 128} with
 * float32 q/k/v; H >= 1.  workspace: device scratch; its size selects the
 * schedule.  bf16, d = 128 (the tensor-core path):
 *  - workspace_bytes >= kda_prefill_workspace_size(): chunk-parallel schedule
 *    (one pass over all (chunk, head) pairs in parallel writes each chunk's
 *    state-free terms, 112.75 KiB per chunk and head, to the workspace; a second
 *    pass runs the state recurrence per (sequence, head) on fp16 tensor-core
 *    operands under exact power-of-two scaling).  The fastest.
 *  - KDA_PREFILL_MIN_WORKSPACE <= workspace_bytes < that: single-pass schedule
 *    (one cluster per (sequence, head) walks its chunks); no scratch beyond
 *    the error word.
 *  - less: KDA_ERR_WORKSPACE.
 * float32, d = 32 or 64: with kda_prefill_workspace_size() bytes the same
 * chunk-parallel schedule (tensor cores, the channels d..127 taken as zero,
 * which leaves every result exact); with less (NULL included) the per-token
 * recurrence on CUDA cores.  float32, d = 128: the per-token recurrence.
 * The first 4 bytes of the workspace are the call's error word: kda_prefill
 * and kda_prefill_records clear it on the stream before their kernels run,
 * kda_prefill_scan does not (a records call's word stays visible through its
 * scans), and a bounded wait inside a kernel that gives up sets it; read it
 * with kda_get_last_device_error.  The per-token CUDA-core path needs no
 * workspace (may be NULL) and has no waits.
 */
#define KDA_PREFILL_MIN_WORKSPACE 256
typedef struct {
    int num_seqs;
    int T_total;
    int H, dk, dv;
    kda_dtype qkv_dtype;
    const int32_t* cu_seqlens;       /* device */
    const int32_t* cu_seqlens_host;  /* host   */
    const void* q;
    const void* k;
    const void* v;
    const float* z;
    const float* beta;
    const float* A;
    float g_min;          /* -5 in every workload */
    float scale;          /* readout scale, 1.0 in every workload */
    int qk_l2norm;        /* 1: L2-normalise q and k in FP32 (eps 1e-6) */
    const float* S0;
    void* o;
    float* S_T;
    const void* g_in;
    const float* norm_w;
    float norm_eps;       /* RMSNorm epsilon, 1e-6 in every workload */
    void* y;
    void* workspace;
    size_t workspace_bytes;
    /* Prefix-cache snapshots (optional): when S_snap is non-NULL, the FP32
     * state of sequence n after every snap_interval of its tokens is written to
     * S_snap [rows, H, dk, dv]: the state after token j*snap_interval (counted
     * from the sequence start), j = 1 .. floor(len_n / snap_interval), goes to
     * row snap_base(n) + j - 1, where snap_base(n) sums floor(len_m /
     * snap_interval) over the sequences m < n.  snap_interval must be a
     * positive multiple of 64 (the chunk length), so snapshots sit on chunk
     * boundaries and a later prefill can resume from any of them through S0.
     * kda_prefill_snapshot_count() gives the number of rows.  Errors: another
     * snap_interval -> KDA_ERR_SHAPE; S_snap not 16-byte aligned ->
     * KDA_ERR_ALIGN.  S_snap must not overlap any other argument.  Ignored
     * (and snap_interval unread) when S_snap is NULL. */
    int snap_interval;
    float* S_snap;
    int gate_mode;        /* kda_gate; KDA_ERR_UNSUPPORTED for other values */
} kda_prefill_args;

size_t kda_prefill_workspace_size(const kda_prefill_args* args);
/* Rows S_snap must hold for these arguments (0 when snapshots are off or the
 * arguments are invalid); computed on the host from cu_seqlens_host. */
long kda_prefill_snapshot_count(const kda_prefill_args* args);
kda_status kda_prefill(const kda_prefill_args* args, void* stream);

/*
 * The chunk-parallel prefill in its two halves, so that one set of chunk
 * records serves several state passes over the same tokens.  KDA context
 * parallelism ("Kimi K3" page, Sec. 10.2) runs a rank's segment three times:
 * its transition M (from S0 = I with v = 0), its state S~ from zero, and its
 * outputs from the entry state; the records depend only on q, k, v, z, beta,
 * A, cu_seqlens, qk_l2norm, g_min and gate_mode, never on S0.
 *
 * kda_prefill_records: writes the chunk records of args' sequences into
 *   args->workspace, which must hold kda_prefill_workspace_size(args) bytes
 *   (else KDA_ERR_WORKSPACE).  S0, S_T, o, g_in, norm_w, y and the snapshot
 *   fields are not read.  Inputs and their validation as for kda_prefill;
 *   KDA_ERR_UNSUPPORTED for inputs the chunk-parallel schedule does not take
 *   (other than bf16 q/k/v with d = 128 or float32 q/k/v with d = 32, 64).
 * kda_prefill_scan: the state recurrence over the records that
 *   kda_prefill_records wrote into args->workspace, producing o, S_T, y and
 *   snapshots exactly as kda_prefill (bit for bit) from args->S0.  The record
 *   inputs of args must be those of the kda_prefill_records call (the library
 *   cannot check this); S0 and the outputs may differ from call to call.  The
 *   workspace is only read, so any number of scans may follow one records
 *   call, each on any stream ordered after it.  flags: 0, or KDA_SCAN_ZERO_V:
 *   evaluate the operator with v = 0 (the records' U parts are not read; the
 *   outputs are those of kda_prefill with a zero v, not bit for bit: this
 *   scan also follows the decaying state's magnitude chunk by chunk, so that
 *   a transition matrix keeps its precision until it has decayed below about
 *   2^-24 of |S0|).  Other flags -> KDA_ERR_SHAPE.
 */
#define KDA_SCAN_ZERO_V 1
kda_status kda_prefill_records(const kda_prefill_args* args, void* stream);
kda_status kda_prefill_scan(const kda_prefill_args* args, int flags, void* stream);

/*
 * kda_prefill for callers that cannot allocate device memory.  (Library
 * plumbing: the KDA pages have no counterpart of this entry point.)
 *
 * Some callers cannot call cudaMalloc at all -- for example a serving engine
 * or plugin host that reserves all device memory for its own pool up front and
 * forbids allocation while requests run -- and so cannot provide the
 * workspace kda_prefill asks for.  This entry point takes the same arguments
 * but ignores args->workspace / args->workspace_bytes and uses instead a fixed
 * array of KDA_NOALLOC_SCRATCH_BYTES bytes in the library's own device memory
 * (every GPU that loads the library holds it until the process exits).  It
 * allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - It runs the schedule that needs the least scratch (on the tensor-core
 *    path the single-pass one, KDA_PREFILL_MIN_WORKSPACE bytes); calls whose
 *    least scratch exceeds KDA_NOALLOC_SCRATCH_BYTES are rejected with
 *    KDA_ERR_WORKSPACE (the message is in kda_last_error_string()).
 *  - All calls share the one array; it keeps the previous call's contents and
 *    each call clears what must start at zero (with cudaMemsetAsync on the
 *    caller's stream).  Calls that overlap on the GPU (different streams with
 *    no ordering between them) race on the array: serialise them.
 *  - Each call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress: no allocation, nothing cached across calls, so a
 *    device reset that reloads the library's module leaves no stale address).
 *    The first call on a device loads the module there; make that first call
 *    before any stream capture.
 *  - A bounded wait that gives up is recorded in the array's error word; read
 *    it with kda_get_last_device_error(NULL, stream).  The size check above
 *    cannot reject a call at the current sizes (the single-pass schedule
 *    needs KDA_PREFILL_MIN_WORKSPACE bytes, the CUDA-core path none); it
 *    guards future schedules.
 * Inputs and outputs are the caller's, exactly as for kda_prefill.
 */
#define KDA_NOALLOC_SCRATCH_BYTES 4096
kda_status kda_prefill_noalloc(const kda_prefill_args* args, void* stream);

/*
 * kda_prefill of one sequence whose inputs and outputs are in HOST memory, the
 * copies overlapped with the compute.  (Library plumbing: the pages have no
 * counterpart.)
 *
 * args as for kda_prefill with num_seqs = 1 and T_total tokens, except that q,
 * k, v, z, beta, A, S0 (may be NULL), g_in (may be NULL), norm_w (may be NULL),
 * o, y and S_T are HOST pointers (page-locked memory, e.g. cudaHostAlloc, for
 * the copies to overlap; pageable memory works but serialises them);
 * cu_seqlens, cu_seqlens_host, workspace and workspace_bytes are ignored;
 * snapshots are not taken (S_snap must be NULL, else KDA_ERR_UNSUPPORTED).
 * With T_total = 0 the token arrays may be NULL and S_T receives S0 (or 0).
 * The sequence is cut into slabs of `slab` tokens (a positive multiple of 64,
 * else KDA_ERR_SHAPE); slab i resumes from the state slab i - 1 left, exactly
 * as one kda_prefill call over the whole sequence would up to the power-of-two
 * scales each slab's scan picks for its fp16 operands (equal to about 1e-6
 * relative).  Host-to-device copies run one slab ahead and device-to-host
 * copies one slab behind, on two streams the library creates for the call;
 * the compute runs on `stream`, which on return is ordered after every copy:
 * synchronise it before reading o, y, S_T or reusing the inputs.
 *
 * staging: caller-owned device memory of
 * kda_prefill_from_host_staging_size(args, slab) bytes (16-byte aligned, else
 * KDA_ERR_ALIGN; smaller -> KDA_ERR_WORKSPACE): double-buffered slab inputs and
 * outputs, the carried state, and one slab's prefill workspace (the
 * chunk-parallel schedule).  The staging is in use until `stream` completes.
 * Errors: those of kda_prefill for the slab calls, KDA_ERR_CUDA for a failed
 * copy or stream operation.
 */
size_t kda_prefill_from_host_staging_size(const kda_prefill_args* args, int slab);
kda_status kda_prefill_from_host(const kda_prefill_args* args, int slab, void* staging, size_t staging_bytes,
                                 void* stream);

/*
 * The same operator as kda_prefill, always evaluated by the per-token
 * recurrence on CUDA cores (one CTA per sequence and head, the state held in
 * registers).  Same arguments, layouts, validation and status codes as
 * kda_prefill; the workspace is not used.  Exported to cross-check the
 * chunked tensor-core path on the GPU; it is sequential in the tokens of each
 * sequence and therefore slow for long sequences.
 */
kda_status kda_prefill_recurrent(const kda_prefill_args* args, void* stream);

/*
 * Batched single-token decode step (Sec. 2.1 recurrence, one token per
 * sequence), states updated IN PLACE.
 *
 *   q, k, z [N, H, dk] (q, k bf16; z float32); v [N, H, dv] bf16;
 *   beta [N, H] float32; A [H] float32;
 *   state [num_slots, H, dk, dv] float32, read and overwritten;
 *   slots [N] int32 row of `state` used by sequence n, or NULL (row n,
 *         then num_slots >= N is required); slots must be distinct.  The
 *         kernel range-checks every slot on the device and skips a sequence
 *         whose slot lies outside [0, num_slots): its state row, o and y are
 *         left untouched (no fault, no error code, since the slots live in
 *         device memory and are not read on the host).
 *   o [N, H, dv] bf16 output or NULL; g_in/norm_w/y as in prefill
 *   (y required iff g_in).  At least one of o, y must be given.
 * Supported: dk = dv = 128.
 */
typedef struct {
    int N, H, dk, dv, num_slots;
    const void* q;
    const void* k;
    const void* v;
    const float* z;
    const float* beta;
    const float* A;
    float g_min;
    float scale;
    int qk_l2norm;
    float* state;
    const int32_t* slots;
    void* o;
    const void* g_in;
    const float* norm_w;
    float norm_eps;
    void* y;
    int gate_mode;        /* kda_gate; KDA_ERR_UNSUPPORTED for other values */
} kda_decode_args;

kda_status kda_decode_step(const kda_decode_args* args, void* stream);

/*
 * Output gate alone (Sec. 2.3): y = Sigmoid(g_in) (.) w (.) o / sqrt(mean(o^2)+eps),
 * the mean taken over the dv channels of each (token, head) row.
 *   o, g_in, y [rows, dv] (rows = tokens * H) with dtype `dtype` (bf16 or
 *   float32; all three the same); w [dv] float32 or NULL (ones).
 * Supported: dv in {32, 64, 128, 256}.
 */
kda_status kda_gate_norm(const void* o, const void* g_in, const float* norm_w, float eps,
                         void* y, long rows, int dv, kda_dtype dtype, void* stream);

/*
 * ShortConv + Swish prologue (Sec. 2.1: q and k pass through ShortConv, Swish
 * and L2Norm before the recurrence, v through ShortConv and Swish; Sec. 5:
 * Swish(z) = z * Sigmoid(z); "Kimi-K3 深度技术分析" (liuhc.cn), prefill-decode
 * section: decode keeps a sliding-window state of the convolution).  The pages
 * give no width; any W in 1..8.  Per channel c of each packed sequence n:
 *   pre[t, c] = sum_{i=0}^{W-1} weight[c*W + i] * x[t - (W-1) + i, c] + bias[c]
 *   y[t, c]   = Swish(pre[t, c])  (activation = 1)  or  pre[t, c]  (activation = 0)
 * where positions before the sequence's first token read state_in[n] (the W-1
 * inputs that preceded it, oldest first; zeros when state_in is NULL), and
 * state_out[n] receives the last W-1 entries of [state_in[n], x of sequence n].
 *   x, y                 [T_total, channels]  dtype (bf16 or float32; y != x)
 *   weight               [channels, W] float32;  bias [channels] float32 or NULL
 *   state_in, state_out  [num_seqs, W-1, channels] float32 or NULL (must differ)
 * cu_seqlens / cu_seqlens_host as for kda_prefill.  channels: a multiple of 8.
 * The L2Norm of q and k is kda_prefill's qk_l2norm.  Errors: KDA_ERR_SHAPE
 * (width, channels), KDA_ERR_SEQLENS, KDA_ERR_NULL, KDA_ERR_ALIGN (16 bytes),
 * KDA_ERR_DTYPE.
 */
typedef struct {
    int num_seqs;
    int T_total;
    int channels;
    int width;
    kda_dtype dtype;
    const int32_t* cu_seqlens;       /* device */
    const int32_t* cu_seqlens_host;  /* host   */
    const void* x;
    const float* weight;
    const float* bias;
    const float* state_in;
    float* state_out;
    void* y;
    int activation;
} kda_short_conv_args;

kda_status kda_short_conv(const kda_short_conv_args* args, void* stream);

/*
 * One decode step of the prologue: x, y [N, channels] (one token per sequence),
 * state [num_slots, W-1, channels] float32 updated in place (row slots[i] for
 * token i, or row i when slots is NULL; slots must be distinct):
 *   y = Swish(conv([state, x]))  then  state <- last W-1 entries of [state, x].
 */
typedef struct {
    int N;
    int channels;
    int width;
    int num_slots;
    kda_dtype dtype;
    const void* x;
    const float* weight;
    const float* bias;
    float* state;
    const int32_t* slots;
    void* y;
    int activation;
} kda_short_conv_step_args;

kda_status kda_short_conv_step(const kda_short_conv_step_args* args, void* stream);

/*
 * KDA context parallelism (Sec. 10.2): a segment acts on the state as
 * S_exit = M S_entry + S~ with M = M_T ... M_1, M_t = (I - beta_t k_t k_t^T)
 * Diag(alpha_t), and S~ the segment's state from zero.  Both come from
 * kda_prefill run state-only (o = NULL): M is the final state with v = 0 and
 * S0 = I (dv = dk), S~ the final state with S0 = NULL.  A rank's entry state is
 * the earlier segments' pairs applied in order, S <- M_j S + S~_j, and pairs
 * compose as (M2, S2) o (M1, S1) = (M2 M1, S2 + M2 S1).
 *
 * kda_kcp_apply: for every head h, X[h] <- M[h] X[h] + add[h], in FP32.
 *   M [H, d, d], X [H, d, n] (in/out), add [H, d, n] or NULL; X must not
 *   overlap M or add; 1 <= d <= 256, n >= 1; all device memory, 16-byte aligned.
 */
kda_status kda_kcp_apply(const float* M, float* X, const float* add, int H, int d, int n, void* stream);

/*
 * Device-side error report of the tensor-core prefill (library plumbing: the
 * KDA pages have no counterpart).  Every wait of a prefill kernel on an
 * asynchronous copy, a tensor-core operation or a peer CTA is bounded; a wait
 * that runs out records it in the call's error word, stops issuing new
 * asynchronous work, waits (again bounded) for the copies and tensor-core
 * operations it has already issued, and lets the kernel finish, so the CUDA
 * context stays usable.  The call's outputs are then invalid.
 *
 * kda_get_last_device_error waits for the work queued on `stream`, then reads
 * and clears the error word of `workspace` (the workspace the prefill calls
 * used), or, with workspace == NULL, of the fixed array kda_prefill_noalloc
 * uses on the current device.  Returns KDA_OK when no wait gave up,
 * KDA_ERR_TIMEOUT when one did, KDA_ERR_CUDA when the read failed.  It
 * allocates nothing.  Call it on the stream of the prefill calls (or after
 * synchronising them); calls on other streams that use the same workspace
 * must not run concurrently.
 */
kda_status kda_get_last_device_error(void* workspace, void* stream);

/*
 * Test hook: the number of polls after which a bounded wait of the prefill
 * kernels on a copy or a tensor-core operation gives up, for every launch
 * that follows (from any thread).  KDA_WAIT_LIMIT_DEFAULT restores the
 * default (about 4 million polls: seconds); 0 makes every such wait give up
 * at once, which exercises, deterministically, the path that
 * kda_get_last_device_error reports.  Waits between the CTAs of a cluster and
 * the final waits before a CTA exits keep their default bound.  Returns the
 * previous setting.
 */
#define KDA_WAIT_LIMIT_DEFAULT 0xFFFFFFFFu
uint32_t kda_debug_set_wait_limit(uint32_t polls);

/* Static description of a status code. */
const char* kda_status_str(kda_status s);

/* Text of the last CUDA error seen by this thread inside the library. */
const char* kda_last_error_string(void);

/* Number of kernel launches this library has enqueued from the calling host
 * thread since the thread first called into it (a monotone counter, for
 * accounting launches inside a timed region). */
uint64_t kda_launch_count(void);

/* Library build description (architecture, version). */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H_ */
