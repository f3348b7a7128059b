// Chunk-parallel KDA prefill on the sm_103a tensor cores: the state-free part
// of every chunk runs in parallel over all chunks, and only the state recurrence
// runs sequentially.
//
// Operator: "Kimi K3: KDA, attention residuals and Stable LatentMoE"
// (hs-black.github.io) Sec. 2.1 chunked form with the Sec. 2.2 bounded gate and
// 16-token sub-chunks and the Sec. 2.3 output gate.  Per chunk of C = 64 tokens
// (notation as in the single-pass kernel):
//   [U | W ; U_o | P Gamma K] = [T Diag(beta) ; P Diag(beta)] . [V | Gamma K]
//   [V' ; O] = [U ; U_o] + [-W ; Gamma Q - P Gamma K] . S
//   S_next   = Diag(gamma_C) S + (K gamma_C / Gamma)^T V'
// Everything in the first line, and the operands of the other two, depends on
// the chunk's own tokens only.  Unrolled over chunks, the state obeys
//   S_{c+1} = E_c S_c + F_c,  E_c = Diag(gamma_C) - (K gamma_C/Gamma)^T W,
//                             F_c = (K gamma_C/Gamma)^T U,
// which is the per-segment transition pair of the pages' context parallelism
// (Sec. 10.2: S_exit = M S_entry + S~) at the granularity of one chunk, kept in
// factored (rank-64) form so that applying it costs two thin products.
//
// Three launches on the caller's stream:
//   plan  -- chunk offsets of the packed sequences (exclusive scan of
//            ceil(len / 64)) into the workspace;
//   prep  -- persistent, one CTA per SM, a loop over (chunk, head) records:
//            gate, Gram sub-blocks, blockwise UT solve and MMA 1 (the single-
//            pass kernel's arithmetic; the solve's block merge by doubling),
//            then writes the record [-W ; Gamma Q - P Gamma K] (fp16, output
//            rows scaled by powers of two), [U ; U_o] (fp32), (K gamma_C /
//            Gamma)^T (fp16), gamma_C and the rows' factors, most of it by TMA
//            stores that drain while the next record runs;
//   scan  -- a cluster of four CTAs per (sequence, head), CTA r owning value
//            columns [32r, 32r+32): per chunk MMA 2 (A from shared memory by
//            TMA, accumulating onto [U ; U_o] preloaded into TMEM), V' to the
//            MMA 3 operand, O to o and the fused output gate, MMA 3, and the
//            FP32 state update in TMEM, the MMAs on fp16 operands under per-
//            column power-of-two scaling.  The records of the next chunks are
//            fetched while the current one is processed.
#include <mutex>

#include "kda_common.cuh"
#include "tcgen05.cuh"
#include "tma_host.cuh"

namespace kda {
namespace spl {

constexpr int C = 64;     // chunk length
constexpr int D = 128;    // dk = dv
constexpr int NT = 256;   // threads per CTA
constexpr int AS = 68;    // padded row stride (floats) of the 64x64 Gram tiles
constexpr int SCAN_R = 4; // scan: CTAs (value-column blocks) per (sequence, head)

// one record per (chunk, head), in four arrays of the workspace: the two MMA
// operands in fp16 (the tf32 mantissa; their range is bounded, see the scan),
// the additive terms and the decay in FP32
constexpr size_t AW_ELEMS = 128 * 128;    // [-W ; Gamma Q - P Gamma K]  [row][d]  fp16
constexpr size_t UU_FLOATS = 128 * 128;   // [U ; U_o]                   [row][e]  FP32
constexpr size_t KT_ELEMS = 128 * 64;     // (K gamma_C / Gamma)^T       [d][t]    fp16
constexpr size_t GM_FLOATS = 192;         // [gamma_C ; rho]             [d] [t]   FP32

struct Work {
    const int* chunk_base;   // [num_seqs + 1] first global chunk of each sequence
    int* vmax;               // [num_seqs][H][128] max |v| of each value column (FP32 bits)
    uint16_t* aw;
    float* uu;
    uint16_t* kt;
    float* gm;
    int* err;                // error word: tc::ERR_WAIT | tc::ERR_DRAIN
    long nrec;               // chunks * H
    int zero_v;              // scan: take v as zero (the U records are not read)
    uint32_t wait_limit;     // polls before a wait on a local copy or MMA gives up
};

TC_DEV uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(tc::smem_u32(p)), "r"(rank));
    return r;
}
TC_DEV void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
TC_DEV void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// byte offset of bf16 element (row, col) in a [rows][64] tile written by TMA with the 128-B swizzle
TC_DEV uint32_t sw128_bf16(int row, int col) {
    return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}
TC_DEV float4 ld_f4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
// byte offset of fp32 element (row, col) in a [rows][32] tile written by TMA with the 128-B swizzle
TC_DEV uint32_t sw128_f32(int row, int col) {
    return (uint32_t)(row * 128 + ((((col >> 2) ^ (row & 7))) << 4) + ((col & 3) << 2));
}
// 2^e as a float, e in [-126, 127]
TC_DEV float exp2i(int e) { return __int_as_float((e + 127) << 23); }
// 16 values as fp16 in one 32-byte streaming store (p 32-byte aligned)
TC_DEV void st_stream_h16(uint16_t* p, const float* v) {
    float w8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w8[i] = __uint_as_float(tc::pack_f16x2(v[2 * i], v[2 * i + 1]));
    st_stream_f8(reinterpret_cast<float*>(p), w8);
}
// four 8 x 4 fp32 matrices from shared memory (ldmatrix on 16-bit pairs): lane l
// passes the address of row l & 7 of matrix l >> 3 (16-byte aligned) and gets
// word (l & 3) of row (l >> 2) of each matrix -- the tf32 m16n8k8 fragment order
TC_DEV void ldsm_x4(const float* p, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(tc::smem_u32(p)) : "memory");
}

// ---------------------------------------------------------------------------
// plan: chunk_base[n] = sum_{m < n} ceil(len_m / C), n = 0..num_seqs (one CTA);
// also clears the call's error word
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_kernel(const int* cu, int num_seqs, int* chunk_base, int* vmax,
                                                     long nvmax, int* err) {
    __shared__ int s_warp[32];
    __shared__ int s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_carry = 0;
        *err = 0;   // the call's error word starts clear (the kernels after this one set it)
    }
    __syncthreads();
    for (int base = 0; base < num_seqs; base += 1024) {
        const int n = base + tid;
        const int v = n < num_seqs ? (cu[n + 1] - cu[n] + C - 1) / C : 0;
        int x = v;   // inclusive scan inside the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = s_warp[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const int carry = s_carry;
        const int incl = carry + x + (warp > 0 ? s_warp[warp - 1] : 0);
        if (n < num_seqs) chunk_base[n] = incl - v;
        __syncthreads();
        if (tid == 1023) s_carry = incl;
        __syncthreads();
    }
    if (tid == 0) chunk_base[num_seqs] = s_carry;
    for (long i = tid; i < nvmax; i += 1024) vmax[i] = 0;   // prep takes maxima into it
}

// record -> (sequence, first token, tokens, head); chunk_base has num_seqs + 1 entries
struct Loc { int t0, nc, h, n; };
TC_DEV Loc locate(long rec, int H, const int* cu, const int* cb, int num_seqs) {
    const int g = (int)(rec / H);
    Loc l;
    l.h = (int)(rec - (long)g * H);
    int lo = 0, hi = num_seqs;          // largest n with cb[n] <= g (cb[num_seqs] > g)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cb[mid] <= g) lo = mid; else hi = mid;
    }
    l.t0 = cu[lo] + C * (g - cb[lo]);
    l.nc = min(C, cu[lo + 1] - l.t0);
    l.n = lo;
    return l;
}

// Row i and column j (j <= i) of the p-th entry of a 16 x 16 lower triangle, row-major.
__host__ __device__ constexpr int tri_row(int p) { int i = 0; while ((i + 1) * (i + 2) / 2 <= p) ++i; return i; }
__host__ __device__ constexpr int tri_col(int p) { return p - tri_row(p) * (tri_row(p) + 1) / 2; }

// Warp reduce-scatter of 32 values: afterwards lane l holds the sum over the
// warp of v[l] (five exchange rounds, 31 shuffles).  v is overwritten.
TC_DEV float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < m; ++k) {
            const float send = up ? v[k] : v[k + m];
            const float keep = up ? v[k + m] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    return v[0];
}

// ---------------------------------------------------------------------------
// prep: the state-free part of every chunk
// ---------------------------------------------------------------------------
namespace prep {
// Region RB, in turn: the raw q, k, z tiles; the Gram's B operand (the key versions);
// the Gram tiles and the solve's scratch; then, from the end of the solve, the next
// record's raw q, k, z.  B_pre = [V | Gamma K]^T, MMA 1's B operand, comes in two
// halves: V^T in region QK once the Gram has read [Q~ ; K~], (Gamma K)^T in a region
// of its own, written while the Gram runs.
constexpr int KV_ROWS = 160;                        // key versions: 16 (a + 1) rows for a = 0..3
constexpr int RB_BYTES = KV_ROWS * D * 4;           // 80 KB
constexpr int OFF_RB = 0;
constexpr int OFF_RAWQ = OFF_RB;                    // [C][D] bf16
constexpr int OFF_RAWK = OFF_RB + C * D * 2;        // [C][D] bf16
constexpr int OFF_RAWZ = OFF_RB + 2 * C * D * 2;    // [C][D] f32
constexpr int OFF_KV = OFF_RB;                      // SW128 [160 rows][D]
constexpr int OFF_AQK = OFF_RB;
constexpr int OFF_AKK = OFF_RB + C * AS * 4;
constexpr int OFF_QK = OFF_RB + RB_BYTES;           // the Gram's A operand [Q~ ; K~], SW128 [128 rows][D]
constexpr int OFF_BPRE = OFF_QK;                    // V^T, SW128 [128 rows][C]
constexpr int OFF_RAWV = OFF_QK + 2 * C * D * 4;    // two [C][64] bf16 tiles, 128-B swizzle
constexpr int OFF_GK = OFF_RAWV + 2 * C * 64 * 2;   // (Gamma K)^T, SW128 [128 rows][C]
constexpr int OFF_SMALL = OFF_GK + D * C * 4;
constexpr int SM_BETA = 0, SM_RQ = 64, SM_RK = 128, SM_TAU = 192, SM_EXPS = SM_TAU + 4 * D,
              SM_GAM = SM_EXPS + 4 * D,
              SM_DIAG = SM_GAM + D,                     // [4 sub-chunks][9 batches][4 warps][32]
              SM_EA = SM_DIAG + 4 * 9 * 4 * 32,         // exp(A_h) of heads 0..EA_HEADS-1
              SM_LOC = SM_EA + 128,                     // record walk (ints), see prep_kernel
              SM_FLOATS = SM_LOC + 16;
constexpr int EA_HEADS = 128;
constexpr int SMEM_BYTES = OFF_SMALL + SM_FLOATS * 4 + 64 + 1024;
static_assert(OFF_RAWV % 1024 == 0 && OFF_BPRE % 1024 == 0 && OFF_QK % 1024 == 0 && OFF_KV % 1024 == 0 &&
              OFF_GK % 1024 == 0, "swizzled tiles need 1024-B alignment");
static_assert(2 * C * D * 2 + C * D * 4 <= RB_BYTES, "region RB");
static_assert(3 * C * AS * 4 + (NT / 32) * 16 * 16 * 4 <= RB_BYTES, "region RB holds the solve tiles");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr uint32_t BYTES_QKZ = 2 * C * D * 2 + C * D * 4;
constexpr uint32_t BYTES_V = C * D * 2;
// float32 inputs with d_k = d_v = DIN <= 64: compact [C][DIN] fp32 tiles in the same
// slots (q, k, z: 16 KB at most each, v: 16 KB at most); channels DIN..127 read as 0
constexpr int DIN_MAX = 64;
constexpr int NTP = 512;         // threads per CTA (16 warps; warps w, w+4, w+8, w+12 share TMEM lanes)
constexpr uint32_t TM_D = 0;     // 256 cols: [U | W ; U_o | P Gamma K - Gamma Q]
constexpr uint32_t TM_A2 = 256;  // 64 cols: [T beta ; P beta]
constexpr uint32_t TM_G = 320;   // 160 cols: [Q~ ; K~] . (key versions)^T
constexpr uint32_t TM_COLS = 512;
// first row of key version a (keys of sub-chunks 0..a referred to the start of sub-chunk a)
__host__ __device__ constexpr int kv_row0(int a) { return 8 * a * (a + 1); }
}  // namespace prep

// GATE 0: K3's bounded gate; 1: Kimi Linear's Softplus gate, whose diagonal Gram
// sub-blocks are formed pair by pair (their sub-chunk factors can exceed fp32).
// IN32 0: bf16 q, k, v with d = 128; 1: float32 q, k, v with d = a.dk <= 64, the
// channels from d to 127 taken as zero (every record term they touch is then 0, so
// the d = 128 records and scan carry the smaller operator exactly).
template <int GATE, int IN32>
__global__ void __launch_bounds__(prep::NTP, 1)
prep_kernel(kda_prefill_args a, Work w,
            const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_v,
            const __grid_constant__ CUtensorMap tm_uu, const __grid_constant__ CUtensorMap tm_aw) {
    using namespace prep;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sBpre = sm + OFF_BPRE;
    uint8_t* sGK = sm + OFF_GK;
    const uint16_t* sRawQ = reinterpret_cast<const uint16_t*>(sm + OFF_RAWQ);
    const uint16_t* sRawK = reinterpret_cast<const uint16_t*>(sm + OFF_RAWK);
    const float* sRawZ = reinterpret_cast<const float*>(sm + OFF_RAWZ);
    const uint8_t* sRawV = sm + OFF_RAWV;
    const int din = IN32 ? a.dk : D;   // input channels
    // raw input element (token t, channel d) of the staged tiles
    auto raw_q = [&](int t, int d) -> float {
        if (IN32) return d < din ? reinterpret_cast<const float*>(sRawQ)[t * din + d] : 0.f;
        return bf16_to_f(sRawQ[t * D + d]);
    };
    auto raw_k = [&](int t, int d) -> float {
        if (IN32) return d < din ? reinterpret_cast<const float*>(sRawK)[t * din + d] : 0.f;
        return bf16_to_f(sRawK[t * D + d]);
    };
    auto raw_z = [&](int t, int d) -> float {
        if (IN32) return d < din ? sRawZ[t * din + d] : 0.f;
        return sRawZ[t * D + d];
    };
    auto raw_v = [&](int t, int e) -> float {
        if (IN32) return e < din ? reinterpret_cast<const float*>(sRawV)[t * din + e] : 0.f;
        return bf16_to_f(*reinterpret_cast<const uint16_t*>(sRawV + (e >> 6) * (C * 128) + sw128_bf16(t, e & 63)));
    };

    uint8_t* sQK = sm + OFF_QK;   // [Q~ ; K~]: rows t = q_t exp(G_t - G_start), rows 64 + t = k_t exp(...)
    uint8_t* sKV = sm + OFF_KV;   // key versions
    auto qk_at = [&](int r, int d) -> float& { return *reinterpret_cast<float*>(sQK + tc::sw128_offset(r, d, 2 * C)); };
    float* sAqk = reinterpret_cast<float*>(sm + OFF_AQK);
    float* sAkk = reinterpret_cast<float*>(sm + OFF_AKK);
    float* fs = reinterpret_cast<float*>(sm + OFF_SMALL);
    float* s_beta = fs + SM_BETA;
    float* s_rq = fs + SM_RQ;
    float* s_rk = fs + SM_RK;
    float* s_tau = fs + SM_TAU;
    float* s_expS = fs + SM_EXPS;
    float* s_gam = fs + SM_GAM;
    float* s_diag = fs + SM_DIAG;
    float* s_eA = fs + SM_EA;
    // s_loc: [0..2] this record's {t0, nc, h}, [3..5] the next one's, [6], [7] their
    // sequences; [8..15] the walk
    // at the next record: chunk g (long), head, sequence n, cb[n], cb[n+1], cu[n], cu[n+1]
    int* s_loc = reinterpret_cast<int*>(fs + SM_LOC);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(fs + SM_FLOATS);
    uint64_t* bar_in = mbar + 1;
    uint64_t* bar_v = mbar + 2;
    uint32_t* tbase_ptr = reinterpret_cast<uint32_t*>(mbar + 3);
    const uint32_t bytes_qkz = IN32 ? 3u * C * din * 4 : BYTES_QKZ;
    const uint32_t bytes_v = IN32 ? (uint32_t)C * din * 4 : BYTES_V;
    auto load_qkz = [&](const Loc& l) {   // thread 0
        tc::mbar_arrive_expect_tx(bar_in, bytes_qkz);
        tc::tma_load_2d(sm + OFF_RAWQ, &tm_q, l.h * din, l.t0, bar_in);
        tc::tma_load_2d(sm + OFF_RAWK, &tm_k, l.h * din, l.t0, bar_in);
        tc::tma_load_2d(sm + OFF_RAWZ, &tm_z, l.h * din, l.t0, bar_in);
    };
    auto load_v = [&](const Loc& l) {     // thread 0
        tc::mbar_arrive_expect_tx(bar_v, bytes_v);
        tc::tma_load_2d(sm + OFF_RAWV, &tm_v, l.h * din, l.t0, bar_v);
        if (!IN32) tc::tma_load_2d(sm + OFF_RAWV + C * 128, &tm_v, l.h * D + 64, l.t0, bar_v);
    };

    const int H = a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, grp = warp >> 2;   // TMEM lane quarter, column quarter
    const int row = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const long stride = gridDim.x;
    long rec = blockIdx.x;
    Loc cur = locate(rec, H, a.cu_seqlens, w.chunk_base, a.num_seqs);

    if (warp == 0) { tc::tmem_alloc(tbase_ptr, TM_COLS); tc::tmem_relinquish(); }
    if (tid < EA_HEADS && tid < H) s_eA[tid] = __expf(a.A[tid]);
    // records are visited with a fixed stride: the walk advances (g, h) without a
    // division and searches the sequence table only when it leaves a sequence
    const long step_g = stride / H;
    const int step_h = (int)(stride - step_g * H);
    if (tid == NTP - 1) {
        s_loc[0] = cur.t0; s_loc[1] = cur.nc; s_loc[2] = cur.h; s_loc[6] = cur.n;
        const long rn = rec + stride;
        const long g = rn / H;
        const int hn = (int)(rn - g * H);
        int n = 0;
        if (rn < w.nrec) {
            int hi = a.num_seqs;
            while (hi - n > 1) { const int mid = (n + hi) >> 1; if (w.chunk_base[mid] <= g) n = mid; else hi = mid; }
        }
        *reinterpret_cast<long*>(s_loc + 8) = g;
        s_loc[10] = hn; s_loc[11] = n;
        s_loc[12] = w.chunk_base[n]; s_loc[13] = w.chunk_base[n + 1];
        s_loc[14] = a.cu_seqlens[n]; s_loc[15] = a.cu_seqlens[n + 1];
        const int t0 = s_loc[14] + C * (int)(g - s_loc[12]);
        s_loc[3] = t0; s_loc[4] = min(C, s_loc[15] - t0); s_loc[5] = hn; s_loc[7] = n;
    }
    // thread 0 issues every copy and MMA; it counts the phases it issued on each
    // mbarrier, for the give-up path at the end
    uint32_t n_in = 0, n_v = 0, n_mma = 0;
    if (tid == 0) {
        tc::mbar_init(mbar, 1);
        tc::mbar_init(bar_in, 1);
        tc::mbar_init(bar_v, 1);
        tc::mbar_fence_init();
        tc::tma_prefetch_desc(&tm_q);
        tc::tma_prefetch_desc(&tm_k);
        tc::tma_prefetch_desc(&tm_z);
        tc::tma_prefetch_desc(&tm_v);
        if (rec < w.nrec) {
            load_qkz(cur);
            load_v(cur);
            n_in = n_v = 1;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t T0 = *tbase_ptr;
    uint32_t ph_mma = 0, ph_in = 0, ph_v = 0;
    bool timed_out = false;
    // A wait that gives up records it; this thread then skips every later wait,
    // and thread 0 issues no further copy or MMA, so the kernel runs to its end
    // quickly (its results are then invalid) and drains what was issued.
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!timed_out && !tc::mbar_wait_bounded(bar, parity, w.wait_limit)) timed_out = true;
    };
    float beta_next = 0.f;
    if (rec < w.nrec && tid < C && tid < cur.nc) beta_next = a.beta[(size_t)(cur.t0 + tid) * H + cur.h];

    // the four column groups' largest |A| and |U_o| of each output row (phase 6; the
    // diagonal-block buffer is free then)
    float* s_rmax = s_diag;
    // the record's TMA stores are issued and awaited by a thread that has no part in the
    // L2 norms (step 1a), so that the wait for the previous record's stores overlaps them
    constexpr int TID_ST = NTP - 32;
    bool stores_out = false;   // thread TID_ST: the previous record's A-tile store may still read its tile

    for (; rec < w.nrec; rec += stride) {
        // the previous record's [U ; U_o] tile (region QK) is rewritten in 1b, its A tile
        // (the (Gamma K)^T region) in step 2: their stores, in that order, in two groups
        if (tid == TID_ST && stores_out) tc::bulk_wait_read_but1();
        const bool has_next = rec + stride < w.nrec;
        cur = Loc{s_loc[0], s_loc[1], s_loc[2], s_loc[6]};
        const Loc nxt = has_next ? Loc{s_loc[3], s_loc[4], s_loc[5], s_loc[7]} : cur;
        const int nc = cur.nc, h = cur.h;
        const float eA = h < EA_HEADS ? s_eA[h] : __expf(__ldg(a.A + h));
        if (tid < C) {
            s_beta[tid] = beta_next;
            beta_next = (has_next && tid < nxt.nc) ? a.beta[(size_t)(nxt.t0 + tid) * H + nxt.h] : 0.f;
        }
        wait(bar_in, ph_in);
        ph_in ^= 1u;

        // ---- 1a. q/k L2 norms: threads 2v and 2v+1 cover vector v (q of token v for
        //          v < 64, else k of token v - 64), 64 dims each, reading 16-byte chunks in
        //          a rotated order so that each quarter-warp hits 8 distinct bank groups
        if (tid < 2 * D) {
            const int v = tid >> 1, half = tid & 1;
            const int t = v & (C - 1);
            const uint16_t* rowp = (v < C ? sRawQ : sRawK) + t * D + half * (D / 2);
            float ssum = 0.f;
            if (IN32 && t < nc) {   // channels half * din/2 .. +din/2 of the fp32 row
                for (int c = half * (din >> 1); c < (half + 1) * (din >> 1); ++c) {
                    const float x = v < C ? raw_q(t, c) : raw_k(t, c);
                    ssum = fmaf(x, x, ssum);
                }
            } else if (!IN32 && t < nc) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = (i + 2 * v + half) & 7;
                    const uint4 u = *reinterpret_cast<const uint4*>(rowp + 8 * c);
                    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float lo = __uint_as_float(wv[j] << 16), hi = __uint_as_float(wv[j] & 0xffff0000u);
                        ssum = fmaf(lo, lo, fmaf(hi, hi, ssum));
                    }
                }
            }
            ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
            if (half == 0) (v < C ? s_rq : s_rk)[t] = a.qk_l2norm ? rsqrtf(ssum + 1e-6f) : 1.f;
        }
        __syncthreads();

        // ---- 1b. gate and sub-chunk-relative decay factors (thread: channel d, sub-chunk b);
        //          q~, k~ (tf32) into the Gram's A operand, k_t exp(G_end(b) - G_t) kept in kf2
        float kf2[16];
        {
            const int d = tid & (D - 1);
#pragma unroll 1
            for (int b = tid >> 7; b < (tid >> 7) + 1; ++b) {   // channel d, sub-chunk b
                float al[16], kv[16], qv[16], Lc[16];
                float F1 = 1.f, L = 0.f;
                const float c1 = -eA * 1.4426950408889634f, c2 = a.g_min * 1.4426950408889634f;   // log2(e)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int t = 16 * b + i;
                    float alpha = 1.f, q = 0.f, k = 0.f;
                    if (t < nc) {
                        if (GATE) {
                            const float g = log_decay_softplus(raw_z(t, d), eA);
                            alpha = __expf(g);
                            L += g;
                        } else {   // exp(g_min Sigmoid(eA z)) in base 2: the two scalings folded
                            const float sg = __fdividef(1.f, 1.f + exp2f(c1 * raw_z(t, d)));
                            alpha = exp2f(c2 * sg);
                        }
                        q = raw_q(t, d) * s_rq[t];
                        k = raw_k(t, d) * s_rk[t];
                    }
                    F1 *= alpha;                   // exp(G_t - G_start(b))
                    al[i] = alpha;
                    kv[i] = k;
                    qv[i] = q;
                    Lc[i] = L;                     // G_t - G_start(b), log domain
                    qk_at(t, d) = tc::to_tf32(q * F1);
                    qk_at(C + t, d) = tc::to_tf32(k * F1);
                }
                float F2 = 1.f;                    // exp(G_end(b) - G_t)
#pragma unroll
                for (int i = 15; i >= 0; --i) {
                    kf2[i] = kv[i] * F2;
                    F2 *= al[i];
                }
                s_tau[b * D + d] = F1;
                if (GATE) {
                    // diagonal sub-block b pair by pair: this channel's share of
                    // A_qk(i,j) = sum_d q_i k_j exp(G_i - G_j) (j <= i) and of A_kk
                    // (j < i), 16 pairs per batch, reduce-scattered over the warp's
                    // 32 channels; the four warps of a sub-chunk add up later
                    float* dst = s_diag + (b * 9 * 4 + (warp & 3)) * 32 + lane;
#pragma unroll
                    for (int bt = 0; bt < 9; ++bt) {
                        float vals[32];
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int p = 16 * bt + u;
                            if (p < 136) {
                                const int i = tri_row(p), j = tri_col(p);
                                const float kj = (i == j) ? kv[j] : kv[j] * __expf(Lc[i] - Lc[j]);
                                vals[u] = qv[i] * kj;
                                vals[16 + u] = (i == j) ? 0.f : kv[i] * kj;
                            } else {
                                vals[u] = 0.f;
                                vals[16 + u] = 0.f;
                            }
                        }
                        dst[bt * 4 * 32] = warp_reduce_scatter32(vals, lane);
                    }
                }
            }
        }
        // the previous record's A-tile store has read the (Gamma K)^T region, rewritten in step 2
        if (tid == TID_ST && stores_out) { tc::bulk_wait_read(); stores_out = false; }
        __syncthreads();   // raw q/k/z are dead from here on

        // ---- 2. Gram sub-blocks on the tensor cores.  Block (a, b), b <= a, of A_qk and A_kk is
        //         sum_d q~_i k_j c_ab[d] / k~_i k_j c_ab[d] with k_j = k exp(G_end(b) - G_j) and
        //         c_ab = exp(G_start(a) - G_end(b)) (<= 1 for b < a; 1/tau_a < e^80 for b = a: the
        //         dense diagonal sub-blocks of the bounded gate).  Key version a holds the keys of
        //         sub-chunks 0..a times c_ab; one MMA, [Q~ ; K~] (128 rows) x versions (160 rows),
        //         leaves every block in TMEM, and each row reads the version of its own sub-chunk.
        {
            const int d = tid & (D - 1), b = tid >> 7;
            // channel d's sub-chunk decays tau_m: es = prod_{m < b}, ec = prod_{m > b},
            // gamma_C = prod_m, c_ab = prod_{b < m < a} (1 / tau_b for a = b)
            float tau[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) tau[m] = s_tau[m * D + d];
            float es = 1.f, ec = 1.f;
#pragma unroll
            for (int m = 0; m < 4; ++m)
                if (m < b) es *= tau[m];
#pragma unroll
            for (int m = 3; m >= 0; --m)
                if (m > b) ec *= tau[m];
            s_expS[b * D + d] = es;   // for the -Gamma Q accumulator
            if (b == 0) s_gam[d] = ((tau[0] * tau[1]) * tau[2]) * tau[3];
#pragma unroll
            for (int av = 0; av < 4; ++av) {
                if (av < b) continue;
                // the softplus gate's diagonal blocks come pair by pair (their factor can overflow)
                float cf = 1.f;
                if (av == b) cf = GATE ? 0.f : __fdividef(1.f, tau[b]);
                else {
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (m > b && m < av) cf *= tau[m];
                }
                const int r0 = kv_row0(av) + 16 * b;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    *reinterpret_cast<float*>(sKV + tc::sw128_offset(r0 + i, d, KV_ROWS)) = tc::to_tf32(kf2[i] * cf);
            }
            // the record's (K gamma_C / Gamma)^T: row d, the 16 tokens of sub-chunk b
            float k16[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) k16[u] = kf2[u] * ec;
            st_stream_h16(w.kt + rec * KT_ELEMS + (size_t)d * C + 16 * b, k16);
            // (Gamma K)^T, MMA 1's second B operand: row d, the 16 tokens of sub-chunk b
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const int t = 16 * b + i;
                float4 w4;
                w4.x = tc::to_tf32(qk_at(C + t, d) * es);
                w4.y = tc::to_tf32(qk_at(C + t + 1, d) * es);
                w4.z = tc::to_tf32(qk_at(C + t + 2, d) * es);
                w4.w = tc::to_tf32(qk_at(C + t + 3, d) * es);
                *reinterpret_cast<float4*>(sGK + tc::sw128_offset(d, t, D)) = w4;
            }
            tc::fence_proxy_async();
        }
        __syncthreads();
        if (tid == 0 && !timed_out) {
            ++n_mma;
            tc::fence_after_sync();
            const uint32_t ab = tc::smem_u32(sQK), bb = tc::smem_u32(sKV);
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks)
                tc::mma_tf32_ss(T0 + TM_G, tc::sw128_desc_k(ab, 2 * C, ks), tc::sw128_desc_k(bb, KV_ROWS, ks),
                                tc::idesc_tf32(2 * C, KV_ROWS), ks > 0);
            tc::mma_commit(mbar);
        }
        // while the Gram runs: D[:, 128:256] <- [0 ; -Gamma Q], onto which MMA 1 adds
        // [T beta ; P beta] . Gamma K (the output rows then hold minus the A tile's rows)
        {
            float v[16];
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                if (row >= C) {
                    const int t = row - C;
                    const float* es = s_expS + (t >> 4) * D;
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const int d = 32 * grp + c + j;
                        const float4 q4 = *reinterpret_cast<const float4*>(&qk_at(t, d));
                        const float4 e4 = *reinterpret_cast<const float4*>(es + d);
                        v[j] = -(q4.x * e4.x);
                        v[j + 1] = -(q4.y * e4.y);
                        v[j + 2] = -(q4.z * e4.z);
                        v[j + 3] = -(q4.w * e4.w);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                }
                tc::tmem_st16(T0 + TM_D + lane_base + D + 32 * grp + c, v);
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
        }
        wait(mbar, ph_mma);
        ph_mma ^= 1u;
        tc::fence_after_sync();
        {
            // row `row` of the result: A_qk row t (row < 64) or A_kk row t (row >= 64), t = row & 63,
            // of sub-chunk av; its blocks (av, 0..av) are version av's columns.  Quarters 0, 2 of the
            // lanes (sub-chunks 0, 1) need columns 0..47, quarters 1, 3 (sub-chunks 2, 3) 48..159:
            // the four warps of a quarter take the 16-column groups in turn.
            const int t = row & (C - 1), av = t >> 4;
            const bool kkrow = row >= C;
            float* Out = kkrow ? sAkk : sAqk;
            const float bt = kkrow ? s_beta[t] : 0.f;
            const int g_lo = (quad & 1) ? 3 : 0, g_hi = (quad & 1) ? 10 : 3;
            for (int g = g_lo + grp; g < g_hi; g += 4) {
                float v[16];
                tc::tmem_ld16(T0 + TM_G + lane_base + 16 * g, v);
                tc::tmem_ld_wait();
                const int gv = g >= 6 ? 3 : g >= 3 ? 2 : g >= 1 ? 1 : 0;   // version of the group
                const int j0 = 16 * g - kv_row0(av);                          // key index of column 0
                // this row's version only; the softplus gate's diagonal comes pair by pair
                if (gv == av && !(GATE && j0 == 16 * av)) {
#pragma unroll
                    for (int u = 0; u < 16; u += 4) {
                        float4 o4;
                        float* op = &o4.x;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int J = j0 + u + e;
                            op[e] = kkrow ? ((J < t) ? v[u + e] * bt : 0.f) : ((J <= t) ? v[u + e] : 0.f);
                        }
                        *reinterpret_cast<float4*>(Out + t * AS + j0 + u) = o4;
                    }
                }
                __syncwarp();   // the next group's TMEM load is warp-collective
            }
            if (GATE) {   // diagonal blocks from the pair-by-pair sums: 2 x 4 blocks of 16 x 16
#pragma unroll 1
                for (int x = tid; x < 2 * 4 * 256; x += NTP) {
                    const int kkb = x >> 10, bb = (x >> 8) & 3, i = (x >> 4) & 15, j = x & 15;
                    float val = 0.f;
                    if (j <= i && (j < i || !kkb)) {
                        const int p = i * (i + 1) / 2 + j, btc = p >> 4, slot = (p & 15) + 16 * kkb;
                        const float* src = s_diag + ((bb * 9 + btc) * 4) * 32 + slot;
                        val = (src[0] + src[32]) + (src[64] + src[96]);
                        if (kkb) val *= s_beta[16 * bb + i];
                    }
                    (kkb ? sAkk : sAqk)[(16 * bb + i) * AS + 16 * bb + j] = val;
                }
            }
        }
        __syncthreads();

        // ---- 3. blockwise UT solve: T = (I + A_kk)^{-1}, P = A_qk T (16x16 blocks)
        {
            float* sT = sAkk + C * AS;
            float* sW = sT + C * AS;
            const int g = lane >> 2, t4 = lane & 3;
            float* wsc = sW + warp * 16 * 16;
            auto blk = [&](float* M, int a_, int b_) { return M + (16 * a_) * AS + 16 * b_; };
            const int mi = lane >> 3, mr = lane & 7;   // ldmatrix: this lane's matrix and row
            auto mma16 = [&](float (&acc)[2][4], const float* X, const float* Y, int ly) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int k0 = 8 * ks + t4, k1 = k0 + 4;
                    uint32_t ra4[4];   // X rows (0..7 | 8..15), columns 8 ks + (0..3 | 4..7); X has row stride AS
                    ldsm_x4(X + (mr + 8 * (mi & 1)) * AS + 8 * ks + 4 * (mi >> 1), ra4);
                    const float af[4] = {tc::to_tf32(__uint_as_float(ra4[0])), tc::to_tf32(__uint_as_float(ra4[1])),
                                         tc::to_tf32(__uint_as_float(ra4[2])), tc::to_tf32(__uint_as_float(ra4[3]))};
#pragma unroll
                    for (int nh = 0; nh < 2; ++nh) {
                        const int nn = 8 * nh + g;
                        const float bfr[2] = {tc::to_tf32(Y[k0 * ly + nn]), tc::to_tf32(Y[k1 * ly + nn])};
                        tc::mma_m16n8k8_tf32(acc[nh], af, bfr);
                    }
                }
            };
            auto zero = [&](float (&acc)[2][4]) {
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) acc[nh][q4] = 0.f;
            };
            auto store = [&](const float (&acc)[2][4], float* Y, int ly, float sgn) {
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        Y[(g + (q4 >= 2 ? 8 : 0)) * ly + 8 * nh + 2 * t4 + (q4 & 1)] = sgn * acc[nh][q4];
            };
            auto t_block = [&](int a_, int b_) {
                float acc[2][4];
                zero(acc);
#pragma unroll 1
                for (int c_ = b_; c_ < a_; ++c_) mma16(acc, blk(sAkk, a_, c_), blk(sT, c_, b_), AS);
                store(acc, wsc, 16, 1.f);
                __syncwarp();
                float acc2[2][4];
                zero(acc2);
                mma16(acc2, blk(sT, a_, a_), wsc, 16);
                store(acc2, blk(sT, a_, b_), AS, -1.f);
                __syncwarp();
            };
            if (tid < C) {
                const int aa = tid >> 4, i = tid & 15;
                const float* Ad = blk(sAkk, aa, aa);
                float x[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) x[j] = (j == i) ? 1.f : 0.f;
#pragma unroll
                for (int kk = 15; kk >= 1; --kk) {
                    const float xk = x[kk];
#pragma unroll
                    for (int j = 0; j < kk; ++j) x[j] = fmaf(-xk, Ad[kk * AS + j], x[j]);
                }
                float* Td = blk(sT, aa, aa) + i * AS;
#pragma unroll
                for (int j = 0; j < 16; ++j) Td[j] = x[j];
            }
            __syncthreads();
            // Off-diagonal blocks by doubling on the 32 x 32 halves: T10 and T32 first,
            // then Y = A[2:4, 0:2] T[0:2, 0:2] (kept in T's unused upper blocks: Y_ab at
            // T's block (b, a)), then T[2:4, 0:2] = -T[2:4, 2:4] Y.  P = A_qk T: each of
            // warps 6..15 owns one P block, accumulated as its T blocks appear and stored
            // over A_qk's once every A_qk block has been read.  Four levels, the longest
            // two products deep.
            float acc[2][4];
            zero(acc);
            switch (warp) {   // level 1: T's diagonal blocks are in
                case 0: t_block(1, 0); break;                                                   // T10
                case 1: t_block(3, 2); break;                                                   // T32
                case 2: mma16(acc, blk(sAkk, 2, 1), blk(sT, 1, 1), AS); store(acc, blk(sT, 1, 2), AS, 1.f); break;  // Y21
                case 3: mma16(acc, blk(sAkk, 3, 1), blk(sT, 1, 1), AS); store(acc, blk(sT, 1, 3), AS, 1.f); break;  // Y31
                case 4: mma16(acc, blk(sAkk, 2, 0), blk(sT, 0, 0), AS); break;                  // Y20 (part)
                case 5: mma16(acc, blk(sAkk, 3, 0), blk(sT, 0, 0), AS); break;                  // Y30 (part)
                case 6: mma16(acc, blk(sAqk, 0, 0), blk(sT, 0, 0), AS); break;                  // P00
                case 7: mma16(acc, blk(sAqk, 1, 1), blk(sT, 1, 1), AS); break;                  // P11
                case 8: mma16(acc, blk(sAqk, 2, 2), blk(sT, 2, 2), AS); break;                  // P22
                case 9: mma16(acc, blk(sAqk, 3, 3), blk(sT, 3, 3), AS); break;                  // P33
                case 10: mma16(acc, blk(sAqk, 1, 0), blk(sT, 0, 0), AS); break;                 // P10 (part)
                case 11: mma16(acc, blk(sAqk, 2, 1), blk(sT, 1, 1), AS); break;                 // P21 (part)
                case 12: mma16(acc, blk(sAqk, 3, 2), blk(sT, 2, 2), AS); break;                 // P32 (part)
                case 13: mma16(acc, blk(sAqk, 2, 0), blk(sT, 0, 0), AS); break;                 // P20 (part)
                case 14: mma16(acc, blk(sAqk, 3, 1), blk(sT, 1, 1), AS); break;                 // P31 (part)
                default: mma16(acc, blk(sAqk, 3, 0), blk(sT, 0, 0), AS); break;                 // P30 (part)
            }
            __syncthreads();
            switch (warp) {   // level 2: T10, T32 are in
                case 4: mma16(acc, blk(sAkk, 2, 1), blk(sT, 1, 0), AS); store(acc, blk(sT, 0, 2), AS, 1.f); break;  // Y20
                case 5: mma16(acc, blk(sAkk, 3, 1), blk(sT, 1, 0), AS); store(acc, blk(sT, 0, 3), AS, 1.f); break;  // Y30
                case 10: mma16(acc, blk(sAqk, 1, 1), blk(sT, 1, 0), AS); break;                 // P10
                case 12: mma16(acc, blk(sAqk, 3, 3), blk(sT, 3, 2), AS); break;                 // P32
                case 13: mma16(acc, blk(sAqk, 2, 1), blk(sT, 1, 0), AS); break;                 // P20 (part)
                case 15: mma16(acc, blk(sAqk, 3, 1), blk(sT, 1, 0), AS); break;                 // P30 (part)
                default: break;
            }
            __syncthreads();
            if (warp < 4) {   // level 3: T[2:4, 0:2] = -T[2:4, 2:4] Y
                const int a_ = 2 + (warp >> 1), b_ = warp & 1;
                float tt[2][4];
                zero(tt);
                mma16(tt, blk(sT, a_, 2), blk(sT, b_, 2), AS);
                if (a_ == 3) mma16(tt, blk(sT, 3, 3), blk(sT, b_, 3), AS);
                store(tt, blk(sT, a_, b_), AS, -1.f);
            }
            __syncthreads();
            switch (warp) {   // level 4: T20, T21, T30, T31 are in
                case 11: mma16(acc, blk(sAqk, 2, 2), blk(sT, 2, 1), AS); break;                 // P21
                case 13: mma16(acc, blk(sAqk, 2, 2), blk(sT, 2, 0), AS); break;                 // P20
                case 14: mma16(acc, blk(sAqk, 3, 2), blk(sT, 2, 1), AS);
                         mma16(acc, blk(sAqk, 3, 3), blk(sT, 3, 1), AS); break;                 // P31
                case 15: mma16(acc, blk(sAqk, 3, 2), blk(sT, 2, 0), AS);
                         mma16(acc, blk(sAqk, 3, 3), blk(sT, 3, 0), AS); break;                 // P30
                default: break;
            }
            __syncthreads();
            if (warp >= 6) {
                // warp -> its P block: 6..9 the diagonal ones, then 10 (1,0), 11 (2,1),
                // 12 (3,2), 13 (2,0), 14 (3,1), 15 (3,0)
                constexpr unsigned long long PA = 0x3323213210ull, PB = 0x0102103210ull;   // 4 bits a warp
                const int k4 = 4 * (warp - 6);
                store(acc, blk(sAqk, (int)((PA >> k4) & 15u), (int)((PB >> k4) & 15u)), AS, 1.f);
            }
            __syncthreads();
            // rows of [T ; P] scaled by beta on the columns -> TMEM operand A2
            const int i = row & 63;
            const float* src = (row < C ? sT : sAqk) + i * AS;
            float v[16];
            {
                const int c = 16 * grp;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = c + j;
                    v[j] = (col <= i) ? tc::to_tf32(src[col] * s_beta[col]) : 0.f;
                }
                tc::tmem_st16(T0 + TM_A2 + lane_base + c, v);
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
        }
        __syncthreads();   // the Gram tiles are dead from here on
        // region RB is free: fetch the next record's q, k, z into it; MMA 1's Gamma K
        // half (its operands are all in) runs while V^T is built
        bool gk_issued = false;   // thread 0
        if (tid == 0 && !timed_out) {
            if (has_next) {
                ++n_in;
                tc::fence_proxy_async();
                load_qkz(nxt);
            }
            tc::fence_after_sync();
            const uint32_t bk = tc::smem_u32(sGK);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks)
                tc::mma_tf32_ts(T0 + TM_D + D, T0 + TM_A2 + 8 * ks, tc::sw128_desc_k(bk, D, ks),
                                tc::idesc_tf32(128, D), 1u);
            gk_issued = true;
        }
        wait(bar_v, ph_v);
        ph_v ^= 1u;

        // ---- 4. V^T (B_pre's first half, in region QK: the Gram has read it) and the
        //         record's gamma_C (thread: value column e, a quarter of the tokens)
        {
            const int e = tid & (D - 1), th = tid >> 7;
            float vm = 0.f;   // max |v| of this column over the quarter's tokens
#pragma unroll
            for (int t = 16 * th; t < 16 * th + 16; t += 4) {
                float4 w4;
                float* wp = &w4.x;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    wp[u] = (t + u < nc) ? raw_v(t + u, e) : 0.f;
                    vm = fmaxf(vm, fabsf(wp[u]));
                }
                *reinterpret_cast<float4*>(sBpre + tc::sw128_offset(e, t, D)) = w4;
            }
            // the sequence's column maximum, for the scan's operand scaling
            // (non-negative floats order like their bit patterns)
            if (vm > 0.f) atomicMax(w.vmax + ((size_t)cur.n * H + h) * D + e, __float_as_int(vm));
            if (th == 0) w.gm[rec * GM_FLOATS + e] = s_gam[e];
            tc::tmem_st_wait();
            tc::fence_proxy_async();
            tc::fence_before_sync();
        }
        __syncthreads();
        // the raw v tiles are consumed: fetch the next record's
        if (tid == 0 && has_next && !timed_out) {
            ++n_v;
            tc::fence_proxy_async();
            load_v(nxt);
        }

        // ---- 5. MMA 1: D[:, 0:128] = [T beta ; P beta] . V (the Gamma K half, D[:, 128:256]
        //         += [T beta ; P beta] . Gamma K, was issued after step 3); one commit for both
        if (tid == 0 && (gk_issued || !timed_out)) {
            if (!timed_out) {
                tc::fence_after_sync();
                const uint32_t bv = tc::smem_u32(sBpre);
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_tf32_ts(T0 + TM_D, T0 + TM_A2 + 8 * ks, tc::sw128_desc_k(bv, D, ks),
                                    tc::idesc_tf32(128, D), ks > 0);
            }
            ++n_mma;
            tc::mma_commit(mbar);
        }
        wait(mbar, ph_mma);
        ph_mma ^= 1u;
        tc::fence_after_sync();

        // ---- 6. the record: [U ; U_o] (fp32) and [-W ; Gamma Q - P Gamma K] (fp16; TMEM
        //      holds its negative) into shared memory as SW128 tiles -- [U ; U_o] in region
        //      QK, the A tile in the (Gamma K)^T region, both free once MMA 1 has read them
        //      -- and out by TMA (row = lane, 32 columns).  Output row t of both is stored
        //      times 2^s_t, s_t >= 0, and rho_t = 2^-s_t goes with gamma_C: a row whose every
        //      decay factor is small would otherwise sit among the fp16 subnormals and keep
        //      only a few bits, and times a large state its product with S is not small.  A
        //      row whose largest entry is below 2^-7 is raised to [1/2, 1) (by at most 2^96,
        //      and U_o's row stays below 2^120); the others keep s_t = 0, rho_t = 1 (their
        //      entries below the fp16 normals are under 2^-7 of the row's largest).  The scan
        //      multiplies the row's sum back by rho_t.
        {
            float v[16];
            uint8_t* sU = sm + OFF_QK;
            uint8_t* sA = sGK;
            if (row >= C) {   // the row's largest |A| and |U_o|, this thread's 32 columns
                float ma = 0.f, mu = 0.f;
#pragma unroll
                for (int c = 0; c < 32; c += 16) {
                    tc::tmem_ld16(T0 + TM_D + lane_base + D + 32 * grp + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) ma = fmaxf(ma, fabsf(v[j]));
                    tc::tmem_ld16(T0 + TM_D + lane_base + 32 * grp + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) mu = fmaxf(mu, fabsf(v[j]));
                }
                s_rmax[grp * C + row - C] = ma;
                s_rmax[4 * C + grp * C + row - C] = mu;
            }
            __syncthreads();
            float up = 1.f;   // 2^s_t
            if (row >= C) {
                const int t = row - C;
                const float ma = fmaxf(fmaxf(s_rmax[t], s_rmax[C + t]), fmaxf(s_rmax[2 * C + t], s_rmax[3 * C + t]));
                const float* sm2 = s_rmax + 4 * C;
                const float mu = fmaxf(fmaxf(sm2[t], sm2[C + t]), fmaxf(sm2[2 * C + t], sm2[3 * C + t]));
                // m = f 2^e with f in [1/2, 1): e from the exponent bits (a subnormal ma
                // reads as e = -126, beyond the cap)
                const int eu = (mu > 0.f && mu <= 3.0e38f) ? (int)((__float_as_uint(mu) >> 23) & 0xffu) - 126 : 0;
                const int st = (ma > 0.f && ma < 0.0078125f)
                                   ? max(0, min(min(96, 126 - (int)((__float_as_uint(ma) >> 23) & 0xffu)), 120 - eu))
                                   : 0;
                up = __int_as_float((127 + st) << 23);
                if (grp == 0) w.gm[rec * GM_FLOATS + D + t] = __int_as_float((127 - st) << 23);
            }
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                tc::tmem_ld16(T0 + TM_D + lane_base + 32 * grp + c, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4*>(sU + tc::sw128_offset(row, 32 * grp + c + j, 128)) =
                        make_float4(v[j] * up, v[j + 1] * up, v[j + 2] * up, v[j + 3] * up);
            }
            const float nup = -up;
#pragma unroll
            for (int c = 0; c < 32; c += 16) {
                tc::tmem_ld16(T0 + TM_D + lane_base + D + 32 * grp + c, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; j += 8)
                    *reinterpret_cast<uint4*>(sA + tc::sw128_offset_h(row, 32 * grp + c + j, 128)) =
                        make_uint4(tc::pack_f16x2(v[j] * nup, v[j + 1] * nup), tc::pack_f16x2(v[j + 2] * nup, v[j + 3] * nup),
                                   tc::pack_f16x2(v[j + 4] * nup, v[j + 5] * nup), tc::pack_f16x2(v[j + 6] * nup, v[j + 7] * nup));
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
        }
        __syncthreads();
        if (tid == TID_ST && !timed_out) {
            uint8_t* sU = sm + OFF_QK;
            const int y = (int)(rec * 128);
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) tc::tma_store_2d(&tm_uu, 32 * sl, y, sU + sl * (128 * 128));
            tc::bulk_commit();
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) tc::tma_store_2d(&tm_aw, 64 * sl, y, sGK + sl * (128 * 128));
            tc::bulk_commit();
            stores_out = true;
        }
        if (tid == NTP - 1 && has_next) {   // advance the walk: this record <- the next, next <- one stride on
            s_loc[0] = s_loc[3]; s_loc[1] = s_loc[4]; s_loc[2] = s_loc[5]; s_loc[6] = s_loc[7];
            long g = *reinterpret_cast<const long*>(s_loc + 8) + step_g;
            int hh = s_loc[10] + step_h;
            if (hh >= H) { hh -= H; ++g; }
            if (rec + 2 * stride < w.nrec) {
                if (g >= s_loc[13]) {           // past this sequence: largest n with cb[n] <= g
                    int n = s_loc[11] + 1, hi = a.num_seqs;
                    while (hi - n > 1) { const int mid = (n + hi) >> 1; if (w.chunk_base[mid] <= g) n = mid; else hi = mid; }
                    s_loc[11] = n;
                    s_loc[12] = w.chunk_base[n]; s_loc[13] = w.chunk_base[n + 1];
                    s_loc[14] = a.cu_seqlens[n]; s_loc[15] = a.cu_seqlens[n + 1];
                }
                const int t0 = s_loc[14] + C * (int)(g - s_loc[12]);
                s_loc[3] = t0; s_loc[4] = min(C, s_loc[15] - t0); s_loc[5] = hh; s_loc[7] = s_loc[11];
            }
            *reinterpret_cast<long*>(s_loc + 8) = g;
            s_loc[10] = hh;
        }
        __syncthreads();
    }
    if (tid == TID_ST) tc::bulk_wait_all();   // every record store has landed before the CTA exits
    // give-up path: wait for the copies and the MMA thread 0 issued before any
    // of this CTA's shared memory or TMEM is released
    if (__syncthreads_or(timed_out) && tid == 0) {
        const bool drained = tc::drain_phase(bar_in, n_in) & tc::drain_phase(bar_v, n_v) &
                             tc::drain_phase(mbar, n_mma);
        atomicOr(w.err, drained ? tc::ERR_WAIT : tc::ERR_WAIT | tc::ERR_DRAIN);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(T0, TM_COLS);
}

// ---------------------------------------------------------------------------
// scan: the state recurrence over one sequence's records
// ---------------------------------------------------------------------------
// scan shared-memory / TMEM layout for a cluster of R CTAs per (sequence, head),
// each owning NE = 128 / R value columns.  Ten warps: 0..7 the epilogue
// (warp w reaches TMEM lanes 32 (w % 4) .. +31 and takes column half w / 4),
// 8 issues the MMAs and TMEM copies, 9 the TMA loads.
template <int R>
struct ScanCfg {
    static constexpr int NE = D / R;
    static constexpr int WARP_MMA = 8, WARP_LOAD = 9, NTS = 320;
    // MMA operands in fp16, SW128 K-major
    static constexpr int AW_TILE = 128 * 128 * 2;            // [128 rows][128 K]
    static constexpr int OFF_AW0 = 0;
    static constexpr int OFF_AW1 = AW_TILE;
    static constexpr int OFF_SOP = 2 * AW_TILE;              // S operand [e][d]
    static constexpr int OFF_VOP = OFF_SOP + NE * D * 2;     // V' operand [e][t]
    static constexpr int G_TILE = C * NE * 2;                // g_in tile, [C][NE] bf16
    static constexpr int OFF_G = OFF_VOP + NE * C * 2;       // two g_in tiles, one per chunk parity
    static constexpr int KT_BYTES = 128 * C * 2;             // (K gamma_C / Gamma)^T [128 rows][C]
    static constexpr int OFF_K0 = OFF_G + 2 * G_TILE;        // MMA 3's A operand, one buffer per chunk parity
    static constexpr int OFF_K1 = OFF_K0 + KT_BYTES;
    static constexpr int GFS = NE + 4;                       // row stride (floats) of a gate-factor tile
    static constexpr int GF_TILE = C * GFS * 4;              // w Sigmoid(g_in) of the output rows, [C][GFS] fp32
    static constexpr int OFF_GF0 = OFF_K1 + KT_BYTES;        // one tile per chunk parity
    static constexpr int OFF_GF1 = OFF_GF0 + GF_TILE;
    // [U ; U_o] rows of a chunk (the CTA's NE columns, SW128 fp32 [128 rows][NE]) and
    // [gamma_C ; rho] (192 floats) by TMA into a ring of NU buffers, loaded two chunks ahead
    static constexpr int NU = 3;
    static constexpr int U_TILE = 128 * NE * 4;
    static constexpr int U_BUF = U_TILE + (int)GM_FLOATS * 4;
    static constexpr int OFF_U = (OFF_GF1 + GF_TILE + 1023) / 1024 * 1024;
    static constexpr int OFF_SMALL = OFF_U + NU * ((U_BUF + 1023) / 1024 * 1024);
    // small region (floats): peers' row sums of squares [2 parity][R source][C], this
    // CTA's half-row sums [2 parity][2 half][C], RMSNorm weights of this CTA's columns
    // [NE], the columns' scale factors 2^-c and 2^c [NE each], the columns' largest
    // |S0| [NE] (ints), the state warps' largest |S| [8] (ints)
    static constexpr int SM_ROWSQ = 0, SM_ROWPART = 2 * R * C, SM_NORMW = SM_ROWPART + 4 * C;
    static constexpr int SM_VSC = SM_NORMW + NE, SM_VINV = SM_VSC + NE, SM_CMAX = SM_VINV + NE;
    static constexpr int SM_WMAX = SM_CMAX + NE;
    static constexpr int SM_FLOATS = SM_WMAX + 8;
    static constexpr int SMEM_BYTES = OFF_SMALL + SM_FLOATS * 4 + 256 + 1024;
    static constexpr uint32_t TM_D = 0;                      // 2 x NE cols: [U ; U_o] -> [V' ; O]
    static constexpr uint32_t TM_DS = 2 * NE;                // NE cols: state increment
    static constexpr uint32_t TM_S = TM_DS + NE;             // NE cols: FP32 state
    static constexpr uint32_t TM_COLS = (TM_S + NE) <= 128 ? 128 : 256;
    static_assert(OFF_SOP % 1024 == 0 && OFF_VOP % 1024 == 0 && OFF_G % 1024 == 0 && OFF_K0 % 1024 == 0,
                  "1024-B aligned operands");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(TM_S + NE <= TM_COLS, "TMEM budget");
};

// 4-byte store into a peer CTA's shared memory that completes 4 transaction bytes
// on the peer's mbarrier (no fence: the mbarrier phase carries the data)
TC_DEV void st_async_f32(uint32_t addr, float v, uint32_t mbar_addr) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 :: "r"(addr), "r"(__float_as_uint(v)), "r"(mbar_addr) : "memory");
}
TC_DEV void mbar_arrive_local(uint64_t* mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(tc::smem_u32(mbar)) : "memory");
}
TC_DEV bool mbar_try_wait_cluster(uint64_t* mbar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(tc::smem_u32(mbar)), "r"(parity) : "memory");
    return ok != 0;
}
// named barrier among `count` threads.  Every participant syncs (none only arrives):
// a producer that could pass the barrier without waiting might, when its own waits are
// skipped after a timeout, run a chunk ahead and add its arrivals to the wrong
// generation; syncing keeps all participants in lockstep in every case, and costs
// nothing here since the MMA-issuing warp is always waiting when the others arrive
TC_DEV void nbar_sync(int id, int count) { asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory"); }

// byte offset of bf16 element (row, col) in a g_in tile of NE columns: the 128-byte
// rows of NE = 64 come swizzled by TMA, narrower rows are plain
template <int NE>
TC_DEV uint32_t gtile_offset(int row, int col) {
    if constexpr (NE == 64) return sw128_bf16(row, col);
    else return (uint32_t)(row * NE * 2 + col * 2);
}

// Per chunk, the recurrence path is MMA 2 -> V' operand -> MMA 3 -> state update.
// Warp specialisation keeps everything else off it: warp 8 only issues the two
// MMAs, released by two named barriers (the V' operand of this chunk is written;
// the state operand of the next chunk is written); warp 9 only issues the TMA
// loads, each as soon as the buffer it refills is free; the epilogue warps never
// wait for the other warps except through those barriers.  Both MMAs read their
// A operand from shared memory, where TMA puts it, so the tensor pipe does
// nothing but the 24 MMA instructions of the chunk.  The chunk's output rows
// take no part in the path: the epilogue of chunk j only forms their sums of
// squares, and o, y of chunk j are written during chunk j+1's MMA 2 from the TMEM
// buffer that still holds them.  The R CTAs' row sums meet in each peer's shared
// memory through st.async on mbarriers.
// TRANS: a transition scan (v = 0, the KCP pairs' M): the state exponent x follows
// the state; otherwise x = 0
template <int R, bool TRANS>
__global__ void __cluster_dims__(R, 1, 1) __launch_bounds__(ScanCfg<R>::NTS, 1)
scan_kernel(kda_prefill_args a, Work w, const __grid_constant__ CUtensorMap tm_aw,
            const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_kt,
            const __grid_constant__ CUtensorMap tm_uu) {
    using Cfg = ScanCfg<R>;
    constexpr int NE = Cfg::NE;
    constexpr int HW = NE / 2;           // value columns per epilogue thread
    constexpr int NB_V = 1, NB_S = 2, NB_O = 3, NB_X = 4;   // named barriers
    constexpr int NV = 5 * 32;           // V' warps (0, 1, 4, 5) + the MMA warp
    constexpr int NS = 9 * 32;           // epilogue warps + the MMA warp
    constexpr int NO = 4 * 32;           // output-row warps (2, 3, 6, 7)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sSop = sm + Cfg::OFF_SOP;
    uint8_t* sVop = sm + Cfg::OFF_VOP;
    float* fs = reinterpret_cast<float*>(sm + Cfg::OFF_SMALL);
    float* s_rowsq = fs + Cfg::SM_ROWSQ;      // [2][R][C] peers' row sums, by parity and source
    float* s_rowpart = fs + Cfg::SM_ROWPART;  // [2][2][C] this CTA's, by parity and half
    float* s_normw = fs + Cfg::SM_NORMW;      // [NE] RMSNorm weights (ones without norm_w)
    // The fp16 operands S and V' have the tf32 mantissa but a narrower range.  The
    // recurrence is linear in (v, S0) column by column, so the scan carries column e of
    // S, V', U and U_o (in TMEM and in the operands) times 2^(x_j - c_e), and only the
    // boundary (S0, U in; o, S_T, snapshots out) rescales, by exact powers of two.
    // 2^c_e is the power of two just above the column's largest |v| (the state then
    // stays near 1), raised if needed to keep the largest |S0| below 2^12: content at
    // the scale of v keeps the full fp16 mantissa while |S0| / |v| < 2^26.  A column
    // with v = 0 takes 2^c_e from S0 alone.  In a transition scan (TRANS: v = 0, the
    // state only decays or mixes) x_j, one exponent for the CTA's columns, follows
    // the largest |S| chunk by chunk, so that the state's fp16 copy stays near 1
    // however fast it decays; otherwise x_j = 0.  An output row of the A tile whose
    // entries are all small comes raised by 1 / rho (prep's row scaling), so the row's
    // sum is multiplied by rho on the way out.  (Terms below 2^-24 of the record
    // operands' own scale -- a chunk's contraction terms under very fast decay --
    // are lost to fp16 whatever x: a transition matrix is exact to about 2^-24 of
    // |S0|, not relative to itself once it has decayed below that.)
    float* s_vsc = fs + Cfg::SM_VSC;          // [NE] 2^-c
    float* s_vinv = fs + Cfg::SM_VINV;        // [NE] 2^c
    int* s_cmax = reinterpret_cast<int*>(fs + Cfg::SM_CMAX);  // [NE] largest |S0|
    uint32_t* s_wmax = reinterpret_cast<uint32_t*>(fs + Cfg::SM_WMAX);  // [8] per state warp
    uint64_t* bars = reinterpret_cast<uint64_t*>(fs + Cfg::SM_FLOATS);
    uint64_t* bar_m2 = bars;             // MMA 2 of chunk j done (phase j)
    uint64_t* bar_m3 = bars + 1;         // MMA 3 of chunk j done (phase j)
    uint64_t* bar_aw = bars + 2;         // [2] A tile of chunk j landed in buffer j & 1

    uint64_t* bar_full = bars + 6;       // [2] peers' row sums of chunk j landed in s_rowsq[j & 1]
    uint64_t* bar_k = bars + 8;          // [2] (K gamma_C / Gamma)^T of chunk j landed in buffer j & 1
    uint64_t* bar_awfree = bar_k + 2;    // [2] MMA 2 has read A-tile buffer b (one phase per use)
    uint64_t* bar_kfree = bar_awfree + 2;   // [2] MMA 3 has read K buffer b (one phase per use)
    uint64_t* bar_g = bar_kfree + 2;     // [2] g_in tile of chunk j landed in buffer j & 1 (one phase per use)
    uint64_t* bar_gfree = bar_g + 2;     // [2] the V' warps have read g_in buffer b (one phase per use)
    uint64_t* bar_u = bar_gfree + 2;     // [NU] U rows and gamma_C of chunk j landed in buffer j % NU
    uint64_t* bar_ufree = bar_u + Cfg::NU;   // [NU] the state warps have read buffer k (one phase per use)
    uint32_t* tbase_ptr = reinterpret_cast<uint32_t*>(bar_ufree + Cfg::NU);

    const int r = blockIdx.x;            // value-column block == cluster rank
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const int H = a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp < 8;
    const int quad = warp & 3, hf = (warp >> 2) & 1;
    const int row = quad * 32 + lane;
    const int c_lo = hf * HW;
    const bool vrow = epi && quad < 2;   // V' rows (tokens) 0..63; else output rows 64..127
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int t_begin = a.cu_seqlens[n], t_end = a.cu_seqlens[n + 1];
    const int g0 = w.chunk_base[n];
    const int nch = w.chunk_base[n + 1] - g0;
    const bool gate = a.g_in != nullptr;
    const int din = a.dk;            // 128, or a float32 operator's d <= 64 (the rest is zero padding)
    auto rec_of = [&](int j) { return (long)(g0 + j) * H + h; };
    auto aw_buf = [&](int b) { return sm + (b ? Cfg::OFF_AW1 : Cfg::OFF_AW0); };
    auto k_buf = [&](int b) { return sm + (b ? Cfg::OFF_K1 : Cfg::OFF_K0); };
    auto g_buf = [&](int b) { return sm + Cfg::OFF_G + b * Cfg::G_TILE; };
    auto u_buf = [&](int k) { return sm + Cfg::OFF_U + k * ((Cfg::U_BUF + 1023) / 1024 * 1024); };
    auto gf_buf = [&](int b) { return reinterpret_cast<float*>(sm + (b ? Cfg::OFF_GF1 : Cfg::OFF_GF0)); };

    if (warp == 0) { tc::tmem_alloc(tbase_ptr, Cfg::TM_COLS); tc::tmem_relinquish(); }
    const int vmx = (tid < NE && !w.zero_v) ? w.vmax[((size_t)n * H + h) * D + NE * r + tid] : 0;
    if (tid < NE) {
        s_normw[tid] = a.norm_w ? a.norm_w[NE * r + tid] : 1.f;
        s_cmax[tid] = 0;
    }
    if (tid == 0) {
        tc::mbar_init(bar_m2, 1);
        for (int k = 0; k < Cfg::NU; ++k) {
            tc::mbar_init(bar_u + k, 1);
            tc::mbar_init(bar_ufree + k, 8);          // one arrival per epilogue warp
        }
        tc::mbar_init(bar_m3, 1);

        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(bar_aw + b, 1);
            tc::mbar_init(bar_full + b, 1);
            tc::mbar_init(bar_k + b, 1);
            tc::mbar_init(bar_awfree + b, 1);
            tc::mbar_init(bar_kfree + b, 1);
            tc::mbar_init(bar_g + b, 1);
            tc::mbar_init(bar_gfree + b, 4);          // one arrival per V' warp
        }
        tc::mbar_fence_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (a.S0) {   // the columns' largest |S0|
        for (int i = tid; i < din * NE; i += Cfg::NTS) {
            const int d = i / NE, c = i - d * NE;
            if (NE * r + c < din)
                atomicMax(s_cmax + c, __float_as_int(fabsf(a.S0[(((size_t)n * H + h) * din + d) * din + NE * r + c])));
        }
    }
    __syncthreads();
    if (tid < NE) {   // m = f 2^ex with f in [1/2, 1)
        const float ms = __int_as_float(s_cmax[tid]), mv = __int_as_float(vmx);
        const bool hs = ms > 0.f && ms <= 3.0e38f, hv = mv > 0.f && mv <= 3.0e38f;
        int es = 0, ev = 0;
        if (hs) frexpf(ms, &es);
        if (hv) frexpf(mv, &ev);
        int ex = hv ? (hs ? max(ev, es - 12) : ev) : es;
        ex = max(-120, min(120, ex));
        s_vsc[tid] = ldexpf(1.f, -ex);
        s_vinv[tid] = ldexpf(1.f, ex);
    }
    __syncthreads();
    const uint32_t T0 = *tbase_ptr;
    if (gate) cluster_sync_all();   // every peer's mbarriers are initialised before the first remote access

    // A wait on a local copy or MMA that gives up records it in timed_out: this
    // thread then skips every later such wait, and the issuing lanes (warp 8 and
    // warp 9, lane 0) issue no further copy or MMA, so the kernel runs to its end
    // (its results are invalid) and drains what was issued.  The named barriers
    // and the row-sum exchange with the peer CTAs keep running (their data are
    // then meaningless, their protocol intact), so that no warp or peer is left
    // waiting and nothing lands after a CTA has exited; a wait of the exchange
    // that gives up (a peer that stopped) sets xdead, after which this thread
    // stops exchanging.
    bool timed_out = false, xdead = false;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!timed_out && !tc::mbar_wait_bounded(bar, parity, w.wait_limit)) timed_out = true;
    };
    auto wait_cl = [&](uint64_t* bar, uint32_t parity) {
        for (uint32_t i = 0; !xdead && !mbar_try_wait_cluster(bar, parity); )
            if (++i == tc::WAIT_POLLS) xdead = true;
    };
    // phases each issuing lane armed or issued on each mbarrier, for the drain
    uint32_t n_aw[2] = {0, 0}, n_k[2] = {0, 0}, n_full[2] = {0, 0}, n_g[2] = {0, 0}, n_u[Cfg::NU] = {};
    uint32_t n_m2 = 0, n_m3 = 0, n_awf[2] = {0, 0}, n_kf[2] = {0, 0};

    if (warp == Cfg::WARP_LOAD) {
        // ------------------------------------------------------------------ TMA loads
        if (lane == 0) {
            tc::tma_prefetch_desc(&tm_aw);
            tc::tma_prefetch_desc(&tm_kt);
            tc::tma_prefetch_desc(&tm_uu);
            if (gate) tc::tma_prefetch_desc(&tm_g);
            auto load_aw = [&](int j) {
                const int b = j & 1;
                ++n_aw[b];
                tc::mbar_arrive_expect_tx(bar_aw + b, Cfg::AW_TILE);
                for (int s = 0; s < 2; ++s)   // two 64-column slabs
                    tc::tma_load_2d(aw_buf(b) + s * (Cfg::AW_TILE / 2), &tm_aw, 64 * s, (int)(rec_of(j) * 128), bar_aw + b);
            };
            auto load_g = [&](int j) {   // into buffer j & 1
                const int b = j & 1;
                ++n_g[b];
                tc::mbar_arrive_expect_tx(bar_g + b, Cfg::G_TILE);
                tc::tma_load_2d(g_buf(b), &tm_g, h * D + NE * r, t_begin + C * j, bar_g + b);
            };
            auto load_k = [&](int j) {   // chunk j's K^T: one 64-token slab
                const int b = j & 1;
                ++n_k[b];
                tc::mbar_arrive_expect_tx(bar_k + b, Cfg::KT_BYTES);
                tc::tma_load_2d(k_buf(b), &tm_kt, 0, (int)(rec_of(j) * 128), bar_k + b);
            };
            auto load_u = [&](int j) {   // chunk j's U rows (this CTA's columns) and gamma_C
                const int k = j % Cfg::NU;
                ++n_u[k];
                tc::mbar_arrive_expect_tx(bar_u + k, (w.zero_v ? 0 : Cfg::U_TILE) + (uint32_t)GM_FLOATS * 4);
                if (!w.zero_v) tc::tma_load_2d(u_buf(k), &tm_uu, NE * r, (int)(rec_of(j) * 128), bar_u + k);
                tc::bulk_load(u_buf(k) + Cfg::U_TILE, w.gm + rec_of(j) * GM_FLOATS, (uint32_t)GM_FLOATS * 4, bar_u + k);
            };
            for (int j = 0; j < Cfg::NU && j < nch; ++j) load_u(j);
            for (int j = 0; j < 2 && j < nch; ++j) { load_aw(j); load_k(j); }
            for (int j = 0; gate && j < 2 && j < nch; ++j) load_g(j);
            for (int j = 0; j < nch && !timed_out; ++j) {
                // buffers j & 1 of chunk j + 2 once MMA 2 / MMA 3 of chunk j have read them
                // (barriers of those buffers' own: their next phases need these very loads,
                // so they cannot run a phase ahead of the waits)
                if (j + 2 < nch) { wait(bar_awfree + (j & 1), (j >> 1) & 1); if (!timed_out) load_aw(j + 2); }
                if (j + 2 < nch) { wait(bar_kfree + (j & 1), (j >> 1) & 1); if (!timed_out) load_k(j + 2); }
                // the g_in tile of chunk j + 1 once the outputs of chunk j are written
                // the g_in tile of chunk j + 2 once the V' warps have read chunk j's
                if (gate && j + 2 < nch) { wait(bar_gfree + (j & 1), (j >> 1) & 1); if (!timed_out) load_g(j + 2); }
                // chunk j + NU's U rows once the state warps have read chunk j's (in chunk j - 1)
                if (j + Cfg::NU < nch) {
                    wait(bar_ufree + j % Cfg::NU, (j / Cfg::NU) & 1);
                    if (!timed_out) load_u(j + Cfg::NU);
                }
            }
        }
        __syncwarp();
    } else if (warp == Cfg::WARP_MMA) {
        // ------------------------------------------------------------------ MMA issue
#pragma unroll 1
        for (int j = 0; j < nch; ++j) {
            const int b = j & 1;
            nbar_sync(NB_S, NS);   // the state operand of chunk j is written
            if (lane == 0) {
                wait(bar_aw + b, (j >> 1) & 1);
                if (!timed_out) {   // MMA 2: [V' ; O] = [U ; U_o] + [-W ; Gamma Q - P Gamma K] . S
                    tc::fence_after_sync();
                    const uint32_t ab = tc::smem_u32(aw_buf(b));
                    const uint32_t sb = tc::smem_u32(sSop);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        tc::mma_f16_ss(T0 + Cfg::TM_D + NE * b, tc::sw128_desc_k(ab, 128, ks),
                                       tc::sw128_desc_k(sb, NE, ks), tc::idesc_f16(128, NE),
                                       (ks > 0 || !w.zero_v) ? 1u : 0u);
                    ++n_m2;
                    tc::mma_commit(bar_m2);
                    ++n_awf[b];
                    tc::mma_commit(bar_awfree + b);
                }
                wait(bar_k + b, (j >> 1) & 1);   // lands long before: loaded two chunks ahead
            }
            __syncwarp();
            nbar_sync(NB_V, NV);   // the V' operand of chunk j is written
            if (lane == 0 && !timed_out) {   // MMA 3: dS = (K gamma_C / Gamma)^T . V'
                tc::fence_after_sync();
                const uint32_t kb = tc::smem_u32(k_buf(b));
                const uint32_t vb = tc::smem_u32(sVop);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    tc::mma_f16_ss(T0 + Cfg::TM_DS, tc::sw128_desc_k(kb, 128, ks), tc::sw128_desc_k(vb, NE, ks),
                                   tc::idesc_f16(128, NE), ks > 0);
                ++n_m3;
                tc::mma_commit(bar_m3);
                ++n_kf[b];
                tc::mma_commit(bar_kfree + b);
            }
            __syncwarp();
        }
        nbar_sync(NB_S, NS);       // the epilogue's last arrival
    } else {
        // ------------------------------------------------------------------ epilogue
        // this thread's columns' scale factors 2^-c and 2^c, kept in registers
        float vsc_r[HW], vinv_r[HW];
#pragma unroll
        for (int c = 0; c < HW; ++c) { vsc_r[c] = s_vsc[c_lo + c]; vinv_r[c] = s_vinv[c_lo + c]; }
        // chunk j's record rows from U-ring buffer j % NU into TMEM buffer j & 1
        // ([U ; U_o] row `row`, this thread's HW columns, scaled by 2^-c); returns
        // gamma_C[row] of the chunk and, for an output row, rho (the power of two by
        // which the row's sum comes out too large)
        auto store_rec = [&](int j) -> float2 {
            const int k = j % Cfg::NU;
            wait(bar_u + k, (j / Cfg::NU) & 1);
            const uint8_t* ub = u_buf(k);
            const float* gr = reinterpret_cast<const float*>(ub + Cfg::U_TILE);
            const float rho = vrow ? 1.f : gr[D + row - C];
            if (!w.zero_v) {
#pragma unroll
                for (int i = 0; i < HW; i += 16) {
                    float v[16];
#pragma unroll
                    for (int q = 0; q < 16; q += 4) {
                        const float4 u4 = *reinterpret_cast<const float4*>(ub + sw128_f32(row, c_lo + i + q));
                        v[q] = u4.x * vsc_r[i + q];
                        v[q + 1] = u4.y * vsc_r[i + q + 1];
                        v[q + 2] = u4.z * vsc_r[i + q + 2];
                        v[q + 3] = u4.w * vsc_r[i + q + 3];
                    }
                    tc::tmem_st16(T0 + Cfg::TM_D + NE * (j & 1) + lane_base + c_lo + i, v);
                }
            }
            const float2 g = make_float2(gr[row], rho);
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar_ufree + k);
            return g;
        };
        // o and y of chunk jo from its TMEM buffer (output-row threads)
        auto emit_outputs = [&](int jo, int xo, float rho_o) {   // the chunk's exponent, the row's rho
            const int bo = jo & 1;
            const int t = row - C;
            const int c0o = t_begin + C * jo;
            const int nco = min(C, t_end - c0o);
            float o[HW];
#pragma unroll
            for (int c = 0; c < HW; c += 16) tc::tmem_ld16(T0 + Cfg::TM_D + NE * bo + lane_base + c_lo + c, o + c);
            tc::tmem_ld_wait();
            if (rho_o != 1.f) {
#pragma unroll
                for (int c = 0; c < HW; ++c) o[c] *= rho_o;
            }
#pragma unroll
            for (int c = 0; c < HW; ++c) o[c] *= a.scale * vinv_r[c] * exp2i(-xo);
            if (t < nco && a.o) {
                if (din == D) {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(a.o) + ((size_t)(c0o + t) * H + h) * D + NE * r + c_lo;
#pragma unroll
                    for (int c = 0; c < HW; c += 8) store8_bf16(dst + c, o + c);
                } else {       // float32 o of d_v = din < 128 columns
                    float* dst = reinterpret_cast<float*>(a.o) + ((size_t)(c0o + t) * H + h) * din;
#pragma unroll
                    for (int c = 0; c < HW; ++c)
                        if (NE * r + c_lo + c < din) dst[NE * r + c_lo + c] = o[c];
                }
            }
            if (gate) {
                wait_cl(bar_full + bo, (jo >> 1) & 1);
                if (t < nco) {
                    float tot = s_rowpart[(bo * 2) * C + t] + s_rowpart[(bo * 2 + 1) * C + t];
#pragma unroll
                    for (int p = 0; p < R; ++p)
                        if (p != r) tot += s_rowsq[(bo * R + p) * C + t];
                    const float rr = rsqrtf(tot * (1.0f / D) + a.norm_eps);
                    uint16_t* yp = reinterpret_cast<uint16_t*>(a.y) + ((size_t)(c0o + t) * H + h) * D + NE * r + c_lo;
                    const float* gf = gf_buf(bo) + t * Cfg::GFS + c_lo;   // w Sigmoid(g_in), by the V' warps
#pragma unroll
                    for (int c = 0; c < HW; c += 8) {
                        const float4 fa = reinterpret_cast<const float4*>(gf + c)[0];
                        const float4 fb = reinterpret_cast<const float4*>(gf + c)[1];
                        const float fv[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
                        float yv[8];
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) yv[jj] = o[c + jj] * rr * fv[jj];
                        store8_bf16(yp + c, yv);
                    }
                }
            }
        };

        // ---- initial state -> TMEM master copy and the fp16 operand copy
        float2 gm_next = make_float2(0.f, 1.f);   // gamma_C and rho of the next chunk, one chunk ahead
        float rho_prev = 1.f;                     // rho of the previous chunk
        int x_prev = 0, x_cur = 0, x_next = 0;   // the exponent x of the previous, this, the next chunk
        {
            const int d = row;
            const size_t sb = (((size_t)n * H + h) * din + d) * din + NE * r;
            float v[16];
#pragma unroll
            for (int c = c_lo; c < c_lo + HW; c += 16) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    v[jj] = (a.S0 && d < din && NE * r + c + jj < din) ? a.S0[sb + c + jj] * s_vsc[c + jj] : 0.f;
                tc::tmem_st16(T0 + Cfg::TM_S + lane_base + c, v);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    *reinterpret_cast<uint16_t*>(sSop + tc::sw128_offset_h(c + jj, d, NE)) = tc::f32_to_f16(v[jj]);
            }
            if (nch > 0) gm_next = store_rec(0);
            tc::tmem_st_wait();
            tc::fence_proxy_async();
            tc::fence_before_sync();
        }
        nbar_sync(NB_S, NS);

#pragma unroll 1
        for (int j = 0; j < nch; ++j) {
            const int b = j & 1;
            const int c0 = t_begin + C * j;
            const int nc = min(C, t_end - c0);
            const float gm = gm_next.x, rho = gm_next.y;

            // ---- while MMA 2 runs: outputs of the previous chunk (their buffer is
            //      refilled next), the next record into the other TMEM buffer, the one
            //      after it into registers
            if (!vrow) {
                if (j > 0 && (a.o || gate)) emit_outputs(j - 1, x_prev, rho_prev);
                // arm this chunk's exchange barrier (its phase for chunk j - 2 completed:
                // this thread waited for it in emit_outputs; a peer that stopped leaves
                // it open, and then it is not armed again)
                if (gate && warp == 2 && lane == 0 && !xdead) {
                    if (j >= 2 && !tc::mbar_try_wait(bar_full + b, ((j - 2) >> 1) & 1)) xdead = true;
                    else { ++n_full[b]; tc::mbar_arrive_expect_tx(bar_full + b, (R - 1) * C * 4); }
                }
            }
            if (j + 1 < nch) gm_next = store_rec(j + 1);
            // (the U rows' TMEM stores complete before this chunk's state barrier, where
            // the state update waits for all of this thread's TMEM stores)
            wait(bar_m2, j & 1);
            tc::fence_after_sync();

            // ---- V' -> MMA 3 operand (smem); output rows: half-row sums of squares
            if (vrow) {
                const int t = row;
                float v[16];
#pragma unroll
                for (int c = c_lo; c < c_lo + HW; c += 16) {
                    tc::tmem_ld16(T0 + Cfg::TM_D + NE * b + lane_base + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        *reinterpret_cast<uint16_t*>(sVop + tc::sw128_offset_h(c + jj, t, NE)) = tc::f32_to_f16(v[jj]);
                }
                tc::fence_proxy_async();
                tc::fence_before_sync();
                nbar_sync(NB_V, NV);
            } else if (gate) {
                const int t = row - C;
                float v[16], ss = 0.f;
#pragma unroll
                for (int c = c_lo; c < c_lo + HW; c += 16) {
                    tc::tmem_ld16(T0 + Cfg::TM_D + NE * b + lane_base + c, v);
                    tc::tmem_ld_wait();
                    if (rho != 1.f) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) v[jj] *= rho;
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float x = v[jj] * (vinv_r[c - c_lo + jj] * exp2i(-x_cur));
                        ss = fmaf(x, x, ss);
                    }
                }
                ss *= a.scale * a.scale;
                s_rowpart[(b * 2 + hf) * C + t] = ss;
                nbar_sync(NB_O, NO);   // both halves of this chunk's sums are in s_rowpart
                // the row's sum over this CTA's columns into every peer's s_rowsq[b], by the
                // first half's thread.  What this CTA wrote there for chunk j - 2 has been
                // read: every peer read it (emit_outputs of chunk j - 2, both halves, then
                // the peer's NB_O) before it sent its sums of chunk j - 1, whose arrival
                // this thread awaited in emit_outputs of chunk j - 1; the st.async
                // complete-tx releases at cluster scope and that wait acquires at cluster
                // scope, so each peer's reads happen before these writes.
                if (hf == 0) {
                    const float own = ss + s_rowpart[(b * 2 + 1) * C + t];
                    if (!xdead) {
#pragma unroll
                        for (int p = 1; p < R; ++p)
                            st_async_f32(cluster_map(s_rowsq + (b * R + r) * C + t, (r + p) % R), own,
                                         cluster_map(bar_full + b, (r + p) % R));
                    }
                }
            }

            // ---- S = Diag(gamma_C) S + dS (FP32 in TMEM), refresh the fp16 operand copy
            //      (in a transition scan first moved to the next chunk's exponent); a
            //      chunk that closes a prefix-cache interval also writes S out
            wait(bar_m3, j & 1);
            tc::fence_after_sync();
            {
                const int d = row;
                float* snap = nullptr;
                if (a.S_snap && (c0 + nc - t_begin) % a.snap_interval == 0) {
                    const long srow = snapshot_row_base(a.cu_seqlens, n, a.snap_interval) +
                                      (c0 + nc - t_begin) / a.snap_interval - 1;
                    snap = a.S_snap + ((srow * H + h) * din + d) * din + NE * r;
                }
                static_assert(HW == 16, "one 16-column group per state thread");
                float dv[16], sv[16];
                const int c = c_lo;
                tc::tmem_ld16(T0 + Cfg::TM_DS + lane_base + c, dv);
                tc::tmem_ld16(T0 + Cfg::TM_S + lane_base + c, sv);
                tc::tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) sv[jj] = fmaf(gm, sv[jj], dv[jj]);
                x_next = x_cur;
                if (TRANS) {
                    // the largest |S| over the CTA's state warps (non-negative floats
                    // order like their bit patterns) brings x back to [1/2, 1) when it
                    // left [2^-6, 2^6)
                    float mx = 0.f;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) mx = fmaxf(mx, fabsf(sv[jj]));
                    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
                    if (lane == 0) s_wmax[warp] = wm;
                    nbar_sync(NB_X, 8 * 32);
                    uint32_t m8 = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) m8 = max(m8, s_wmax[k]);
                    const float m = __uint_as_float(m8);
                    if (m > 0.f && m <= 3.0e38f) {
                        int ex;
                        frexpf(m, &ex);
                        if (ex < -5 || ex > 6) x_next = max(-100, min(100, x_cur - max(-60, min(60, ex))));
                    }
                    const float px = exp2i(x_next - x_cur);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) sv[jj] *= px;
                }
                const float pu = exp2i(-x_next);
                {
                    tc::tmem_st16(T0 + Cfg::TM_S + lane_base + c, sv);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        *reinterpret_cast<uint16_t*>(sSop + tc::sw128_offset_h(c + jj, d, NE)) = tc::f32_to_f16(sv[jj]);
                    if (snap) {
                        float su[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) su[jj] = sv[jj] * (s_vinv[c + jj] * pu);
                        if (din == D) {
#pragma unroll
                            for (int jj = 0; jj < 16; jj += 4)
                                *reinterpret_cast<float4*>(snap + c + jj) = make_float4(su[jj], su[jj + 1], su[jj + 2], su[jj + 3]);
                        } else if (d < din) {
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                if (NE * r + c + jj < din) snap[c + jj] = su[jj];
                        }
                    }
                }
                tc::tmem_st_wait();
                tc::fence_proxy_async();
                tc::fence_before_sync();
            }
            // ---- V' rows, off the recurrence path: w Sigmoid(g_in) of output row t =
            //      row of this chunk (this thread's columns), read by the output thread
            //      of the same row and columns in the next chunk
            if (gate && vrow) {
                wait(bar_g + b, (j >> 1) & 1);
                const int t = row;
                const uint8_t* sg = g_buf(b);
                float* gf = gf_buf(b) + t * Cfg::GFS + c_lo;
#pragma unroll
                for (int c = 0; c < HW; c += 8) {
                    const uint4 g8 = *reinterpret_cast<const uint4*>(sg + gtile_offset<NE>(t, c_lo + c));
                    const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w};
                    float fv[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const float gv = __uint_as_float((jj & 1) ? (gw[jj >> 1] & 0xffff0000u) : (gw[jj >> 1] << 16));
                        fv[jj] = __fdividef(s_normw[c_lo + c + jj], 1.0f + __expf(-gv));
                    }
                    reinterpret_cast<float4*>(gf + c)[0] = make_float4(fv[0], fv[1], fv[2], fv[3]);
                    reinterpret_cast<float4*>(gf + c)[1] = make_float4(fv[4], fv[5], fv[6], fv[7]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_local(bar_gfree + b);
            }
            nbar_sync(NB_S, NS);
            x_prev = x_cur;
            x_cur = x_next;
            rho_prev = rho;
        }
        // outputs of the last chunk
        if (nch > 0 && !vrow && (a.o || gate)) emit_outputs(nch - 1, x_prev, rho_prev);

        // ---- final state
        if (a.S_T) {
            const int d = row;
            float* dst = a.S_T + (((size_t)n * H + h) * din + d) * din + NE * r;
            float v[16];
#pragma unroll
            for (int c = c_lo; c < c_lo + HW; c += 16) {
                tc::tmem_ld16(T0 + Cfg::TM_S + lane_base + c, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) v[jj] *= s_vinv[c + jj] * exp2i(-x_cur);
                if (din == D) {
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 4)
                        *reinterpret_cast<float4*>(dst + c + jj) = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
                } else if (d < din) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        if (NE * r + c + jj < din) dst[c + jj] = v[jj];
                }
            }
        }
    }

    // give-up path: each issuing lane waits for the copies and tensor-core work it
    // issued, and the lane that armed the exchange barriers for the peers' sums,
    // before any of this CTA's shared memory or TMEM is released
    if (__syncthreads_or(timed_out || xdead)) {
        bool drained = true;
        if (warp == Cfg::WARP_MMA && lane == 0)
            drained = tc::drain_phase(bar_m2, n_m2) & tc::drain_phase(bar_m3, n_m3) &
                      tc::drain_phase(bar_awfree, n_awf[0]) & tc::drain_phase(bar_awfree + 1, n_awf[1]) &
                      tc::drain_phase(bar_kfree, n_kf[0]) & tc::drain_phase(bar_kfree + 1, n_kf[1]);
        if (warp == Cfg::WARP_LOAD && lane == 0) {
            drained = tc::drain_phase(bar_g, n_g[0]) & tc::drain_phase(bar_g + 1, n_g[1]);
            for (int k = 0; k < Cfg::NU; ++k) drained = drained & tc::drain_phase(bar_u + k, n_u[k]);
#pragma unroll
            for (int b = 0; b < 2; ++b)
                drained = drained & tc::drain_phase(bar_aw + b, n_aw[b]) & tc::drain_phase(bar_k + b, n_k[b]);
        }
        if (warp == 2 && lane == 0)
            drained = tc::drain_phase(bar_full, n_full[0]) & tc::drain_phase(bar_full + 1, n_full[1]);
        if ((warp == Cfg::WARP_MMA || warp == Cfg::WARP_LOAD || warp == 2) && lane == 0)
            atomicOr(w.err, drained ? tc::ERR_WAIT : tc::ERR_WAIT | tc::ERR_DRAIN);
    }
    tc::fence_before_sync();
    __syncthreads();
    cluster_sync_all();   // no CTA leaves while a peer may still write to its shared memory
    if (warp == 0) tc::tmem_dealloc(T0, Cfg::TM_COLS);
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static long total_chunks(const kda_prefill_args& a) {
    long c = 0;
    for (int n = 0; n < a.num_seqs; ++n) c += (a.cu_seqlens_host[n + 1] - a.cu_seqlens_host[n] + C - 1) / C;
    return c;
}

// workspace: error word at 0, chunk offsets at 256, the value-column maxima,
// then the record arrays from the first 1024-byte aligned address after them
// (the size allows for the slack)
struct Layout { size_t base, vmax, rec_start, aw, uu, kt, gm, total; long nrec, nvmax; };
static Layout layout(const kda_prefill_args& a) {
    Layout l;
    l.nrec = total_chunks(a) * a.H;
    l.nvmax = (long)a.num_seqs * a.H * D;
    l.base = 256;
    l.vmax = align_up(l.base + 4 * (size_t)(a.num_seqs + 1), 16);
    l.rec_start = l.vmax + 4 * (size_t)l.nvmax;
    l.aw = 0;                                               // relative to the aligned record start
    l.uu = l.aw + (size_t)l.nrec * AW_ELEMS * 2;
    l.kt = l.uu + (size_t)l.nrec * UU_FLOATS * 4;
    l.gm = l.kt + (size_t)l.nrec * KT_ELEMS * 2;
    l.total = l.rec_start + 1024 + l.gm + (size_t)l.nrec * GM_FLOATS * 4;
    return l;
}

static int sm_count() {
    static int count[256] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!count[dev]) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
    return count[dev];
}

}  // namespace spl

size_t prefill_split_workspace_size(const kda_prefill_args& a) { return spl::layout(a).total; }

// bf16 q/k/v with d = 128, or float32 q/k/v with d = 32 or 64 (zero-padded to 128)
bool prefill_split_supported(const kda_prefill_args& a) {
    if (a.dk != a.dv) return false;
    if (a.qkv_dtype == KDA_BF16) return a.dk == spl::D;
    return a.qkv_dtype == KDA_F32 && (a.dk == 32 || a.dk == spl::prep::DIN_MAX);
}

// parts: bit 0 = plan + prep (the records), bit 1 = scan; scan_flags: KDA_SCAN_*
cudaError_t launch_prefill_split_parts(const kda_prefill_args& a, int parts, int scan_flags, cudaStream_t s) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        auto set = [](const void* f, int bytes) {
            return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        };
        attr_err = set((const void*)spl::prep_kernel<0, 0>, spl::prep::SMEM_BYTES);
        if (attr_err == cudaSuccess) attr_err = set((const void*)spl::prep_kernel<1, 0>, spl::prep::SMEM_BYTES);
        if (attr_err == cudaSuccess) attr_err = set((const void*)spl::prep_kernel<0, 1>, spl::prep::SMEM_BYTES);
        if (attr_err == cudaSuccess) attr_err = set((const void*)spl::prep_kernel<1, 1>, spl::prep::SMEM_BYTES);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(spl::scan_kernel<spl::SCAN_R, false>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, spl::ScanCfg<spl::SCAN_R>::SMEM_BYTES);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(spl::scan_kernel<spl::SCAN_R, true>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, spl::ScanCfg<spl::SCAN_R>::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (a.num_seqs == 0) return cudaSuccess;
    const spl::Layout L = spl::layout(a);
    uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
    spl::Work w;
    w.err = reinterpret_cast<int*>(ws);
    w.chunk_base = reinterpret_cast<const int*>(ws + L.base);
    uint8_t* recs = reinterpret_cast<uint8_t*>(spl::align_up(reinterpret_cast<uintptr_t>(ws) + L.rec_start, 1024));
    w.vmax = reinterpret_cast<int*>(ws + L.vmax);
    w.aw = reinterpret_cast<uint16_t*>(recs + L.aw);
    w.uu = reinterpret_cast<float*>(recs + L.uu);
    w.kt = reinterpret_cast<uint16_t*>(recs + L.kt);
    w.gm = reinterpret_cast<float*>(recs + L.gm);
    w.nrec = L.nrec;
    w.zero_v = (scan_flags & KDA_SCAN_ZERO_V) ? 1 : 0;
    w.wait_limit = wait_limit();

    const bool f32 = a.qkv_dtype == KDA_F32;
    const uint32_t din = (uint32_t)a.dk;
    const uint64_t rowq = (uint64_t)a.H * din;
    const uint64_t rows = (uint64_t)a.T_total;
    CUtensorMap mq, mk, mz, mv, mg, maw;
    cudaError_t e;
    const CUtensorMapDataType tq = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const size_t eq = f32 ? 4 : 2;
    if ((e = make_map(&mq, tq, eq, a.q, rowq, rows, din, spl::C, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
    if ((e = make_map(&mk, tq, eq, a.k, rowq, rows, din, spl::C, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
    if ((e = make_map(&mz, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.z, rowq, rows, din, spl::C,
                      CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
    if ((e = make_map(&mv, tq, eq, a.v, rowq, rows, f32 ? din : 64, spl::C,
                      f32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
    constexpr int NE = spl::ScanCfg<spl::SCAN_R>::NE;
    if ((e = make_map(&mg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.g_in ? a.g_in : a.v, rowq, rows, NE, spl::C,
                      NE == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
    if ((e = make_map(&maw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.aw, 128, (uint64_t)L.nrec * 128, 64, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
    CUtensorMap mkt, muu;
    if ((e = make_map(&muu, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, w.uu, 128, (uint64_t)L.nrec * 128, NE, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
    if ((e = make_map(&mkt, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.kt, spl::C, (uint64_t)L.nrec * 128, 64, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;

    int launched = 0;
    if (parts & 1) {
        spl::plan_kernel<<<1, 1024, 0, s>>>(a.cu_seqlens, a.num_seqs, const_cast<int*>(w.chunk_base), w.vmax,
                                             L.nvmax, w.err);
        ++launched;
        if (L.nrec > 0) {
            const int nsm = spl::sm_count();
            const long grid = L.nrec < (long)(nsm > 0 ? nsm : 148) ? L.nrec : (long)(nsm > 0 ? nsm : 148);
            const bool sp = a.gate_mode == KDA_GATE_SOFTPLUS, f32 = a.qkv_dtype == KDA_F32;
            auto kern = sp ? (f32 ? spl::prep_kernel<1, 1> : spl::prep_kernel<1, 0>)
                           : (f32 ? spl::prep_kernel<0, 1> : spl::prep_kernel<0, 0>);
            kern<<<(unsigned)grid, spl::prep::NTP, spl::prep::SMEM_BYTES, s>>>(a, w, mq, mk, mz, mv, muu, maw);
            ++launched;
        }
    }
    if (parts & 2) {
        dim3 grid(spl::SCAN_R, a.H, a.num_seqs);
        auto kern = w.zero_v ? spl::scan_kernel<spl::SCAN_R, true> : spl::scan_kernel<spl::SCAN_R, false>;
        kern<<<grid, spl::ScanCfg<spl::SCAN_R>::NTS, spl::ScanCfg<spl::SCAN_R>::SMEM_BYTES, s>>>(a, w, maw, mg, mkt,
                                                                                                   muu);
        ++launched;
    }
    count_launches(launched);
    return cudaGetLastError();
}

cudaError_t launch_prefill_split(const kda_prefill_args& a, cudaStream_t s) {
    return launch_prefill_split_parts(a, 3, 0, s);
}

}  // namespace kda
