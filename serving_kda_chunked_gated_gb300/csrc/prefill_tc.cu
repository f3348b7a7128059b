// Chunked KDA prefill on the sm_103a tensor cores.
//
// Operator: "Kimi K3: KDA, attention residuals and Stable LatentMoE"
// (hs-black.github.io) Sec. 2.1 chunked form
//     O = (Gamma (.) Q) S + Tril[(Q (.) Gamma)(K / Gamma)^T] (U - W S),
// with the Sec. 2.2 bounded gate and 16-token sub-chunks (every Gamma-ratio
// formed inside one sub-chunk stays below e^80), and the Sec. 2.3 output gate.
//
// Per chunk of C = 64 tokens with entry state S (dk x dv), Gamma_t the
// cumulative retention inside the chunk, beta the write strengths:
//   A_kk = StrictTril(Diag(beta)(Gamma K)(K/Gamma)^T),  A_qk = Tril((Gamma Q)(K/Gamma)^T)
//   T = (I + A_kk)^{-1},  P = A_qk T Diag(beta)
//   [U | W ; U_o | P Gamma K] = [T Diag(beta) ; P] . [V | Gamma K]          (MMA 1)
//   [V' ; O] = [U ; U_o] + [-W ; Gamma Q - P Gamma K] . S                   (MMA 2)
//   S_next = Diag(gamma_C) S + (K (.) gamma_C / Gamma)^T V'                 (MMA 3)
// (O = (Gamma Q) S + A_qk V' rearranged so that one MMA yields V' and O.)
//
// Work decomposition: a cluster of two CTAs (8 warps each) per (sequence,
// head); CTA r owns value columns [64r, 64r+64).  Both CTAs compute the
// d_k-wide chunk terms; the only exchange is the per-row sum of squares for
// the RMSNorm of the fused output gate (over distributed shared memory).
//
// Data movement: each chunk's q, k, z tiles (64 x 128) and this CTA's v and
// g_in tiles (64 x 64) arrive by TMA bulk tensor copies into shared memory,
// issued one chunk ahead (q/k/z as soon as the previous chunk's first MMA has
// consumed their buffer, v/g_in after the previous chunk's epilogue), so the
// CUDA-core prologue reads shared memory only.
//
// Precision: every contraction runs as tcgen05 kind::tf32 (the 16x16 Gram
// sub-blocks as mma.sync tf32) with FP32 accumulation; operands are rounded to
// tf32 (nearest) when staged; the gate, cumulative decays, the triangular
// solve and the state carry stay FP32 (the state lives in TMEM in FP32 across
// chunks and is only rounded for its copy used as an MMA operand).
#include <mutex>

#include "kda_common.cuh"
#include "tcgen05.cuh"
#include "tma_host.cuh"

namespace kda {
namespace tcp {

constexpr int C = 64;     // chunk length
constexpr int D = 128;    // dk = dv
constexpr int NE = 64;    // value columns per CTA
constexpr int NT = 256;   // threads per CTA (8 warps; warps w and w+4 share TMEM lanes)
constexpr int QS = 132;   // padded row stride (floats) of the scaled q/k tiles
constexpr int AS = 68;    // padded row stride (floats) of the 64x64 Gram tiles
constexpr int NPAIR = 10; // sub-block pairs (a >= b) of a chunk

// shared memory map (offsets from a 1024-aligned base)
constexpr int SOP_BYTES = NE * D * 4;                 // S operand, SW128 [e][d]            32 KB
constexpr int RB_BYTES = 65536;                       // raw q,k,z | Gram tiles | [V|GK]^T  64 KB
constexpr int TILE_BYTES = C * QS * 4;                // one scaled q/k tile                33 KB
constexpr int VG_BYTES = 2 * C * NE * 2;              // raw v, g_in halves (bf16, swizzled) 16 KB
constexpr int OFF_SOP = 0;
constexpr int OFF_RB = OFF_SOP + SOP_BYTES;
constexpr int OFF_RAWQ = OFF_RB;                      // [C][D] bf16
constexpr int OFF_RAWK = OFF_RB + C * D * 2;          // [C][D] bf16
constexpr int OFF_RAWZ = OFF_RB + 2 * C * D * 2;      // [C][D] f32
constexpr int OFF_AQK = OFF_RB;                       // Gram tiles
constexpr int OFF_AKK = OFF_RB + C * AS * 4;
constexpr int OFF_BPRE = OFF_RB;                      // [V | Gamma K]^T, SW128 [n][t]
constexpr int OFF_QH = OFF_RB + RB_BYTES;             // q * exp(G - G_subchunk_start)
constexpr int OFF_KR = OFF_QH + TILE_BYTES;           // k * exp(G - G_subchunk_start)
constexpr int OFF_KH = OFF_KR + TILE_BYTES;           // k * exp(G_subchunk_end - G)
constexpr int OFF_VOP = OFF_KR;                       // V' operand [e][t] (aliases KR)
constexpr int OFF_RAWV = OFF_KH + TILE_BYTES;         // [C][NE] bf16, 128-B swizzle
constexpr int OFF_RAWG = OFF_RAWV + C * NE * 2;       // [C][NE] bf16, 128-B swizzle
constexpr int OFF_SMALL = OFF_RAWV + VG_BYTES;
// small region (floats)
constexpr int SM_BETA = 0, SM_RQ = 64, SM_RK = 128, SM_TAU = 192, SM_EXPS = SM_TAU + 4 * D,
              SM_EXPCE = SM_EXPS + 4 * D, SM_GAM = SM_EXPCE + 4 * D, SM_ROWSQ = SM_GAM + D,
              SM_ROWPART = SM_ROWSQ + 2 * C, SM_CTAB = SM_ROWPART + 2 * C, SM_FLOATS = SM_CTAB + NPAIR * D;
constexpr int SMEM_BYTES = OFF_SMALL + SM_FLOATS * 4 + 64 /*mbarriers, tmem base*/ + 1024 /*align*/;
static_assert(OFF_VOP % 1024 == 0 && OFF_BPRE % 1024 == 0, "SW128 operands need 1024-B alignment");
static_assert(OFF_RAWV % 1024 == 0 && OFF_RAWG % 1024 == 0, "128-B swizzled TMA tiles need 1024-B alignment");
static_assert(2 * C * AS * 4 <= RB_BYTES && (NE + D) * C * 4 <= RB_BYTES && 2 * C * D * 2 + C * D * 4 <= RB_BYTES,
              "region RB holds the raw tiles, the Gram tiles and [V|GK]^T in turn");
static_assert(3 * C * AS * 4 + (NT / 32) * 16 * 16 * 4 <= RB_BYTES,
              "region RB holds A_qk, A_kk, T and the per-warp solve scratch");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t BYTES_QKZ = 2 * C * D * 2 + C * D * 4;   // one chunk of q, k, z
constexpr uint32_t BYTES_V = C * NE * 2;                    // one chunk of the v (or g_in) half

// TMEM columns
constexpr uint32_t TM_D = 0;      // 192 cols: [U;U_o] -> [V';O] (0..63), [W;P Gamma K] -> A1 (64..191)
constexpr uint32_t TM_A2 = 192;   // 64 cols: [T beta ; P]
constexpr uint32_t TM_A3 = 256;   // 64 cols: (K gamma_C / Gamma)^T
constexpr uint32_t TM_DS = 320;   // 64 cols: state increment
constexpr uint32_t TM_S = 384;    // 64 cols: FP32 state (master copy)
constexpr uint32_t TM_COLS = 512;

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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NT, 1)
prefill_tc_kernel(kda_prefill_args a, int* err, uint32_t wait_limit,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sSop = sm + OFF_SOP;
    uint8_t* sBpre = sm + OFF_BPRE;
    uint8_t* sVop = sm + OFF_VOP;
    const uint16_t* sRawQ = reinterpret_cast<const uint16_t*>(sm + OFF_RAWQ);
    const uint16_t* sRawK = reinterpret_cast<const uint16_t*>(sm + OFF_RAWK);
    const float* sRawZ = reinterpret_cast<const float*>(sm + OFF_RAWZ);
    const uint8_t* sRawV = sm + OFF_RAWV;
    const uint8_t* sRawG = sm + OFF_RAWG;
    float* sQ = reinterpret_cast<float*>(sm + OFF_QH);
    float* sKr = reinterpret_cast<float*>(sm + OFF_KR);
    float* sK = reinterpret_cast<float*>(sm + OFF_KH);
    float* sAqk = reinterpret_cast<float*>(sm + OFF_AQK);
    float* sAkk = reinterpret_cast<float*>(sm + OFF_AKK);
    float* fs = reinterpret_cast<float*>(sm + OFF_SMALL);
    float* s_beta = fs + SM_BETA;
    float* s_rq = fs + SM_RQ;
    float* s_rk = fs + SM_RK;
    float* s_tau = fs + SM_TAU;      // [4][D] retention product of each sub-chunk
    float* s_expS = fs + SM_EXPS;    // [4][D] exp(G at sub-chunk start)
    float* s_expCE = fs + SM_EXPCE;  // [4][D] exp(G_C - G at sub-chunk end)
    float* s_gam = fs + SM_GAM;      // [D]    exp(G_C)
    float* s_rowsq = fs + SM_ROWSQ;  // [2][C] peer's row sums of squares (by chunk parity)
    float* s_rowpart = fs + SM_ROWPART;  // [2][C] this CTA's row sums of squares, per column half
    float* s_ctab = fs + SM_CTAB;    // [NPAIR][D] exp(G_start(a) - G_end(b)), b < a; 1/tau_a for b = a
    uint64_t* mbar = reinterpret_cast<uint64_t*>(fs + SM_FLOATS);
    uint64_t* bar_in = mbar + 1;
    uint64_t* bar_vg = mbar + 2;
    uint32_t* tbase_ptr = reinterpret_cast<uint32_t*>(mbar + 3);

    const int r = blockIdx.x;          // value half == cluster rank
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const int H = a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // TMEM access: warp w reaches lanes 32*(w%4)..+31; warps w and w+4 split the columns
    const int quad = warp & 3, hf = warp >> 2;
    const int row = quad * 32 + lane;  // TMEM lane == operand row owned by this thread
    const int t_begin = a.cu_seqlens[n], t_end = a.cu_seqlens[n + 1];
    const float eA = __expf(a.A[h]);
    const bool gate = a.g_in != nullptr;
    const uint32_t bytes_vg = gate ? 2 * BYTES_V : BYTES_V;

    if (warp == 0) { tc::tmem_alloc(tbase_ptr, TM_COLS); tc::tmem_relinquish(); }
    // thread 0 issues every copy and MMA; it counts the phases it issued on each
    // mbarrier, for the give-up path at the end
    uint32_t n_in = 0, n_vg = 0, n_mma = 0;
    if (tid == 0) {
        tc::mbar_init(mbar, 1);
        tc::mbar_init(bar_in, 1);
        tc::mbar_init(bar_vg, 1);
        tc::mbar_fence_init();
        tc::tma_prefetch_desc(&tm_q);
        tc::tma_prefetch_desc(&tm_k);
        tc::tma_prefetch_desc(&tm_z);
        tc::tma_prefetch_desc(&tm_v);
        if (gate) tc::tma_prefetch_desc(&tm_g);
        if (t_begin < t_end) {
            tc::mbar_arrive_expect_tx(bar_in, BYTES_QKZ);
            tc::tma_load_2d(sm + OFF_RAWQ, &tm_q, h * D, t_begin, bar_in);
            tc::tma_load_2d(sm + OFF_RAWK, &tm_k, h * D, t_begin, bar_in);
            tc::tma_load_2d(sm + OFF_RAWZ, &tm_z, h * D, t_begin, bar_in);
            tc::mbar_arrive_expect_tx(bar_vg, bytes_vg);
            tc::tma_load_2d(sm + OFF_RAWV, &tm_v, h * D + NE * r, t_begin, bar_vg);
            if (gate) tc::tma_load_2d(sm + OFF_RAWG, &tm_g, h * D + NE * r, t_begin, bar_vg);
            n_in = n_vg = 1;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t T0 = *tbase_ptr;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int c_lo = hf * (NE / 2);    // this thread's half of a 64-column TMEM region
    uint32_t ph_mma = 0, ph_in = 0, ph_vg = 0;
    // A wait that gives up records it; this thread then skips every later wait,
    // and thread 0 issues no further copy or MMA, so the kernel runs to its end
    // (its results are invalid) and drains what was issued.  The cluster
    // barriers are unconditional, so the peer CTA is never left waiting.
    bool timed_out = false;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!timed_out && !tc::mbar_wait_bounded(bar, parity, wait_limit)) timed_out = true;
    };
    auto mma_wait = [&]() {
        wait(mbar, ph_mma);
        ph_mma ^= 1u;
        tc::fence_after_sync();
    };
    // write strengths of the next chunk, prefetched into a register one chunk ahead
    float beta_next = 0.f;
    if (tid < C && t_begin + tid < t_end) beta_next = a.beta[(size_t)(t_begin + tid) * H + h];

    // ---- initial state -> TMEM master copy and the tf32 operand copy (row d, 32 columns)
    {
        const int d = row;
        const size_t sb = (((size_t)n * H + h) * D + d) * D + NE * r;
        float v[16];
#pragma unroll
        for (int c = c_lo; c < c_lo + NE / 2; c += 16) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = a.S0 ? a.S0[sb + c + j] : 0.f;
            tc::tmem_st16(T0 + TM_S + lane_base + c, v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                *reinterpret_cast<float*>(sSop + tc::sw128_offset(c + j, d, NE)) = tc::to_tf32(v[j]);
        }
        tc::tmem_st_wait();
        tc::fence_proxy_async();
    }
    tc::fence_before_sync();
    __syncthreads();

    for (int c0 = t_begin; c0 < t_end; c0 += C) {
        const int nc = min(C, t_end - c0);
        const int par = ((c0 - t_begin) / C) & 1;
        const bool has_next = c0 + C < t_end;

        if (tid < C) {
            s_beta[tid] = beta_next;
            beta_next = (c0 + C + tid < t_end) ? a.beta[(size_t)(c0 + C + tid) * H + h] : 0.f;
        }
        wait(bar_in, ph_in);
        ph_in ^= 1u;

        // ---- 1a. q/k L2 norms (warp w: tokens 8w..8w+7) from the staged tiles
#pragma unroll 4
        for (int i = 0; i < 8; ++i) {
            const int t = warp * 8 + i;
            float sq = 0.f, sk = 0.f;
            if (t < nc) {
                const uint2 qa = *reinterpret_cast<const uint2*>(sRawQ + t * D + 4 * lane);
                const uint2 ka = *reinterpret_cast<const uint2*>(sRawK + t * D + 4 * lane);
                const float q0 = __uint_as_float(qa.x << 16), q1 = __uint_as_float(qa.x & 0xffff0000u),
                            q2 = __uint_as_float(qa.y << 16), q3 = __uint_as_float(qa.y & 0xffff0000u);
                const float k0 = __uint_as_float(ka.x << 16), k1 = __uint_as_float(ka.x & 0xffff0000u),
                            k2 = __uint_as_float(ka.y << 16), k3 = __uint_as_float(ka.y & 0xffff0000u);
                sq = q0 * q0 + q1 * q1 + q2 * q2 + q3 * q3;
                sk = k0 * k0 + k1 * k1 + k2 * k2 + k3 * k3;
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            if (lane == 0) {
                s_rq[t] = a.qk_l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
                s_rk[t] = a.qk_l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
            }
        }
        __syncthreads();

        // ---- 1b. gate and sub-chunk-relative decay factors: thread (channel d, half hf)
        //          handles sub-chunks 2hf and 2hf+1 (the decay products restart at each
        //          sub-chunk, so the halves are independent)
        {
            const int d = tid & (D - 1);
#pragma unroll 1
            for (int b = 2 * (tid >> 7); b < 2 * (tid >> 7) + 2; ++b) {
                float al[16], kv[16];
                float F1 = 1.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int t = 16 * b + i;
                    float alpha = 1.f, q = 0.f, k = 0.f;
                    if (t < nc) {
                        alpha = __expf(log_decay(sRawZ[t * D + d], eA, a.g_min));
                        q = bf16_to_f(sRawQ[t * D + d]) * s_rq[t];
                        k = bf16_to_f(sRawK[t * D + d]) * s_rk[t];
                    }
                    F1 *= alpha;                   // exp(G_t - G_start(b))
                    al[i] = alpha;
                    kv[i] = k;
                    sQ[t * QS + d] = q * F1;
                    sKr[t * QS + d] = k * F1;
                }
                float F2 = 1.f;                    // exp(G_end(b) - G_t)
#pragma unroll
                for (int i = 15; i >= 0; --i) {
                    sK[(16 * b + i) * QS + d] = kv[i] * F2;
                    F2 *= al[i];
                }
                s_tau[b * D + d] = F1;
            }
        }
        __syncthreads();   // the raw q/k/z tiles are dead from here on
        if (tid < D) {     // per-channel constants of the chunk (thread = channel d)
            const int d = tid;
            float tau[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) tau[b] = s_tau[b * D + d];
            float pre = 1.f;
#pragma unroll
            for (int b = 0; b < 4; ++b) { s_expS[b * D + d] = pre; pre *= tau[b]; }
            s_gam[d] = pre;
            float suf = 1.f;
#pragma unroll
            for (int b = 3; b >= 0; --b) { s_expCE[b * D + d] = suf; suf *= tau[b]; }
            // factor joining the row reference (start of sub-chunk a) and the key
            // reference (end of sub-chunk b): exp(G_start(a) - G_end(b))
#pragma unroll
            for (int aa = 0; aa < 4; ++aa) {
#pragma unroll
                for (int bb = 0; bb <= aa; ++bb) {
                    float cf = 1.f;
                    if (aa == bb) cf = __fdividef(1.f, tau[aa]);
                    else {
#pragma unroll
                        for (int m = bb + 1; m < aa; ++m) cf *= tau[m];
                    }
                    s_ctab[(aa * (aa + 1) / 2 + bb) * D + d] = cf;
                }
            }
        }
        // cluster-wide: the peer writes its Gram blocks into region RB only after both
        // CTAs have consumed their raw q/k/z tiles there
        cluster_sync_all();

        // ---- 2. Gram sub-blocks with mma.sync (tf32), split over the cluster: CTA 0
        //         forms A_qk, CTA 1 forms A_kk (10 blocks of 16x16 each; warp w owns pairs
        //         w and w+8) and writes every block to its own and to its peer's tile.
        {
            const int g = lane >> 2, t4 = lane & 3;
            const bool kk_pass = r == 1;
            const float* Arows = kk_pass ? sKr : sQ;
            float* Out = kk_pass ? sAkk : sAqk;
            const uint32_t out_peer = cluster_map(Out, r ^ 1);
            const int n_it = warp < NPAIR - 8 ? 2 : 1;
            float acc[2][2][4];
#pragma unroll
            for (int it = 0; it < 2; ++it)
#pragma unroll
                for (int nh = 0; nh < 2; ++nh)
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) acc[it][nh][q4] = 0.f;
            int ia[2], ib[2];
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int pr = warp + 8 * it;                 // pair index a(a+1)/2 + b
                const int aa = pr >= 6 ? 3 : pr >= 3 ? 2 : pr >= 1 ? 1 : 0;
                ia[it] = aa;
                ib[it] = pr - aa * (aa + 1) / 2;
            }
#pragma unroll 2
            for (int ks = 0; ks < 16; ++ks) {
                const int k0 = 8 * ks + t4, k1 = k0 + 4;
#pragma unroll
                for (int it = 0; it < 2; ++it) {
                    if (it < n_it) {
                        const int ra = 16 * ia[it] + g;
                        const float af[4] = {tc::to_tf32(Arows[ra * QS + k0]), tc::to_tf32(Arows[(ra + 8) * QS + k0]),
                                             tc::to_tf32(Arows[ra * QS + k1]), tc::to_tf32(Arows[(ra + 8) * QS + k1])};
                        const float* ct = s_ctab + (ia[it] * (ia[it] + 1) / 2 + ib[it]) * D;
                        const float c0f = ct[k0], c1f = ct[k1];
#pragma unroll
                        for (int nh = 0; nh < 2; ++nh) {
                            const int j = 16 * ib[it] + 8 * nh + g;
                            const float bfr[2] = {tc::to_tf32(sK[j * QS + k0] * c0f), tc::to_tf32(sK[j * QS + k1] * c1f)};
                            tc::mma_m16n8k8_tf32(acc[it][nh], af, bfr);
                        }
                    }
                }
            }
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                if (it < n_it) {
#pragma unroll
                    for (int nh = 0; nh < 2; ++nh) {
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int I = 16 * ia[it] + g + 8 * hr;
                            const int J = 16 * ib[it] + 8 * nh + 2 * t4;
                            float v0 = acc[it][nh][2 * hr], v1 = acc[it][nh][2 * hr + 1];
                            if (!kk_pass) { if (J > I) v0 = 0.f; if (J + 1 > I) v1 = 0.f; }
                            else {
                                const float bI = s_beta[I];
                                v0 = (J >= I) ? 0.f : v0 * bI;
                                v1 = (J + 1 >= I) ? 0.f : v1 * bI;
                            }
                            const int off = I * AS + J;
                            *reinterpret_cast<float2*>(Out + off) = make_float2(v0, v1);
                            asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};"
                                         :: "r"(out_peer + 4u * (uint32_t)off), "f"(v0), "f"(v1) : "memory");
                        }
                    }
                }
            }
        }
        cluster_sync_all();   // both halves of the Gram are in both CTAs

        // ---- 3. UT solve, blockwise on 16x16 sub-blocks:
        //         T = (I + A_kk)^{-1}:  T_aa = (I + A_aa)^{-1} (FP32 substitution),
        //                               T_ab = -T_aa sum_{c=b}^{a-1} A_ac T_cb  (a > b)
        //         P = A_qk T:           P_ab = sum_{c=b}^{a} Aqk_ac T_cb
        //         The block products run as mma.sync tf32 in five dependency phases.
        {
            float* sT = sAkk + C * AS;                 // T tile (region RB, after the Gram tiles)
            float* sW = sT + C * AS;                   // per-warp 16x16 scratch for chained products
            const int g = lane >> 2, t4 = lane & 3;
            float* wsc = sW + warp * 16 * 16;
            auto blk = [&](float* M, int a_, int b_) { return M + (16 * a_) * AS + 16 * b_; };
            // acc += X(16x16, ld AS) * Y(16x16, ld ly)
            auto mma16 = [&](float (&acc)[2][4], const float* X, const float* Y, int ly) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int k0 = 8 * ks + t4, k1 = k0 + 4;
                    const float af[4] = {tc::to_tf32(X[g * AS + k0]), tc::to_tf32(X[(g + 8) * AS + k0]),
                                         tc::to_tf32(X[g * AS + k1]), tc::to_tf32(X[(g + 8) * AS + k1])};
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
            // T_ab = -T_aa * (sum_{c=b}^{a-1} A_ac T_cb)
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
            // P_ab = sum_{c=b}^{a} Aqk_ac T_cb, kept in registers until every read of Aqk is done
            auto p_block = [&](float (&acc)[2][4], int a_, int b_) {
                zero(acc);
#pragma unroll 1
                for (int c_ = b_; c_ <= a_; ++c_) mma16(acc, blk(sAqk, a_, c_), blk(sT, c_, b_), AS);
            };

            // phase A: diagonal inverses, thread (a, i) -> row i of (I + A_aa)^{-1}
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
            // P blocks held in registers until every read of A_qk is done:
            //   warp 2: P21   warp 3: P00 P32   warp 4: P11 P20   warp 5: P22 P31
            //   warp 6: P33 P30   warp 7: P10
            float pA[2][4], pB[2][4];
            // phase B: T10 T21 T32 (warps 0-2), P00 P11 P22 P33 (warps 3-6)
            if (warp < 3) t_block(warp + 1, warp);
            else if (warp < 7) p_block(pA, warp - 3, warp - 3);
            __syncthreads();
            // phase C: T20 T31 (warps 0-1), P21 (warp 2), P32 (warp 3), P10 (warp 7)
            if (warp < 2) t_block(warp + 2, warp);
            else if (warp == 2) p_block(pA, 2, 1);
            else if (warp == 3) p_block(pB, 3, 2);
            else if (warp == 7) p_block(pA, 1, 0);
            __syncthreads();
            // phase D: T30 (warp 0), P20 (warp 4), P31 (warp 5)
            if (warp == 0) t_block(3, 0);
            else if (warp == 4) p_block(pB, 2, 0);
            else if (warp == 5) p_block(pB, 3, 1);
            __syncthreads();
            // phase E: P30 (warp 6)
            if (warp == 6) p_block(pB, 3, 0);
            __syncthreads();   // every read of A_qk is done: overwrite it with P
            switch (warp) {
                case 2: store(pA, blk(sAqk, 2, 1), AS, 1.f); break;
                case 3: store(pA, blk(sAqk, 0, 0), AS, 1.f); store(pB, blk(sAqk, 3, 2), AS, 1.f); break;
                case 4: store(pA, blk(sAqk, 1, 1), AS, 1.f); store(pB, blk(sAqk, 2, 0), AS, 1.f); break;
                case 5: store(pA, blk(sAqk, 2, 2), AS, 1.f); store(pB, blk(sAqk, 3, 1), AS, 1.f); break;
                case 6: store(pA, blk(sAqk, 3, 3), AS, 1.f); store(pB, blk(sAqk, 3, 0), AS, 1.f); break;
                case 7: store(pA, blk(sAqk, 1, 0), AS, 1.f); break;
                default: break;
            }
            __syncthreads();
            // rows of [T ; P] scaled by beta on the columns -> TMEM operand A2 (32 columns each)
            const int i = row & 63;
            const float* src = (row < C ? sT : sAqk) + i * AS;
            float v[16];
#pragma unroll
            for (int c = c_lo; c < c_lo + C / 2; c += 16) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = c + j;
                    v[j] = (col <= i) ? tc::to_tf32(src[col] * s_beta[col]) : 0.f;
                }
                tc::tmem_st16(T0 + TM_A2 + lane_base + c, v);
            }
        }
        __syncthreads();   // Gram tiles are dead from here on
        wait(bar_vg, ph_vg);
        ph_vg ^= 1u;

        // ---- 4. B_pre = [V_half | Gamma K]^T (smem) and A3 = (K gamma_C / Gamma)^T (TMEM)
        {
            if (tid < NE) {                      // rows 0..63: this CTA's value columns
                const int e = tid;
#pragma unroll 4
                for (int t = 0; t < C; t += 4) {
                    float4 w4;
                    float* wp = &w4.x;
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        wp[u] = (t + u < nc)
                            ? bf16_to_f(*reinterpret_cast<const uint16_t*>(sRawV + sw128_bf16(t + u, e))) : 0.f;
                    *reinterpret_cast<float4*>(sBpre + tc::sw128_offset(e, t, NE + D)) = w4;
                }
            } else if (tid < NE + D) {           // rows 64..191: (Gamma K)^T
                const int d = tid - NE;
#pragma unroll 4
                for (int t = 0; t < C; t += 4) {
                    float4 w4;
                    float* wp = &w4.x;
                    const float es = s_expS[(t >> 4) * D + d];
#pragma unroll
                    for (int u = 0; u < 4; ++u) wp[u] = tc::to_tf32(sKr[(t + u) * QS + d] * es);
                    *reinterpret_cast<float4*>(sBpre + tc::sw128_offset(NE + d, t, NE + D)) = w4;
                }
            }
            const int d = row;                   // A3: lane d, this thread's 32 token columns
            float v[16];
#pragma unroll
            for (int c = c_lo; c < c_lo + C / 2; c += 16) {
                const float ec = s_expCE[(c >> 4) * D + d];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = tc::to_tf32(sK[(c + j) * QS + d] * ec);
                tc::tmem_st16(T0 + TM_A3 + lane_base + c, v);
            }
            tc::tmem_st_wait();
            tc::fence_proxy_async();
            tc::fence_before_sync();
        }
        __syncthreads();

        // ---- 5. MMA 1: D[:, 0:192] = [T beta ; P] . [V_half | Gamma K]
        if (tid == 0 && !timed_out) {
            ++n_mma;
            tc::fence_after_sync();
            const uint32_t bb = tc::smem_u32(sBpre);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks)
                tc::mma_tf32_ts(T0 + TM_D, T0 + TM_A2 + 8 * ks, tc::sw128_desc_k(bb, NE + D, ks),
                                tc::idesc_tf32(128, NE + D), ks > 0);
            tc::mma_commit(mbar);
        }
        mma_wait();
        // region RB is free again: fetch the next chunk's q, k, z into it
        if (tid == 0 && has_next && !timed_out) {
            ++n_in;
            tc::fence_proxy_async();
            tc::mbar_arrive_expect_tx(bar_in, BYTES_QKZ);
            tc::tma_load_2d(sm + OFF_RAWQ, &tm_q, h * D, c0 + C, bar_in);
            tc::tma_load_2d(sm + OFF_RAWK, &tm_k, h * D, c0 + C, bar_in);
            tc::tma_load_2d(sm + OFF_RAWZ, &tm_z, h * D, c0 + C, bar_in);
        }

        // ---- 6. A1 = [-W ; Gamma Q - P Gamma K] in place of D[:, 64:192]
        //         (row = lane, this thread's 64 of the 128 columns)
        {
            float v[16];
            const int cbeg = NE + hf * (D / 2);
            if (row < C) {
#pragma unroll 1
                for (int c = cbeg; c < cbeg + D / 2; c += 16) {
                    tc::tmem_ld16(T0 + TM_D + lane_base + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = tc::to_tf32(-v[j]);
                    tc::tmem_st16(T0 + TM_D + lane_base + c, v);
                }
            } else {
                const int t = row - C;
                const float* es = s_expS + (t >> 4) * D;
#pragma unroll 1
                for (int c = cbeg; c < cbeg + D / 2; c += 16) {
                    tc::tmem_ld16(T0 + TM_D + lane_base + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int d = c - NE + j;
                        v[j] = tc::to_tf32(sQ[t * QS + d] * es[d] - v[j]);
                    }
                    tc::tmem_st16(T0 + TM_D + lane_base + c, v);
                }
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
        }
        __syncthreads();

        // ---- 7. MMA 2: [V' ; O] = [U ; U_o] + A1 . S
        if (tid == 0 && !timed_out) {
            ++n_mma;
            tc::fence_after_sync();
            const uint32_t sb = tc::smem_u32(sSop);
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks)
                tc::mma_tf32_ts(T0 + TM_D, T0 + TM_D + NE + 8 * ks, tc::sw128_desc_k(sb, NE, ks),
                                tc::idesc_tf32(128, NE), 1);
            tc::mma_commit(mbar);
        }
        mma_wait();

        // ---- 8. V' -> operand (smem), O -> o and the fused output gate (32 columns per thread)
        {
            float v[16];
            float o[NE / 2];
            float ss = 0.f;
            if (row < C) {
                const int t = row;
#pragma unroll
                for (int c = c_lo; c < c_lo + NE / 2; c += 16) {
                    tc::tmem_ld16(T0 + TM_D + lane_base + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        *reinterpret_cast<float*>(sVop + tc::sw128_offset(c + j, t, C)) = tc::to_tf32(v[j]);
                }
            } else {
                const int t = row - C;
#pragma unroll
                for (int c = 0; c < NE / 2; c += 16) {
                    tc::tmem_ld16(T0 + TM_D + lane_base + c_lo + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) { o[c + j] = a.scale * v[j]; ss += o[c + j] * o[c + j]; }
                }
                if (t < nc && a.o) {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(a.o) + ((size_t)(c0 + t) * H + h) * D + NE * r + c_lo;
#pragma unroll
                    for (int c = 0; c < NE / 2; c += 8) store8_bf16(dst + c, o + c);
                }
                if (gate) s_rowpart[hf * C + t] = ss;
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            if (gate) {
                __syncthreads();
                if (row >= C && hf == 0) {
                    const int t = row - C;
                    st_cluster_f32(cluster_map(s_rowsq + par * C + t, r ^ 1), s_rowpart[t] + s_rowpart[C + t]);
                }
                cluster_sync_all();
                if (row >= C) {
                    const int t = row - C;
                    if (t < nc) {
                        const float tot = s_rowpart[t] + s_rowpart[C + t] + s_rowsq[par * C + t];
                        const float rr = rsqrtf(tot * (1.0f / D) + a.norm_eps);
                        uint16_t* yp = reinterpret_cast<uint16_t*>(a.y) + ((size_t)(c0 + t) * H + h) * D + NE * r + c_lo;
#pragma unroll
                        for (int c = 0; c < NE / 2; c += 8) {
                            const uint4 g8 = *reinterpret_cast<const uint4*>(sRawG + sw128_bf16(t, c_lo + c));
                            const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w};
                            float yv[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float gv = __uint_as_float((j & 1) ? (gw[j >> 1] & 0xffff0000u) : (gw[j >> 1] << 16));
                                const float wn = a.norm_w ? a.norm_w[NE * r + c_lo + c + j] : 1.f;
                                yv[j] = sigmoidf_fast(gv) * wn * o[c + j] * rr;
                            }
                            store8_bf16(yp + c, yv);
                        }
                    }
                }
            }
        }
        __syncthreads();
        // v and g_in of this chunk are consumed: fetch the next chunk's
        if (tid == 0 && has_next && !timed_out) {
            ++n_vg;
            tc::fence_proxy_async();
            tc::mbar_arrive_expect_tx(bar_vg, bytes_vg);
            tc::tma_load_2d(sm + OFF_RAWV, &tm_v, h * D + NE * r, c0 + C, bar_vg);
            if (gate) tc::tma_load_2d(sm + OFF_RAWG, &tm_g, h * D + NE * r, c0 + C, bar_vg);
        }

        // ---- 9. MMA 3: dS = (K gamma_C / Gamma)^T . V'
        if (tid == 0 && !timed_out) {
            ++n_mma;
            tc::fence_after_sync();
            const uint32_t vb = tc::smem_u32(sVop);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks)
                tc::mma_tf32_ts(T0 + TM_DS, T0 + TM_A3 + 8 * ks, tc::sw128_desc_k(vb, NE, ks),
                                tc::idesc_tf32(128, NE), ks > 0);
            tc::mma_commit(mbar);
        }
        mma_wait();

        // ---- 10. S = Diag(gamma_C) S + dS  (FP32 in TMEM), refresh the tf32 operand copy;
        //          a chunk that closes a prefix-cache interval also writes S out
        {
            const int d = row;
            const float gm = s_gam[d];
            float* snap = nullptr;
            if (a.S_snap && (c0 + nc - t_begin) % a.snap_interval == 0) {
                const long srow = snapshot_row_base(a.cu_seqlens, n, a.snap_interval) +
                                  (c0 + nc - t_begin) / a.snap_interval - 1;
                snap = a.S_snap + ((srow * H + h) * D + d) * D + NE * r;
            }
            float dv[16], sv[16];
#pragma unroll
            for (int c = c_lo; c < c_lo + NE / 2; c += 16) {
                tc::tmem_ld16(T0 + TM_DS + lane_base + c, dv);
                tc::tmem_ld16(T0 + TM_S + lane_base + c, sv);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) sv[j] = fmaf(gm, sv[j], dv[j]);
                tc::tmem_st16(T0 + TM_S + lane_base + c, sv);
                if (snap) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        *reinterpret_cast<float4*>(snap + c + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    *reinterpret_cast<float*>(sSop + tc::sw128_offset(c + j, d, NE)) = tc::to_tf32(sv[j]);
            }
            tc::tmem_st_wait();
            tc::fence_proxy_async();
            tc::fence_before_sync();
        }
        __syncthreads();
    }

    // ---- final state
    if (a.S_T) {
        const int d = row;
        float* dst = a.S_T + (((size_t)n * H + h) * D + d) * D + NE * r;
        float v[16];
#pragma unroll
        for (int c = c_lo; c < c_lo + NE / 2; c += 16) {
            tc::tmem_ld16(T0 + TM_S + lane_base + c, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(dst + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    // give-up path: wait for the copies and MMAs thread 0 issued before any of
    // this CTA's shared memory or TMEM is released
    if (__syncthreads_or(timed_out) && tid == 0) {
        const bool drained = tc::drain_phase(bar_in, n_in) & tc::drain_phase(bar_vg, n_vg) &
                             tc::drain_phase(mbar, n_mma);
        atomicOr(err, drained ? tc::ERR_WAIT : tc::ERR_WAIT | tc::ERR_DRAIN);
    }
    tc::fence_before_sync();
    __syncthreads();
    cluster_sync_all();   // no CTA leaves while its peer may still write to its shared memory
    if (warp == 0) tc::tmem_dealloc(T0, TM_COLS);
}

}  // namespace tcp

bool prefill_tc_supported(const kda_prefill_args& a) {
    return a.qkv_dtype == KDA_BF16 && a.dk == tcp::D && a.dv == tcp::D;
}

// The workspace holds one int error word (a bounded wait that gave up sets it).
size_t prefill_tc_workspace_size(const kda_prefill_args&) { return 256; }

cudaError_t launch_prefill_tc(const kda_prefill_args& a, cudaStream_t s) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tcp::prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        tcp::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (a.num_seqs == 0) return cudaSuccess;
    const uint64_t row = (uint64_t)a.H * tcp::D;
    const uint64_t rows = (uint64_t)a.T_total;
    CUtensorMap mq, mk, mz, mv, mg;
    cudaError_t e;
    if ((e = make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, row, rows, tcp::D, tcp::C,
                           CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
    if ((e = make_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, row, rows, tcp::D, tcp::C,
                           CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
    if ((e = make_map(&mz, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.z, row, rows, tcp::D, tcp::C,
                           CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess) return e;
    if ((e = make_map(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, row, rows, tcp::NE, tcp::C,
                           CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
    if ((e = make_map(&mg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.g_in ? a.g_in : a.v, row, rows, tcp::NE,
                           tcp::C, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
    // the call's error word starts clear (the kernel sets it when a wait gives up)
    if ((e = cudaMemsetAsync(a.workspace, 0, sizeof(int), s)) != cudaSuccess) return e;
    dim3 grid(2, a.H, a.num_seqs);
    tcp::prefill_tc_kernel<<<grid, tcp::NT, tcp::SMEM_BYTES, s>>>(a, reinterpret_cast<int*>(a.workspace),
                                                                  wait_limit(), mq, mk, mz, mv, mg);
    count_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free variant (kda_prefill_noalloc): the scratch this kernel needs
// lives in a fixed array of the library's own device memory instead of a
// caller-provided workspace.  Every GPU that loads the library holds the
// array until the process exits; all calls share it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  In host code the
// symbol's name is only a host-side stand-in, never a device address, so it is
// looked up with that device current -- on every call: the lookup allocates
// nothing, and an address cached across calls would go stale if the device's
// context were reset and the library's module loaded again.  The first lookup
// on a device loads the module there.
cudaError_t noalloc_scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

size_t prefill_noalloc_scratch_needed(const kda_prefill_args& a) {
    return prefill_tc_supported(a) ? prefill_tc_workspace_size(a) : 0;
}

cudaError_t launch_prefill_tc_noalloc(const kda_prefill_args& a, cudaStream_t s) {
    void* scratch = nullptr;
    cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    // the array keeps the previous call's contents; the launch below clears the
    // error word, the only part of it that must start at zero
    kda_prefill_args b = a;
    b.workspace = scratch;
    b.workspace_bytes = KDA_NOALLOC_SCRATCH_BYTES;
    return launch_prefill_tc(b, s);
}

}  // namespace kda
