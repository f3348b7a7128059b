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
// Work decomposition: a cluster of two CTAs per (sequence, head); CTA r owns
// value columns [64r, 64r+64).  Both CTAs compute the d_k-wide chunk terms;
// the only exchange is the per-row sum of squares for the RMSNorm of the
// fused output gate (over distributed shared memory).
//
// Precision: every contraction runs as tcgen05 kind::tf32 (the 16x16 Gram
// sub-blocks as mma.sync tf32) with FP32 accumulation; operands are rounded to
// tf32 (nearest) when staged; the gate, cumulative decays, the triangular
// solve and the state carry stay FP32 (the state lives in TMEM in FP32 across
// chunks and is only rounded for its copy used as an MMA operand).
#include <mutex>

#include "kda_common.cuh"
#include "tcgen05.cuh"

namespace kda {
namespace tcp {

constexpr int C = 64;     // chunk length
constexpr int D = 128;    // dk = dv
constexpr int NE = 64;    // value columns per CTA
constexpr int NT = 128;   // threads per CTA
constexpr int QS = 132;   // padded row stride (floats) of the scaled q/k tiles
constexpr int AS = 68;    // padded row stride (floats) of the 64x64 Gram tiles

// shared memory map (offsets from a 1024-aligned base)
constexpr int SOP_BYTES = NE * D * 4;                 // S operand, SW128 [e][d]      32 KB
constexpr int BPRE_BYTES = (NE + D) * C * 4;          // [V | Gamma K]^T, SW128 [n][t] 48 KB
constexpr int TILE_BYTES = C * QS * 4;                // one scaled q/k tile           33 KB
constexpr int OFF_SOP = 0;
constexpr int OFF_BPRE = OFF_SOP + SOP_BYTES;
constexpr int OFF_QH = OFF_BPRE + BPRE_BYTES;         // q * exp(G - G_subchunk_start)
constexpr int OFF_KR = OFF_QH + TILE_BYTES;           // k * exp(G - G_subchunk_start)
constexpr int OFF_KH = OFF_KR + TILE_BYTES;           // k * exp(G_subchunk_end - G)
constexpr int OFF_VOP = OFF_KR;                       // V' operand [e][t] (aliases KR)
constexpr int OFF_AQK = OFF_BPRE;                     // Gram tiles (alias B_pre)
constexpr int OFF_AKK = OFF_BPRE + C * AS * 4;
constexpr int OFF_SMALL = OFF_KH + TILE_BYTES;
// small region (floats)
constexpr int SM_BETA = 0, SM_RQ = 64, SM_RK = 128, SM_TAU = 192, SM_EXPS = SM_TAU + 4 * D,
              SM_EXPCE = SM_EXPS + 4 * D, SM_GAM = SM_EXPCE + 4 * D, SM_ROWSQ = SM_GAM + D,
              SM_FLOATS = SM_ROWSQ + 2 * C;
constexpr int SMEM_BYTES = OFF_SMALL + SM_FLOATS * 4 + 64 /*mbarrier, tmem base*/ + 1024 /*align*/;
static_assert(OFF_VOP % 1024 == 0 && OFF_BPRE % 1024 == 0, "SW128 operands need 1024-B alignment");
static_assert(2 * C * AS * 4 <= BPRE_BYTES, "Gram tiles must fit in the B_pre region");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NT, 1)
prefill_tc_kernel(kda_prefill_args a, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sSop = sm + OFF_SOP;
    uint8_t* sBpre = sm + OFF_BPRE;
    uint8_t* sVop = sm + OFF_VOP;
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
    uint64_t* mbar = reinterpret_cast<uint64_t*>(fs + SM_FLOATS);
    uint32_t* tbase_ptr = reinterpret_cast<uint32_t*>(mbar + 1);

    const int r = blockIdx.x;          // value half == cluster rank
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const int H = a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t_begin = a.cu_seqlens[n], t_end = a.cu_seqlens[n + 1];
    const uint16_t* qp = reinterpret_cast<const uint16_t*>(a.q);
    const uint16_t* kp = reinterpret_cast<const uint16_t*>(a.k);
    const uint16_t* vp = reinterpret_cast<const uint16_t*>(a.v);
    const float eA = __expf(a.A[h]);
    const bool gate = a.g_in != nullptr;

    if (warp == 0) { tc::tmem_alloc(tbase_ptr, TM_COLS); tc::tmem_relinquish(); }
    if (tid == 0) { tc::mbar_init(mbar, 1); tc::mbar_fence_init(); }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t T0 = *tbase_ptr;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t phase = 0;
    bool timed_out = false;
    auto mma_wait = [&]() {
        if (!tc::mbar_wait_bounded(mbar, phase, 1u << 22)) timed_out = true;
        phase ^= 1u;
        tc::fence_after_sync();
    };

    // ---- initial state -> TMEM master copy and the tf32 operand copy
    {
        const int d = tid;
        const size_t sb = (((size_t)n * H + h) * D + d) * D + NE * r;
        float v[16];
#pragma unroll
        for (int c = 0; c < NE; c += 16) {
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

        // ---- 1a. write strengths and q/k L2 norms (warp w: tokens 16w..16w+15)
        if (tid < C) s_beta[tid] = tid < nc ? a.beta[(size_t)(c0 + tid) * H + h] : 0.f;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            const int t = warp * 16 + i;
            float sq = 0.f, sk = 0.f;
            if (t < nc) {
                const size_t base = ((size_t)(c0 + t) * H + h) * D + 4 * lane;
                const uint2 qa = *reinterpret_cast<const uint2*>(qp + base);
                const uint2 ka = *reinterpret_cast<const uint2*>(kp + base);
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

        // ---- 1b. gate, sub-chunk-relative decay factors, scaled q/k tiles (thread = channel d)
        {
            const int d = tid;
            float pre = 1.f;                       // exp(G at the start of sub-chunk b)
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
                float al[16], kv[16];
                float F1 = 1.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int t = 16 * b + i;
                    float alpha = 1.f, q = 0.f, k = 0.f;
                    if (t < nc) {
                        const size_t e = ((size_t)(c0 + t) * H + h) * D + d;
                        alpha = __expf(log_decay(a.z[e], eA, a.g_min));
                        q = bf16_to_f(qp[e]) * s_rq[t];
                        k = bf16_to_f(kp[e]) * s_rk[t];
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
                s_expS[b * D + d] = pre;
                pre *= F1;
            }
            s_gam[d] = pre;
            float suf = 1.f;
#pragma unroll
            for (int b = 3; b >= 0; --b) { s_expCE[b * D + d] = suf; suf *= s_tau[b * D + d]; }
        }
        __syncthreads();

        // ---- 2. Gram sub-blocks with mma.sync (tf32): warp w -> QK row block w, KK row block 3-w
        {
            const int g = lane >> 2, t4 = lane & 3;
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {
                const int ab = pass == 0 ? warp : 3 - warp;
                const float* Arow = pass == 0 ? sQ : sKr;
                float* Out = pass == 0 ? sAqk : sAkk;
#pragma unroll 1
                for (int b = 0; b <= ab; ++b) {
                    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 4
                    for (int ks = 0; ks < 16; ++ks) {
                        const int k0 = 8 * ks + t4, k1 = k0 + 4;
                        // per-channel factor joining the two references: exp(G_start(ab) - G_end(b))
                        float c0f, c1f;
                        if (ab == b) {
                            c0f = __fdividef(1.f, s_tau[b * D + k0]);
                            c1f = __fdividef(1.f, s_tau[b * D + k1]);
                        } else {
                            c0f = 1.f; c1f = 1.f;
                            for (int m = b + 1; m < ab; ++m) { c0f *= s_tau[m * D + k0]; c1f *= s_tau[m * D + k1]; }
                        }
                        const int ra = 16 * ab + g;
                        float af[4] = {tc::to_tf32(Arow[ra * QS + k0]), tc::to_tf32(Arow[(ra + 8) * QS + k0]),
                                       tc::to_tf32(Arow[ra * QS + k1]), tc::to_tf32(Arow[(ra + 8) * QS + k1])};
#pragma unroll
                        for (int nh = 0; nh < 2; ++nh) {
                            const int j = 16 * b + 8 * nh + g;
                            float bfr[2] = {tc::to_tf32(sK[j * QS + k0] * c0f), tc::to_tf32(sK[j * QS + k1] * c1f)};
                            tc::mma_m16n8k8_tf32(acc[nh], af, bfr);
                        }
                    }
#pragma unroll
                    for (int nh = 0; nh < 2; ++nh) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int I = 16 * ab + g + (q4 >= 2 ? 8 : 0);
                            const int J = 16 * b + 8 * nh + 2 * t4 + (q4 & 1);
                            float val = acc[nh][q4];
                            if (pass == 0) { if (J > I) val = 0.f; }
                            else { val = (J >= I) ? 0.f : val * s_beta[I]; }
                            Out[I * AS + J] = val;
                        }
                    }
                }
            }
        }
        __syncthreads();

        // ---- 3. UT solve: rows of T = (I + A_kk)^{-1} (threads 0..63) and of
        //         A_qk (I + A_kk)^{-1} (threads 64..127), then scale columns by beta
        {
            const int i = tid & 63;
            const bool isP = tid >= 64;
            float x[C];
#pragma unroll
            for (int j = 0; j < C; ++j) x[j] = isP ? (j <= i ? sAqk[i * AS + j] : 0.f) : (j == i ? 1.f : 0.f);
            // x (I + A) = rhs, A strictly lower: x_j = rhs_j - sum_{k>j} x_k A[k][j]
#pragma unroll
            for (int kk = C - 1; kk >= 1; --kk) {
                const float xk = x[kk];
#pragma unroll
                for (int j = 0; j < kk; ++j) x[j] = fmaf(-xk, sAkk[kk * AS + j], x[j]);
            }
            float v[16];
#pragma unroll
            for (int c = 0; c < C; c += 16) {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = tc::to_tf32(x[c + j] * s_beta[c + j]);
                tc::tmem_st16(T0 + TM_A2 + lane_base + c, v);
            }
        }
        __syncthreads();   // Gram tiles (aliasing B_pre) are dead from here on

        // ---- 4. B_pre = [V_half | Gamma K]^T (smem) and A3 = (K gamma_C / Gamma)^T (TMEM)
        {
            if (tid < NE) {
                const int e = tid;
#pragma unroll 2
                for (int t = 0; t < C; t += 4) {
                    float4 w4;
                    float* wp = &w4.x;
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        wp[u] = (t + u < nc) ? bf16_to_f(vp[((size_t)(c0 + t + u) * H + h) * D + NE * r + e]) : 0.f;
                    *reinterpret_cast<float4*>(sBpre + tc::sw128_offset(e, t, NE + D)) = w4;
                }
            }
            const int d = tid;
#pragma unroll 2
            for (int t = 0; t < C; t += 4) {
                float4 w4;
                float* wp = &w4.x;
                const float es = s_expS[(t >> 4) * D + d];
#pragma unroll
                for (int u = 0; u < 4; ++u) wp[u] = tc::to_tf32(sKr[(t + u) * QS + d] * es);
                *reinterpret_cast<float4*>(sBpre + tc::sw128_offset(NE + d, t, NE + D)) = w4;
            }
            float v[16];
#pragma unroll
            for (int c = 0; c < C; c += 16) {
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
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t bb = tc::smem_u32(sBpre);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks)
                tc::mma_tf32_ts(T0 + TM_D, T0 + TM_A2 + 8 * ks, tc::sw128_desc_k(bb, NE + D, ks),
                                tc::idesc_tf32(128, NE + D), ks > 0);
            tc::mma_commit(mbar);
        }
        mma_wait();

        // ---- 6. A1 = [-W ; Gamma Q - P Gamma K] in place of D[:, 64:192]
        {
            float v[16];
            if (tid < C) {
#pragma unroll 1
                for (int c = NE; c < NE + D; c += 16) {
                    tc::tmem_ld16(T0 + TM_D + lane_base + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = tc::to_tf32(-v[j]);
                    tc::tmem_st16(T0 + TM_D + lane_base + c, v);
                }
            } else {
                const int t = tid - C;
                const float* es = s_expS + (t >> 4) * D;
#pragma unroll 1
                for (int c = NE; c < NE + D; c += 16) {
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
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t sb = tc::smem_u32(sSop);
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks)
                tc::mma_tf32_ts(T0 + TM_D, T0 + TM_D + NE + 8 * ks, tc::sw128_desc_k(sb, NE, ks),
                                tc::idesc_tf32(128, NE), 1);
            tc::mma_commit(mbar);
        }
        mma_wait();

        // ---- 8. V' -> operand (smem), O -> o and the fused output gate
        {
            float v[16];
            float o[NE];
            float ss = 0.f;
            if (tid < C) {
                const int t = tid;
#pragma unroll
                for (int c = 0; c < NE; c += 16) {
                    tc::tmem_ld16(T0 + TM_D + lane_base + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        *reinterpret_cast<float*>(sVop + tc::sw128_offset(c + j, t, C)) = tc::to_tf32(v[j]);
                }
            } else {
                const int t = tid - C;
#pragma unroll
                for (int c = 0; c < NE; c += 16) {
                    tc::tmem_ld16(T0 + TM_D + lane_base + c, v);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) { o[c + j] = a.scale * v[j]; ss += o[c + j] * o[c + j]; }
                }
                if (t < nc) {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(a.o) + ((size_t)(c0 + t) * H + h) * D + NE * r;
#pragma unroll
                    for (int c = 0; c < NE; c += 8) store8_bf16(dst + c, o + c);
                }
                if (gate) st_cluster_f32(cluster_map(s_rowsq + par * C + t, r ^ 1), ss);
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            if (gate) {
                cluster_sync_all();
                if (tid >= C) {
                    const int t = tid - C;
                    if (t < nc) {
                        const float tot = ss + s_rowsq[par * C + t];
                        const float rr = rsqrtf(tot * (1.0f / D) + a.norm_eps);
                        const size_t rowoff = ((size_t)(c0 + t) * H + h) * D + NE * r;
                        const uint16_t* gp = reinterpret_cast<const uint16_t*>(a.g_in) + rowoff;
                        uint16_t* yp = reinterpret_cast<uint16_t*>(a.y) + rowoff;
#pragma unroll
                        for (int c = 0; c < NE; c += 8) {
                            float gv[8], yv[8];
                            load8_bf16(gp + c, gv);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float wn = a.norm_w ? a.norm_w[NE * r + c + j] : 1.f;
                                yv[j] = sigmoidf_fast(gv[j]) * wn * o[c + j] * rr;
                            }
                            store8_bf16(yp + c, yv);
                        }
                    }
                }
            }
        }
        __syncthreads();

        // ---- 9. MMA 3: dS = (K gamma_C / Gamma)^T . V'
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t vb = tc::smem_u32(sVop);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks)
                tc::mma_tf32_ts(T0 + TM_DS, T0 + TM_A3 + 8 * ks, tc::sw128_desc_k(vb, NE, ks),
                                tc::idesc_tf32(128, NE), ks > 0);
            tc::mma_commit(mbar);
        }
        mma_wait();

        // ---- 10. S = Diag(gamma_C) S + dS  (FP32 in TMEM), refresh the tf32 operand copy
        {
            const int d = tid;
            const float gm = s_gam[d];
            float dv[16], sv[16];
#pragma unroll
            for (int c = 0; c < NE; c += 16) {
                tc::tmem_ld16(T0 + TM_DS + lane_base + c, dv);
                tc::tmem_ld16(T0 + TM_S + lane_base + c, sv);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) sv[j] = fmaf(gm, sv[j], dv[j]);
                tc::tmem_st16(T0 + TM_S + lane_base + c, sv);
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
        const int d = tid;
        float* dst = a.S_T + (((size_t)n * H + h) * D + d) * D + NE * r;
        float v[16];
#pragma unroll
        for (int c = 0; c < NE; c += 16) {
            tc::tmem_ld16(T0 + TM_S + lane_base + c, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(dst + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    if (timed_out && err) atomicOr(err, 1);
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
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(tcp::prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             tcp::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (a.num_seqs == 0) return cudaSuccess;
    dim3 grid(2, a.H, a.num_seqs);
    tcp::prefill_tc_kernel<<<grid, tcp::NT, tcp::SMEM_BYTES, s>>>(a, reinterpret_cast<int*>(a.workspace));
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

// Device address of g_noalloc_scratch on the current device, looked up once per
// device with that device current (in host code the symbol name is only a
// host-side stand-in, never a device address).
static cudaError_t noalloc_scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

size_t prefill_noalloc_scratch_needed(const kda_prefill_args& a) {
    return prefill_tc_supported(a) ? prefill_tc_workspace_size(a) : 0;
}

cudaError_t launch_prefill_tc_noalloc(const kda_prefill_args& a, cudaStream_t s) {
    void* scratch = nullptr;
    cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    const size_t need = prefill_tc_workspace_size(a);
    // the error word must start at zero; the array keeps the previous call's contents
    e = cudaMemsetAsync(scratch, 0, need, s);
    if (e != cudaSuccess) return e;
    kda_prefill_args b = a;
    b.workspace = scratch;
    b.workspace_bytes = KDA_NOALLOC_SCRATCH_BYTES;
    return launch_prefill_tc(b, s);
}

}  // namespace kda
