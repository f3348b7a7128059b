// KDA prefill by the per-token recurrence on CUDA cores ("Kimi K3" page,
// Sec. 2.1 recurrence, Sec. 2.2 gate, Sec. 2.3 output gate).
//
// This is the path for float32 inputs and head sizes 32/64/128 (the tensor-core
// chunked kernel covers bf16 with dk = dv = 128), and it is exported on its own
// as kda_prefill_recurrent for cross-checking the chunked kernel on the GPU.
// One CTA of 256 threads per (sequence, head); the D x D FP32 state stays in
// registers for the whole sequence (thread t: column group t % (D/4) of four
// columns, row group t / (D/4)).
#include "kda_common.cuh"

namespace kda {

template <int D, bool BF16>
__global__ void __launch_bounds__(256)
prefill_recurrent_kernel(kda_prefill_args a) {
    constexpr int NT = 256;
    constexpr int CG = D / 4;              // column groups of 4
    constexpr int RG = NT / CG;            // row groups
    constexpr int RPG = D / RG;            // rows per row group
    constexpr int NW = NT / 32;
    const int h = blockIdx.x % a.H;
    const int n = blockIdx.x / a.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % CG, rg = tid / CG;
    const int t0 = a.cu_seqlens[n], t1 = a.cu_seqlens[n + 1];

    __shared__ float s_alpha[D], s_k[D], s_q[D], s_u[D], s_v[D];
    __shared__ float s_part[2][RG][D];
    __shared__ float s_red[4][NW];

    const size_t sbase = ((size_t)n * a.H + h) * (size_t)D * D;
    float4 st[RPG];
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
        if (a.S0) st[r] = *reinterpret_cast<const float4*>(a.S0 + sbase + (size_t)(rg * RPG + r) * D + 4 * cg);
        else st[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float eA = __expf(a.A[h]);
    // prefix-cache snapshots: the next row to write and the tokens until it is due
    long snap_row = a.S_snap ? snapshot_row_base(a.cu_seqlens, n, a.snap_interval) : 0;
    int snap_left = a.snap_interval;

    for (int t = t0; t < t1; ++t) {
        const size_t tok = (size_t)t * a.H + h;
        float qi = 0.f, ki = 0.f;
        if (tid < D) {
            if (BF16) {
                qi = bf16_to_f(reinterpret_cast<const uint16_t*>(a.q)[tok * D + tid]);
                ki = bf16_to_f(reinterpret_cast<const uint16_t*>(a.k)[tok * D + tid]);
                s_v[tid] = bf16_to_f(reinterpret_cast<const uint16_t*>(a.v)[tok * D + tid]);
            } else {
                qi = reinterpret_cast<const float*>(a.q)[tok * D + tid];
                ki = reinterpret_cast<const float*>(a.k)[tok * D + tid];
                s_v[tid] = reinterpret_cast<const float*>(a.v)[tok * D + tid];
            }
            s_alpha[tid] = __expf(log_decay_mode(a.z[tok * D + tid], eA, a.g_min, a.gate_mode));
        }
        float qq = warp_sum(qi * qi), kk = warp_sum(ki * ki), kq = warp_sum(qi * ki);
        if (lane == 0) { s_red[0][warp] = qq; s_red[1][warp] = kk; s_red[2][warp] = kq; }
        __syncthreads();
        float sq = 0.f, sk = 0.f, skq = 0.f;
#pragma unroll
        for (int j = 0; j < NW; ++j) { sq += s_red[0][j]; sk += s_red[1][j]; skq += s_red[2][j]; }
        float rq = 1.f, rk = 1.f;
        if (a.qk_l2norm) { rq = rsqrtf(sq + 1e-6f); rk = rsqrtf(sk + 1e-6f); }
        if (tid < D) { s_q[tid] = qi * rq; s_k[tid] = ki * rk; }
        const float kqn = skq * rq * rk;
        __syncthreads();

        float4 wk = make_float4(0.f, 0.f, 0.f, 0.f), wq = wk;
#pragma unroll
        for (int r = 0; r < RPG; ++r) {
            const int i = rg * RPG + r;
            const float al = s_alpha[i], kn = s_k[i], qn = s_q[i];
            float4 s = st[r];
            s.x *= al; s.y *= al; s.z *= al; s.w *= al;
            st[r] = s;
            wk.x += kn * s.x; wk.y += kn * s.y; wk.z += kn * s.z; wk.w += kn * s.w;
            wq.x += qn * s.x; wq.y += qn * s.y; wq.z += qn * s.z; wq.w += qn * s.w;
        }
        *reinterpret_cast<float4*>(&s_part[0][rg][4 * cg]) = wk;
        *reinterpret_cast<float4*>(&s_part[1][rg][4 * cg]) = wq;
        __syncthreads();

        float o_e = 0.f;
        if (tid < D) {
            float w = 0.f, qs = 0.f;
#pragma unroll
            for (int j = 0; j < RG; ++j) { w += s_part[0][j][tid]; qs += s_part[1][j][tid]; }
            const float u = a.beta[tok] * (s_v[tid] - w);
            s_u[tid] = u;
            o_e = a.scale * (qs + kqn * u);
            if (a.o) {
                if (BF16) reinterpret_cast<uint16_t*>(a.o)[tok * D + tid] = f_to_bf16(o_e);
                else reinterpret_cast<float*>(a.o)[tok * D + tid] = o_e;
            }
        }
        float ss = warp_sum(o_e * o_e);
        if (lane == 0) s_red[3][warp] = ss;
        __syncthreads();
        const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * cg]);
#pragma unroll
        for (int r = 0; r < RPG; ++r) {
            const float kn = s_k[rg * RPG + r];
            st[r].x += kn * u4.x; st[r].y += kn * u4.y; st[r].z += kn * u4.z; st[r].w += kn * u4.w;
        }
        if (a.g_in && tid < D) {
            float ms = 0.f;
#pragma unroll
            for (int j = 0; j < NW; ++j) ms += s_red[3][j];
            const float r = rsqrtf(ms * (1.0f / D) + a.norm_eps);
            const float gi = bf16_to_f(reinterpret_cast<const uint16_t*>(a.g_in)[tok * D + tid]);
            const float wn = a.norm_w ? a.norm_w[tid] : 1.0f;
            reinterpret_cast<uint16_t*>(a.y)[tok * D + tid] = f_to_bf16(sigmoidf_fast(gi) * wn * o_e * r);
        }
        if (a.S_snap && --snap_left == 0) {
            float* dst = a.S_snap + ((size_t)snap_row * a.H + h) * (size_t)D * D;
#pragma unroll
            for (int r = 0; r < RPG; ++r)
                *reinterpret_cast<float4*>(dst + (size_t)(rg * RPG + r) * D + 4 * cg) = st[r];
            ++snap_row;
            snap_left = a.snap_interval;
        }
        __syncthreads();   // shared buffers are rewritten by the next token
    }
    if (a.S_T) {
#pragma unroll
        for (int r = 0; r < RPG; ++r)
            *reinterpret_cast<float4*>(a.S_T + sbase + (size_t)(rg * RPG + r) * D + 4 * cg) = st[r];
    }
}

template <int D, bool BF16>
static cudaError_t launch_rec(const kda_prefill_args& a, cudaStream_t s) {
    prefill_recurrent_kernel<D, BF16><<<(unsigned)((long)a.num_seqs * a.H), 256, 0, s>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_prefill_recurrent(const kda_prefill_args& a, cudaStream_t s) {
    if ((long)a.num_seqs * a.H == 0) return cudaSuccess;
    const bool bf = a.qkv_dtype == KDA_BF16;
    switch (a.dk) {
        case 32: return bf ? launch_rec<32, true>(a, s) : launch_rec<32, false>(a, s);
        case 64: return bf ? launch_rec<64, true>(a, s) : launch_rec<64, false>(a, s);
        case 128: return bf ? launch_rec<128, true>(a, s) : launch_rec<128, false>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kda
