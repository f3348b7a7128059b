// Batched single-token KDA decode step ("Kimi K3" page, Sec. 2.1 recurrence with
// the Sec. 2.2 gate and the Sec. 2.3 output gate), states updated in place.
//
// One CTA of 256 threads per (sequence, head).  The 128x128 FP32 state is read
// once with 128-bit coalesced streaming loads into registers (64 floats per
// thread: warp w owns rows 16w..16w+15, lane l owns columns 4l..4l+3), used for
// both reductions S_bar^T k and S_bar^T q, and written back once:
//     S_bar = Diag(alpha) S,  u = beta (v - S_bar^T k),
//     S_new = S_bar + k u^T,  o = S_bar^T q + (k.q) u.
#include "kda_common.cuh"

namespace kda {

constexpr int DEC_D = 128;
constexpr int DEC_THREADS = 256;
constexpr int DEC_ROWS_PER_WARP = DEC_D / (DEC_THREADS / 32);  // 16

__global__ void __launch_bounds__(DEC_THREADS)
decode_step_kernel(kda_decode_args a) {
    const int h = blockIdx.x % a.H;
    const int n = blockIdx.x / a.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = a.slots ? a.slots[n] : n;
    if (slot < 0 || slot >= a.num_slots) return;   // out-of-range slot: skipped

    __shared__ float s_alpha[DEC_D], s_k[DEC_D], s_q[DEC_D], s_u[DEC_D];
    __shared__ float s_part[2][DEC_THREADS / 32][DEC_D];
    __shared__ float s_red[3][4];

    float* S = a.state + ((size_t)slot * a.H + h) * (size_t)DEC_D * DEC_D;
    const int row0 = warp * DEC_ROWS_PER_WARP;

    // Issue the state loads first (64 KiB in flight per CTA).
    float4 st[DEC_ROWS_PER_WARP];
#pragma unroll
    for (int r = 0; r < DEC_ROWS_PER_WARP; ++r)
        st[r] = ld_stream_f4(S + (size_t)(row0 + r) * DEC_D + 4 * lane);

    const size_t tok = (size_t)n * a.H + h;
    // Gate and L2 norms: thread i < 128 owns channel i.
    if (tid < DEC_D) {
        const uint16_t* q = reinterpret_cast<const uint16_t*>(a.q) + tok * DEC_D;
        const uint16_t* k = reinterpret_cast<const uint16_t*>(a.k) + tok * DEC_D;
        float qi = bf16_to_f(q[tid]), ki = bf16_to_f(k[tid]);
        float zi = a.z[tok * DEC_D + tid];
        s_alpha[tid] = __expf(log_decay_mode(zi, __expf(a.A[h]), a.g_min, a.gate_mode));
        float qq = warp_sum(qi * qi), kk = warp_sum(ki * ki);
        if (lane == 0) { s_red[0][warp] = qq; s_red[1][warp] = kk; }
        s_q[tid] = qi;
        s_k[tid] = ki;
    }
    __syncthreads();
    if (tid < DEC_D) {
        float rq = 1.0f, rk = 1.0f;
        if (a.qk_l2norm) {
            rq = rsqrtf(s_red[0][0] + s_red[0][1] + s_red[0][2] + s_red[0][3] + 1e-6f);
            rk = rsqrtf(s_red[1][0] + s_red[1][1] + s_red[1][2] + s_red[1][3] + 1e-6f);
        }
        float qn = s_q[tid] * rq, kn = s_k[tid] * rk;
        float kq = warp_sum(qn * kn);
        __syncwarp();
        s_q[tid] = qn;
        s_k[tid] = kn;
        if (lane == 0) s_red[2][warp] = kq;
    }
    __syncthreads();

    // S_bar = Diag(alpha) S ; partial column sums of k_i S_bar_i and q_i S_bar_i.
    float4 wk = make_float4(0.f, 0.f, 0.f, 0.f), wq = wk;
#pragma unroll
    for (int r = 0; r < DEC_ROWS_PER_WARP; ++r) {
        const int i = row0 + r;
        const float al = s_alpha[i], ki = s_k[i], qi = s_q[i];
        float4 s = st[r];
        s.x *= al; s.y *= al; s.z *= al; s.w *= al;
        st[r] = s;
        wk.x += ki * s.x; wk.y += ki * s.y; wk.z += ki * s.z; wk.w += ki * s.w;
        wq.x += qi * s.x; wq.y += qi * s.y; wq.z += qi * s.z; wq.w += qi * s.w;
    }
    *reinterpret_cast<float4*>(&s_part[0][warp][4 * lane]) = wk;
    *reinterpret_cast<float4*>(&s_part[1][warp][4 * lane]) = wq;
    __syncthreads();

    float o_e = 0.f;
    if (tid < DEC_D) {
        const int e = tid;
        float w = 0.f, qs = 0.f;
#pragma unroll
        for (int j = 0; j < DEC_THREADS / 32; ++j) { w += s_part[0][j][e]; qs += s_part[1][j][e]; }
        const uint16_t* v = reinterpret_cast<const uint16_t*>(a.v) + tok * DEC_D;
        const float beta = a.beta[tok];
        const float u = beta * (bf16_to_f(v[e]) - w);
        s_u[e] = u;
        const float kq = s_red[2][0] + s_red[2][1] + s_red[2][2] + s_red[2][3];
        o_e = a.scale * (qs + kq * u);
    }
    __syncthreads();

    // S_new = S_bar + k u^T, written back once.
    const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * lane]);
#pragma unroll
    for (int r = 0; r < DEC_ROWS_PER_WARP; ++r) {
        const float ki = s_k[row0 + r];
        float4 s = st[r];
        s.x += ki * u4.x; s.y += ki * u4.y; s.z += ki * u4.z; s.w += ki * u4.w;
        st_stream_f4(S + (size_t)(row0 + r) * DEC_D + 4 * lane, s);
    }

    // Outputs: o (bf16) and the fused output gate y = Sigmoid(g_in) w o / rms(o).
    if (tid < DEC_D) {
        const int e = tid;
        if (a.o) reinterpret_cast<uint16_t*>(a.o)[tok * DEC_D + e] = f_to_bf16(o_e);
        float ss = warp_sum(o_e * o_e);
        if (lane == 0) s_red[0][warp] = ss;
    }
    if (a.y) {
        __syncthreads();
        if (tid < DEC_D) {
            const int e = tid;
            const float ms = (s_red[0][0] + s_red[0][1] + s_red[0][2] + s_red[0][3]) * (1.0f / DEC_D);
            const float r = rsqrtf(ms + a.norm_eps);
            const float gi = bf16_to_f(reinterpret_cast<const uint16_t*>(a.g_in)[tok * DEC_D + e]);
            const float wn = a.norm_w ? a.norm_w[e] : 1.0f;
            reinterpret_cast<uint16_t*>(a.y)[tok * DEC_D + e] = f_to_bf16(sigmoidf_fast(gi) * wn * o_e * r);
        }
    }
}

cudaError_t launch_decode_step(const kda_decode_args& a, cudaStream_t stream) {
    const long blocks = (long)a.N * a.H;
    if (blocks == 0) return cudaSuccess;
    decode_step_kernel<<<(unsigned)blocks, DEC_THREADS, 0, stream>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
