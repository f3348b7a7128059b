// ShortConv + Swish prologue ("Kimi K3: KDA, attention residuals and Stable
// LatentMoE", Sec. 2.1: q and k pass through ShortConv, Swish and L2Norm, v
// through ShortConv and Swish; Swish(z) = z Sigmoid(z) as defined in Sec. 5).
//
// A causal depthwise convolution of width W along each packed sequence:
//   pre[t, c] = sum_i w[c, i] x[t - (W-1) + i, c] + b[c],  y = Swish(pre),
// positions before a sequence's first token read its conv state.
//
// Streaming, HBM-bound: each thread owns 8 consecutive channels (one 16-byte
// bf16 or two 16-byte f32 accesses per token, coalesced across the warp) and
// walks a segment of SEG packed tokens with the last W-1 inputs in registers;
// at a sequence start it reloads the window from that sequence's state.  One
// lane per warp prefetches the warp's row slices into L2 a few tokens ahead.  A
// second launch writes the new states; the decode step shifts a state in place.
#include "kda_common.cuh"

namespace kda {
namespace conv {

constexpr int NT = 128;     // threads per block; each covers 8 channels
constexpr int SEG = 128;    // packed tokens per thread

template <bool BF16>
KDA_DEV void load8(const void* base, size_t idx, float* v) {
    if (BF16) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(base) + idx));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
        const float4 a = __ldcs(p), b = __ldcs(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

template <bool BF16>
KDA_DEV void store8(void* base, size_t idx, const float* v) {
    if (BF16) {
        store8_bf16(reinterpret_cast<uint16_t*>(base) + idx, v);
    } else {
        float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx);
        __stcs(p, make_float4(v[0], v[1], v[2], v[3]));
        __stcs(p + 1, make_float4(v[4], v[5], v[6], v[7]));
    }
}

KDA_DEV float swish(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// largest n with cu[n] <= t among n < num_seqs (sequence holding packed token t)
KDA_DEV int seq_of(const int* cu, int num_seqs, int t) {
    int lo = 0, hi = num_seqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

template <int W, bool BF16>
__global__ void __launch_bounds__(NT) short_conv_kernel(kda_short_conv_args a) {
    const int C = a.channels;
    const int c0 = (blockIdx.x * NT + threadIdx.x) * 8;
    if (c0 >= C) return;
    const int t_begin = blockIdx.y * SEG;
    const int t_end = min(a.T_total, t_begin + SEG);
    if (t_begin >= t_end) return;
    float wt[W][8], bs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        bs[j] = a.bias ? a.bias[c0 + j] : 0.f;
#pragma unroll
        for (int i = 0; i < W; ++i) wt[i][j] = a.weight[(size_t)(c0 + j) * W + i];
    }
    int n = seq_of(a.cu_seqlens, a.num_seqs, t_begin);
    int s_start = a.cu_seqlens[n], s_end = a.cu_seqlens[n + 1];
    // window: hist[i] = input at position t - (W-1) + i, i < W-1
    float hist[W > 1 ? W - 1 : 1][8];
    auto fill = [&](int t) {   // window for token t of sequence n
#pragma unroll
        for (int i = 0; i < W - 1; ++i) {
            const int p = t - (W - 1) + i;
            if (p >= s_start) {
                load8<BF16>(a.x, (size_t)p * C + c0, hist[i]);
            } else if (a.state_in) {
                const float* st = a.state_in + ((size_t)n * (W - 1) + (p - s_start + (W - 1))) * C + c0;
                const float4 u = *reinterpret_cast<const float4*>(st), v = *reinterpret_cast<const float4*>(st + 4);
                hist[i][0] = u.x; hist[i][1] = u.y; hist[i][2] = u.z; hist[i][3] = u.w;
                hist[i][4] = v.x; hist[i][5] = v.y; hist[i][6] = v.z; hist[i][7] = v.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) hist[i][j] = 0.f;
            }
        }
    };
    fill(t_begin);
    // lane 0 has the warp's row slice (its 32 threads' channels, clamped at the row
    // end) prefetched into L2 PF tokens ahead of the loads: memory parallelism
    // without registers
    constexpr int PF = 8;
    const bool pf_lane = (threadIdx.x & 31) == 0;
    const int cw0 = c0;   // lane 0: the warp's first channel
    const uint32_t pf_bytes = (uint32_t)(min(256, C - cw0) * (BF16 ? 2 : 4));
    // one token: y from the window and x, then slide the window
    auto step = [&](int t, const float* xv) {
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float pre = fmaf(wt[W - 1][j], xv[j], bs[j]);
#pragma unroll
            for (int i = 0; i < W - 1; ++i) pre = fmaf(wt[i][j], hist[i][j], pre);
            y[j] = a.activation ? swish(pre) : pre;
        }
        store8<BF16>(a.y, (size_t)t * C + c0, y);
#pragma unroll
        for (int i = 0; i + 1 < W - 1; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) hist[i][j] = hist[i + 1][j];
        if (W > 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) hist[W > 1 ? W - 2 : 0][j] = xv[j];
        }
    };
    int t = t_begin;
#pragma unroll 1
    while (t < t_end) {
        if (t >= s_end) {   // the next sequence starts here (skip empty ones)
            while (t >= a.cu_seqlens[n + 1]) ++n;
            s_start = a.cu_seqlens[n];
            s_end = a.cu_seqlens[n + 1];
            fill(t);
        }
        const int stop = min(t_end, s_end);   // this sequence's tokens in the segment
        // U tokens per round: their loads are issued together, then consumed in order
        constexpr int U = 4;
#pragma unroll 1
        for (; t + U <= stop; t += U) {
            if (pf_lane && t + PF + U <= t_end) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const void* pp = reinterpret_cast<const uint8_t*>(a.x) + ((size_t)(t + PF + u) * C + cw0) * (BF16 ? 2 : 4);
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(pp), "r"(pf_bytes) : "memory");
                }
            }
            float xv[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u) load8<BF16>(a.x, (size_t)(t + u) * C + c0, xv[u]);
#pragma unroll
            for (int u = 0; u < U; ++u) step(t + u, xv[u]);
        }
#pragma unroll 1
        for (; t < stop; ++t) {
            float xv[8];
            load8<BF16>(a.x, (size_t)t * C + c0, xv);
            step(t, xv);
        }
    }
}

// state_out[n] = last W-1 entries of [state_in[n], x of sequence n]
template <bool BF16>
__global__ void __launch_bounds__(NT) short_conv_state_kernel(kda_short_conv_args a) {
    const int C = a.channels, W = a.width;
    const int c0 = (blockIdx.x * NT + threadIdx.x) * 8;
    const int n = blockIdx.y;
    if (c0 >= C) return;
    const int s_start = a.cu_seqlens[n], L = a.cu_seqlens[n + 1] - s_start;
    for (int s = 0; s < W - 1; ++s) {
        float v[8];
        if (L + s >= W - 1) {
            load8<BF16>(a.x, (size_t)(s_start + L + s - (W - 1)) * C + c0, v);
        } else if (a.state_in) {
            const float* st = a.state_in + ((size_t)n * (W - 1) + (L + s)) * C + c0;
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = st[j];
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0.f;
        }
        float* dst = a.state_out + ((size_t)n * (W - 1) + s) * C + c0;
        *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
}

template <int W, bool BF16>
__global__ void __launch_bounds__(NT) short_conv_step_kernel(kda_short_conv_step_args a) {
    const int C = a.channels;
    const int c0 = (blockIdx.x * NT + threadIdx.x) * 8;
    const int i = blockIdx.y;
    if (c0 >= C) return;
    const int slot = a.slots ? a.slots[i] : i;
    float xv[8], y[8];
    load8<BF16>(a.x, (size_t)i * C + c0, xv);
    float hist[W > 1 ? W - 1 : 1][8];
    float* st = a.state + (size_t)slot * (W - 1) * C + c0;
#pragma unroll
    for (int s = 0; s < W - 1; ++s)
#pragma unroll
        for (int j = 0; j < 8; ++j) hist[s][j] = st[(size_t)s * C + j];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float pre = fmaf(a.weight[(size_t)(c0 + j) * W + W - 1], xv[j], a.bias ? a.bias[c0 + j] : 0.f);
#pragma unroll
        for (int s = 0; s < W - 1; ++s) pre = fmaf(a.weight[(size_t)(c0 + j) * W + s], hist[s][j], pre);
        y[j] = a.activation ? swish(pre) : pre;
    }
    store8<BF16>(a.y, (size_t)i * C + c0, y);
#pragma unroll
    for (int s = 0; s < W - 1; ++s)
#pragma unroll
        for (int j = 0; j < 8; ++j) st[(size_t)s * C + j] = (s + 1 < W - 1) ? hist[s + 1][j] : xv[j];
}

template <int W>
static cudaError_t launch_w(const kda_short_conv_args& a, cudaStream_t s) {
    const dim3 grid((a.channels / 8 + NT - 1) / NT, (a.T_total + SEG - 1) / SEG);
    if (a.T_total > 0) {
        if (a.dtype == KDA_BF16) short_conv_kernel<W, true><<<grid, NT, 0, s>>>(a);
        else short_conv_kernel<W, false><<<grid, NT, 0, s>>>(a);
        count_launches(1);
    }
    if (a.state_out && W > 1) {
        const dim3 g2((a.channels / 8 + NT - 1) / NT, a.num_seqs);
        if (a.dtype == KDA_BF16) short_conv_state_kernel<true><<<g2, NT, 0, s>>>(a);
        else short_conv_state_kernel<false><<<g2, NT, 0, s>>>(a);
        count_launches(1);
    }
    return cudaGetLastError();
}

template <int W>
static cudaError_t launch_step_w(const kda_short_conv_step_args& a, cudaStream_t s) {
    const dim3 grid((a.channels / 8 + NT - 1) / NT, a.N);
    if (a.dtype == KDA_BF16) short_conv_step_kernel<W, true><<<grid, NT, 0, s>>>(a);
    else short_conv_step_kernel<W, false><<<grid, NT, 0, s>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace conv

cudaError_t launch_short_conv(const kda_short_conv_args& a, cudaStream_t s) {
    switch (a.width) {
        case 1: return conv::launch_w<1>(a, s);
        case 2: return conv::launch_w<2>(a, s);
        case 3: return conv::launch_w<3>(a, s);
        case 4: return conv::launch_w<4>(a, s);
        case 5: return conv::launch_w<5>(a, s);
        case 6: return conv::launch_w<6>(a, s);
        case 7: return conv::launch_w<7>(a, s);
        case 8: return conv::launch_w<8>(a, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_short_conv_step(const kda_short_conv_step_args& a, cudaStream_t s) {
    if (a.N == 0) return cudaSuccess;
    switch (a.width) {
        case 1: return conv::launch_step_w<1>(a, s);
        case 2: return conv::launch_step_w<2>(a, s);
        case 3: return conv::launch_step_w<3>(a, s);
        case 4: return conv::launch_step_w<4>(a, s);
        case 5: return conv::launch_step_w<5>(a, s);
        case 6: return conv::launch_step_w<6>(a, s);
        case 7: return conv::launch_step_w<7>(a, s);
        case 8: return conv::launch_step_w<8>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kda
