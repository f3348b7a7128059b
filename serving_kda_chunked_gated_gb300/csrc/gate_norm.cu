// Output gate of the "Kimi K3" page, Sec. 2.3, applied on its own:
//   y = Sigmoid(g_in) (.) w (.) o / sqrt(mean(o^2) + eps)   per (token, head) row of dv.
// One warp per row; each lane holds dv/32 consecutive channels.
#include "kda_common.cuh"

namespace kda {

template <int DV, bool BF16>
__global__ void __launch_bounds__(256)
gate_norm_kernel(const void* __restrict__ o, const void* __restrict__ g_in,
                 const float* __restrict__ w, float eps, void* __restrict__ y, long rows) {
    constexpr int PER = DV / 32;
    const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const size_t base = (size_t)row * DV + (size_t)lane * PER;
    float ov[PER], gv[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        if (BF16) {
            ov[i] = bf16_to_f(reinterpret_cast<const uint16_t*>(o)[base + i]);
            gv[i] = bf16_to_f(reinterpret_cast<const uint16_t*>(g_in)[base + i]);
        } else {
            ov[i] = reinterpret_cast<const float*>(o)[base + i];
            gv[i] = reinterpret_cast<const float*>(g_in)[base + i];
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) ss += ov[i] * ov[i];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss * (1.0f / DV) + eps);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const float wn = w ? w[lane * PER + i] : 1.0f;
        const float val = sigmoidf_fast(gv[i]) * wn * ov[i] * r;
        if (BF16) reinterpret_cast<uint16_t*>(y)[base + i] = f_to_bf16(val);
        else reinterpret_cast<float*>(y)[base + i] = val;
    }
}

template <int DV>
static cudaError_t launch_gn(const void* o, const void* g, const float* w, float eps, void* y,
                             long rows, bool bf16, cudaStream_t s) {
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    count_launches(1);
    if (bf16) gate_norm_kernel<DV, true><<<blocks, 256, 0, s>>>(o, g, w, eps, y, rows);
    else gate_norm_kernel<DV, false><<<blocks, 256, 0, s>>>(o, g, w, eps, y, rows);
    return cudaGetLastError();
}

cudaError_t launch_gate_norm(const void* o, const void* g, const float* w, float eps, void* y,
                             long rows, int dv, bool bf16, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    switch (dv) {
        case 32: return launch_gn<32>(o, g, w, eps, y, rows, bf16, s);
        case 64: return launch_gn<64>(o, g, w, eps, y, rows, bf16, s);
        case 128: return launch_gn<128>(o, g, w, eps, y, rows, bf16, s);
        case 256: return launch_gn<256>(o, g, w, eps, y, rows, bf16, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kda
