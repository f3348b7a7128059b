// KDA context parallelism (KCP) combine step ("Kimi K3: KDA, attention
// residuals and Stable LatentMoE", Sec. 10.2): a segment of tokens acts on the
// state as S_exit = M S_entry + S~, M the product of the per-token transitions
// (I - beta k k^T) Diag(alpha) and S~ the segment's state from zero.  A rank
// recovers its entry state by applying the earlier segments' pairs in order,
// S <- M_j S + S~_j, and pairs compose as (M2, S2) o (M1, S1) = (M2 M1, S2 + M2 S1).
//
// kcp_apply: per head, X <- M X + Add (M d x d, X and Add d x n), FP32 with a
// fixed summation order.  Off the hot path (P - 1 small products per rank), so
// CUDA cores: one CTA per (32-column tile, head) copies its X tile to shared
// memory and each thread forms 16 outputs of one row.
#include "kda_common.cuh"

namespace kda {
namespace kcp {

constexpr int NT = 256;
constexpr int TILE = 32;    // columns of X per CTA

__global__ void __launch_bounds__(NT) apply_kernel(const float* __restrict__ M, float* X, const float* Add,
                                                   int d, int n) {
    extern __shared__ float sX[];                 // [d][TILE]
    const int h = blockIdx.y, c0 = blockIdx.x * TILE;
    const float* Mh = M + (size_t)h * d * d;
    float* Xh = X + (size_t)h * d * n;
    for (int e = threadIdx.x; e < d * TILE; e += NT) {
        const int r = e / TILE, c = e % TILE;
        sX[e] = (c0 + c < n) ? Xh[(size_t)r * n + c0 + c] : 0.f;
    }
    __syncthreads();
    // thread -> (row, half of the tile): rows d / (NT / 2) per pass
    const int half = threadIdx.x & 1;
    for (int i = threadIdx.x >> 1; i < d; i += NT / 2) {
        float acc[TILE / 2];
#pragma unroll
        for (int c = 0; c < TILE / 2; ++c) acc[c] = 0.f;
        const float* mrow = Mh + (size_t)i * d;
        for (int kk = 0; kk < d; ++kk) {
            const float m = __ldg(mrow + kk);
            const float* xr = sX + kk * TILE + half * (TILE / 2);
#pragma unroll
            for (int c = 0; c < TILE / 2; ++c) acc[c] = fmaf(m, xr[c], acc[c]);
        }
#pragma unroll
        for (int c = 0; c < TILE / 2; ++c) {
            const int col = c0 + half * (TILE / 2) + c;
            if (col < n) {
                const size_t idx = (size_t)i * n + col;
                Xh[idx] = acc[c] + (Add ? Add[(size_t)h * d * n + idx] : 0.f);
            }
        }
    }
}

}  // namespace kcp

cudaError_t launch_kcp_apply(const float* M, float* X, const float* Add, int H, int d, int n, cudaStream_t s) {
    if (H == 0 || n == 0) return cudaSuccess;
    const dim3 grid((n + kcp::TILE - 1) / kcp::TILE, H);
    kcp::apply_kernel<<<grid, kcp::NT, (size_t)d * kcp::TILE * sizeof(float), s>>>(M, X, Add, d, n);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
