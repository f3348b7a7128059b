// Device helpers shared by the KDA kernels (decay gate, bf16 I/O, reductions).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"   // include/ is on the include path

#define KDA_DEV __device__ __forceinline__

namespace kda {

// launch accounting (api.cu): every launch wrapper reports the kernels it enqueued
void count_launches(int n);
// poll bound of the prefill kernels' waits on local copies and MMAs (api.cu;
// kda_debug_set_wait_limit)
uint32_t wait_limit();
kda_status cuda_failure(cudaError_t e);   // records the CUDA error string, returns KDA_ERR_CUDA

// Logistic function through the hardware exp2 / fast-divide path.
KDA_DEV float sigmoidf_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// Bounded decay gate ("Kimi K3" page, Sec. 2.2): log-retention
//   g = g_min * Sigmoid(exp(A_h) * z), g in (g_min, 0).
// eA is exp(A_h), computed once per head.
KDA_DEV float log_decay(float z, float eA, float g_min) { return g_min * sigmoidf_fast(eA * z); }

// Kimi Linear's gate, the one K3's replaces (same page, Sec. 2.2):
//   g = -exp(A_h) * Softplus(z), Softplus(x) = log(1 + e^x), unbounded below.
KDA_DEV float log_decay_softplus(float z, float eA) {
    return -eA * (fmaxf(z, 0.f) + log1pf(__expf(-fabsf(z))));
}
// gate_mode 0: bounded (K3), 1: softplus (Kimi Linear)
KDA_DEV float log_decay_mode(float z, float eA, float g_min, int gate_mode) {
    return gate_mode ? log_decay_softplus(z, eA) : log_decay(z, eA, g_min);
}

KDA_DEV float bf16_to_f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// round-to-nearest-even float -> bf16 bits (finite inputs)
KDA_DEV uint16_t f_to_bf16(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// First prefix-cache snapshot row of sequence n: the whole snapshot intervals in
// the sequences before it.  Called by every lane of a warp; all get the value.
KDA_DEV long snapshot_row_base(const int* cu_seqlens, int n, int interval) {
    long s = 0;
    for (int m = threadIdx.x & 31; m < n; m += 32) s += (cu_seqlens[m + 1] - cu_seqlens[m]) / interval;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

KDA_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Load 8 consecutive bf16 (16 bytes) as floats.
KDA_DEV void load8_bf16(const uint16_t* p, float* out) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

KDA_DEV void store8_bf16(uint16_t* p, const float* in) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // one round-to-nearest-even conversion per pair, in[2i] in the low half
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Streaming (read-once / write-once) 128-bit accesses for large state tensors.
KDA_DEV float4 ld_stream_f4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
KDA_DEV void st_stream_f4(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

// 32 bytes (8 floats) per thread in one access, a whole 32-B sector per lane when
// lanes touch different rows; p must be 32-byte aligned.
KDA_DEV void st_stream_f8(float* p, const float* v) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}
KDA_DEV void ld_nc_f8(const float* p, float* v) {
    asm("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                 : "l"(p));
}

}  // namespace kda
