// gdn_device.cuh -- device helpers shared by the forward kernels: bf16 packing, the per-token
// gate and beta transforms, state stores and cu_seqlens reads.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"

namespace la {

__device__ __forceinline__ uint32_t pack_bf16(float x0, float x1) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    return *reinterpret_cast<uint32_t*>(&h);
}
// Eight consecutive floats of a 16-byte-aligned shared array, as two vector loads.
__device__ __forceinline__ void ld8(float* dst, const float* src) {
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 b = *reinterpret_cast<const float4*>(src + 4);
    dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
    dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f_to_bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Per-token gate and beta as the recurrence uses them: the natural-log decay and beta in
// [0, 1], after the optional input transforms (cudnn-frontend PR #616, in-kernel fusions):
// softplus gate -exp(a_log) softplus(g + dt_bias) (gA = -exp(a_log[h]), gdt = dt_bias[h]),
// bounded gate lower_bound * sigmoid(g), beta = sigmoid(beta) from bf16 or fp32 logits.
__device__ __forceinline__ float gate_at(const ChunkArgs& a, int64_t t, int h, float gA, float gdt) {
    const float x = a.g[t * a.g_st + h * a.g_sh];
    if (a.gate_mode == LA_GATE_SOFTPLUS) {
        const float z = x + gdt;
        return gA * (z > 20.f ? z : log1pf(expf(z)));
    }
    if (a.gate_mode == LA_GATE_SIGMOID_BOUND) return a.gate_lb / (1.f + expf(-x));
    return x;
}
// The log decay of update row r: on the update timeline of Gated DeltaProduct (gdp_n > 1 rows
// per token) a token's gate enters at its first update and the others carry no decay.
template <bool kGdp>
__device__ __forceinline__ float gate_row(const ChunkArgs& a, int64_t r, int h, float gA, float gdt) {
    if (kGdp) return (r % a.gdp_n == 0) ? gate_at(a, r / a.gdp_n, h, gA, gdt) : 0.f;
    return gate_at(a, r, h, gA, gdt);
}
__device__ __forceinline__ float beta_at(const ChunkArgs& a, int64_t t, int h) {
    const int64_t i = t * a.b_st + h * a.b_sh;
    const float x = a.beta_bf16 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(a.beta)[i]) << 16)
                                : a.beta[i];
    return a.beta_sigmoid ? 1.f / (1.f + expf(-x)) : x;
}

// One element of the end state: fp32, or bf16 when it goes back into a bf16 state pool.
__device__ __forceinline__ void store_state(const ChunkArgs& a, int64_t i, float x) {
    if (a.final_bf16) reinterpret_cast<uint16_t*>(a.final_state)[i] = f_to_bf16_bits(x);
    else a.final_state[i] = x;
}

__device__ __forceinline__ int64_t cu_get(const void* cu, int cu64, int64_t i) {
    return cu64 ? static_cast<const int64_t*>(cu)[i] : static_cast<int64_t>(static_cast<const int32_t*>(cu)[i]);
}

// Stores 8 floats as bf16 (hi part) and, if lo != nullptr, the bf16 residual (lo part).
__device__ __forceinline__ void store8_split(uint8_t* hi, uint8_t* lo, const float* x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        h[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
        if (lo) l[e] = pack_bf16(x[2 * e] - bf16_lo(h[e]), x[2 * e + 1] - bf16_hi(h[e]));
    }
    *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
    if (lo) *reinterpret_cast<uint4*>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

}  // namespace la
