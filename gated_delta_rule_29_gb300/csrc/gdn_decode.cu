// gdn_decode.cu -- one Gated DeltaNet recurrence step per sequence against a state pool.
//
// Method (cuDNN Linear Attention page: the GDN recurrence, and "States and checkpoints":
// state_indices turns the initial state into a pool addressed per sequence and written back
// in place).  For a sequence with one new token, head h, S = pool[slot, h] (K x V):
//
//   a = exp(g),  x = a S^T k_hat,  u = beta (v - x),  S' = a S + k_hat u^T,
//   o = scale S'^T q_hat = scale (a S^T q_hat + u (k_hat . q_hat))
//
// which is S' = exp(g)(I - beta k_hat k_hat^T) S + beta k_hat v^T expanded so that S is read
// once and written once.  The step is bound by those two passes over the state (HBM), so
// the kernel is shaped for memory-level parallelism: one CTA per (sequence, head), every
// thread owning a 4-column strip of a band of rows, all its state loads issued before any
// arithmetic, the state kept in registers between the read and the write.
#include <cuda_bf16.h>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"

namespace la {
namespace {

constexpr int kDecThreads = 128;

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f2bf(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Sum over the CTA of three values; every thread gets the totals.
__device__ __forceinline__ void block_sum3(float& a, float& b, float& c, float (*red)[3]) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
        c += __shfl_xor_sync(0xffffffffu, c, off);
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[w][0] = a;
        red[w][1] = b;
        red[w][2] = c;
    }
    __syncthreads();
    a = b = c = 0.f;
#pragma unroll
    for (int i = 0; i < kDecThreads / 32; ++i) {
        a += red[i][0];
        b += red[i][1];
        c += red[i][2];
    }
}

template <int KD, int VD>
__global__ void __launch_bounds__(kDecThreads) gdn_decode_kernel(const DecodeArgs a) {
    constexpr int NC = VD / 4;              // threads across the columns (4 columns each)
    constexpr int NG = kDecThreads / NC;    // row bands
    constexpr int RPT = KD / NG;            // rows per thread
    __shared__ float kh[KD], qh[KD];
    __shared__ float red[kDecThreads / 32][3];
    __shared__ float px[NG][VD], pq[NG][VD];
    __shared__ float us[VD];

    const int tid = threadIdx.x;
    const int cg = tid % NC, rg = tid / NC;
    const int i = blockIdx.x / a.HV, h = blockIdx.x % a.HV;
    const int hk = h / a.group;
    int64_t slot = i;
    if (a.idx) {
        slot = a.idx[i];
        if (slot < 0 || slot >= a.pool_size) {
            if (tid == 0 && a.status) atomicCAS(a.status, LA_OK, LA_ERR_BAD_STATE_INDEX);
            return;
        }
    }
    const int64_t sbase = (slot * a.HV + h) * static_cast<int64_t>(KD) * VD + 4 * cg;
    const int r0 = rg * RPT;

    // the state band: every load in flight before anything waits on one
    float4 s[RPT];
    if (a.pool_bf16) {
        const uint16_t* P = static_cast<const uint16_t*>(a.pool);
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const uint2 w = *reinterpret_cast<const uint2*>(P + sbase + static_cast<int64_t>(r0 + j) * VD);
            s[j] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                               __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
        }
    } else {
        const float* P = static_cast<const float*>(a.pool);
#pragma unroll
        for (int j = 0; j < RPT; ++j) s[j] = *reinterpret_cast<const float4*>(P + sbase + static_cast<int64_t>(r0 + j) * VD);
    }

    // k, q, norms, gate and beta while the state loads are in flight
    float kv = 0.f, qv = 0.f;
    if (tid < KD) {
        kv = bf16f(a.k[i * a.k_sn + hk * a.k_sh + tid]);
        qv = bf16f(a.q[i * a.q_sn + hk * a.q_sh + tid]);
    }
    float ssk = kv * kv, ssq = qv * qv, kq = kv * qv;
    block_sum3(ssk, ssq, kq, red);
    const float rk = a.l2norm ? 1.0f / sqrtf(ssk + 1e-6f) : 1.f;
    const float rq = a.l2norm ? 1.0f / sqrtf(ssq + 1e-6f) : 1.f;
    if (tid < KD) {
        kh[tid] = kv * rk;
        qh[tid] = qv * rq;
    }
    float gl = a.g[i * a.g_sn + h * a.g_sh];
    if (a.gate_mode == LA_GATE_SOFTPLUS) {
        const float z = gl + a.dt_bias[h];
        gl = -expf(a.a_log[h]) * (z > 20.f ? z : log1pf(expf(z)));
    } else if (a.gate_mode == LA_GATE_SIGMOID_BOUND) {
        gl = a.gate_lb / (1.f + expf(-gl));
    }
    const float decay = expf(gl);
    const int64_t bi = i * a.b_sn + h * a.b_sh;
    float beta = a.beta_bf16 ? bf16f(static_cast<const uint16_t*>(a.beta)[bi]) : static_cast<const float*>(a.beta)[bi];
    if (a.beta_sigmoid) beta = 1.f / (1.f + expf(-beta));
    const float kdotq = kq * rk * rq;
    __syncthreads();

    // partial S^T k_hat and S^T q_hat over this thread's rows
    float4 ax = make_float4(0.f, 0.f, 0.f, 0.f), aq = ax;
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const float kr = kh[r0 + j], qr = qh[r0 + j];
        ax.x = fmaf(s[j].x, kr, ax.x); ax.y = fmaf(s[j].y, kr, ax.y);
        ax.z = fmaf(s[j].z, kr, ax.z); ax.w = fmaf(s[j].w, kr, ax.w);
        aq.x = fmaf(s[j].x, qr, aq.x); aq.y = fmaf(s[j].y, qr, aq.y);
        aq.z = fmaf(s[j].z, qr, aq.z); aq.w = fmaf(s[j].w, qr, aq.w);
    }
    *reinterpret_cast<float4*>(&px[rg][4 * cg]) = ax;
    *reinterpret_cast<float4*>(&pq[rg][4 * cg]) = aq;
    __syncthreads();
    if (tid < VD) {
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            x += px[gi][tid];
            y += pq[gi][tid];
        }
        const float vv = bf16f(a.v[i * a.v_sn + h * a.v_sh + tid]);
        const float u = beta * (vv - decay * x);
        us[tid] = u;
        a.o[i * a.o_sn + h * a.o_sh + tid] = f2bf(a.scale * (decay * y + u * kdotq));
    }
    __syncthreads();

    // S' = a S + k_hat u^T, back into the same slot
    const float4 u4 = *reinterpret_cast<const float4*>(&us[4 * cg]);
    if (a.pool_bf16) {
        uint16_t* P = static_cast<uint16_t*>(a.pool);
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const float kr = kh[r0 + j];
            const float4 n = make_float4(fmaf(decay, s[j].x, kr * u4.x), fmaf(decay, s[j].y, kr * u4.y),
                                         fmaf(decay, s[j].z, kr * u4.z), fmaf(decay, s[j].w, kr * u4.w));
            uint2 w;
            w.x = static_cast<uint32_t>(f2bf(n.x)) | (static_cast<uint32_t>(f2bf(n.y)) << 16);
            w.y = static_cast<uint32_t>(f2bf(n.z)) | (static_cast<uint32_t>(f2bf(n.w)) << 16);
            *reinterpret_cast<uint2*>(P + sbase + static_cast<int64_t>(r0 + j) * VD) = w;
        }
    } else {
        float* P = static_cast<float*>(a.pool);
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const float kr = kh[r0 + j];
            *reinterpret_cast<float4*>(P + sbase + static_cast<int64_t>(r0 + j) * VD) =
                make_float4(fmaf(decay, s[j].x, kr * u4.x), fmaf(decay, s[j].y, kr * u4.y),
                            fmaf(decay, s[j].z, kr * u4.z), fmaf(decay, s[j].w, kr * u4.w));
        }
    }
}

template <int KD, int VD>
cudaError_t launch_decode_kv(const DecodeArgs& a, cudaStream_t s) {
    const int64_t grid = static_cast<int64_t>(a.N) * a.HV;
    if (grid == 0) return cudaSuccess;
    gdn_decode_kernel<KD, VD><<<static_cast<unsigned>(grid), kDecThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    if (a.K == 128) return a.V == 128 ? launch_decode_kv<128, 128>(a, s) : launch_decode_kv<128, 64>(a, s);
    return a.V == 128 ? launch_decode_kv<64, 128>(a, s) : launch_decode_kv<64, 64>(a, s);
}

}  // namespace la
