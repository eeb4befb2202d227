// gdn_gdp.cu -- Gated DeltaProduct (several delta updates per token) on the update timeline.
//
// Method (cuDNN Linear Attention page: GDP runs on two timelines, q and g with one row per
// token, k, v and beta with n rows per token, update-major; num_householder == 1 is GDN).
// Per token t the state decays once, takes the token's n delta updates in order, and the
// output reads the state after the last one.  That is the GDN recurrence on the update
// timeline (T * n steps) with the log decay g_t at each token's first update and 0 at the
// others, and the query at each token's last update.  The chunk kernel walks that timeline
// natively for n <= 64; for larger n these kernels build it (query rows, gate rows, sequence
// boundaries) so the plain forward runs it unchanged, and gather the per-token outputs
// afterwards.
#include <cuda_bf16.h>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"

namespace la {
namespace {

__global__ void gdp_expand_kernel(const GdpArgs a) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int n = a.n;
    // query rows: row t * n + n - 1 is q[t]; the other rows are zero (16-byte pieces of 8 bf16)
    const int chunks = a.K / 8;
    const int64_t qtotal = a.T * n * a.HK * chunks;
    for (int64_t e = t0; e < qtotal; e += stride) {
        const int c8 = static_cast<int>(e % chunks);
        const int64_t rh = e / chunks;
        const int hk = static_cast<int>(rh % a.HK);
        const int64_t r = rh / a.HK;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (r % n == n - 1) w = *reinterpret_cast<const uint4*>(a.q + (r / n) * a.q_st + hk * a.q_sh + 8 * c8);
        *reinterpret_cast<uint4*>(a.qe + (r * a.HK + hk) * a.K + 8 * c8) = w;
    }
    // gate rows: the token's log decay at its first update (after the optional transform)
    const int64_t gtotal = a.T * n * a.HO;
    for (int64_t e = t0; e < gtotal; e += stride) {
        const int h = static_cast<int>(e % a.HO);
        const int64_t r = e / a.HO;
        float gl = 0.f;
        if (r % n == 0) {
            gl = a.g[(r / n) * a.g_st + h * a.g_sh];
            if (a.gate_mode == LA_GATE_SOFTPLUS) {
                const float z = gl + a.dt_bias[h];
                gl = -expf(a.a_log[h]) * (z > 20.f ? z : log1pf(expf(z)));
            } else if (a.gate_mode == LA_GATE_SIGMOID_BOUND) {
                gl = a.gate_lb / (1.f + expf(-gl));
            }
        }
        a.ge[e] = gl;
    }
    // sequence boundaries on the update timeline
    for (int64_t e = t0; e <= a.N; e += stride) {
        const int64_t c = a.cu64 ? static_cast<const int64_t*>(a.cu)[e] : static_cast<const int32_t*>(a.cu)[e];
        a.cue[e] = c * n;
    }
}

__global__ void gdp_gather_kernel(const GdpArgs a) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t total = a.T * a.HO * a.V;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total; e += stride) {
        const int v = static_cast<int>(e % a.V);
        const int64_t th = e / a.V;
        const int h = static_cast<int>(th % a.HO);
        const int64_t t = th / a.HO;
        a.o[t * a.o_st + h * a.o_sh + v] = a.oe[((t * a.n + a.n - 1) * a.HO + h) * a.V + v];
    }
}

}  // namespace

cudaError_t launch_gdp_expand(const GdpArgs& a, cudaStream_t s) {
    gdp_expand_kernel<<<1216, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gdp_gather(const GdpArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    gdp_gather_kernel<<<1216, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace la
