// gdn_compose.cu -- composition of span summaries (context parallelism over sequence spans).
//
// cuDNN Linear Attention page, "Summaries": a span's end state from a zero start and its
// transition compose across consecutive spans as S_final = S_init * transition + S_H; with the
// library's orientation (transition = P^T, states [K][V]) the state leaving span r is
//     S_{r+1}[b][v] = sum_a transition_r[a][b] S_r[a][v] + end_r[b][v].
// The backward moves a state gradient the other way: d_r[a][v] = term_r[a][v] +
// sum_b transition_r[a][b] d_{r+1}[b][v], term_r being span r's own entering-state gradient.
// One CTA of 256 threads per (head, 32 value columns) walks the spans in order (forward) or in
// reverse (backward) with the running state tile in shared memory; every output is a K-term
// fp32 dot product in ascending index order, so results do not depend on the launch shape.
#include "../../include/liblinattn.h"
#include "gdn_kernel.h"

namespace la {
namespace {

constexpr int kCT = 256;  // threads
constexpr int kVW = 32;   // value columns per CTA
constexpr int kKC = 32;   // transition rows (forward) or columns (backward) staged per step

template <int KD>
__global__ void __launch_bounds__(kCT) gdn_compose_kernel(ComposeArgs a) {
    __shared__ float Sx[KD][kVW];   // the running state (or gradient) tile
    __shared__ float Tc[KD][kKC + 1];  // a slice of the transition (padded against bank conflicts)
    const int tid = threadIdx.x;
    const int h = blockIdx.x;
    const int v0 = blockIdx.y * kVW;
    const int HO = a.HO, V = a.V;
    // thread t owns output row t / 2 (all KD rows: 256 threads x 16 = KD x 32 outputs for KD =
    // 128; for KD = 64 threads 128-255 own nothing) and columns (t & 1) * 16 .. + 15
    const int row = tid >> 1;
    const int c0 = (tid & 1) * 16;
    const bool owner = row < KD;
    const size_t kv = static_cast<size_t>(KD) * V;

    // the starting tile: `start` (the initial state, or the cotangent after the last span) or 0
    for (int e = tid; e < KD * kVW; e += kCT) {
        const int k = e / kVW, c = e % kVW;
        const int v = v0 + c;
        Sx[k][c] = (a.start && v < V) ? a.start[static_cast<size_t>(h) * kv + static_cast<size_t>(k) * V + v] : 0.f;
    }
    __syncthreads();
    auto store = [&](int slot) {
        if (!owner) return;
        float* o = a.out + (static_cast<size_t>(slot) * HO + h) * kv + static_cast<size_t>(row) * V;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (v0 + c0 + j < V) o[v0 + c0 + j] = Sx[row][c0 + j];
    };
    if (!a.backward) store(0);

    for (int step = 0; step < a.R; ++step) {
        const int r = a.backward ? a.R - 1 - step : step;
        if (a.backward) store(r);  // the gradient leaving span r
        const float* tr = a.transitions + (static_cast<size_t>(r) * HO + h) * KD * KD;
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
        for (int m0 = 0; m0 < KD; m0 += kKC) {
            // forward: rows m0 .. m0 + 31 of the transition (Tc[b][m] = tr[m0 + m][b]);
            // backward: its columns m0 .. m0 + 31 (Tc[a][m] = tr[a][m0 + m])
            for (int e = tid; e < KD * kKC; e += kCT) {
                if (a.backward) {
                    const int i = e / kKC, m = e % kKC;
                    Tc[i][m] = tr[static_cast<size_t>(i) * KD + m0 + m];
                } else {
                    const int m = e / KD, i = e % KD;
                    Tc[i][m] = tr[static_cast<size_t>(m0 + m) * KD + i];
                }
            }
            __syncthreads();
            if (owner) {
#pragma unroll 4
                for (int m = 0; m < kKC; ++m) {
                    const float t = Tc[row][m];
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = fmaf(t, Sx[m0 + m][c0 + j], acc[j]);
                }
            }
            __syncthreads();
        }
        if (owner) {
            const float* term = a.terms + (static_cast<size_t>(r) * HO + h) * kv + static_cast<size_t>(row) * V;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int v = v0 + c0 + j;
                Sx[row][c0 + j] = acc[j] + (v < V ? term[v] : 0.f);
            }
        }
        __syncthreads();
        if (!a.backward) store(r + 1);  // the state leaving span r
    }
    if (a.backward) store(a.R);  // the gradient entering span 0
}

}  // namespace

cudaError_t launch_compose(const ComposeArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.HO), static_cast<unsigned>((a.V + kVW - 1) / kVW));
    if (a.K == 128) gdn_compose_kernel<128><<<grid, kCT, 0, s>>>(a);
    else gdn_compose_kernel<64><<<grid, kCT, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace la
