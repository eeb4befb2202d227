// gdn_ckpt.cu -- checkpoint rows for the backward (cuDNN Linear Attention page, "States and
// checkpoints": the backward reuses rows at the chunk cadence and regenerates the dense series
// from any other rows).
//
// gdn_ckpt_widen_kernel: bf16 rows at the chunk cadence -> fp32 (the backward's operand).
// gdn_ckpt_segments_kernel: for rows every n > 64 tokens, the pseudo-sequences that cut every
// sequence at multiples of n, and their start states (the given rows).  A forward launch over
// them with fp32 checkpoints every 64 tokens then writes the states entering every chunk in the
// order the backward reads them: segment j of sequence i owns the rows of offsets j n, j n + 64,
// ... (n is a multiple of 64), and the segments of a sequence are consecutive.
#include <cuda_bf16.h>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"

namespace la {

__device__ __forceinline__ float ckpt_elem(const CkptArgs& a, int64_t i) {
    return a.src_bf16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(a.src)[i]) << 16)
                      : static_cast<const float*>(a.src)[i];
}

__global__ void gdn_ckpt_widen_kernel(const CkptArgs a) {
    if (a.hdr->status != LA_OK) return;
    int64_t rows = a.hdr->ckpt_rows;
    if (rows > a.max_rows) rows = a.max_rows;
    const int64_t n = rows * a.row_elems;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        a.dst[i] = ckpt_elem(a, i);
}

__global__ void gdn_ckpt_segments_kernel(const CkptArgs a) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool ok = a.hdr->status == LA_OK;
    int64_t rows = ok ? a.hdr->ckpt_rows : 0;
    if (rows > a.max_seg) rows = a.max_seg;
    // boundaries: sequence i's segments are pseudo-sequences ckpt_off_n[i] .. + ceil(L_i / n) - 1
    for (int64_t i = tid; i < (ok ? a.N : 0); i += stride) {
        const int64_t c0 = a.cu64 ? static_cast<const int64_t*>(a.cu)[i] : static_cast<const int32_t*>(a.cu)[i];
        const int64_t c1 = a.cu64 ? static_cast<const int64_t*>(a.cu)[i + 1] : static_cast<const int32_t*>(a.cu)[i + 1];
        const int64_t segs = (c1 - c0 + a.n - 1) / a.n;
        const int64_t base = a.ckpt_off_n[i];
        for (int64_t j = 0; j < segs && base + j < a.max_seg; ++j) a.cu_seg[base + j] = c0 + j * a.n;
    }
    // the closing boundary and the empty pseudo-sequences after the last segment (all of them,
    // with boundary 0, when the batch's cu_seqlens were rejected: nothing then runs)
    for (int64_t k = rows + tid; k <= a.max_seg; k += stride) a.cu_seg[k] = ok ? a.T : 0;
    // start states: the given rows, zero for the empty pseudo-sequences
    const int64_t total = (a.max_seg) * a.row_elems;
    const int64_t given = rows * a.row_elems;
    for (int64_t e = tid; e < total; e += stride) a.s0_seg[e] = e < given ? ckpt_elem(a, e) : 0.f;
}

cudaError_t launch_ckpt_widen(const CkptArgs& a, cudaStream_t s) {
    gdn_ckpt_widen_kernel<<<1024, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_ckpt_segments(const CkptArgs& a, cudaStream_t s) {
    gdn_ckpt_segments_kernel<<<1024, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace la
