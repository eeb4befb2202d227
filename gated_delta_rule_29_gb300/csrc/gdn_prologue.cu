// gdn_prologue.cu -- device prologue of gdn_fwd / gdn_summary.
//
// One CTA, launched before the chunk kernel on the same stream:
//   * validates cu_seqlens (starts at 0, nondecreasing, ends at T) and writes the
//     status word (the chunk kernel does nothing when it is non-zero);
//   * resets the unit ticket of the persistent chunk kernel;
//   * computes each sequence's first checkpoint row, an exclusive prefix sum of
//     ceil(L_i / n) (entries are the states entering offsets 0, n, 2n, ... < L_i),
//     and for the two-pass forward each sequence's first chunk, the same sum with
//     n = 64;
//   * orders sequences longest-first (ties by index) so the persistent kernel
//     hands out the longest (sequence, head) units first.  The order only decides
//     which unit starts when, never how a unit is computed, so results stay
//     bitwise independent of the batch;
//   * records whether the sequences' chunk counts are close enough for the
//     forward's range launches to pay (the same bits either way).
#include "gdn_kernel.h"
#include "../../include/liblinattn.h"

namespace la {

__device__ __forceinline__ int64_t cu_at(const void* cu, int cu64, int i) {
    return cu64 ? static_cast<const int64_t*>(cu)[i] : static_cast<int64_t>(static_cast<const int32_t*>(cu)[i]);
}

// Exclusive block-wide scan of one int64 per thread; `total` receives the block sum.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* warp_sums, int64_t& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int64_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
        int64_t s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        if (lane < nw) warp_sums[lane] = s;
    }
    __syncthreads();
    const int64_t prefix = w > 0 ? warp_sums[w - 1] : 0;
    total = warp_sums[nw - 1];
    __syncthreads();
    return prefix + incl - v;
}

__global__ void __launch_bounds__(kPrologueThreads) gdn_prologue_kernel(PrologueArgs a) {
    extern __shared__ uint64_t skeys[];
    __shared__ int bad;
    __shared__ int64_t warp_sums[32];
    const int tid = threadIdx.x;
    const int N = a.N;
    if (tid == 0) {
        bad = 0;
        a.hdr->ticket = 0ull;
    }
    __syncthreads();
    for (int i = tid; i <= N; i += blockDim.x) {
        const int64_t c = cu_at(a.cu, a.cu64, i);
        if (i == 0 && c != 0) bad = 1;
        if (i == N && c != a.T) bad = 1;
        if (i < N && cu_at(a.cu, a.cu64, i + 1) < c) bad = 1;
    }
    __syncthreads();
    const int32_t status = bad ? LA_ERR_BAD_SEQLENS : LA_OK;
    if (tid == 0) {
        a.hdr->status = status;
        if (a.user_status) *a.user_status = status;
    }
    if (bad) return;

    if (a.ckpt_n > 0) {
        int64_t carry = 0;
        for (int base = 0; base < N; base += blockDim.x) {
            const int i = base + tid;
            int64_t rows = 0;
            if (i < N) {
                const int64_t L = cu_at(a.cu, a.cu64, i + 1) - cu_at(a.cu, a.cu64, i);
                rows = (L + a.ckpt_n - 1) / a.ckpt_n;
            }
            int64_t total;
            const int64_t ex = block_exclusive_scan(rows, warp_sums, total);
            if (i < N) a.ckpt_off[i] = carry + ex;
            carry += total;
        }
        if (tid == 0) a.hdr->ckpt_rows = static_cast<int32_t>(carry);
    }
    if (a.chunk_off) {
        // the two-pass schedule numbers the batch's chunks sequence by sequence (GDP's on the
        // update timeline, chunk_rows rows per token)
        int64_t carry = 0;
        for (int base = 0; base < N; base += blockDim.x) {
            const int i = base + tid;
            int64_t nch = 0;
            if (i < N) nch = ((cu_at(a.cu, a.cu64, i + 1) - cu_at(a.cu, a.cu64, i)) * a.chunk_rows + kChunk - 1) / kChunk;
            int64_t total;
            const int64_t ex = block_exclusive_scan(nch, warp_sums, total);
            if (i < N) a.chunk_off[i] = carry + ex;
            carry += total;
        }
        if (tid == 0) {
            a.chunk_off[N] = carry;
            a.hdr->total_chunks = carry;
            a.hdr->wy_ticket = 0ull;
        }
    }

    const uint32_t P = next_pow2(static_cast<uint32_t>(N > 0 ? N : 1));
    volatile uint64_t* keys = P <= kSmemSortMax ? skeys : a.keys;
    for (uint32_t i = tid; i < P; i += blockDim.x) {
        uint64_t key = ~0ull;
        if (i < static_cast<uint32_t>(N)) {
            const int64_t L = cu_at(a.cu, a.cu64, i + 1) - cu_at(a.cu, a.cu64, i);
            const uint64_t chunks = static_cast<uint64_t>((L + kChunk - 1) / kChunk);
            key = ((0xFFFFFFFFull - (chunks & 0xFFFFFFFFull)) << 32) | i;
        }
        keys[i] = key;
    }
    __syncthreads();
    for (uint32_t k = 2; k <= P; k <<= 1) {
        for (uint32_t j = k >> 1; j > 0; j >>= 1) {
            for (uint32_t i = tid; i < P; i += blockDim.x) {
                const uint32_t ixj = i ^ j;
                if (ixj > i) {
                    const bool up = (i & k) == 0;
                    const uint64_t x = keys[i], y = keys[ixj];
                    if ((x > y) == up) {
                        keys[i] = y;
                        keys[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < N; i += blockDim.x) a.order[i] = static_cast<int32_t>(keys[i] & 0xFFFFFFFFull);
    if (tid == 0) {
        // the forward's chunk ranges are cut at the longest range of each wave: they pay only
        // when the sequences' chunk counts are within 1/8 of each other
        const uint64_t cmax = N > 0 ? 0xFFFFFFFFull - (keys[0] >> 32) : 0;
        const uint64_t cmin = N > 0 ? 0xFFFFFFFFull - (keys[N - 1] >> 32) : 0;
        a.hdr->ranges_ok = (N > 0 && cmin * 8 >= cmax * 7) ? 1 : 0;
    }
    if (a.chunk_off && N > 0) {
        // chunk_seq[g] = the sequence whose chunks include g: the last i with chunk_off[i] <= g
        // (empty sequences share their successor's offset), by binary search over the offsets,
        // staged in the sort keys' shared memory when they fit
        __syncthreads();
        const int64_t* off = a.chunk_off;
        if (P <= kSmemSortMax) {
            int64_t* soff = reinterpret_cast<int64_t*>(skeys);
            for (int i = tid; i < N; i += blockDim.x) soff[i] = a.chunk_off[i];
            __syncthreads();
            off = soff;
        }
        const int64_t total = a.chunk_off[N];
        for (int64_t gch = tid; gch < total; gch += blockDim.x) {
            int lo = 0, hi = N - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (off[mid] <= gch) lo = mid;
                else hi = mid - 1;
            }
            a.chunk_seq[gch] = lo;
        }
    }
}

cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t s) {
    const uint32_t P = next_pow2(static_cast<uint32_t>(a.N > 0 ? a.N : 1));
    const size_t smem = P <= kSmemSortMax ? P * sizeof(uint64_t) : 0;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(gdn_prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemSortMax * sizeof(uint64_t)));
        if (e != cudaSuccess) return e;
    }
    gdn_prologue_kernel<<<1, kPrologueThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace la
