// gdn_chunk.cu -- the fused, persistent chunked Gated DeltaNet kernel for sm_103a.
//
// Method (cuDNN Linear Attention page: the GDN recurrence; chunked form of the
// delta rule with 64-token chunks restarting at each sequence start).  Within a
// chunk, with b_i the inclusive cumulative sum of g_j * log2(e), gamma_i = 2^{b_i},
// rk/rq the per-row inverse L2 norms and S0 the state entering the chunk:
//
//   A  = strict_tril( beta_i rk_i rk_j (k_i . k_j) 2^{b_i - b_j} )        (64 x 64)
//   T  = (I + A)^{-1}                                   forward substitution, fp32
//   X  = beta (.) V - (beta gamma rk) (.) (K S0)                          (64 x V)
//   D  = T X                                                   (the delta rows)
//   O  = (scale rq gamma) (.) (Q S0) + P D,
//        P = tril_incl( scale rq_i rk_j (q_i . k_j) 2^{b_i - b_j} )
//   S1 = 2^{b_C} S0 + K^T ( (2^{b_C - b_j} rk_j) (.) D )
//
// which equals the token-by-token recurrence exactly (up to rounding order).
//
// Mapping.  One CTA (256 threads) per SM walks a ticket-ordered list of units
// (sequence, head, tile).  Every product runs on the 5th-generation tensor cores
// (tcgen05.mma kind::f16, bf16 operands, fp32 accumulators in TMEM, M = 128) in
// transposed form so that M is the value dimension (padded to 128) or the
// stacked [K; Q] token rows.  q/k/v tiles arrive by TMA (128-byte swizzle,
// double buffered).  The state S stays in fp32 registers: thread (r, hf) holds
// column v = r of S for half hf of the k rows.  X and the decayed delta rows
// are split into bf16 hi + lo parts so the state update keeps ~16 bits.
//
// Tiles: a forward unit has one value tile.  A summary unit has a value tile
// (the span end state from the given start) and a transition tile: the same
// recurrence on P with v = 0 and P0 = I, stored transposed.  Summaries also
// split the state operand of K S into bf16 hi + lo: the transition's small
// off-diagonal entries need it to stay within the fp32-state tolerance.
#include <cuda_bf16.h>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"
#include "ptx.cuh"

namespace la {

// ------------------------------------------------------------------ shared memory map
constexpr uint32_t SM_KQ0 = 0;         // [region 0..1][128 rows: K 0-63, Q 64-127][128 B]
constexpr uint32_t SM_KQ1 = 32768;
constexpr uint32_t SM_V0 = 65536;      // [region 0..1][64 rows][128 B]
constexpr uint32_t SM_V1 = 81920;
constexpr uint32_t SM_WB = 98304;      // S^T bf16 [2][128][128 B] | X^T hi,lo | Ddec^T hi,lo
constexpr uint32_t SM_DT = 131072;     // A fp32 [64][64] during the solve | D^T bf16 [128][128 B]
constexpr uint32_t SM_TF = 147456;     // T fp32 [64][64]
constexpr uint32_t SM_PB = 163840;     // P bf16 [64][128 B]
constexpr uint32_t SM_TB = 172032;     // T bf16 [64][128 B]
constexpr uint32_t SM_SCAL = 180224;   // Scalars
constexpr uint32_t SM_SLO = 188416;    // summary only: S^T bf16 residual (lo part), same layout as WB
__host__ __device__ constexpr uint32_t smem_alloc(int mode) {
    return (mode == kModeSummary ? SM_SLO + 32768 : SM_SCAL + 8192) + 1024;
}

// TMEM columns (fp32 accumulators, 128 lanes)
constexpr uint32_t COL_G = 0;     // [K;Q] K^T            (64 columns)
constexpr uint32_t COL_D = 0;     // D^T                   (64)
constexpr uint32_t COL_SU = 0;    // K^T Ddec, transposed  (128)
constexpr uint32_t COL_KS = 128;  // (K S)^T               (64)
constexpr uint32_t COL_QS = 192;  // (Q' S)^T, then += D^T P^T = O^T
constexpr uint32_t TMEM_COLS = 256;

constexpr float kLog2e = 1.4426950408889634f;

struct Scalars {
    float b[64];    // chunk-local inclusive cumsum of g * log2(e)
    float bw[64];   // per-warp partial scans
    float rk[64];   // inverse key norms (0 on rows past the sequence end)
    float rq[64];   // inverse query norms
    float bet[64];  // beta (0 past the end)
    float sx[64];   // beta_j 2^{b_j} rk_j
    float sq[64];   // scale rq_i 2^{b_i}
    float sd[64];   // 2^{b_C - b_j} rk_j
    float red[256]; // norm partial sums
    float Y[768];   // solve scratch
    uint64_t tma_bar[2];
    uint64_t mma_bar;
    uint32_t tmem_base;
    int32_t unit_lo, unit_hi;
};
static_assert(sizeof(Scalars) <= 8192, "scalar area");

__device__ __forceinline__ int aidx(int i, int j) { return i * 64 + (j ^ (i & 31)); }

__device__ __forceinline__ uint32_t pack_bf16(float x0, float x1) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f_to_bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
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

// T = (I + A)^{-1} for strictly lower-triangular A (fp32, 64 x 64): 16 x 16 diagonal
// blocks by substitution, off-diagonal blocks by block forward substitution
//   T[bi][bj] = -T[bi][bi] * sum_{m=bj}^{bi-1} A[bi][m] T[m][bj].
// Writes T as bf16 (K-major, 128-byte swizzle) into tb.  All 256 threads.
__device__ void solve_unit_lower(const float* A, float* TF, float* Y, uint8_t* tb, int tid) {
    if (tid < 64) {
        const int o = 16 * (tid >> 4), c = tid & 15;
        float t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < i; ++j) acc = fmaf(-A[aidx(o + i, o + j)], t[j], acc);
            t[i] = acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) TF[aidx(o + i, o + c)] = t[i];
    }
    __syncthreads();
    for (int d = 1; d < 4; ++d) {
        const int ne = (4 - d) * 256;
        for (int e = tid; e < ne; e += kThreads) {
            const int p = e >> 8, i = (e >> 4) & 15, j = e & 15;
            const int rowA = 16 * (p + d) + i, colT = 16 * p + j;
            float acc = 0.f;
            for (int m = 16 * p; m < 16 * (p + d); ++m) acc = fmaf(A[aidx(rowA, m)], TF[aidx(m, colT)], acc);
            Y[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < ne; e += kThreads) {
            const int p = e >> 8, i = (e >> 4) & 15, j = e & 15;
            const int bi = 16 * (p + d);
            float acc = 0.f;
            for (int m = 0; m <= i; ++m) acc = fmaf(TF[aidx(bi + i, bi + m)], Y[(p << 8) + (m << 4) + j], acc);
            TF[aidx(bi + i, 16 * p + j)] = -acc;
        }
        __syncthreads();
    }
    {
        const int i = tid >> 2;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int jc = (tid & 3) * 2 + cc;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = jc * 8 + e;
                x[e] = (j <= i) ? TF[aidx(i, j)] : 0.f;
            }
            store8_split(tb + sw128_off(i, jc), nullptr, x);
        }
    }
}

template <int KD, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_chunk_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const ChunkArgs a) {
    constexpr int KH = KD / 2;  // state rows held per thread
    constexpr bool kFwd = MODE == kModeFwd;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Scalars& sc = *reinterpret_cast<Scalars*>(sm + SM_SCAL);
    float* Asm = reinterpret_cast<float*>(sm + SM_DT);
    float* TF = reinterpret_cast<float*>(sm + SM_TF);
    uint8_t* WB = sm + SM_WB;
    uint8_t* DT = sm + SM_DT;
    uint8_t* PB = sm + SM_PB;
    uint8_t* TB = sm + SM_TB;
    uint8_t* SLO = kFwd ? nullptr : sm + SM_SLO;

    const int tid = threadIdx.x;
    const int r = tid & 127;   // TMEM lane / value column / stacked token row
    const int hf = tid >> 7;   // column half
    const int HO = a.HV;

    if (*reinterpret_cast<volatile int32_t*>(&a.hdr->status) != LA_OK) return;

    if (tid < 32) {
        tmem_alloc(&sc.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sc.tma_bar[0], 1);
        mbar_init(&sc.tma_bar[1], 1);
        mbar_init(&sc.mma_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sc.tmem_base;
    const uint32_t trow = tmem + (static_cast<uint32_t>(r & ~31) << 16);

    uint32_t tma_phase = 0, mma_phase = 0;  // parity of the next wait per barrier
    uint32_t tma_pending = 0;               // stages with an issued, unconsumed load
    bool mma_pending = false;
    bool failed = false;
    const uint64_t budget = a.wait_budget_ns;
    const int64_t per_seq = static_cast<int64_t>(HO) * a.tiles_per_head;

    for (;;) {
        if (tid == 0) {
            const unsigned long long u = atomicAdd(reinterpret_cast<unsigned long long*>(&a.hdr->ticket), 1ull);
            sc.unit_lo = static_cast<int32_t>(u & 0xFFFFFFFFull);
            sc.unit_hi = static_cast<int32_t>(u >> 32);
        }
        __syncthreads();
        const int64_t unit = (static_cast<int64_t>(sc.unit_hi) << 32) | static_cast<uint32_t>(sc.unit_lo);
        __syncthreads();  // every thread has read the ticket before thread 0 may take the next one
        if (unit >= a.num_units) break;
        const int seq = a.order[unit / per_seq];
        const int rem = static_cast<int>(unit % per_seq);
        const int h = rem / a.tiles_per_head;
        const int tile = rem % a.tiles_per_head;
        const int hk = h / a.group;
        const bool value_tile = kFwd || tile == kTileValue;
        const int64_t ts = cu_get(a.cu, a.cu64, seq);
        const int64_t L = cu_get(a.cu, a.cu64, seq + 1) - ts;
        const int nchunks = static_cast<int>((L + kChunk - 1) / kChunk);
        const int64_t unit_state = (static_cast<int64_t>(seq) * HO + h);
        const uint32_t tile_bytes = (kFwd ? 2u : 1u) * KD * 128u + (value_tile ? static_cast<uint32_t>(a.V) * 128u : 0u);

        // ---- initial state: thread (r, hf) holds S[k][r], k = hf*KH + i
        float st[KH];
#pragma unroll
        for (int i = 0; i < KH; ++i) st[i] = 0.f;
        if (value_tile) {
            if (a.s0 && r < a.V) {
                const int64_t base = unit_state * KD * a.V + r;
#pragma unroll
                for (int i = 0; i < KH; ++i) {
                    const int64_t idx = base + static_cast<int64_t>(hf * KH + i) * a.V;
                    st[i] = a.s0_bf16 ? bf16_bits_to_f(static_cast<const uint16_t*>(a.s0)[idx])
                                      : static_cast<const float*>(a.s0)[idx];
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < KH; ++i) st[i] = (hf * KH + i == r) ? 1.f : 0.f;
        }
        // S^T bf16 -> WB (A operand of the K S / Q S products)
#pragma unroll
        for (int c8 = 0; c8 < KH / 8; ++c8) {
            const int kc = (hf * KH) / 8 + c8;  // 16-byte chunk index along k
            const uint32_t off = (kc >> 3) * 16384 + sw128_off(r, kc & 7);
            store8_split(WB + off, kFwd ? nullptr : SLO + off, &st[c8 * 8]);
        }

        // ---- first chunk's tiles and per-token scalars
        if (tid == 0 && nchunks > 0) {
            uint8_t* KQ = sm + SM_KQ0;
            mbar_arrive_expect_tx(&sc.tma_bar[0], tile_bytes);
#pragma unroll
            for (int rg = 0; rg < KD / 64; ++rg) {
                tma_load_3d(KQ + rg * 16384, &kmap, &sc.tma_bar[0], rg * 64, hk, static_cast<int>(ts));
                if (kFwd) tma_load_3d(KQ + rg * 16384 + 8192, &qmap, &sc.tma_bar[0], rg * 64, hk, static_cast<int>(ts));
            }
            if (value_tile)
                for (int rg = 0; rg < (a.V + 63) / 64; ++rg)
                    tma_load_3d(sm + SM_V0 + rg * 8192, &vmap, &sc.tma_bar[0], rg * 64, h, static_cast<int>(ts));
        }
        if (nchunks > 0) tma_pending |= 1u;
        float g_nx = 0.f, b_nx = 0.f;
        if (tid < 64 && tid < L) {
            g_nx = a.g[(ts + tid) * a.g_st + h * a.g_sh];
            b_nx = a.beta[(ts + tid) * a.b_st + h * a.b_sh];
        }

        for (int c = 0; c < nchunks; ++c) {
            const int64_t t0 = ts + static_cast<int64_t>(c) * kChunk;
            const int64_t left = L - static_cast<int64_t>(c) * kChunk;
            const int n = left < kChunk ? static_cast<int>(left) : kChunk;
            const int s = c & 1;
            uint8_t* KQ = sm + (s ? SM_KQ1 : SM_KQ0);
            uint8_t* VT = sm + (s ? SM_V1 : SM_V0);
            const float g_cur = g_nx, b_cur = b_nx;

            // prefetch chunk c+1 (tiles by TMA, scalars into registers)
            if (c + 1 < nchunks) {
                const int64_t t1 = t0 + kChunk;
                if (tid == 0) {
                    uint8_t* KQn = sm + (s ? SM_KQ0 : SM_KQ1);
                    uint8_t* VTn = sm + (s ? SM_V0 : SM_V1);
                    uint64_t* bar = &sc.tma_bar[s ^ 1];
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(bar, tile_bytes);
#pragma unroll
                    for (int rg = 0; rg < KD / 64; ++rg) {
                        tma_load_3d(KQn + rg * 16384, &kmap, bar, rg * 64, hk, static_cast<int>(t1));
                        if (kFwd) tma_load_3d(KQn + rg * 16384 + 8192, &qmap, bar, rg * 64, hk, static_cast<int>(t1));
                    }
                    if (value_tile)
                        for (int rg = 0; rg < (a.V + 63) / 64; ++rg)
                            tma_load_3d(VTn + rg * 8192, &vmap, bar, rg * 64, h, static_cast<int>(t1));
                }
                tma_pending |= 1u << (s ^ 1);
                g_nx = b_nx = 0.f;
                if (tid < 64 && static_cast<int64_t>(c + 1) * kChunk + tid < L) {
                    g_nx = a.g[(t1 + tid) * a.g_st + h * a.g_sh];
                    b_nx = a.beta[(t1 + tid) * a.b_st + h * a.b_sh];
                }
            }

            bool ok = mbar_wait(&sc.tma_bar[s], (tma_phase >> s) & 1u, budget);
            if (ok) {
                tma_phase ^= 1u << s;
                tma_pending &= ~(1u << s);
            }

            // ---- row norms (partial over a feature half) and the gate scan
            {
                float ss = 0.f;
                if (r < 64 || kFwd) {
#pragma unroll
                    for (int c8 = 0; c8 < KH / 8; ++c8) {
                        const int kc = (hf * KH) / 8 + c8;
                        const uint4 w = *reinterpret_cast<const uint4*>(KQ + (kc >> 3) * 16384 + sw128_off(r, kc & 7));
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = bf16_lo(ww[e]), x1 = bf16_hi(ww[e]);
                            ss = fmaf(x0, x0, fmaf(x1, x1, ss));
                        }
                    }
                }
                sc.red[tid] = ss;
                if (tid < 64) {
                    float x = (tid < n) ? g_cur * kLog2e : 0.f;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, x, off);
                        if ((tid & 31) >= off) x += y;
                    }
                    sc.bw[tid] = x;
                }
            }
            if (__syncthreads_or(!ok)) { failed = true; break; }
            if (tid < 64) {
                const int i = tid;
                const bool valid = i < n;
                float rk = 0.f, rq = 0.f;
                if (valid) {
                    rk = a.l2norm ? 1.0f / sqrtf(sc.red[i] + sc.red[128 + i] + 1e-6f) : 1.f;
                    rq = a.l2norm ? 1.0f / sqrtf(sc.red[64 + i] + sc.red[192 + i] + 1e-6f) : 1.f;
                }
                const float bi = sc.bw[i] + (i >= 32 ? sc.bw[31] : 0.f);
                const float bC = sc.bw[31] + sc.bw[63];
                const float bet = valid ? b_cur : 0.f;
                const float gam = exp2f(bi);
                sc.b[i] = bi;
                sc.rk[i] = rk;
                sc.rq[i] = rq;
                sc.bet[i] = bet;
                sc.sx[i] = bet * gam * rk;
                sc.sq[i] = a.scale * rq * gam;
                sc.sd[i] = exp2f(bC - bi) * rk;
            }
            __syncthreads();

            // ---- G = [K; Q] K^T  (M = 128 stacked rows, N = 64 key rows, contraction over K)
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
                const uint32_t kq = smem_u32(KQ);
#pragma unroll
                for (int kk = 0; kk < KD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    umma_bf16(tmem + COL_G, sdesc_sw128(kq + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024), idesc,
                              kk > 0);
                }
                umma_commit(&sc.mma_bar);
            }
            mma_pending = true;

            // checkpoint: the state entering this chunk, at token offsets that are multiples of n
            if (kFwd && a.ckpt && (static_cast<int64_t>(c) * kChunk) % a.ckpt_n == 0 && r < a.V) {
                const int64_t row = a.ckpt_off[seq] + static_cast<int64_t>(c) * kChunk / a.ckpt_n;
                const int64_t base = ((row * HO + h) * KD) * a.V + r;
#pragma unroll
                for (int i = 0; i < KH; ++i) {
                    const int64_t idx = base + static_cast<int64_t>(hf * KH + i) * a.V;
                    if (a.ckpt_bf16) static_cast<uint16_t*>(a.ckpt)[idx] = f_to_bf16_bits(st[i]);
                    else static_cast<float*>(a.ckpt)[idx] = st[i];
                }
            }

            ok = mbar_wait(&sc.mma_bar, mma_phase, budget);
            if (ok) {
                mma_phase ^= 1u;
                mma_pending = false;
            }
            tc_fence_after();
            {
                float gv[32];
                tmem_ld16(trow + COL_G + 32 * hf, *reinterpret_cast<float(*)[16]>(&gv[0]));
                tmem_ld16(trow + COL_G + 32 * hf + 16, *reinterpret_cast<float(*)[16]>(&gv[16]));
                tmem_wait_ld();
                if (r < 64) {
                    // A row i = r (strictly lower), fp32 for the solve
                    const int i = r;
                    const float ci = sc.bet[i] * sc.rk[i], bi = sc.b[i];
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int j = 32 * hf + jj;
                        Asm[aidx(i, j)] = (j < i) ? ci * sc.rk[j] * gv[jj] * exp2f(bi - sc.b[j]) : 0.f;
                    }
                } else if (kFwd) {
                    // P row i = r - 64 (lower incl. diagonal), bf16 K-major
                    const int i = r - 64;
                    const float ci = a.scale * sc.rq[i], bi = sc.b[i];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = 32 * hf + 8 * cc + e;
                            x[e] = (j <= i) ? ci * sc.rk[j] * gv[8 * cc + e] * exp2f(bi - sc.b[j]) : 0.f;
                        }
                        store8_split(PB + sw128_off(i, 4 * hf + cc), nullptr, x);
                    }
                }
            }
            if (kFwd) {
                // Q' = (scale rq gamma) (.) Q in place: the B rows 64-127 of the next product
                constexpr int kQChunks = 64 * (KD / 8);
                for (int e = tid; e < kQChunks; e += kThreads) {
                    const int row = e / (KD / 8), cc = e % (KD / 8);
                    uint4* p = reinterpret_cast<uint4*>(KQ + (cc >> 3) * 16384 + (64 + row) * 128 + (cc & 7) * 16);
                    const float f = sc.sq[row];
                    uint4 w = *p;
                    w.x = pack_bf16(bf16_lo(w.x) * f, bf16_hi(w.x) * f);
                    w.y = pack_bf16(bf16_lo(w.y) * f, bf16_hi(w.y) * f);
                    w.z = pack_bf16(bf16_lo(w.z) * f, bf16_hi(w.z) * f);
                    w.w = pack_bf16(bf16_lo(w.w) * f, bf16_hi(w.w) * f);
                    *p = w;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }

            // ---- (K S)^T and (Q' S)^T = S^T [K; Q']^T  (M = 128 value rows)
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, kFwd ? 128 : 64, false, false);
                const uint32_t wb = smem_u32(WB), kq = smem_u32(KQ);
#pragma unroll
                for (int kk = 0; kk < KD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    umma_bf16(tmem + COL_KS, sdesc_sw128(wb + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024), idesc,
                              kk > 0);
                }
                if (!kFwd) {
                    const uint32_t slo = smem_u32(SLO);
#pragma unroll
                    for (int kk = 0; kk < KD / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        umma_bf16(tmem + COL_KS, sdesc_sw128(slo + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024),
                                  idesc, 1u);
                    }
                }
                umma_commit(&sc.mma_bar);
            }
            mma_pending = true;

            // T = (I + A)^{-1} on the CUDA cores while the tensor cores run
            solve_unit_lower(Asm, TF, sc.Y, TB, tid);

            ok = mbar_wait(&sc.mma_bar, mma_phase, budget);
            if (ok) {
                mma_phase ^= 1u;
                mma_pending = false;
            }
            tc_fence_after();
            {
                // X^T[v][j] = beta_j V[j][v] - sx_j (K S)^T[v][j], split into bf16 hi + lo
                float ks[32];
                tmem_ld16(trow + COL_KS + 32 * hf, *reinterpret_cast<float(*)[16]>(&ks[0]));
                tmem_ld16(trow + COL_KS + 32 * hf + 16, *reinterpret_cast<float(*)[16]>(&ks[16]));
                tmem_wait_ld();
                const int v = r;
                const bool has_v = value_tile && v < a.V;
                const uint8_t* vcol = VT + (v >> 6) * 8192 + (v & 7) * 2;
                const uint32_t vchunk = (v & 63) >> 3;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 32 * hf + 8 * cc + e;
                        const float vv =
                            has_v ? bf16_bits_to_f(*reinterpret_cast<const uint16_t*>(vcol + sw128_off(j, vchunk))) : 0.f;
                        x[e] = sc.bet[j] * vv - sc.sx[j] * ks[8 * cc + e];
                    }
                    store8_split(WB + sw128_off(v, 4 * hf + cc), WB + 16384 + sw128_off(v, 4 * hf + cc), x);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }

            // ---- D^T = X^T T^T  (hi and lo parts accumulate; contraction over 64 tokens)
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
                const uint32_t wb = smem_u32(WB), tb = smem_u32(TB);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + COL_D, sdesc_sw128(wb + part * 16384 + kk * 32, 16, 1024),
                                  sdesc_sw128(tb + kk * 32, 16, 1024), idesc, (part | kk) != 0);
                umma_commit(&sc.mma_bar);
            }
            mma_pending = true;
            ok = mbar_wait(&sc.mma_bar, mma_phase, budget);
            if (ok) {
                mma_phase ^= 1u;
                mma_pending = false;
            }
            tc_fence_after();
            {
                float dd[32];
                tmem_ld16(trow + COL_D + 32 * hf, *reinterpret_cast<float(*)[16]>(&dd[0]));
                tmem_ld16(trow + COL_D + 32 * hf + 16, *reinterpret_cast<float(*)[16]>(&dd[16]));
                tmem_wait_ld();
                const int v = r;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = sc.sd[32 * hf + 8 * cc + e] * dd[8 * cc + e];
                    if (kFwd) store8_split(DT + sw128_off(v, 4 * hf + cc), nullptr, &dd[8 * cc]);
                    store8_split(WB + sw128_off(v, 4 * hf + cc), WB + 16384 + sw128_off(v, 4 * hf + cc), x);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }

            // ---- O^T += D^T P^T (fwd) and SU = Ddec^T K (state update, K read MN-major)
            if (tid == 0) {
                tc_fence_after();
                const uint32_t wb = smem_u32(WB), kq = smem_u32(KQ);
                if (kFwd) {
                    const uint32_t idesc_o = idesc_bf16_f32(128, 64, false, false);
                    const uint32_t dt = smem_u32(DT), pb = smem_u32(PB);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + COL_QS, sdesc_sw128(dt + kk * 32, 16, 1024), sdesc_sw128(pb + kk * 32, 16, 1024),
                                  idesc_o, 1u);
                }
                const uint32_t idesc_s = idesc_bf16_f32(128, KD, false, true);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + COL_SU, sdesc_sw128(wb + part * 16384 + kk * 32, 16, 1024),
                                  sdesc_sw128(kq + kk * 2048, 16384, 1024), idesc_s, (part | kk) != 0);
                umma_commit(&sc.mma_bar);
            }
            mma_pending = true;
            ok = mbar_wait(&sc.mma_bar, mma_phase, budget);
            if (ok) {
                mma_phase ^= 1u;
                mma_pending = false;
            }
            tc_fence_after();
            if (kFwd) {
                float ov[32];
                tmem_ld16(trow + COL_QS + 32 * hf, *reinterpret_cast<float(*)[16]>(&ov[0]));
                tmem_ld16(trow + COL_QS + 32 * hf + 16, *reinterpret_cast<float(*)[16]>(&ov[16]));
                tmem_wait_ld();
                if (r < a.V) {
                    uint16_t* op = a.o + (t0 + 32 * hf) * a.o_st + static_cast<int64_t>(h) * a.o_sh + r;
#pragma unroll
                    for (int ii = 0; ii < 32; ++ii)
                        if (32 * hf + ii < n) op[static_cast<int64_t>(ii) * a.o_st] = f_to_bf16_bits(ov[ii]);
                }
            }
            {
                const float gC = exp2f(sc.b[63]);
#pragma unroll
                for (int c16 = 0; c16 < KH / 16; ++c16) {
                    float su[16];
                    tmem_ld16(trow + COL_SU + hf * KH + 16 * c16, su);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) st[16 * c16 + e] = fmaf(gC, st[16 * c16 + e], su[e]);
                }
#pragma unroll
                for (int c8 = 0; c8 < KH / 8; ++c8) {
                    const int kc = (hf * KH) / 8 + c8;
                    const uint32_t off = (kc >> 3) * 16384 + sw128_off(r, kc & 7);
                    store8_split(WB + off, kFwd ? nullptr : SLO + off, &st[c8 * 8]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        if (failed) break;

        // ---- end of unit: final state / span end state / transition
        if (value_tile) {
            if (a.final_state && r < a.V) {
                float* fp = a.final_state + unit_state * KD * a.V + r;
#pragma unroll
                for (int i = 0; i < KH; ++i) fp[static_cast<int64_t>(hf * KH + i) * a.V] = st[i];
            }
        } else if (r < KD) {
            // transition[j][k] = P[k][j]: thread row r = j holds column j of P
            float* tp = a.transition + (unit_state * KD + r) * KD + hf * KH;
#pragma unroll
            for (int i = 0; i < KH; i += 4)
                *reinterpret_cast<float4*>(tp + i) = make_float4(st[i], st[i + 1], st[i + 2], st[i + 3]);
        }
    }

    if (failed) {
        // Let in-flight copies and products finish (bounded) before TMEM and shared memory go away.
        for (int s = 0; s < 2; ++s)
            if (tma_pending & (1u << s)) mbar_wait(&sc.tma_bar[s], (tma_phase >> s) & 1u, budget);
        if (mma_pending) mbar_wait(&sc.mma_bar, mma_phase, budget);
        if (tid == 0) {
            atomicCAS(&a.hdr->status, LA_OK, LA_ERR_TIMEOUT);
            if (a.user_status) atomicCAS(a.user_status, LA_OK, LA_ERR_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ host side
template <int KD, int MODE>
static cudaError_t launch_one(const ChunkArgs& a, const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                              int grid, cudaStream_t s) {
    auto* fn = gdn_chunk_kernel<KD, MODE>;
    constexpr uint32_t smem = smem_alloc(MODE);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, s>>>(qm, km, vm, a);
    return cudaGetLastError();
}

int chunk_kernel_grid(int device, int64_t num_units) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0) sms = 1;
    return static_cast<int>(num_units < sms ? num_units : sms);
}

cudaError_t launch_chunk_kernel(const ChunkArgs& a, const CUtensorMap& qm, const CUtensorMap& km,
                                const CUtensorMap& vm, int mode, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int grid = chunk_kernel_grid(dev, a.num_units);
    if (grid <= 0) return cudaSuccess;
    if (a.K == 128) return mode == kModeFwd ? launch_one<128, kModeFwd>(a, qm, km, vm, grid, s)
                                            : launch_one<128, kModeSummary>(a, qm, km, vm, grid, s);
    return mode == kModeFwd ? launch_one<64, kModeFwd>(a, qm, km, vm, grid, s)
                            : launch_one<64, kModeSummary>(a, qm, km, vm, grid, s);
}

}  // namespace la
