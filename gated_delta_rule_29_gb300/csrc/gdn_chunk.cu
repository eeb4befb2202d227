// gdn_chunk.cu -- the fused, persistent chunked Gated DeltaNet kernel for sm_103a.
//
// Method (cuDNN Linear Attention page: the GDN recurrence; chunked form of the
// delta rule with 64-token chunks restarting at each sequence start).  Within a
// chunk, with b_i the inclusive cumulative sum of g_j * log2(e), gamma_i = 2^{b_i},
// rk/rq the per-row inverse L2 norms and S0 the state entering the chunk:
//
//   A  = strict_tril( beta_i rk_i rk_j (k_i . k_j) 2^{b_i - b_j} )        (64 x 64)
//   T  = (I + A)^{-1}                                      block substitution, fp32/tf32
//   X  = beta (.) V - (beta gamma rk) (.) (K S0)                          (64 x V)
//   D  = T X                                                   (the delta rows)
//   O  = (scale rq gamma) (.) (Q S0) + P D,
//        P = tril_incl( scale rq_i rk_j (q_i . k_j) 2^{b_i - b_j} )
//   S1 = 2^{b_C} S0 + K^T ( (2^{b_C - b_j} rk_j) (.) D )
//
// which equals the token-by-token recurrence exactly (up to rounding order).
//
// Mapping.  Persistent CTAs of 128 threads (two per SM) take units (sequence, head,
// tile) from a ticket.  Thread r owns TMEM lane r.  The state S lives in TMEM as
// fp32 S^T (lane = value column, column = k) and is updated in place by the
// tensor core.  Every product is a tcgen05.mma (kind::f16, bf16 operands, fp32
// accumulation, M = 128) in transposed form: M is the value dimension (padded to
// 128) or the stacked [K; Q] token rows.  q/k/v tiles arrive by TMA (128-byte
// swizzle).  X and the decayed delta rows are split into bf16 hi + lo parts so
// the state keeps ~16 bits per update; summaries also split the state operand of
// K S (the transition's small entries need it).  The 64 x 64 unit-lower-
// triangular inverse runs on the CUDA cores: 16 x 16 diagonal blocks by
// substitution, the off-diagonal blocks by tf32 warp MMAs.
//
// Tiles: a forward unit has one value tile.  A summary unit has a value tile
// (the span end state from the given start) and a transition tile: the same
// recurrence on P with v = 0 and P0 = I, stored transposed.  When the summary's
// units outnumber one wave (it runs one CTA per SM), each unit's chunks run as
// four consecutive ranges in successive launches, a range starting from the
// exact fp32 state the previous one left in the outputs: the same bits as one
// walk, in fewer waves.  The forward does the same when its units fill between
// one and four waves and the final state is kept in fp32 (the hand-over goes
// through it): a range ending inside its sequence writes the state it reached
// there, and the checkpoint row if the boundary is one.
//
// Gated DeltaProduct (mode kModeGdp, 2 <= n <= 64 updates per token): the same
// recurrence walked on the update timeline (n rows per token of k, v, beta; a
// token's gate at its first update, no decay at the others).  A 64-row chunk's
// query tokens are those whose last update row lies in it; their queries occupy
// the first rows of the query half of the K/Q tile, each read after its token's
// last update row, and the outputs go to the token rows of o.
#include <cuda_bf16.h>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"
#include "ptx.cuh"
#include "gdn_device.cuh"

namespace la {

constexpr int kCta = 128;  // threads per CTA (the state passes: two per TMEM lane, below)
constexpr int kSumPieces = 4;  // chunk ranges per summary unit when the units outnumber one wave

// Threads of a chunk-kernel CTA: the state passes of the two-pass schedules (no solve, only the
// chain's per-chunk phases) run two threads per TMEM lane, splitting each lane's columns (the
// chunk's tokens, the state's key columns) in halves; the fused kernel one.
__host__ __device__ constexpr int chunk_threads(int mode) {
    return (mode == kModeFwdSplit || mode == kModeSummarySplit || mode == kModeGdpSplit) ? 2 * kCta : kCta;
}

// ------------------------------------------------------------------ shared memory map
// Byte offsets from the 1024-aligned base, per mode:
//   kq   [region 0..1][128 rows: K 0-63, Q 64-127][128 B], regions kq_region bytes apart
//   v    V tile [region 0..1][64 rows][128 B] | later T fp32 [64][64]
//   wb   S^T bf16 [2][128][128 B] | X^T hi,lo | Ddec^T hi,lo
//   m    A fp32 [64][64] | T bf16 [64][128 B] | D^T bf16 [128][128 B]
//   pb   P bf16 [64][128 B]
//   sc   Scalars (7 KB; without the solve's scratch in the summary's state pass)
//   slo  summary only: S^T bf16 residual (lo part), same layout as wb
// The summary's state pass loads only K (two 8 KB regions), keeps only T (bf16) in m and has no
// P: 109 KB, so two CTAs share an SM.
struct SmemMap {
    uint32_t kq, kq_region, v, wb, m, pb, sc, slo, total;
};
__host__ __device__ constexpr SmemMap smem_map(int mode) {
    return mode == kModeSummarySplit
               ? SmemMap{0u, 8192u, 16384u, 32768u, 65536u, 0u, 73728u, 77824u, 77824u + 32768u + 1024u}
               : SmemMap{0u, 16384u, 32768u, 49152u, 81920u, 98304u, 106496u, 114688u,
                         (mode == kModeSummary ? 114688u + 32768u : 106496u + 7168u) + 1024u};
}

// TMEM columns (fp32, 128 lanes)
constexpr uint32_t COL_S = 0;     // S^T (K columns)
constexpr uint32_t COL_R1 = 128;  // G (128 columns with R2) -> (K S)^T -> D^T
constexpr uint32_t COL_R2 = 192;  // (Q S)^T, scaled per query row in place, then += D^T P^T = O^T
constexpr uint32_t TMEM_COLS = 256;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFastRange = 100.f;  // factorised decays when |b_i - b_31| <= this (log2 units)

struct __align__(16) Scalars {
    float b[64];    // chunk-local inclusive cumsum of g * log2(e)
    float bw[64];   // per-warp partial scans
    float rk[64];   // inverse key norms (0 on rows past the sequence end)
    float rq[64];   // inverse query norms
    float bet[64];  // beta (0 past the end)
    float sx[64];   // beta_j 2^{b_j} rk_j
    float sq[64];   // scale rq_i 2^{b_i}
    float sd[64];   // 2^{b_C - b_j} rk_j
    float u[64];    // rk_j 2^{b_31 - b_j}           (factorised decay, column factor)
    float cA[64];   // beta_i rk_i 2^{b_i - b_31}    (row factor of A)
    float cP[64];   // scale rq_i 2^{b_i - b_31}     (row factor of P)
    float gsum[2];    // per-warp sums of the next chunk's g * log2(e)
    uint64_t bar_kq, bar_v, bar_mma, bar_o, bar_f;
    uint32_t tmem_base;
    int32_t unit_lo, unit_hi;
    int32_t status0;
    int32_t ranges_ok;
    float Y[4][256];  // per-warp 16 x 16 solve scratch (last: the WY pass keeps it elsewhere)
};
static_assert(sizeof(Scalars) <= 7168, "scalar area");
constexpr uint32_t kScalarsNoY = static_cast<uint32_t>(sizeof(Scalars) - sizeof(float[4][256]));
static_assert(smem_map(kModeSummarySplit).sc + kScalarsNoY <= smem_map(kModeSummarySplit).slo,
              "the summary state pass's scalars overlap its residual buffer");

// fp32 64 x 64 tiles (A, T): 16-byte chunks XOR-swizzled by row to spread rows over the banks.
__device__ __forceinline__ int midx(int r, int c) { return r * 64 + ((((c >> 2) ^ (r & 15)) << 2) | (c & 3)); }

// y (16 x 16, as two m16n8 accumulator fragments) = sum over KS steps of 8 of
// la(row, m) * lb(m, col), on tf32 warp MMAs; every operand is loaded before the products.
template <int KS, class LA, class LB>
__device__ __forceinline__ void mma16x16(float (&y)[2][4], LA la, LB lb, int g, int q) {
    uint32_t af[KS][4], bf[KS][2][2];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        const int m0 = 8 * s;
        af[s][0] = to_tf32(la(g, m0 + q));
        af[s][1] = to_tf32(la(g + 8, m0 + q));
        af[s][2] = to_tf32(la(g, m0 + q + 4));
        af[s][3] = to_tf32(la(g + 8, m0 + q + 4));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            bf[s][nt][0] = to_tf32(lb(m0 + q, 8 * nt + g));
            bf[s][nt][1] = to_tf32(lb(m0 + q + 4, 8 * nt + g));
        }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) y[nt][0] = y[nt][1] = y[nt][2] = y[nt][3] = 0.f;
#pragma unroll
    for (int s = 0; s < KS; ++s)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma_tf32_16x8x8(y[nt], af[s], bf[s][nt]);
}

// A 16 x 16 accumulator (two m16n8 fragments) into a row-major 16 x 16 scratch tile.
__device__ __forceinline__ void store_frag16(float* Y, const float (&y)[2][4], int g, int q) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        Y[g * 16 + 8 * nt + 2 * q] = y[nt][0];
        Y[g * 16 + 8 * nt + 2 * q + 1] = y[nt][1];
        Y[(g + 8) * 16 + 8 * nt + 2 * q] = y[nt][2];
        Y[(g + 8) * 16 + 8 * nt + 2 * q + 1] = y[nt][3];
    }
}

// One off-diagonal block of T = (I + A)^{-1}, on tf32 warp MMAs (one warp, 16 x 16 result):
//   T[bj + D][bj] = -T[bj + D][bj + D] * sum_{m = bj}^{bj + D - 1} A[bj + D][m] T[m][bj]
// (16-row block indices).  It reads only T blocks of column bj computed earlier by the same
// warp and the diagonal block T[bj + D][bj + D], so consecutive stages of one warp need no
// block-wide barrier.  The k loops have compile-time lengths so every operand load can be
// issued ahead of the products.
template <int D>
__device__ __forceinline__ void solve_stage(const float* M, float* Tf, float* Y, int bj, int g, int q) {
    const int r0 = 16 * (bj + D), c0 = 16 * bj;
    float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    uint32_t af[2 * D][4], bf[2 * D][2][2];
#pragma unroll
    for (int s = 0; s < 2 * D; ++s) {
        const int m0 = c0 + 8 * s;
        af[s][0] = to_tf32(M[midx(r0 + g, m0 + q)]);
        af[s][1] = to_tf32(M[midx(r0 + g + 8, m0 + q)]);
        af[s][2] = to_tf32(M[midx(r0 + g, m0 + q + 4)]);
        af[s][3] = to_tf32(M[midx(r0 + g + 8, m0 + q + 4)]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            bf[s][nt][0] = to_tf32(Tf[midx(m0 + q, c0 + 8 * nt + g)]);
            bf[s][nt][1] = to_tf32(Tf[midx(m0 + q + 4, c0 + 8 * nt + g)]);
        }
    }
#pragma unroll
    for (int s = 0; s < 2 * D; ++s)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma_tf32_16x8x8(y[nt], af[s], bf[s][nt]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        Y[g * 16 + 8 * nt + 2 * q] = y[nt][0];
        Y[g * 16 + 8 * nt + 2 * q + 1] = y[nt][1];
        Y[(g + 8) * 16 + 8 * nt + 2 * q] = y[nt][2];
        Y[(g + 8) * 16 + 8 * nt + 2 * q + 1] = y[nt][3];
    }
    __syncwarp();
    float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) {
        const uint32_t a[4] = {to_tf32(Tf[midx(r0 + g, r0 + k0 + q)]), to_tf32(Tf[midx(r0 + g + 8, r0 + k0 + q)]),
                               to_tf32(Tf[midx(r0 + g, r0 + k0 + q + 4)]),
                               to_tf32(Tf[midx(r0 + g + 8, r0 + k0 + q + 4)])};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b[2] = {to_tf32(Y[(k0 + q) * 16 + 8 * nt + g]), to_tf32(Y[(k0 + q + 4) * 16 + 8 * nt + g])};
            mma_tf32_16x8x8(o[nt], a, b);
        }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int cc = c0 + 8 * nt + 2 * q;
        Tf[midx(r0 + g, cc)] = -o[nt][0];
        Tf[midx(r0 + g, cc + 1)] = -o[nt][1];
        Tf[midx(r0 + g + 8, cc)] = -o[nt][2];
        Tf[midx(r0 + g + 8, cc + 1)] = -o[nt][3];
    }
    __syncwarp();
}

// T = (I + A)^{-1} for the strictly lower-triangular A held (fp32) in the packed buffer M.
// T's blocks on and below the diagonal are written (fp32 [64][64], same swizzle) into Tf;
// the blocks above it are never written (the caller writes zeros there).  128 threads.
//   diagonal 16 x 16 blocks, one warp per block: 8 x 8 diagonal blocks by right-looking
//   substitution (lane = column; each step updates all later rows at once, and the next
//   column of A is loaded while the current one is applied), then the 8 x 8 block below;
//   then by doubling: the two 32 x 32 diagonal blocks (T[1][0], T[3][2]: solve_stage), and
//   the 32 x 32 block below them, T_BA = -T_BB A_BA T_AA, as two products over all four warps.
__device__ void solve_unit_lower(const float* M, float* Tf, float (*Ys)[256], int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    {
        // diagonal 16 x 16 block o of warp w, itself by doubling: its two 8 x 8 diagonal blocks by
        // substitution (lanes 0-7 and 8-15, lane = column), then the lower-left 8 x 8 block
        // T10 = -T11 A10 T00 on all 32 lanes; lanes 16-31 meanwhile clear the upper-right block
        const int o = 16 * warp;
        if (lane < 16) {
            const int b = o + 8 * (lane >> 3), c = lane & 7;
            float acc[8], col[8], nxt[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
            for (int i = 1; i < 8; ++i) col[i] = M[midx(b + i, b)];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int i = j + 2; i < 8; ++i) nxt[i] = M[midx(b + i, b + j + 1)];
                const float tj = ((j == c) ? 1.f : 0.f) - acc[j];
                Tf[midx(b + j, b + c)] = tj;
#pragma unroll
                for (int i = j + 1; i < 8; ++i) acc[i] = fmaf(col[i], tj, acc[i]);
#pragma unroll
                for (int i = j + 2; i < 8; ++i) col[i] = nxt[i];
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int idx = (lane - 16) * 4 + e;  // 0 .. 63
                Tf[midx(o + (idx >> 3), o + 8 + (idx & 7))] = 0.f;
            }
        }
        __syncwarp();
        float* Y = Ys[warp];
        const int i = lane >> 2, c = 2 * (lane & 3);
        {
            float a8[8], y0 = 0.f, y1 = 0.f;
#pragma unroll
            for (int m = 0; m < 8; ++m) a8[m] = M[midx(o + 8 + i, o + m)];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                y0 = fmaf(a8[m], Tf[midx(o + m, o + c)], y0);
                y1 = fmaf(a8[m], Tf[midx(o + m, o + c + 1)], y1);
            }
            Y[i * 8 + c] = y0;
            Y[i * 8 + c + 1] = y1;
        }
        __syncwarp();
        {
            float t8[8], z0 = 0.f, z1 = 0.f;
#pragma unroll
            for (int m = 0; m < 8; ++m) t8[m] = Tf[midx(o + 8 + i, o + 8 + m)];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                z0 = fmaf(t8[m], Y[m * 8 + c], z0);
                z1 = fmaf(t8[m], Y[m * 8 + c + 1], z1);
            }
            Tf[midx(o + 8 + i, o + c)] = -z0;
            Tf[midx(o + 8 + i, o + c + 1)] = -z1;
        }
    }
    __syncthreads();
    const int g = lane >> 2, q = lane & 3;
    // 32 x 32 diagonal blocks: T[1][0] (warp 0) and T[3][2] (warp 1)
    if (warp <= 1) solve_stage<1>(M, Tf, Ys[warp], 2 * warp, g, q);
    __syncthreads();
    // the 32 x 32 block below them, T_BA = -T_BB A_BA T_AA (A = rows 0-31, B = rows 32-63), as
    // 2 x 2 blocks of 16: warp (i, j) forms Y[i][j] = sum_m A[32 + 16 i ..][m] T[m][16 j ..]
    // over m = 16 j .. 31 (T_AA is block lower triangular) ...
    const int bi = warp >> 1, bj = warp & 1;
    {
        float y[2][4];
        const int r0 = 32 + 16 * bi, c0 = 16 * bj;
        auto la = [&](int r, int m) { return M[midx(r0 + r, c0 + m)]; };
        auto lb = [&](int m, int c) { return Tf[midx(c0 + m, c0 + c)]; };
        if (bj == 0) mma16x16<4>(y, la, lb, g, q);
        else mma16x16<2>(y, la, lb, g, q);
        store_frag16(Ys[warp], y, g, q);
    }
    __syncthreads();
    // ... then T[32 + 16 i ..][16 j ..] = -sum_{k <= i} T[32 + 16 i ..][32 + 16 k ..] Y[k][j]
    {
        float z[2][4];
        const int r0 = 32 + 16 * bi;
        auto la = [&](int r, int m) { return Tf[midx(r0 + r, 32 + m)]; };
        auto lb = [&](int m, int c) { return Ys[(m >> 4) * 2 + bj][(m & 15) * 16 + c]; };
        if (bi == 0) mma16x16<2>(z, la, lb, g, q);
        else mma16x16<4>(z, la, lb, g, q);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int cc = 16 * bj + 8 * nt + 2 * q;
            Tf[midx(r0 + g, cc)] = -z[nt][0];
            Tf[midx(r0 + g, cc + 1)] = -z[nt][1];
            Tf[midx(r0 + g + 8, cc)] = -z[nt][2];
            Tf[midx(r0 + g + 8, cc + 1)] = -z[nt][3];
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------ state-independent phases
// (shared by the fused kernel and the WY pass, so both compute the same bits)

// Rows of G = [K; Q] [K; Q]^T (at TMEM column col) into g64 (thread r: row r's first 64
// columns, the products with the key rows), and the inverse row norms from G's diagonal: rk (key
// rows, threads 0-63) and rq (query rows, threads 64-127; the forward only); rows past the
// chunk's tokens get 0.
template <bool kFwd>
__device__ __forceinline__ void g_rows_and_norms(uint32_t trow, uint32_t col, int r, int n, int nq, int l2norm,
                                                 float (&g64)[64], Scalars& sc) {
    const int lane = r & 31;
    if (r < 64 || kFwd) {
#pragma unroll
        for (int p = 0; p < 4; ++p) tmem_ld16(trow + col + 16 * p, *reinterpret_cast<float(*)[16]>(&g64[16 * p]));
        float nrm = 0.f;
        if (r < 64) {
            tmem_wait_ld();
            if (r < 32) {
#pragma unroll
                for (int e = 0; e < 32; ++e) nrm = (e == lane) ? g64[e] : nrm;
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) nrm = (e == lane) ? g64[32 + e] : nrm;
            }
        } else {
            float d32[32];
            const uint32_t cbase = col + (r & ~31);
            tmem_ld16(trow + cbase, *reinterpret_cast<float(*)[16]>(&d32[0]));
            tmem_ld16(trow + cbase + 16, *reinterpret_cast<float(*)[16]>(&d32[16]));
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) nrm = (e == lane) ? d32[e] : nrm;
        }
        const int row = r & 63;
        const int nvalid = (r < 64) ? n : nq;  // key rows, or the chunk's query tokens
        const float inv = (row < nvalid) ? (l2norm ? 1.0f / sqrtf(nrm + 1e-6f) : 1.f) : 0.f;
        if (r < 64) sc.rk[row] = inv;
        else sc.rq[row] = inv;
    }
}

// Per-token factors of a chunk from the per-warp gate scans (sc.bw), the norms and beta
// (b_cur: this thread's row); returns, block-wide, whether the factorised decays are in range.
template <bool kFwd, bool kGdp>
__device__ __forceinline__ bool chunk_scalars(Scalars& sc, int tid, int n, int nq, int tq0, int rel0, int NH,
                                              float b_cur, float scale) {
    bool in_range = true;
    if (tid < 64) {
        const int i = tid;
        const float bi = sc.bw[i] + (i >= 32 ? sc.bw[31] : 0.f);
        const float b31 = sc.bw[31];
        const float bC = sc.bw[31] + sc.bw[63];
        const float rk = sc.rk[i], rq = kFwd ? sc.rq[i] : 0.f;
        const float bet = i < n ? b_cur : 0.f;
        const float gam = exp2f(bi);
        const float e = exp2f(bi - b31);
        sc.b[i] = bi;
        sc.bet[i] = bet;
        sc.sx[i] = bet * gam * rk;
        sc.sd[i] = exp2f(bC - bi) * rk;
        sc.u[i] = rk * exp2f(b31 - bi);
        sc.cA[i] = bet * rk * e;
        if (kGdp) {
            // query row i is token tok0 + i, read after its last update row ri of the chunk
            const int ri = i < nq ? (tq0 + i) * NH + NH - 1 - rel0 : -1;
            const float bq = ri >= 0 ? sc.bw[ri] + (ri >= 32 ? sc.bw[31] : 0.f) : 0.f;
            sc.sq[i] = ri >= 0 ? scale * rq * exp2f(bq) : 0.f;
            sc.cP[i] = ri >= 0 ? scale * rq * exp2f(bq - b31) : 0.f;
        } else {
            sc.sq[i] = scale * rq * gam;
            sc.cP[i] = scale * rq * e;
        }
        in_range = fabsf(bi - b31) <= kFastRange;
    }
    return __syncthreads_and(in_range) != 0;
}

// A (fp32, strictly lower, into M for the solve) and P (bf16, lower with the diagonal, into PB)
// from this thread's row of G.
template <bool kFwd, bool kGdp>
__device__ __forceinline__ void build_a_p(float (&g64)[64], const Scalars& sc, float* M, uint8_t* PB, bool fast, int r,
                                          int nq, int tq0, int rel0, int NH, float scale) {
    if (r < 64 || kFwd) {
        const int i = r & 63;
        const bool is_a = r < 64;
        const float ci = fast ? (is_a ? sc.cA[i] : sc.cP[i]) : (is_a ? sc.bet[i] * sc.rk[i] : scale * sc.rq[i]);
        // the row's position on the update timeline (GDP query rows: the token's last update;
        // rows past the chunk's tokens are zero and fully masked)
        const int ip = (kGdp && !is_a) ? (i < nq ? (tq0 + i) * NH + NH - 1 - rel0 : -1) : i;
        const float bi = sc.b[ip < 0 ? 0 : ip];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            float* gv = &g64[16 * p];
            if (fast) {
                float uv[16];
                ld8(uv, &sc.u[16 * p]);
                ld8(uv + 8, &sc.u[16 * p + 8]);
#pragma unroll
                for (int e = 0; e < 16; ++e) gv[e] *= ci * uv[e];
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int j = 16 * p + e;
                    const float dec = (j <= ip) ? exp2f(bi - sc.b[j]) : 0.f;
                    gv[e] *= ci * sc.rk[j] * dec;
                }
            }
            if (is_a) {
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                    const int j = 16 * p + 4 * j4;
                    float4 w;
                    w.x = (j + 0 < i) ? gv[4 * j4 + 0] : 0.f;
                    w.y = (j + 1 < i) ? gv[4 * j4 + 1] : 0.f;
                    w.z = (j + 2 < i) ? gv[4 * j4 + 2] : 0.f;
                    w.w = (j + 3 < i) ? gv[4 * j4 + 3] : 0.f;
                    *reinterpret_cast<float4*>(&M[midx(i, j)]) = w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (16 * p + e > ip) gv[e] = 0.f;
                store8_split(PB + sw128_off(i, 2 * p), nullptr, &gv[0]);
                store8_split(PB + sw128_off(i, 2 * p + 1), nullptr, &gv[8]);
            }
        }
    }
}

// T (fp32, from the solve) -> bf16, K-major (128-byte swizzle), into TB; zeros above the
// diagonal blocks.
__device__ __forceinline__ void t_to_bf16(const float* Tf, uint8_t* TB, int tid) {
    const int i = tid >> 1;
#pragma unroll
    for (int cc4 = 0; cc4 < 4; ++cc4) {
        const int cc = (tid & 1) * 4 + cc4;
        if ((cc >> 1) > (i >> 4)) {
            // a block above the diagonal: zeros
            *reinterpret_cast<uint4*>(TB + sw128_off(i, cc)) = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        const float4 lo4 = *reinterpret_cast<const float4*>(&Tf[midx(i, 8 * cc)]);
        const float4 hi4 = *reinterpret_cast<const float4*>(&Tf[midx(i, 8 * cc + 4)]);
        const float x[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
        store8_split(TB + sw128_off(i, cc), nullptr, x);
    }
}

// The bf16 residual T - bf16(T) of the same tile (the lo part the full backward's products add),
// in the 128-byte swizzled byte order of a [64][128 B] tile, so that a bulk copy into a
// 1024-aligned buffer lands it as a swizzled TMA load would; into global memory at dst.
__device__ __forceinline__ void t_lo_store(const float* Tf, uint8_t* dst, int tid) {
    const int i = tid >> 1;
#pragma unroll
    for (int cc4 = 0; cc4 < 4; ++cc4) {
        const int cc = (tid & 1) * 4 + cc4;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if ((cc >> 1) <= (i >> 4)) {
            const float4 lo4 = *reinterpret_cast<const float4*>(&Tf[midx(i, 8 * cc)]);
            const float4 hi4 = *reinterpret_cast<const float4*>(&Tf[midx(i, 8 * cc + 4)]);
            const float x[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
            uint32_t l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t h = pack_bf16(x[2 * e], x[2 * e + 1]);
                l[e] = pack_bf16(x[2 * e] - bf16_lo(h), x[2 * e + 1] - bf16_hi(h));
            }
            w = make_uint4(l[0], l[1], l[2], l[3]);
        }
        *reinterpret_cast<uint4*>(dst + sw128_off(static_cast<uint32_t>(i), static_cast<uint32_t>(cc))) = w;
    }
}

// One WY record into shared memory, on bar_f: T (bf16, into TB's place), P (into PB; the
// summary has none: PBdst null) and the factors beta, sx, sq, sd (into sc.bet .. sc.sd,
// contiguous).  One thread.
__device__ __forceinline__ void load_wy(const ChunkArgs& a, const CUtensorMap& wymap, int64_t chunk, int h,
                                        void* TBdst, void* PBdst, Scalars& sc) {
    const int64_t item = chunk * a.HV + h;
    mbar_arrive_expect_tx(&sc.bar_f, static_cast<uint32_t>(PBdst ? kWyRecordBytes : kWyRecordBytes - kWyTileBytes));
    tma_load_3d(TBdst, &wymap, &sc.bar_f, 0, static_cast<int>(item), 0);
    if (PBdst) tma_load_3d(PBdst, &wymap, &sc.bar_f, 0, static_cast<int>(item), 64);
    bulk_load(sc.bet, a.wy + item * static_cast<int64_t>(kWyRecordBytes) + 2 * kWyTileBytes,
              static_cast<uint32_t>(kWyFactorBytes), &sc.bar_f);
}

template <int KD, int MODE>
__global__ void __launch_bounds__(chunk_threads(MODE), 2)
    gdn_chunk_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                     const __grid_constant__ CUtensorMap wymap, const ChunkArgs a) {
    constexpr bool kSum = MODE == kModeSummary || MODE == kModeSummarySplit;
    constexpr bool kFwd = !kSum;  // queries and outputs (the forward, or GDP's)
    constexpr bool kGdp = MODE == kModeGdp || MODE == kModeGdpSplit;
    // the state pass of the two-pass forward, summary or GDP: T (P) and the factors of every chunk
    // come from the WY pass's records instead of being formed here
    constexpr bool kSplit = MODE == kModeFwdSplit || MODE == kModeSummarySplit || MODE == kModeGdpSplit;
    constexpr SmemMap L = smem_map(MODE);
    constexpr uint32_t RQ = L.kq_region;
    // waits sleep in hardware when another CTA shares the SM (the forward and the summary's state
    // pass run two per SM; the fused summary, with its larger shared-memory footprint, one)
    constexpr bool kSleep = !kSum || kSplit;
    constexpr int KP = KD / 16;  // 16-column pieces of the state
    constexpr int PPT = KP / (chunk_threads(MODE) / kCta);
    // GDP: the tokens whose last update row falls in a chunk of 64 update rows (at most QR of
    // them) have their queries in rows 0 .. QR-1 of the query half of the K/Q tile (the other
    // rows stay zero) and their outputs in columns 0 .. QR-1; when n does not divide 64 a chunk
    // begins or ends inside a token
    const int NH = kGdp ? a.gdp_n : 1;
    const int QR = (kChunk + NH - 1) / NH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Scalars& sc = *reinterpret_cast<Scalars*>(sm + L.sc);  // (no solve scratch in the summary's state pass)
    uint8_t* KQ = sm + L.kq;
    uint8_t* VT = sm + L.v;
    uint8_t* WB = sm + L.wb;
    float* M = reinterpret_cast<float*>(sm + L.m);   // A (fp32) -> T bf16 (TB) -> D^T bf16 (DT)
    uint8_t* TB = sm + L.m;
    uint8_t* DT = sm + L.m;
    float* Tf = reinterpret_cast<float*>(sm + L.v);  // T fp32, in the V tile's space after X
    uint8_t* PB = kFwd ? sm + L.pb : nullptr;
    uint8_t* SLO = kFwd ? nullptr : sm + L.slo;
    uint8_t* OST = sm + L.m;  // O staging for the bulk store, once the O product has read D^T

    const int tid = threadIdx.x;
    constexpr int NT = chunk_threads(MODE);
    constexpr int NHALF = NT / kCta;         // threads per TMEM lane
    const int r = tid & (kCta - 1);          // TMEM lane, value column, stacked token row
    const int hf = tid / kCta;               // this thread's share of the lane's columns:
    constexpr int TPT = kChunk / NHALF;      //   tokens tb .. tb + TPT - 1,
    constexpr int CPT = 8 / NHALF;           //   8-token chunks cb .. cb + CPT - 1,
    const int tb = hf * TPT, cb = hf * CPT;  //   and 16-column state pieces pb .. pb + PPT - 1
    const int HO = a.HV;

    // one read of the status word for the whole CTA (another CTA may set it meanwhile), and of
    // the prologue's decision on forward ranges
    if (tid == 0) {
        sc.status0 = *reinterpret_cast<volatile int32_t*>(&a.hdr->status);
        sc.ranges_ok = a.hdr->ranges_ok;
    }
    __syncthreads();
    if (sc.status0 != LA_OK) return;
    // chunk ranges: the summary's whenever launched so, the forward's unless the prologue found
    // the sequence lengths spread, in which case launch 0 walks whole units and the rest return
    const bool ranged = !kGdp && a.pieces > 1 && (kSum || a.pieces_request > 1 || sc.ranges_ok != 0);
    if (!kGdp && a.pieces > 1 && !ranged && a.item_base > 0) return;

    if (tid < 32) {
        tmem_alloc(&sc.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sc.bar_kq, 1);
        mbar_init(&sc.bar_v, 1);
        mbar_init(&sc.bar_mma, 1);
        mbar_init(&sc.bar_o, 1);
        mbar_init(&sc.bar_f, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sc.tmem_base;
    const uint32_t trow = tmem + (static_cast<uint32_t>(r & ~31) << 16);
    // shared-memory matrix descriptors of the operand buffers; an operand at byte offset off
    // from a buffer uses base + (off >> 4) (the start-address field counts 16-byte units)
    const uint64_t d_kq = sdesc_sw128(smem_u32(KQ), 16, 1024);
    const uint64_t d_kq_mn = sdesc_sw128(smem_u32(KQ), RQ, 1024);  // K read MN-major
    const uint64_t d_wb = sdesc_sw128(smem_u32(WB), 16, 1024);
    const uint64_t d_m = sdesc_sw128(smem_u32(sm + L.m), 16, 1024);   // T bf16, then D^T bf16
    const uint64_t d_pb = kFwd ? sdesc_sw128(smem_u32(PB), 16, 1024) : 0;
    const uint64_t d_slo = kFwd ? 0 : sdesc_sw128(smem_u32(SLO), 16, 1024);
    // (K S)^T and, in the forward, (Q S)^T = S^T [K; Q]^T, one M = 128 product per 16 keys (the
    // summary adds the product with the state's lo part); one thread
    auto issue_state_products = [&]() {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, kFwd ? 128 : 64, false, false);
#pragma unroll
        for (int kk = 0; kk < KD / 16; ++kk) {
            const uint64_t ow = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            const uint64_t oq = ((kk >> 2) * RQ + (kk & 3) * 32) >> 4;
            umma_bf16(tmem + COL_R1, d_wb + ow, d_kq + oq, idesc, kk > 0);
        }
        if (!kFwd) {
#pragma unroll
            for (int kk = 0; kk < KD / 16; ++kk) {
                const uint64_t ow = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                const uint64_t oq = ((kk >> 2) * RQ + (kk & 3) * 32) >> 4;
                umma_bf16(tmem + COL_R1, d_slo + ow, d_kq + oq, idesc, 1u);
            }
        }
        umma_commit(&sc.bar_mma);
    };

    if constexpr (kGdp) {
        // the query rows past a chunk's QR tokens are never written by the tile loads: zero them once
        for (int e = tid; e < (KD / 64) * (64 - QR) * 8; e += NT) {
            const int rg = e / ((64 - QR) * 8), rem = e % ((64 - QR) * 8);
            *reinterpret_cast<uint4*>(KQ + rg * RQ + 8192 + (QR + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncthreads();
    }
    uint32_t ph_kq = 0, ph_v = 0, ph_mma = 0, ph_o = 0, ph_f = 0;  // parity of the next wait on each barrier
    bool pend_kq = false, pend_v = false, pend_mma = false, pend_o = false, pend_f = false;
    bool pend_st = false;  // the state's write-back to TMEM, waited for before the next state update
    bool failed = false;
    const uint64_t budget = a.wait_budget_ns;
    const int64_t per_seq = static_cast<int64_t>(HO) * a.tiles_per_head;
    const uint32_t kq_bytes = KD * 128u + (kFwd ? static_cast<uint32_t>(KD / 64) * QR * 128u : 0u);
    const uint32_t v_bytes = static_cast<uint32_t>(a.V) * 128u;

    for (int iter = 0;; ++iter) {
        if (tid == 0) {
            const unsigned long long u =
                ranged ? (iter == 0 ? static_cast<unsigned long long>(blockIdx.x) : 0x7FFFFFFFFFFFFFFFull)
                       : atomicAdd(reinterpret_cast<unsigned long long*>(&a.hdr->ticket), 1ull);
            sc.unit_lo = static_cast<int32_t>(u & 0xFFFFFFFFull);
            sc.unit_hi = static_cast<int32_t>(u >> 32);
        }
        __syncthreads();
        const int64_t taken = (static_cast<int64_t>(sc.unit_hi) << 32) | static_cast<uint32_t>(sc.unit_lo);
        __syncthreads();  // every thread has read the ticket before thread 0 may take the next one
        if (taken >= (ranged ? a.items : a.num_units)) break;
        const int64_t item = ranged ? a.item_base + taken : taken;
        const int rng = ranged ? static_cast<int>(item / a.num_units) : 0;  // the chunk range
        const int64_t unit = ranged ? item % a.num_units : item;
        const int seq = a.order[unit / per_seq];
        const int rem = static_cast<int>(unit % per_seq);
        const int h = rem / a.tiles_per_head;
        const int tile = rem % a.tiles_per_head;
        const int hk = h / a.group;
        const bool value_tile = kFwd || tile == kTileValue;
        // update rows (GDP: NH per token); tok_s is the sequence's first token
        const int64_t tok_s = cu_get(a.cu, a.cu64, seq);
        const int64_t ts = tok_s * NH;
        const int64_t L = (cu_get(a.cu, a.cu64, seq + 1) - tok_s) * NH;
        const int nchunks = static_cast<int>((L + kChunk - 1) / kChunk);
        // this item's chunks lo .. hi - 1 (all of them unless ranged)
        const int lo = ranged ? static_cast<int>(static_cast<int64_t>(rng) * nchunks / a.pieces) : 0;
        const int hi = ranged ? static_cast<int>(static_cast<int64_t>(rng + 1) * nchunks / a.pieces) : nchunks;
        if (lo == hi && rng > 0) continue;  // an empty later range: the state stays where it is
        const int64_t tlo = static_cast<int64_t>(lo) * kChunk;  // first update row of the range
        const int64_t unit_state = static_cast<int64_t>(seq) * HO + h;
        // the start state's slot, and where the end state goes (the same pool slot when a state
        // pool is used: written back in place)
        int64_t s0_unit = unit_state;
        if (a.state_idx) {
            const int32_t slot = a.state_idx[seq];
            if (slot < 0 || slot >= a.pool_size) {
                if (tid == 0) {
                    atomicCAS(&a.hdr->status, LA_OK, LA_ERR_BAD_STATE_INDEX);
                    if (a.user_status) atomicCAS(a.user_status, LA_OK, LA_ERR_BAD_STATE_INDEX);
                }
                continue;
            }
            s0_unit = static_cast<int64_t>(slot) * HO + h;
        }
        const int64_t fin_unit = a.state_idx ? s0_unit : unit_state;

        // ---- first chunk's tiles (and record): issued before the start state is read, so that
        // their latency overlaps that read
        if (hi > lo) {
            const int64_t tf = ts + tlo;
            if (tid == 0 && !a.test_skip_tile_load) {
                mbar_arrive_expect_tx(&sc.bar_kq, kq_bytes);
#pragma unroll
                for (int rg = 0; rg < KD / 64; ++rg) {
                    tma_load_3d(KQ + rg * RQ, &kmap, &sc.bar_kq, rg * 64, hk, static_cast<int>(tf));
                    if (kFwd)
                        tma_load_3d(KQ + rg * RQ + 8192, &qmap, &sc.bar_kq, rg * 64, hk, static_cast<int>(tf / NH));
                }
            }
            if (tid == 0) {
                if (value_tile) {
                    mbar_arrive_expect_tx(&sc.bar_v, v_bytes);
                    for (int rg = 0; rg < a.V / 64; ++rg)
                        tma_load_3d(VT + rg * 8192, &vmap, &sc.bar_v, rg * 64, h, static_cast<int>(tf));
                }
            }
            pend_kq = !a.test_skip_tile_load;
            pend_v = value_tile;
            if (kSplit) {
                if (tid == 0) load_wy(a, wymap, a.chunk_off[seq] + lo, h, M, PB, sc);
                pend_f = true;
            }
        }
        // ---- chunk 0's gate total: the state kept in TMEM is pre-multiplied by the decay of the
        // chunk it is about to enter, so the state-update product can accumulate onto it
        float g_nx = 0.f, b_nx = 0.f;
        float gA = 0.f, gdt = 0.f;
        if (a.gate_mode == LA_GATE_SOFTPLUS && tid < 64) {
            gA = -expf(a.a_log[h]);
            gdt = a.dt_bias[h];
        }
        if (tid < 64 && tid < L - tlo) {
            g_nx = gate_row<kGdp>(a, ts + tlo + tid, h, gA, gdt);
            b_nx = beta_at(a, ts + tlo + tid, h);
        }
        if (tid < 64) {
            float x = g_nx * kLog2e;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
            if ((tid & 31) == 0) sc.gsum[tid >> 5] = x;
        }
        __syncthreads();
        const float gam0 = hi > lo ? exp2f(sc.gsum[0] + sc.gsum[1]) : 1.f;

        // ---- initial state -> TMEM (fp32 2^{b_C} S^T), WB (bf16 S^T, the A operand of K S),
        // checkpoint entry 0, and the end state of an empty sequence
        {
            const int64_t base = s0_unit * KD * a.V + r;
            const int64_t fbase0 = fin_unit * KD * a.V + r;
            // a later range starts from what the previous range left in the outputs: the end
            // state (fp32, value tile) or the transition (stored transposed: lane r reads row r)
            const bool from_out = ranged && rng > 0;
            const bool ckpt0 = kFwd && a.ckpt && nchunks > 0 && r < a.V && !from_out;
            const int64_t cbase = ckpt0 ? ((a.ckpt_off[seq] * HO + h) * KD) * a.V + r : 0;
            const int pb = hf * PPT;
#pragma unroll 1
            for (int p = pb; p < pb + PPT; ++p) {
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int k = 16 * p + e;
                    float val = 0.f;
                    if (from_out) {
                        if (value_tile) {
                            if (r < a.V) val = a.final_state[fbase0 + static_cast<int64_t>(k) * a.V];
                        } else if (r < KD) {
                            val = a.transition[(unit_state * KD + r) * KD + k];
                        }
                    } else if (value_tile) {
                        if (a.s0 && r < a.V) {
                            const int64_t idx = base + static_cast<int64_t>(k) * a.V;
                            val = a.s0_bf16 ? bf16_bits_to_f(static_cast<const uint16_t*>(a.s0)[idx])
                                            : static_cast<const float*>(a.s0)[idx];
                        }
                    } else {
                        val = (k == r) ? 1.f : 0.f;
                    }
                    x[e] = val;
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int kc = 2 * p + hh;  // 16-byte chunk index along k
                    const uint32_t off = (kc >> 3) * 16384 + sw128_off(r, kc & 7);
                    store8_split(WB + off, kFwd ? nullptr : SLO + off, &x[8 * hh]);
                }
                if (ckpt0) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int64_t idx = cbase + static_cast<int64_t>(16 * p + e) * a.V;
                        if (a.ckpt_bf16) static_cast<uint16_t*>(a.ckpt)[idx] = f_to_bf16_bits(x[e]);
                        else static_cast<float*>(a.ckpt)[idx] = x[e];
                    }
                }
                if (hi == lo) {  // no chunks (an empty sequence, or an empty first range): start = end
                    if (value_tile) {
                        if (a.final_state && r < a.V)
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                store_state(a, fbase0 + static_cast<int64_t>(16 * p + e) * a.V, x[e]);
                    } else if (r < KD) {
                        float* tp = a.transition + (unit_state * KD + r) * KD + 16 * p;
#pragma unroll
                        for (int e = 0; e < 16; e += 4)
                            *reinterpret_cast<float4*>(tp + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) x[e] *= gam0;
                tmem_st16(trow + COL_S + 16 * p, x);
            }
            tmem_wait_st();
        }

        for (int c = lo; c < hi; ++c) {
            const int64_t t0 = ts + static_cast<int64_t>(c) * kChunk;
            const int64_t left = L - static_cast<int64_t>(c) * kChunk;
            const int n = left < kChunk ? static_cast<int>(left) : kChunk;
            const bool last = c + 1 == hi;
            const bool o_tma_chunk = kFwd && a.o_tma && n == kChunk;
            // the chunk's query tokens: tok0 .. tok0 + nq - 1, those whose last update row is in it
            // (32-bit arithmetic relative to the sequence start, which is a token boundary)
            const int rel0 = c * kChunk;
            const int tq0 = kGdp ? rel0 / NH : rel0;
            const int64_t tok0 = tok_s + tq0;
            const int nq = kGdp ? (rel0 + n) / NH - tq0 : n;
            const float g_cur = g_nx, b_cur = b_nx;
            if (!last) {
                g_nx = b_nx = 0.f;
                if (tid < 64 && tid < left - kChunk) {
                    g_nx = gate_row<kGdp>(a, t0 + kChunk + tid, h, gA, gdt);
                    b_nx = beta_at(a, t0 + kChunk + tid, h);
                }
            }

            // ---- S1: K/Q tile; G = [K; Q] [K; Q]^T on the tensor core while the gate scan runs.
            // Its diagonal holds the squared row norms of K (lanes 0-63) and Q (lanes 64-127).
            bool ok = mbar_wait(&sc.bar_kq, ph_kq, budget, kSleep);
            if (ok) {
                ph_kq ^= 1u;
                pend_kq = false;
            }
            if (!kSplit && tid == 0 && ok) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, kFwd ? 128 : 64, false, false);
#pragma unroll
                for (int kk = 0; kk < KD / 16; ++kk) {
                    const uint64_t off = ((kk >> 2) * RQ + (kk & 3) * 32) >> 4;
                    umma_bf16(tmem + COL_R1, d_kq + off, d_kq + off, idesc, kk > 0);
                }
                umma_commit(&sc.bar_mma);
            }
            float g64[64];
            bool fast = true;
            if constexpr (kSplit) {
                // no G: (K S)^T and (Q S)^T are issued as soon as the tile is in (at a range's first
                // chunk once every thread has written its row of the start state's bf16 copy)
                if (c == lo) {
                    fence_proxy_async_smem();
                    tc_fence_before();
                    if (__syncthreads_or(!ok)) { failed = true; break; }
                }
                if (tid == 0 && ok) issue_state_products();
                pend_mma = true;
            } else {
                pend_mma = ok;
                if (tid < 64) {
                    float x = (tid < n) ? g_cur * kLog2e : 0.f;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, x, off);
                        if ((tid & 31) >= off) x += y;
                    }
                    sc.bw[tid] = x;
                }
                {
                    const bool okg = mbar_wait(&sc.bar_mma, ph_mma, budget, kSleep);
                    if (okg) {
                        ph_mma ^= 1u;
                        pend_mma = false;
                    }
                    ok = ok && okg;
                }
                tc_fence_after();
                g_rows_and_norms<kFwd>(trow, COL_R1, r, n, nq, a.l2norm, g64, sc);
                tc_fence_before();
                if (__syncthreads_or(!ok)) { failed = true; break; }
                // ---- S3: (K S)^T and (Q S)^T = S^T [K; Q]^T, issued as soon as every thread holds its row of
                // G (the product reuses G's columns); it runs while the scalars and A / P are formed
                if (tid == 0) issue_state_products();
                pend_mma = true;

                fast = chunk_scalars<kFwd, kGdp>(sc, tid, n, nq, tq0, rel0, NH, b_cur, a.scale);

                // ---- S2: A (fp32, for the solve) and P (bf16) from G
                build_a_p<kFwd, kGdp>(g64, sc, M, PB, fast, r, nq, tq0, rel0, NH, a.scale);
            }  // !kSplit
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }

            // ---- S4: X^T = beta V^T - sx (K S)^T (hi + lo); then T = (I + A)^{-1} in the V tile's space.
            // This thread's column of V (64 bf16, packed in pairs) is read while the K S product runs.
            uint32_t vpk[TPT / 2];
            {
                bool okv = true;
                if (value_tile) {
                    okv = mbar_wait(&sc.bar_v, ph_v, budget, kSleep);
                    if (okv) {
                        ph_v ^= 1u;
                        pend_v = false;
                    }
                }
                const bool has_v = value_tile && okv && r < a.V;
                const uint8_t* vcol = VT + (r >> 6) * 8192 + (r & 7) * 2;
                const uint32_t vchunk = (r & 63) >> 3;
#pragma unroll
                for (int j2 = 0; j2 < TPT / 2; ++j2) {
                    const uint32_t i0 = static_cast<uint32_t>(tb + 2 * j2);
                    const uint32_t lo16 = has_v ? *reinterpret_cast<const uint16_t*>(vcol + sw128_off(i0, vchunk)) : 0u;
                    const uint32_t hi16 = has_v ? *reinterpret_cast<const uint16_t*>(vcol + sw128_off(i0 + 1, vchunk)) : 0u;
                    vpk[j2] = lo16 | (hi16 << 16);
                }
                ok = ok && okv;
            }
            {
                const bool okk = mbar_wait(&sc.bar_mma, ph_mma, budget, kSleep);
                if (okk) {
                    ph_mma ^= 1u;
                    pend_mma = false;
                }
                ok = ok && okk;
            }
            if (kSplit) {
                const bool okf = mbar_wait(&sc.bar_f, ph_f, budget, kSleep);
                if (okf) {
                    ph_f ^= 1u;
                    pend_f = false;
                }
                ok = ok && okf;
            }
            tc_fence_after();
            {
                const int v = r;
                float kx[TPT];
#pragma unroll
                for (int p = 0; p < TPT / 16; ++p)
                    tmem_ld16(trow + COL_R1 + tb + 16 * p, *reinterpret_cast<float(*)[16]>(&kx[16 * p]));
                tmem_wait_ld();
#pragma unroll
                for (int c2 = 0; c2 < CPT; ++c2) {
                    const int cc = cb + c2;
                    float x[8], bt[8], sxv[8];
                    ld8(bt, &sc.bet[8 * cc]);
                    ld8(sxv, &sc.sx[8 * cc]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 8 * c2 + e;  // (relative to tb, which is even)
                        const float vv = __uint_as_float((j & 1) ? (vpk[j >> 1] & 0xFFFF0000u) : (vpk[j >> 1] << 16));
                        x[e] = bt[e] * vv - sxv[e] * kx[j];
                    }
                    store8_split(WB + sw128_off(v, cc), WB + 16384 + sw128_off(v, cc), x);
                }
            }
            if (kFwd) {
                // (Q S)^T -> (scale rq gamma) (Q S)^T in place: column i is query row i
#pragma unroll
                for (int p = tb / 16; p < tb / 16 + TPT / 16; ++p) {
                    float qs[16], f[16];
                    tmem_ld16(trow + COL_R2 + 16 * p, qs);
                    ld8(f, &sc.sq[16 * p]);
                    ld8(f + 8, &sc.sq[16 * p + 8]);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) qs[e] *= f[e];
                    tmem_st16(trow + COL_R2 + 16 * p, qs);
                }
                tmem_wait_st();
                tc_fence_before();
            }
            __syncthreads();  // every V read is done before T takes the tile's space
            if (!kSplit) {
                solve_unit_lower(M, Tf, sc.Y, tid);
                t_to_bf16(Tf, TB, tid);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }
            if (tid == 0 && value_tile && !last) {
                // the V tile's space (T, fp32) is free: fetch the next chunk's V
                mbar_arrive_expect_tx(&sc.bar_v, v_bytes);
                for (int rg = 0; rg < a.V / 64; ++rg)
                    tma_load_3d(VT + rg * 8192, &vmap, &sc.bar_v, rg * 64, h, static_cast<int>(t0 + kChunk));
            }
            if (value_tile && !last) pend_v = true;

            // ---- S5: D^T = X^T T^T (hi + lo)
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + COL_R1, d_wb + ((part * 16384 + kk * 32) >> 4), d_m + ((kk * 32) >> 4), idesc,
                                  (part | kk) != 0);
                umma_commit(&sc.bar_mma);
            }
            pend_mma = true;
            if (tid < 64) {
                // total gate of the next chunk (its values were prefetched at the chunk start)
                float x = last ? 0.f : g_nx * kLog2e;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
                if ((tid & 31) == 0) sc.gsum[tid >> 5] = x;
            }
            ok = mbar_wait(&sc.bar_mma, ph_mma, budget, kSleep);
            if (ok) {
                ph_mma ^= 1u;
                pend_mma = false;
            }
            tc_fence_after();
            {
                const int v = r;
                float dd[TPT];
#pragma unroll
                for (int p = 0; p < TPT / 16; ++p)
                    tmem_ld16(trow + COL_R1 + tb + 16 * p, *reinterpret_cast<float(*)[16]>(&dd[16 * p]));
                tmem_wait_ld();
#pragma unroll
                for (int c2 = 0; c2 < CPT; ++c2) {
                    const int cc = cb + c2;
                    float x[8], sdv[8];
                    ld8(sdv, &sc.sd[8 * cc]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = sdv[e] * dd[8 * c2 + e];
                    if (kFwd) store8_split(DT + sw128_off(v, cc), nullptr, &dd[8 * c2]);
                    store8_split(WB + sw128_off(v, cc), WB + 16384 + sw128_off(v, cc), x);
                }
            }
            if (pend_st) {
                tmem_wait_st();  // the previous chunk's state write-back, which the update accumulates onto
                pend_st = false;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }

            // ---- S6: O^T += D^T P^T (fwd); S^T += Ddec^T K (K read MN-major)
            if (tid == 0) {
                tc_fence_after();
                if (kFwd) {
                    const uint32_t idesc_o = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + COL_R2, d_m + ((kk * 32) >> 4), d_pb + ((kk * 32) >> 4), idesc_o, 1u);
                    umma_commit(&sc.bar_o);
                }
                const uint32_t idesc_s = idesc_bf16_f32(128, KD, false, true);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + COL_S, d_wb + ((part * 16384 + kk * 32) >> 4), d_kq_mn + ((kk * 2048) >> 4),
                                  idesc_s, 1u);
                umma_commit(&sc.bar_mma);
            }
            pend_mma = true;
            pend_o = kFwd;
            if (kFwd) {
                // O is complete before the state update: store it while the update runs
                const bool oko = mbar_wait(&sc.bar_o, ph_o, budget, kSleep);
                if (oko) {
                    ph_o ^= 1u;
                    pend_o = false;
                }
                ok = ok && oko;
                tc_fence_after();
                float o64[TPT];
#pragma unroll
                for (int p = 0; p < TPT / 16; ++p)
                    tmem_ld16(trow + COL_R2 + tb + 16 * p, *reinterpret_cast<float(*)[16]>(&o64[16 * p]));
                tmem_wait_ld();
                if (o_tma_chunk) {
                    // a full chunk: O (bf16) into the free M buffer in the TMA box layout
                    // ([v / 64][64 tokens][128 B], 128-byte swizzle), then one bulk store per 64 columns
                    if (r < a.V) {
                        uint8_t* col = OST + (r >> 6) * 8192 + (r & 7) * 2;
                        const uint32_t vchunk = (r & 63) >> 3;
#pragma unroll
                        for (int i = 0; i < TPT; ++i)
                            if (!kGdp || tb + i < QR)  // (the bulk store needs 64 / n whole tokens: n divides 64)
                                *reinterpret_cast<uint16_t*>(col + sw128_off(static_cast<uint32_t>(tb + i), vchunk)) =
                                    f_to_bf16_bits(o64[i]);
                    }
                    fence_proxy_async_smem();
                    __syncthreads();
                    if (tid == 0) {
                        for (int rg = 0; rg < a.V / 64; ++rg)
                            tma_store_3d(&omap, OST + rg * 8192, rg * 64, h, static_cast<int>(tok0));
                        bulk_commit_group();
                    }
                } else if (r < a.V) {
                    uint16_t* op = a.o + tok0 * a.o_st + static_cast<int64_t>(h) * a.o_sh + r;
#pragma unroll
                    for (int i = 0; i < TPT; ++i)
                        if (tb + i < nq) op[static_cast<int64_t>(tb + i) * a.o_st] = f_to_bf16_bits(o64[i]);
                }
            }
            {
                const bool okm = mbar_wait(&sc.bar_mma, ph_mma, budget, kSleep);
                if (okm) {
                    ph_mma ^= 1u;
                    pend_mma = false;
                }
                ok = ok && okm;
            }
            tc_fence_after();
            if (tid == 0 && ok && !last) {
                // the K/Q tile is free: fetch the next chunk's
                const int t1 = static_cast<int>(t0 + kChunk);
                mbar_arrive_expect_tx(&sc.bar_kq, kq_bytes);
#pragma unroll
                for (int rg = 0; rg < KD / 64; ++rg) {
                    tma_load_3d(KQ + rg * RQ, &kmap, &sc.bar_kq, rg * 64, hk, t1);
                    if (kFwd) tma_load_3d(KQ + rg * RQ + 8192, &qmap, &sc.bar_kq, rg * 64, hk, t1 / NH);
                }
            }
            if (!last) pend_kq = true;
            if (kSplit && !last) {
                // P, the factors and the O staging buffer (the next T's place) are free: fetch the
                // next chunk's record once the bulk store of O has read its staging buffer
                if (tid == 0 && ok) {
                    bulk_wait_read_all();
                    load_wy(a, wymap, a.chunk_off[seq] + c + 1, h, M, PB, sc);
                }
                pend_f = true;
            }
            {
                // new state: bf16 copy for the next K S product, end state or checkpoint entry,
                // then pre-multiplied by the next chunk's decay for its state update
                const float gnext = last ? 1.f : exp2f(sc.gsum[0] + sc.gsum[1]);
                const int64_t fbase = fin_unit * KD * a.V + r;
                // (a range that ends inside its sequence writes the checkpoint row at its end too)
                const bool ckpt = kFwd && a.ckpt && c + 1 < nchunks &&
                                  (static_cast<int64_t>(c + 1) * kChunk) % a.ckpt_n == 0 && r < a.V;
                const int64_t cbase =
                    ckpt ? (((a.ckpt_off[seq] + static_cast<int64_t>(c + 1) * kChunk / a.ckpt_n) * HO + h) * KD) * a.V + r
                         : 0;
                const int pb = hf * PPT;
#pragma unroll 1
                for (int p0 = pb; p0 < pb + PPT; p0 += 4) {
                    float s64[64];
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp)
                        if (p0 + pp < pb + PPT)
                            tmem_ld16(trow + COL_S + 16 * (p0 + pp), *reinterpret_cast<float(*)[16]>(&s64[16 * pp]));
                    tmem_wait_ld();
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        const int p = p0 + pp;
                        if (p >= pb + PPT) break;
                        float* x = &s64[16 * pp];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int kc = 2 * p + hh;
                            const uint32_t off = (kc >> 3) * 16384 + sw128_off(r, kc & 7);
                            store8_split(WB + off, kFwd ? nullptr : SLO + off, &x[8 * hh]);
                        }
                        if (last) {
                            if (value_tile) {
                                if (a.final_state && r < a.V)
#pragma unroll
                                    for (int e = 0; e < 16; ++e)
                                        store_state(a, fbase + static_cast<int64_t>(16 * p + e) * a.V, x[e]);
                                if (ckpt) {
#pragma unroll
                                    for (int e = 0; e < 16; ++e) {
                                        const int64_t idx = cbase + static_cast<int64_t>(16 * p + e) * a.V;
                                        if (a.ckpt_bf16) static_cast<uint16_t*>(a.ckpt)[idx] = f_to_bf16_bits(x[e]);
                                        else static_cast<float*>(a.ckpt)[idx] = x[e];
                                    }
                                }
                            } else if (r < KD) {
                                // transition[j][k] = P[k][j]: lane r = j holds column j of P
                                float* tp = a.transition + (unit_state * KD + r) * KD + 16 * p;
#pragma unroll
                                for (int e = 0; e < 16; e += 4)
                                    *reinterpret_cast<float4*>(tp + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
                            }
                        } else {
                            if (ckpt) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    const int64_t idx = cbase + static_cast<int64_t>(16 * p + e) * a.V;
                                    if (a.ckpt_bf16) static_cast<uint16_t*>(a.ckpt)[idx] = f_to_bf16_bits(x[e]);
                                    else static_cast<float*>(a.ckpt)[idx] = x[e];
                                }
                            }
#pragma unroll
                            for (int e = 0; e < 16; ++e) x[e] *= gnext;
                            tmem_st16(trow + COL_S + 16 * p, *reinterpret_cast<float(*)[16]>(x));
                        }
                    }
                }
                pend_st = !last;
            }
            // the O staging buffer is the next chunk's A: the bulk store must have read it
            if (kFwd && tid == 0) bulk_wait_read_all();
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        if (failed) break;
    }
    if (kFwd && tid == 0) bulk_wait_all();

    if (failed) {
        // Let in-flight copies and products finish (bounded) before TMEM and shared memory go away.
        if (pend_kq) mbar_wait(&sc.bar_kq, ph_kq, budget);
        if (pend_v) mbar_wait(&sc.bar_v, ph_v, budget);
        if (pend_mma) mbar_wait(&sc.bar_mma, ph_mma, budget);
        if (pend_o) mbar_wait(&sc.bar_o, ph_o, budget);
        if (pend_f) mbar_wait(&sc.bar_f, ph_f, budget);
        tmem_wait_st();
        if (tid == 0) {
            atomicCAS(&a.hdr->status, LA_OK, LA_ERR_TIMEOUT);
            if (a.user_status) atomicCAS(a.user_status, LA_OK, LA_ERR_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ WY pass of the two-pass forward
// Every (chunk, head) item of the batch is independent of the state: G, the norms, the
// per-token factors, A, P and T = (I + A)^{-1} are formed exactly as the fused kernel forms them
// (the same functions, so the same bits), and written out as one record per item: T and P as
// bf16 64 x 64 tiles by TMA stores, the factors beta, sx, sq, sd by a bulk copy.  The state pass
// (kModeFwdSplit) then walks each sequence with only the state-dependent products on its chain.
// CTAs of 128 threads, four per SM (52 KB of shared memory, 128 TMEM columns for G, at most 128
// registers a thread); CTA b takes items b, b + grid, ...  Once G is formed the K/Q tile's space
// holds T (fp32), P (bf16) and the solve's scratch; the next item's indices, gates and betas
// are fetched while the current one is formed.
constexpr uint32_t WY_KQ = 0;       // K/Q tile [region][128 rows][128 B] | T fp32 [64][64], P, solve scratch
constexpr uint32_t WY_PB = 16384;   // P bf16 [64][128 B] (in the K/Q tile's space)
constexpr uint32_t WY_Y = 24576;    // solve scratch [4][256] fp32 (in the K/Q tile's space)
constexpr uint32_t WY_M = 32768;    // A fp32 [64][64] | T bf16 [64][128 B]
constexpr uint32_t WY_SC = 49152;   // Scalars without the solve scratch
constexpr uint32_t WY_SMEM = WY_SC + ((kScalarsNoY + 127) & ~127u) + 1024;
constexpr uint32_t WY_TMEM_COLS = 128;

// KIND kWyFwd: the forward's records (queries: P and the query factors); kWySummary: the
// summary's (T and the key factors only, G over the keys alone as the fused summary forms it);
// kWyGdp: Gated DeltaProduct's, chunks of 64 update rows whose query tokens are those whose last
// update row lies in the chunk (at most ceil(64 / n), in the first rows of the query half).
template <int KD, int KIND>
__global__ void __launch_bounds__(kCta, 4)
    gdn_wy_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap wymap, const ChunkArgs a) {
    constexpr bool kQ = KIND != kWySummary;
    constexpr bool kG = KIND == kWyGdp;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Scalars& sc = *reinterpret_cast<Scalars*>(sm + WY_SC);  // (its solve scratch is not used here)
    uint8_t* KQ = sm + WY_KQ;
    float* Tf = reinterpret_cast<float*>(sm + WY_KQ);
    uint8_t* PB = sm + WY_PB;
    float (*Y)[256] = reinterpret_cast<float(*)[256]>(sm + WY_Y);
    float* M = reinterpret_cast<float*>(sm + WY_M);
    uint8_t* TB = sm + WY_M;
    const int tid = threadIdx.x;
    const int r = tid;
    const int HO = a.HV;
    const int NH = kG ? a.gdp_n : 1;            // rows per token on the update timeline
    const int QR = (kChunk + NH - 1) / NH;      // query rows a chunk can hold

    if (tid == 0) sc.status0 = *reinterpret_cast<volatile int32_t*>(&a.hdr->status);
    __syncthreads();
    if (sc.status0 != LA_OK) return;
    const int64_t items = a.hdr->total_chunks * HO;
    if (static_cast<int64_t>(blockIdx.x) >= items) return;

    if (tid < 32) {
        tmem_alloc(&sc.tmem_base, WY_TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sc.bar_kq, 1);
        mbar_init(&sc.bar_mma, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sc.tmem_base;
    const uint32_t trow = tmem + (static_cast<uint32_t>(r & ~31) << 16);
    const uint64_t d_kq = sdesc_sw128(smem_u32(KQ), 16, 1024);
    const uint32_t kq_bytes = KD * 128u + (kQ ? static_cast<uint32_t>(KD / 64) * QR * 128u : 0u);
    const uint64_t budget = a.wait_budget_ns;
    uint32_t ph_kq = 0, ph_mma = 0;
    bool pend_kq = false, pend_mma = false, failed = false;

    // an item's rows: chunk c of sequence seq, head h; first (update) row t0, n valid rows; its
    // query tokens tq0 .. tq0 + nq - 1 relative to the sequence start (GDP), rel0 = 64 c
    auto rows_of = [&](int64_t item, int seq, int64_t& t0, int& n, int& rel0, int& tq0, int& nq) {
        const int64_t chunk = item / HO;
        const int c = static_cast<int>(chunk - a.chunk_off[seq]);
        const int64_t tok_s = cu_get(a.cu, a.cu64, seq);
        const int64_t rows = (cu_get(a.cu, a.cu64, seq + 1) - tok_s) * NH;
        const int64_t left = rows - static_cast<int64_t>(c) * kChunk;
        n = left < kChunk ? static_cast<int>(left) : kChunk;
        rel0 = c * kChunk;
        t0 = tok_s * NH + rel0;
        tq0 = kG ? rel0 / NH : rel0;
        nq = kG ? (rel0 + n) / NH - tq0 : n;
    };
    // a row's gate and beta (threads 0-63)
    auto gates_of = [&](int64_t t0, int n, int h, float& g, float& b) {
        g = b = 0.f;
        if (tid < 64 && tid < n) {
            float gA = 0.f, gdt = 0.f;
            if (a.gate_mode == LA_GATE_SOFTPLUS) {
                gA = -expf(a.a_log[h]);
                gdt = a.dt_bias[h];
            }
            g = gate_row<kG>(a, t0 + tid, h, gA, gdt);
            b = beta_at(a, t0 + tid, h);
        }
    };

    int64_t item = blockIdx.x;
    int64_t t0;
    int n, rel0, tq0, nq;
    rows_of(item, a.chunk_seq[item / HO], t0, n, rel0, tq0, nq);
    float g_cur, b_cur;
    gates_of(t0, n, static_cast<int>(item % HO), g_cur, b_cur);
    for (; item < items; item += gridDim.x) {
        const int h = static_cast<int>(item % HO);
        if (kG && QR < kChunk) {
            // query rows QR .. 63 of the tile get no load: zero them (the space held the previous
            // item's T and scratch), as the fused kernel has them
            for (int e = tid; e < (KD / 64) * (kChunk - QR) * 8; e += kCta) {
                const int rg = e / ((kChunk - QR) * 8), rem = e % ((kChunk - QR) * 8);
                *reinterpret_cast<uint4*>(KQ + rg * 16384 + 8192 + (QR + rem / 8) * 128 + (rem % 8) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // the G product reads them through the async proxy
            __syncthreads();
        }
        if (tid == 0 && !a.test_skip_tile_load) {
            // the previous item's T, P and scratch in this space are dead (the loop ended with a
            // barrier) and its record stores have read their sources
            bulk_wait_read_all();
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sc.bar_kq, kq_bytes);
            const int hk = h / a.group;
#pragma unroll
            for (int rg = 0; rg < KD / 64; ++rg) {
                tma_load_3d(KQ + rg * 16384, &kmap, &sc.bar_kq, rg * 64, hk, static_cast<int>(t0));
                if (kQ)
                    tma_load_3d(KQ + rg * 16384 + 8192, &qmap, &sc.bar_kq, rg * 64, hk, static_cast<int>(t0 / NH));
            }
        }
        pend_kq = !a.test_skip_tile_load;
        // the next item's sequence (its load completes while this item is formed)
        const int64_t nitem = item + gridDim.x;
        const bool has_next = nitem < items;
        const int nseq = has_next ? a.chunk_seq[nitem / HO] : 0;

        bool ok = mbar_wait(&sc.bar_kq, ph_kq, budget, true);
        if (ok) {
            ph_kq ^= 1u;
            pend_kq = false;
        }
        if (tid == 0 && ok) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(128, kQ ? 128 : 64, false, false);
#pragma unroll
            for (int kk = 0; kk < KD / 16; ++kk) {
                const uint64_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                umma_bf16(tmem, d_kq + off, d_kq + off, idesc, kk > 0);
            }
            umma_commit(&sc.bar_mma);
        }
        pend_mma = ok;
        if (tid < 64) {
            float x = (tid < n) ? g_cur * kLog2e : 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if ((tid & 31) >= off) x += y;
            }
            sc.bw[tid] = x;
        }
        {
            const bool okg = mbar_wait(&sc.bar_mma, ph_mma, budget, true);
            if (okg) {
                ph_mma ^= 1u;
                pend_mma = false;
            }
            ok = ok && okg;
        }
        tc_fence_after();
        float g64[64];
        g_rows_and_norms<kQ>(trow, 0, r, n, nq, a.l2norm, g64, sc);
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        const bool fast = chunk_scalars<kQ, kG>(sc, tid, n, nq, tq0, rel0, NH, b_cur, a.scale);
        build_a_p<kQ, kG>(g64, sc, M, PB, fast, r, nq, tq0, rel0, NH, a.scale);
        // the next item's rows, gates and betas (in flight during the solve)
        int64_t nt0 = t0;
        int nn = 0, nrel0 = 0, ntq0 = 0, nnq = 0;
        float g_nx = 0.f, b_nx = 0.f;
        if (has_next) {
            rows_of(nitem, nseq, nt0, nn, nrel0, ntq0, nnq);
            gates_of(nt0, nn, static_cast<int>(nitem % HO), g_nx, b_nx);
        }
        __syncthreads();  // A and P complete; the K/Q tile (read by the finished G product) becomes T's space
        solve_unit_lower(M, Tf, Y, tid);
        t_to_bf16(Tf, TB, tid);
        if (a.wy_tlo) t_lo_store(Tf, a.wy_tlo + item * static_cast<int64_t>(kWyTileBytes), tid);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&wymap, TB, 0, static_cast<int>(item), 0);
            if (kQ) tma_store_3d(&wymap, PB, 0, static_cast<int>(item), 64);
            bulk_store(a.wy + item * static_cast<int64_t>(kWyRecordBytes) + 2 * kWyTileBytes, sc.bet,
                       static_cast<uint32_t>(kWyFactorBytes));
            bulk_commit_group();
        }
        __syncthreads();  // T (fp32) and the scratch are read: the next item's tile may land in their space
        t0 = nt0;
        n = nn;
        rel0 = nrel0;
        tq0 = ntq0;
        nq = nnq;
        g_cur = g_nx;
        b_cur = b_nx;
    }
    if (tid == 0) bulk_wait_all();
    if (failed) {
        if (pend_kq) mbar_wait(&sc.bar_kq, ph_kq, budget);
        if (pend_mma) mbar_wait(&sc.bar_mma, ph_mma, budget);
        if (tid == 0) {
            atomicCAS(&a.hdr->status, LA_OK, LA_ERR_TIMEOUT);
            if (a.user_status) atomicCAS(a.user_status, LA_OK, LA_ERR_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tmem, WY_TMEM_COLS);
}

// ------------------------------------------------------------------ host side
// CTAs of kCta threads resident per SM, at most `cap`: the occupancy API's answer or the one
// from the hardware limits (registers allocated per warp in units of 256, shared memory per SM
// minus the per-block reserve), whichever is larger.  A CTA that cannot be resident yet simply
// starts later and finds no work left, so overestimating costs nothing.
static cudaError_t resident_per_sm(const void* fn, uint32_t smem, int cap, int device, int* out, int threads = kCta) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    int smem_sm = 0, reserve = 0, regs_sm = 0;
    if (cudaFuncGetAttributes(&fa, fn) == cudaSuccess &&
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) == cudaSuccess &&
        cudaDeviceGetAttribute(&reserve, cudaDevAttrReservedSharedMemoryPerBlock, device) == cudaSuccess &&
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, device) == cudaSuccess) {
        const int regs_cta = ((fa.numRegs * 32 + 255) / 256) * 256 * (threads / 32);
        const int by_regs = regs_cta > 0 ? regs_sm / regs_cta : 1;
        const int by_smem = smem_sm / (static_cast<int>(smem) + reserve);
        const int hw = by_regs < by_smem ? by_regs : by_smem;
        if (hw > per_sm) per_sm = hw;
    }
    if (per_sm > cap) per_sm = cap;
    if (per_sm < 1) per_sm = 1;
    *out = per_sm;
    return cudaSuccess;
}

// Ranges per unit for a forward whose units fill between one and four waves: the count in
// 2..8 that minimises the estimated time, waves x (chunks per range + two chunks for a
// launch's start and drain, as measured), against whole units (ceil(units / slots) waves of
// `chunks`), from the mean sequence length.  1 when no count saves at least 5 %.  The kernel
// still walks whole units when the lengths turn out spread (the prologue's decision).
static int fwd_pieces(int64_t units, int64_t slots, int64_t chunks) {
    if (chunks < 2) return 1;
    const double whole = static_cast<double>((units + slots - 1) / slots) * static_cast<double>(chunks);
    int best = 1;
    double best_t = whole;
    for (int p = 2; p <= 8 && p <= chunks; ++p) {
        const int64_t waves = (units * p + slots - 1) / slots;
        const double t = static_cast<double>(waves) * (static_cast<double>(chunks) / p + 2.0);
        if (t < best_t) {
            best_t = t;
            best = p;
        }
    }
    return best_t < 0.95 * whole ? best : 1;
}

template <int KD, int MODE>
static cudaError_t launch_one(const ChunkArgs& a, const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                              const CUtensorMap& om, const CUtensorMap& wm, int device, cudaStream_t s) {
    auto* fn = gdn_chunk_kernel<KD, MODE>;
    constexpr uint32_t smem = smem_map(MODE).total;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // Ask for the largest shared-memory carveout so two CTAs fit per SM.
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = resident_per_sm(reinterpret_cast<const void*>(fn), smem, 2, device, &per_sm, chunk_threads(MODE));
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    const int64_t slots = static_cast<int64_t>(per_sm) * sms;
    ChunkArgs b = a;
    b.pieces = 1;
    b.item_base = 0;
    b.items = 0;
    if ((MODE == kModeSummary || MODE == kModeSummarySplit) && b.num_units > slots) b.pieces = kSumPieces;
    if ((MODE == kModeFwd || MODE == kModeFwdSplit) && b.final_state && !b.final_bf16 && b.num_units > slots) {
        if (a.pieces_request > 0) b.pieces = a.pieces_request;
        else if (b.num_units <= 4 * slots)
            b.pieces = fwd_pieces(b.num_units, slots, (b.T / (b.N > 0 ? b.N : 1) + kChunk - 1) / kChunk);
    }
    if (b.pieces > 1) {
        // ranges of every unit, one wave per launch: item r * units + u's predecessor (u, r - 1)
        // is `units` > `slots` items earlier, so it ran in an earlier launch
        const int64_t items = b.num_units * b.pieces;
        for (int64_t base = 0; base < items; base += slots) {
            b.item_base = base;
            b.items = items - base < slots ? items - base : slots;
            fn<<<static_cast<int>(b.items), chunk_threads(MODE), smem, s>>>(qm, km, vm, om, wm, b);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    const int grid = static_cast<int>(b.num_units < slots ? b.num_units : slots);
    if (grid <= 0) return cudaSuccess;
    fn<<<grid, chunk_threads(MODE), smem, s>>>(qm, km, vm, om, wm, b);
    return cudaGetLastError();
}

cudaError_t launch_chunk_kernel(const ChunkArgs& a, const CUtensorMap& qm, const CUtensorMap& km,
                                const CUtensorMap& vm, const CUtensorMap& om, const CUtensorMap& wm, int mode,
                                cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (a.K == 128) {
        switch (mode) {
            case kModeGdp: return launch_one<128, kModeGdp>(a, qm, km, vm, om, wm, dev, s);
            case kModeFwdSplit: return launch_one<128, kModeFwdSplit>(a, qm, km, vm, om, wm, dev, s);
            case kModeSummary: return launch_one<128, kModeSummary>(a, qm, km, vm, om, wm, dev, s);
            case kModeSummarySplit: return launch_one<128, kModeSummarySplit>(a, qm, km, vm, om, wm, dev, s);
            case kModeGdpSplit: return launch_one<128, kModeGdpSplit>(a, qm, km, vm, om, wm, dev, s);
            default: return launch_one<128, kModeFwd>(a, qm, km, vm, om, wm, dev, s);
        }
    }
    switch (mode) {
        case kModeGdp: return launch_one<64, kModeGdp>(a, qm, km, vm, om, wm, dev, s);
        case kModeFwdSplit: return launch_one<64, kModeFwdSplit>(a, qm, km, vm, om, wm, dev, s);
        case kModeSummary: return launch_one<64, kModeSummary>(a, qm, km, vm, om, wm, dev, s);
        case kModeSummarySplit: return launch_one<64, kModeSummarySplit>(a, qm, km, vm, om, wm, dev, s);
        case kModeGdpSplit: return launch_one<64, kModeGdpSplit>(a, qm, km, vm, om, wm, dev, s);
        default: return launch_one<64, kModeFwd>(a, qm, km, vm, om, wm, dev, s);
    }
}

template <int KD, int KIND>
static cudaError_t launch_wy(const ChunkArgs& a, const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& wm,
                             int device, cudaStream_t s) {
    auto* fn = gdn_wy_kernel<KD, KIND>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, WY_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    // four per SM: their 512 TMEM columns fill the SM's, and registers and shared memory allow it
    e = resident_per_sm(reinterpret_cast<const void*>(fn), WY_SMEM, 4, device, &per_sm);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    // whole waves, at most one CTA per item of the host's bound (a.num_units); the kernel reads
    // the item count the prologue wrote, and CTAs past it return at once
    const int64_t bound = a.num_units;
    int64_t grid = static_cast<int64_t>(per_sm) * sms;
    if (grid > bound) grid = bound;
    if (grid <= 0) return cudaSuccess;
    fn<<<static_cast<int>(grid), kCta, WY_SMEM, s>>>(qm, km, wm, a);
    return cudaGetLastError();
}

cudaError_t launch_wy_kernel(const ChunkArgs& a, const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& wm,
                             int kind, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (kind == kWySummary)
        return a.K == 128 ? launch_wy<128, kWySummary>(a, qm, km, wm, dev, s) : launch_wy<64, kWySummary>(a, qm, km, wm, dev, s);
    if (kind == kWyGdp)
        return a.K == 128 ? launch_wy<128, kWyGdp>(a, qm, km, wm, dev, s) : launch_wy<64, kWyGdp>(a, qm, km, wm, dev, s);
    return a.K == 128 ? launch_wy<128, kWyFwd>(a, qm, km, wm, dev, s) : launch_wy<64, kWyFwd>(a, qm, km, wm, dev, s);
}

}  // namespace la
