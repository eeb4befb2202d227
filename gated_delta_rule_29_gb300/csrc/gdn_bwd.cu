// gdn_bwd.cu -- the backward of the chunked Gated DeltaNet forward.
//
// Method (cuDNN Linear Attention page: every variant has a full backward, which reuses the
// forward's state checkpoints at the chunk cadence).  Within a 64-token chunk with entering
// state S, b_i the inclusive cumsum of g (natural log), gamma_i = e^{b_i}, Gamma_ij =
// e^{b_i - b_j}, Gamma_Cj = e^{b_last - b_j}:
//   A = strict_tril(beta_i (k_i . k_j) Gamma_ij),  T = (I + A)^{-1}
//   x = K S,  Y = diag(beta) V - diag(beta gamma) x,  D = T Y
//   O = scale (diag(gamma) Q S + P D),  P = tril_incl((q_i . k_j) Gamma_ij)
//   S_next = gamma_last S + K^T diag(Gamma_C) D
// Given dO and dS_next, reverse mode gives (all derived from those four lines):
//   dD = scale P^T dO + diag(Gamma_C) K dS_next,  dY = T^T dD,  dV = diag(beta) dY,
//   dx = -diag(beta gamma) dY,  dS = gamma_last dS_next + K^T dx + scale Q^T diag(gamma) dO,
//   dA = -strict_tril(dY D^T),  dP = scale tril_incl(dO D^T),
//   dK = dx S^T + diag(Gamma_C) D dS_next^T + M K + M^T K + H^T Q,  M = dA (.) beta_i Gamma,
//   dQ = scale diag(gamma) dO S^T + H K,  H = dP (.) Gamma,
//   dbeta_i = sum_v dY (V - gamma x) + sum_j dA_ij (k_i . k_j) Gamma_ij,
//   db collects every gamma / Gamma dependence and dg_j = sum_{i >= j} db_i,
// then the L2-norm backward for q and k and the sum over grouped value heads.  K and Q above
// are the normalised rows; the kernel keeps the raw rows (exact bf16 values) and applies the
// inverse norms as row or column scales of the other operand.
//
// Mapping.  One CTA of 256 threads (8 warps) per (sequence, head) walks the chunks in reverse
// and carries dS in a global per-unit buffer.  When the units outnumber the CTAs that fit on the
// GPU at once, each unit's chunks are cut into four consecutive ranges: launch after launch, one
// wave each, the work items are the units' last ranges, then the ranges before them, so that a
// range's dS comes from the previous launch through the global buffer (exact fp32), the results
// are the same bits as one walk, and the units fill 1.75 waves instead of 2 (e.g. 256 on 152).  The value columns are independent chains (each
// column of S evolves on its own), so a chunk is processed in 16-column tiles of S, dS, V and
// dO; the tile-independent parts (K, Q, A, T, P, the decays) are formed once per chunk in
// shared memory and the cross-column sums (dA, dP, dK, dQ, dbeta, db) accumulate over the
// tiles.  The next tile's S, dS, V and dO stream in with cp.async while a tile is computed.
// Every product runs on warp-level tensor-core MMAs (m16n8k8, tf32 operands, fp32
// accumulation) with each inexact fp32 operand split into a tf32 head and a tf32 remainder:
// three products per MMA (head x head, head x rest, rest x head), two when one operand is an
// exact bf16 input (k, q, dO), which keeps fp32-level accuracy; the products that reach only
// the bf16 dq and dk take one MMA on rounded operands.  The dK and dQ rows stay in the warps'
// accumulator fragments for the whole chunk: warps 0-3 own dK rows 16 w .. 16 w + 15, warps 4-7
// the same dQ rows.  The chunk entering states come from the forward kernel run with fp32
// checkpoints every 64 tokens.  With the forward's input transforms the gate and beta are
// transformed as they are loaded and dg, dbeta go back through the chain rule (d_a_log and
// d_dt_bias are per-unit sums added in sequence order by a second small kernel).
//
// State-only mode (gdn_summary_bwd): the recursion of dS needs no forward state, so only
// K dS, dD, dY and the dS update run per tile, no checkpoints are read, and the gradient
// entering the span is the result.
#include <cuda_bf16.h>

#include <atomic>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"
#include "ptx.cuh"

namespace la {
namespace {

constexpr int kBT = 256;   // threads
constexpr int kC = 64;     // chunk
constexpr int kVT = 16;    // value columns per tile

__device__ __forceinline__ uint16_t f2b(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ float b2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Shared-memory layout of the key-length rows (K, Q, S^T, dS^T): the four KD/4-column slices
// are staggered by 4 words, and the row stride is 12 mod 32 words, so that the MMA operand
// fragments of row-major reads (8 rows x 4 columns per warp) hit 32 distinct banks.
template <int KD>
__device__ __forceinline__ int colp(int d) { return d + (d / (KD / 4)) * 4; }

template <int KD>
struct BwdSmem {
    static constexpr int PK = KD + 12;  // row stride of K / Q / S^T / dS^T
    static constexpr int PC = kC + 4;   // row stride of the 64 x 64 matrices and of the tiles read
                                        // along the token index (4 mod 32 words)
    static constexpr int PT = kC + 8;   // row stride of the tiles read along the value column
                                        // (8 mod 32 words): both fragment patterns conflict free
    float Kr[kC * PK];      // raw keys (rows past the end are zero); k_hat = rk k
    float Qr[kC * PK];      // raw queries; q_hat = rq q
    float Tm[kC * PC];      // T = (I + A)^{-1}
    float Pt[kC * PC];      // P transposed: Pt[j][i] = P_ij (P lower incl.)
    // strictly lower part: dA accumulated over the tiles, then M; strictly upper part: the
    // transpose of Gk_ij = (k_hat_i . k_hat_j) Gamma_ij (j < i) stored at [j][i]; diagonal zero
    float dA[kC * PC];
    float dP[kC * PC];      // accumulated over tiles, then H
    // value tiles, stored transposed: row = value column cc, contiguous along the token / key index;
    // S and dS are double buffered so that the next tile streams in while this one is computed
    float SJ[2][kVT * PK];  // S[:, tile]^T
    float dSJ[2][kVT * PK]; // dS_next[:, tile]^T
    // per tile, [cc][i]: Y, dD, dY, dO with stride PC (MMA operands along the tokens), D and
    // copies of dY and dO with stride PT (MMA operands along the value columns)
    float Y[kVT * PC], dD[kVT * PC], dY[kVT * PC], OJ[kVT * PC];
    float D[kVT * PT], dYc[kVT * PT], OJc[kVT * PT];
    uint16_t Vb[kC * kVT], Ob[kC * kVT];  // the next tile's raw V and dO rows (bf16, token-major)
    // per-row partial sums over each 8-column half of the tile, formed in the MMA epilogues:
    // [0] sum dY (V - gamma x), [1] sum dY x, [2] sum dO (Q S), [3] sum (K dS) D
    float part[4][2][kC];
    float beta[kC], b[kC], gam[kC], GC[kC], rk[kC], rq[kC];
    float cx[kC], co[kC];   // -rk beta gamma (K^T dx) and scale rq gamma (Q^T dO) row factors
    float dbeta[kC], db[kC], wv[kC];
    float gt[kC];           // the chunk's log decays (after the gate transform)
    float red[kBT / 32];
};
static_assert(sizeof(BwdSmem<128>) <= 227 * 1024, "backward shared memory exceeds the per-CTA limit");

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// x = head + rest: the head is x with its 13 low mantissa bits cleared (a tf32 value), the rest
// x - head exactly (|rest| < 2^-10 |x|); the tensor core reads the rest's top 19 bits, so the
// split represents x to about 2^-20 relative.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hd, uint32_t& rs) {
    hd = __float_as_uint(x) & 0xFFFFE000u;
    rs = __float_as_uint(x - __uint_as_float(hd));
}
// A fragment (16 x 8, rows m0.., columns k0..) of an element function, rounded to tf32 (for the
// products that only feed the bf16 gradients dq and dk: one MMA, ~2^-11 relative per operand).
template <class F>
__device__ __forceinline__ void frag_a_round(F f, int m0, int k0, int g, int t, uint32_t (&a)[4]) {
    a[0] = to_tf32(f(m0 + g, k0 + t));
    a[1] = to_tf32(f(m0 + g + 8, k0 + t));
    a[2] = to_tf32(f(m0 + g, k0 + t + 4));
    a[3] = to_tf32(f(m0 + g + 8, k0 + t + 4));
}
// A fragment (16 x 8, rows m0.., columns k0..) of an element function, split in two.
template <class F>
__device__ __forceinline__ void frag_a_split(F f, int m0, int k0, int g, int t, uint32_t (&hd)[4], uint32_t (&rs)[4]) {
    split_tf32(f(m0 + g, k0 + t), hd[0], rs[0]);
    split_tf32(f(m0 + g + 8, k0 + t), hd[1], rs[1]);
    split_tf32(f(m0 + g, k0 + t + 4), hd[2], rs[2]);
    split_tf32(f(m0 + g + 8, k0 + t + 4), hd[3], rs[3]);
}
// B fragment (8 x 8, rows k0.., columns n0..) of an element function, split in two.
template <class F>
__device__ __forceinline__ void frag_b_split(F f, int k0, int n0, int g, int t, uint32_t (&hd)[2], uint32_t (&rs)[2]) {
    split_tf32(f(k0 + t, n0 + g), hd[0], rs[0]);
    split_tf32(f(k0 + t + 4, n0 + g), hd[1], rs[1]);
}
// c += A B with both operands split (three products), or with an exact A operand (two).
__device__ __forceinline__ void mma3(float (&c)[4], const uint32_t (&ah)[4], const uint32_t (&ar)[4],
                                     const uint32_t (&bh)[2], const uint32_t (&br)[2]) {
    mma_tf32_16x8x8(c, ar, bh);
    mma_tf32_16x8x8(c, ah, br);
    mma_tf32_16x8x8(c, ah, bh);
}
__device__ __forceinline__ void mma2a(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&bh)[2],
                                      const uint32_t (&br)[2]) {
    mma_tf32_16x8x8(c, a, br);
    mma_tf32_16x8x8(c, a, bh);
}
__device__ __forceinline__ uint32_t fbits(float x) { return __float_as_uint(x); }
// The same three products with the head x head term in c and the two rest terms in r
// (two independent accumulation chains; the caller adds r to c at the end).
__device__ __forceinline__ void mma3s(float (&c)[4], float (&r)[4], const uint32_t (&ah)[4], const uint32_t (&ar)[4],
                                      const uint32_t (&bh)[2], const uint32_t (&br)[2]) {
    mma_tf32_16x8x8(r, ar, bh);
    mma_tf32_16x8x8(r, ah, br);
    mma_tf32_16x8x8(c, ah, bh);
}

// The recurrence's log decay and beta from the raw inputs (the forward's input transforms:
// softplus gate gA softplus(g + gdt) with gA = -exp(a_log[h]), bounded gate lb sigmoid(g), beta
// sigmoid of fp32 or bf16 logits).
__device__ __forceinline__ float raw_gate(const BwdArgs& a, int64_t t, int h) { return a.g[t * a.g_st + h * a.g_sh]; }
__device__ __forceinline__ float raw_beta(const BwdArgs& a, int64_t t, int h) {
    const int64_t i = t * a.b_st + h * a.b_sh;
    return a.beta_bf16 ? b2f(reinterpret_cast<const uint16_t*>(a.beta)[i]) : a.beta[i];
}
__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }
__device__ __forceinline__ float gate_of(const BwdArgs& a, float x, float gA, float gdt) {
    if (a.gate_mode == LA_GATE_SOFTPLUS) {
        const float z = x + gdt;
        return gA * (z > 20.f ? z : log1pf(expf(z)));
    }
    if (a.gate_mode == LA_GATE_SIGMOID_BOUND) return a.gate_lb * sigmoidf_(x);
    return x;
}

// Sum over the four lanes of a quad (the accumulator fragment's column pairs of one row).
__device__ __forceinline__ float quad_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// The 20 lower (16-row, 8-column) output tiles of a 64 x 64 lower-triangular product, in order.
__device__ __forceinline__ void lower_tile(int p, int& mt, int& nt) {
    mt = p < 2 ? 0 : (p < 6 ? 1 : (p < 12 ? 2 : 3));
    nt = p - (mt == 0 ? 0 : (mt == 1 ? 2 : (mt == 2 ? 6 : 12)));
}

template <int KD, int VD>
__global__ void __launch_bounds__(kBT, 1) gdn_bwd_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BwdSmem<KD>& s = *reinterpret_cast<BwdSmem<KD>*>(smem_raw);
    constexpr int PK = BwdSmem<KD>::PK;
    constexpr int PC = BwdSmem<KD>::PC;
    constexpr int PT = BwdSmem<KD>::PT;
    constexpr int NT = KD / 8;    // 8-column key tiles of the dK / dQ rows
    constexpr int MTW = KD / 64;  // 16-row key tiles of dS per warp in the dS update
    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    if (tid == 0) s.red[0] = __int_as_float(*reinterpret_cast<const volatile int32_t*>(&a.hdr->status));
    __syncthreads();
    if (__float_as_int(s.red[0]) != LA_OK) return;  // bad cu_seqlens: the forward ran nothing
    __syncthreads();
    const int HO = a.HV;
    const int U = a.N * HO;
    const int item = a.item_base + static_cast<int>(blockIdx.x);
    const int P = a.pieces;
    const int piece = P - 1 - item / U;  // the unit's chunk range, counted from its start
    const int unit = item % U;
    const int seq = unit / HO, h = unit % HO;
    const int hk = h / a.group;
    const int64_t ts = a.cu64 ? static_cast<const int64_t*>(a.cu)[seq] : static_cast<const int32_t*>(a.cu)[seq];
    const int64_t te = a.cu64 ? static_cast<const int64_t*>(a.cu)[seq + 1] : static_cast<const int32_t*>(a.cu)[seq + 1];
    const int64_t L = te - ts;
    const int nch = static_cast<int>((L + kC - 1) / kC);
    const int lo = static_cast<int>(static_cast<int64_t>(piece) * nch / P);  // chunks lo .. hi - 1
    const int hi = static_cast<int>(static_cast<int64_t>(piece + 1) * nch / P);
    const int64_t KV = static_cast<int64_t>(KD) * VD;
    float* dSg = a.dS_work + static_cast<int64_t>(unit) * KV;  // carried dS (global, L2 resident)

    // dS after the last token: d_final_state or zero (set by the last range, which runs first)
    if (piece == P - 1)
        for (int64_t e = tid; e < KV; e += kBT) dSg[e] = a.dfinal ? a.dfinal[unit * KV + e] : 0.f;
    __syncthreads();

    constexpr int KSL = KD / 4;
    const bool so = a.state_only != 0;  // the entering-state gradient alone

    // Asynchronous fetch of one value tile (chunk cc, columns j0..j0+15) into buffer pb: the
    // S and dS columns (4-byte copies, transposed into the tile layout) and the raw V and dO
    // rows (4-byte copies of bf16 pairs when the operands allow it, else plain loads).
    auto fetch_tile = [&](int cc, int j0, int pb) {
        const int64_t ft0 = ts + static_cast<int64_t>(cc) * kC;
        const int fn = static_cast<int>(L - static_cast<int64_t>(cc) * kC < kC ? L - static_cast<int64_t>(cc) * kC : kC);
        if (!so) {
            const float* Sf = a.ckpt + ((a.ckpt_off[seq] + cc) * HO + h) * KV;
#pragma unroll
            for (int e = tid; e < KD * kVT; e += kBT) {
                const int r = e / kVT, col = e % kVT;
                cp_async4(&s.SJ[pb][col * PK + colp<KD>(r)], Sf + r * VD + j0 + col);
            }
        }
#pragma unroll
        for (int e = tid; e < KD * kVT; e += kBT) {
            const int r = e / kVT, col = e % kVT;
            cp_async4(&s.dSJ[pb][col * PK + colp<KD>(r)], dSg + r * VD + j0 + col);
        }
        for (int e = tid; e < kC * kVT / 2; e += kBT) {
            const int i = e / (kVT / 2), c2 = 2 * (e % (kVT / 2));
            uint16_t* vd = &s.Vb[i * kVT + c2];
            uint16_t* od = &s.Ob[i * kVT + c2];
            if (i >= fn) {
                *reinterpret_cast<uint32_t*>(vd) = 0u;
                *reinterpret_cast<uint32_t*>(od) = 0u;
            } else {
                const uint16_t* os = a.dout + (ft0 + i) * a.do_st + h * a.do_sh + j0 + c2;
                if (a.vo_async) cp_async4(od, os);
                else {
                    od[0] = os[0];
                    od[1] = os[1];
                }
                if (!so) {
                    const uint16_t* vs = a.v + (ft0 + i) * a.v_st + h * a.v_sh + j0 + c2;
                    if (a.vo_async) cp_async4(vd, vs);
                    else {
                        vd[0] = vs[0];
                        vd[1] = vs[1];
                    }
                }
            }
        }
        cp_async_commit();
    };
    int pb = 0;  // buffer of the current tile
    if (hi > lo) fetch_tile(hi - 1, 0, 0);

    const bool kwarp = w < 4;  // owns dK_hat rows (else dQ_hat rows) 16 (w % 4) .. + 15
    const int om0 = 16 * (w & 3);
    const float gA = a.gate_mode == LA_GATE_SOFTPLUS ? -expf(a.a_log[h]) : 0.f;
    const float gdt = a.gate_mode == LA_GATE_SOFTPLUS ? a.dt_bias[h] : 0.f;
    float pa_log = 0.f, pa_dt = 0.f;  // this token slot's sums for d_a_log and d_dt_bias (tid < 64)

    for (int c = hi - 1; c >= lo; --c) {
        const int64_t t0 = ts + static_cast<int64_t>(c) * kC;
        const int n = static_cast<int>(L - static_cast<int64_t>(c) * kC < kC ? L - static_cast<int64_t>(c) * kC : kC);

        // ---- chunk-level quantities: raw rows, norms, decays, Gk, P, T
        {
            // 8 bf16 (16 bytes) per load (k and q rows are 16-byte aligned: TMA operand rules);
            // every load of the thread is issued before the first is used
            constexpr int LPT = kC * KD / 8 / kBT;  // 16-byte pieces per thread and matrix
            uint4 kw[LPT], qw[LPT];
#pragma unroll
            for (int x = 0; x < LPT; ++x) {
                const int e = tid + x * kBT;
                const int i = e / (KD / 8), d = (e % (KD / 8)) * 8;
                kw[x] = qw[x] = make_uint4(0u, 0u, 0u, 0u);
                if (i < n) {
                    kw[x] = *reinterpret_cast<const uint4*>(a.k + (t0 + i) * a.k_st + hk * a.k_sh + d);
                    qw[x] = *reinterpret_cast<const uint4*>(a.q + (t0 + i) * a.q_st + hk * a.q_sh + d);
                }
            }
#pragma unroll
            for (int x = 0; x < LPT; ++x) {
                const int e = tid + x * kBT;
                const int i = e / (KD / 8), d = (e % (KD / 8)) * 8;
                float* kd = &s.Kr[i * PK + colp<KD>(d)];
                float* qd = &s.Qr[i * PK + colp<KD>(d)];
                const uint32_t kk[4] = {kw[x].x, kw[x].y, kw[x].z, kw[x].w}, qq[4] = {qw[x].x, qw[x].y, qw[x].z, qw[x].w};
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    kd[2 * y] = __uint_as_float(kk[y] << 16);
                    kd[2 * y + 1] = __uint_as_float(kk[y] & 0xFFFF0000u);
                    qd[2 * y] = __uint_as_float(qq[y] << 16);
                    qd[2 * y + 1] = __uint_as_float(qq[y] & 0xFFFF0000u);
                }
            }
        }
        if (tid < kC) {
            const int i = tid;
            float bt = 0.f, gt = 0.f;
            if (i < n) {
                bt = raw_beta(a, t0 + i, h);
                if (a.beta_sigmoid) bt = sigmoidf_(bt);
                gt = gate_of(a, raw_gate(a, t0 + i, h), gA, gdt);
            }
            s.beta[i] = bt;
            s.b[i] = gt;
            s.gt[i] = gt;
        }
        __syncthreads();
        {
            // row norms: four threads per row (rows = tid / 4), quarter rows each
            const int i = tid >> 2, q4 = tid & 3;
            float sk = 0.f, sq = 0.f;
#pragma unroll 4
            for (int d = q4 * KSL; d < (q4 + 1) * KSL; d += 4) {
                const float4 kv = ld4(&s.Kr[i * PK + colp<KD>(d)]), qv = ld4(&s.Qr[i * PK + colp<KD>(d)]);
                sk = dot4(kv, kv, sk);
                sq = dot4(qv, qv, sq);
            }
            sk += __shfl_xor_sync(0xffffffffu, sk, 1);
            sk += __shfl_xor_sync(0xffffffffu, sk, 2);
            sq += __shfl_xor_sync(0xffffffffu, sq, 1);
            sq += __shfl_xor_sync(0xffffffffu, sq, 2);
            if (q4 == 0) {
                s.rk[i] = (i < n && a.l2norm) ? 1.0f / sqrtf(sk + 1e-6f) : (i < n ? 1.f : 0.f);
                s.rq[i] = (i < n && a.l2norm) ? 1.0f / sqrtf(sq + 1e-6f) : (i < n ? 1.f : 0.f);
            }
        }
        if (tid < 32) {
            // chunk-local inclusive cumsum of g (rows past the end carry g = 0)
            float x0 = s.b[tid], x1 = s.b[tid + 32];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y0 = __shfl_up_sync(0xffffffffu, x0, off), y1 = __shfl_up_sync(0xffffffffu, x1, off);
                if (tid >= off) {
                    x0 += y0;
                    x1 += y1;
                }
            }
            x1 += __shfl_sync(0xffffffffu, x0, 31);
            s.b[tid] = x0;
            s.b[tid + 32] = x1;
        }
        __syncthreads();
        if (tid < kC) {
            const int i = tid;
            const float bl = s.b[n - 1];
            const float gm = expf(s.b[i]);
            s.gam[i] = gm;
            s.GC[i] = i < n ? expf(bl - s.b[i]) : 0.f;
            s.cx[i] = -s.rk[i] * s.beta[i] * gm;
            s.co[i] = a.scale * s.rq[i] * gm;
            s.dbeta[i] = 0.f;
            s.db[i] = 0.f;
        }
        // Gk = rk_i rk_j (k_i . k_j) Gamma_ij and P = rq_i rk_j (q_i . k_j) Gamma_ij on the
        // lower 16 x 8 tiles (the raw rows are exact in tf32: one product per MMA)
#pragma unroll
        for (int jx = 0; jx < 5; ++jx) {  // five of the 40 (tile, product) jobs per warp
            const int job = w + 8 * jx;
            int mt, nt;
            lower_tile(job >> 1, mt, nt);
            const bool isP = job & 1;
            const float* Ar = isP ? s.Qr : s.Kr;
            const int m0 = 16 * mt, n0 = 8 * nt;
            float cf[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int k0 = 0; k0 < KD; k0 += 8) {
                const int kp = colp<KD>(k0) + t;
                const uint32_t af[4] = {fbits(Ar[(m0 + g) * PK + kp]), fbits(Ar[(m0 + g + 8) * PK + kp]),
                                        fbits(Ar[(m0 + g) * PK + kp + 4]), fbits(Ar[(m0 + g + 8) * PK + kp + 4])};
                const uint32_t bf[2] = {fbits(s.Kr[(n0 + g) * PK + kp]), fbits(s.Kr[(n0 + g) * PK + kp + 4])};
                mma_tf32_16x8x8(cf, af, bf);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = m0 + g + 8 * (e >> 1), j = n0 + 2 * t + (e & 1);
                const float G = j <= i ? expf(s.b[i] - s.b[j]) : 0.f;
                if (isP) {
                    s.Pt[j * PC + i] = s.rq[i] * s.rk[j] * cf[e] * G;
                    s.dP[i * PC + j] = 0.f;
                } else {
                    if (j <= i) s.dA[i * PC + j] = 0.f;                             // dA accumulator, diagonal
                    if (j < i) s.dA[j * PC + i] = s.rk[i] * s.rk[j] * cf[e] * G;   // Gk_ij, transposed
                }
            }
        }
        __syncthreads();
        {
            // T = (I + A)^{-1}, A = strict_tril(beta_i Gk_ij), in 16 x 16 blocks: the diagonal
            // blocks by substitution (warp w, lane = column), then the blocks below by
            // T[bi][bj] = -T[bi][bi] sum_{m = bj}^{bi - 1} A[bi][m] T[m][bj], one level of block
            // distance at a time (scratch: the dD tile, not yet in use)
            if (w < 4 && lane < 16) {
                const int o = 16 * w, cc = lane;
                float acc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float tj = ((j == cc) ? 1.f : 0.f) - acc[j];
                    s.Tm[(o + j) * PC + o + cc] = tj;
#pragma unroll
                    for (int i = j + 1; i < 16; ++i)
                        acc[i] = fmaf(s.beta[o + i] * s.dA[(o + j) * PC + o + i], tj, acc[i]);
                }
            }
            // the blocks above the diagonal are zero
            for (int e = tid; e < 6 * 256; e += kBT) {
                const int blk = e >> 8, i = (e >> 4) & 15, j = e & 15;
                const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                s.Tm[(16 * bi + i) * PC + 16 * bj + j] = 0.f;
            }
            __syncthreads();
            float* Ysc = s.dD + w * 256;
#pragma unroll 1
            for (int d = 1; d < 4; ++d) {
                if (w < 4 - d) {
                    const int bj = w, bi = w + d;
                    const int r = lane >> 1, c0 = (lane & 1) * 8;
                    float y[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) y[x] = 0.f;
                    for (int m = 16 * bj; m < 16 * bi; ++m) {
                        const float am = s.beta[16 * bi + r] * s.dA[m * PC + 16 * bi + r];
#pragma unroll
                        for (int x = 0; x < 8; ++x) y[x] = fmaf(am, s.Tm[m * PC + 16 * bj + c0 + x], y[x]);
                    }
#pragma unroll
                    for (int x = 0; x < 8; ++x) Ysc[r * 16 + c0 + x] = y[x];
                    __syncwarp();
                    float tt[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) tt[x] = 0.f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float tk = s.Tm[(16 * bi + r) * PC + 16 * bi + k];
#pragma unroll
                        for (int x = 0; x < 8; ++x) tt[x] = fmaf(tk, Ysc[k * 16 + c0 + x], tt[x]);
                    }
#pragma unroll
                    for (int x = 0; x < 8; ++x) s.Tm[(16 * bi + r) * PC + 16 * bj + c0 + x] = -tt[x];
                    __syncwarp();
                }
                __syncthreads();
            }
        }

        // dK_hat (warps 0-3) or the unscaled dQ_hat sum (warps 4-7) of rows om0 .. om0 + 15:
        // accumulator fragments, column tile nd holds key columns 8 nd + 2 t, + 1
        float acc[NT][4];
#pragma unroll
        for (int nd = 0; nd < NT; ++nd) acc[nd][0] = acc[nd][1] = acc[nd][2] = acc[nd][3] = 0.f;

        // ---- the value tiles: independent columns of S and dS
        for (int j0 = 0; j0 < VD; j0 += kVT) {
            cp_async_wait_all();
            __syncthreads();  // this tile's S, dS, V, dO have landed; the previous tile is done
            if (tid == 0 && j0 > 0 && !so) {
                // the previous tile's Gamma_C terms of S_next and the decay of S into S_next
                float p = 0.f, wsum = 0.f;
                for (int x = 0; x < kBT / 32; ++x) p += s.red[x];
                for (int j = 0; j < kC; ++j) wsum += s.wv[j];
                s.db[n - 1] += s.gam[n - 1] * p + wsum;
            }
            const float* SJ = s.SJ[pb];
            const float* dSJ = s.dSJ[pb];
            const int mt = w & 3, m0 = 16 * mt, n0 = 8 * (w >> 2);  // this warp's 16 x 8 tile
            const int nh = w >> 2;                                 // its 8-column half
            // values of this thread's four (row, column) elements kept from one phase to the next
            float kds[4], xs[4], zs[4];
            if (so) {
                // K dS_J alone (rows scaled by rk afterwards); dO into its tile
                float cd4[4] = {0.f, 0.f, 0.f, 0.f}, rd4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int k0 = 0; k0 < KD; k0 += 8) {
                    const int kp = colp<KD>(k0) + t;
                    const uint32_t ak[4] = {fbits(s.Kr[(m0 + g) * PK + kp]), fbits(s.Kr[(m0 + g + 8) * PK + kp]),
                                            fbits(s.Kr[(m0 + g) * PK + kp + 4]), fbits(s.Kr[(m0 + g + 8) * PK + kp + 4])};
                    uint32_t dh[2], dr[2];
                    split_tf32(dSJ[(n0 + g) * PK + kp], dh[0], dr[0]);
                    split_tf32(dSJ[(n0 + g) * PK + kp + 4], dh[1], dr[1]);
                    mma_tf32_16x8x8(rd4, ak, dr);
                    mma_tf32_16x8x8(cd4, ak, dh);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = m0 + g + 8 * (e >> 1), cc = n0 + 2 * t + (e & 1);
                    kds[e] = s.rk[i] * (cd4[e] + rd4[e]);
                    const float ov = b2f(s.Ob[i * kVT + cc]);
                    s.OJ[cc * PC + i] = ov;
                    s.OJc[cc * PT + i] = ov;
                }
            } else {
                // x = K S_J, Q S_J, K dS_J (rows scaled by rk / rq afterwards); V, dO into the tiles
                // head and rest products accumulate separately (independent MMA chains)
                float cx4[4] = {0.f, 0.f, 0.f, 0.f}, cq4[4] = {0.f, 0.f, 0.f, 0.f}, cd4[4] = {0.f, 0.f, 0.f, 0.f};
                float rx4[4] = {0.f, 0.f, 0.f, 0.f}, rq4[4] = {0.f, 0.f, 0.f, 0.f}, rd4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
                for (int k0 = 0; k0 < KD; k0 += 8) {
                    const int kp = colp<KD>(k0) + t;
                    const uint32_t ak[4] = {fbits(s.Kr[(m0 + g) * PK + kp]), fbits(s.Kr[(m0 + g + 8) * PK + kp]),
                                            fbits(s.Kr[(m0 + g) * PK + kp + 4]), fbits(s.Kr[(m0 + g + 8) * PK + kp + 4])};
                    const uint32_t aq[4] = {fbits(s.Qr[(m0 + g) * PK + kp]), fbits(s.Qr[(m0 + g + 8) * PK + kp]),
                                            fbits(s.Qr[(m0 + g) * PK + kp + 4]), fbits(s.Qr[(m0 + g + 8) * PK + kp + 4])};
                    uint32_t sh[2], sr[2], dh[2], dr[2];
                    split_tf32(SJ[(n0 + g) * PK + kp], sh[0], sr[0]);
                    split_tf32(SJ[(n0 + g) * PK + kp + 4], sh[1], sr[1]);
                    split_tf32(dSJ[(n0 + g) * PK + kp], dh[0], dr[0]);
                    split_tf32(dSJ[(n0 + g) * PK + kp + 4], dh[1], dr[1]);
                    mma_tf32_16x8x8(rx4, ak, sr);
                    mma_tf32_16x8x8(rq4, aq, sr);
                    mma_tf32_16x8x8(rd4, ak, dr);
                    mma_tf32_16x8x8(cx4, ak, sh);
                    mma_tf32_16x8x8(cq4, aq, sh);
                    mma_tf32_16x8x8(cd4, ak, dh);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    cx4[e] += rx4[e];
                    cq4[e] += rq4[e];
                    cd4[e] += rd4[e];
                }
                float sop[2] = {0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = m0 + g + 8 * (e >> 1), cc = n0 + 2 * t + (e & 1);
                    const float x = s.rk[i] * cx4[e];
                    const float vv = b2f(s.Vb[i * kVT + cc]);
                    const float ov = b2f(s.Ob[i * kVT + cc]);
                    xs[e] = x;
                    zs[e] = vv - s.gam[i] * x;
                    kds[e] = s.rk[i] * cd4[e];
                    s.Y[cc * PC + i] = s.beta[i] * zs[e];
                    s.OJ[cc * PC + i] = ov;
                    s.OJc[cc * PT + i] = ov;
                    sop[e >> 1] = fmaf(ov, s.rq[i] * cq4[e], sop[e >> 1]);
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float v_ = quad_sum(sop[hh]);
                    if (t == 0) s.part[2][nh][m0 + g + 8 * hh] = v_;
                }
            }
            __syncthreads();
            // the next tile (this chunk's next columns, else the previous chunk's first) streams
            // into the other buffer; the staged V / dO rows have been read above
            if (j0 + kVT < VD) fetch_tile(c, j0 + kVT, pb ^ 1);
            else if (c > lo) fetch_tile(c - 1, 0, pb ^ 1);
            {
                // D = T Y (T lower: column tiles up to the diagonal);  dD = scale P^T dO + Gamma_C (K dS_J)
                float cD[4] = {0.f, 0.f, 0.f, 0.f}, cE[4] = {0.f, 0.f, 0.f, 0.f};
                float rD[4] = {0.f, 0.f, 0.f, 0.f}, rE[4] = {0.f, 0.f, 0.f, 0.f};
                for (int kt = 0; kt <= (so ? -1 : 2 * mt + 1); ++kt) {
                    const int k0 = 8 * kt;
                    uint32_t ah[4], ar[4], bh[2], br[2];
                    frag_a_split([&](int i, int m) { return s.Tm[i * PC + m]; }, m0, k0, g, t, ah, ar);
                    frag_b_split([&](int m, int cc) { return s.Y[cc * PC + m]; }, k0, n0, g, t, bh, br);
                    mma3s(cD, rD, ah, ar, bh, br);
                }
                for (int kt = 2 * mt; kt < 8; ++kt) {
                    const int k0 = 8 * kt;
                    uint32_t ah[4], ar[4];
                    frag_a_split([&](int i, int m) { return s.Pt[i * PC + m]; }, m0, k0, g, t, ah, ar);
                    const uint32_t b[2] = {fbits(s.OJ[(n0 + g) * PC + k0 + t]), fbits(s.OJ[(n0 + g) * PC + k0 + t + 4])};
                    mma_tf32_16x8x8(rE, ar, b);
                    mma_tf32_16x8x8(cE, ah, b);
                }
                float wp[2] = {0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = m0 + g + 8 * (e >> 1), cc = n0 + 2 * t + (e & 1);
                    const float dv_ = cD[e] + rD[e];
                    s.D[cc * PT + i] = dv_;
                    s.dD[cc * PC + i] = a.scale * (cE[e] + rE[e]) + s.GC[i] * kds[e];
                    wp[e >> 1] = fmaf(kds[e], dv_, wp[e >> 1]);
                }
                if (!so) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float v_ = quad_sum(wp[hh]);
                        if (t == 0) s.part[3][nh][m0 + g + 8 * hh] = v_;
                    }
                }
            }
            __syncthreads();
            {
                // dY = T^T dD (T^T upper: column tiles from the diagonal); dV = beta dY (final)
                float cY[4] = {0.f, 0.f, 0.f, 0.f}, rY[4] = {0.f, 0.f, 0.f, 0.f};
                for (int kt = 2 * mt; kt < 8; ++kt) {
                    const int k0 = 8 * kt;
                    uint32_t ah[4], ar[4], bh[2], br[2];
                    frag_a_split([&](int i, int m) { return s.Tm[m * PC + i]; }, m0, k0, g, t, ah, ar);
                    frag_b_split([&](int m, int cc) { return s.dD[cc * PC + m]; }, k0, n0, g, t, bh, br);
                    mma3s(cY, rY, ah, ar, bh, br);
                }
                float sbp[2] = {0.f, 0.f}, sgp[2] = {0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = m0 + g + 8 * (e >> 1), cc = n0 + 2 * t + (e & 1);
                    const float dy = cY[e] + rY[e];
                    s.dY[cc * PC + i] = dy;
                    s.dYc[cc * PT + i] = dy;
                    if (!so) {
                        if (i < n) a.dv[(t0 + i) * a.dv_st + h * a.dv_sh + j0 + cc] = f2b(s.beta[i] * dy);
                        sbp[e >> 1] = fmaf(dy, zs[e], sbp[e >> 1]);
                        sgp[e >> 1] = fmaf(dy, xs[e], sgp[e >> 1]);
                    }
                }
                if (!so) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float b_ = quad_sum(sbp[hh]), g_ = quad_sum(sgp[hh]);
                        if (t == 0) {
                            s.part[0][nh][m0 + g + 8 * hh] = b_;
                            s.part[1][nh][m0 + g + 8 * hh] = g_;
                        }
                    }
                }
            }
            __syncthreads();
            if (!so) {
                // gamma_last <dS_J, S_J>: the decay of the entering state into S_next
                float p = 0.f;
                for (int e = tid; e < KD * kVT; e += kBT) {
                    const int r = colp<KD>(e % KD), cc = e / KD;
                    p = fmaf(dSJ[cc * PK + r], SJ[cc * PK + r], p);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
                if (lane == 0) s.red[w] = p;
            }
            if (kwarp && !so) {
                // dK_hat += dx S_J^T + Gamma_C D dS_J^T,  dx = -beta gamma dY (rounded tf32 operands:
                // these sums only reach the bf16 dk)
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const int k0 = 8 * kt;
                    uint32_t xa[4], da[4];
                    frag_a_round([&](int i, int cc) { return -s.beta[i] * s.gam[i] * s.dYc[cc * PT + i]; }, om0, k0, g,
                                 t, xa);
                    frag_a_round([&](int i, int cc) { return s.GC[i] * s.D[cc * PT + i]; }, om0, k0, g, t, da);
#pragma unroll
                    for (int nd = 0; nd < NT; ++nd) {
                        const int dp = colp<KD>(8 * nd) + g;
                        const uint32_t sb[2] = {to_tf32(SJ[(k0 + t) * PK + dp]), to_tf32(SJ[(k0 + t + 4) * PK + dp])};
                        const uint32_t tb[2] = {to_tf32(dSJ[(k0 + t) * PK + dp]), to_tf32(dSJ[(k0 + t + 4) * PK + dp])};
                        mma_tf32_16x8x8(acc[nd], xa, sb);
                        mma_tf32_16x8x8(acc[nd], da, tb);
                    }
                }
                // dA -= dY D^T (strict), dP += scale dO D^T (incl.) on the lower 16 x 8 tiles
                for (int pr = w; pr < 20; pr += 4) {
                    int pmt, pnt;
                    lower_tile(pr, pmt, pnt);
                    const int p0 = 16 * pmt, q0 = 8 * pnt;
                    float ca[4] = {0.f, 0.f, 0.f, 0.f}, cp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kt = 0; kt < 2; ++kt) {
                        const int k0 = 8 * kt;
                        uint32_t yh[4], yr[4], bh[2], br[2];
                        frag_a_split([&](int i, int cc) { return s.dYc[cc * PT + i]; }, p0, k0, g, t, yh, yr);
                        frag_b_split([&](int cc, int j) { return s.D[cc * PT + j]; }, k0, q0, g, t, bh, br);
                        const uint32_t ao[4] = {fbits(s.OJc[(k0 + t) * PT + p0 + g]), fbits(s.OJc[(k0 + t) * PT + p0 + g + 8]),
                                                fbits(s.OJc[(k0 + t + 4) * PT + p0 + g]),
                                                fbits(s.OJc[(k0 + t + 4) * PT + p0 + g + 8])};
                        mma3(ca, yh, yr, bh, br);
                        mma2a(cp, ao, bh, br);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = p0 + g + 8 * (e >> 1), j = q0 + 2 * t + (e & 1);
                        if (j < i) s.dA[i * PC + j] -= ca[e];
                        if (j <= i) s.dP[i * PC + j] += a.scale * cp[e];
                    }
                }
            } else if (!kwarp) {
                if (tid < 128 + kC && !so) {
                    // per-row sums: dbeta (Y's beta), db (Y's gamma, O's gamma); the Gamma_Cj terms
                    // of S_next, w_j = Gamma_Cj sum_v (K dS_J)_jv D_jv, move from b_j to b_last
                    const int i = tid - 128;
                    const float sb = s.part[0][0][i] + s.part[0][1][i], sg = s.part[1][0][i] + s.part[1][1][i];
                    const float so_ = s.part[2][0][i] + s.part[2][1][i], wj = s.part[3][0][i] + s.part[3][1][i];
                    s.dbeta[i] += sb;
                    s.db[i] += s.gam[i] * (a.scale * so_ - s.beta[i] * sg) - wj * s.GC[i];
                    s.wv[i] = wj * s.GC[i];
                }
                // dQ_hat sum += dO S_J^T (the row factor scale gamma_i is applied after the tiles)
#pragma unroll
                for (int kt = 0; kt < (so ? 0 : 2); ++kt) {
                    const int k0 = 8 * kt;
                    const uint32_t ao[4] = {fbits(s.OJc[(k0 + t) * PT + om0 + g]), fbits(s.OJc[(k0 + t) * PT + om0 + g + 8]),
                                            fbits(s.OJc[(k0 + t + 4) * PT + om0 + g]),
                                            fbits(s.OJc[(k0 + t + 4) * PT + om0 + g + 8])};
#pragma unroll
                    for (int nd = 0; nd < NT; ++nd) {
                        const int dp = colp<KD>(8 * nd) + g;
                        const uint32_t sb[2] = {to_tf32(SJ[(k0 + t) * PK + dp]), to_tf32(SJ[(k0 + t + 4) * PK + dp])};
                        mma_tf32_16x8x8(acc[nd], ao, sb);
                    }
                }
                // dS_J <- gamma_last dS_J + K^T (cx (.) dY) + Q^T (co (.) dO): key rows
                // kb .. kb + 16 MTW - 1 of this warp, both 8-column halves of the tile
                const int kb = 16 * MTW * (w - 4);
                const float gl = s.gam[n - 1];
                float cs[MTW][2][4];
#pragma unroll
                for (int mi = 0; mi < MTW; ++mi)
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int d = kb + 16 * mi + g + 8 * (e >> 1), cc = 8 * h2 + 2 * t + (e & 1);
                            cs[mi][h2][e] = gl * dSJ[cc * PK + colp<KD>(d)];
                        }
#pragma unroll 2
                for (int kt = 0; kt < 8; ++kt) {
                    const int k0 = 8 * kt;
                    uint32_t xh[2][2], xr[2][2], oh[2][2], orr[2][2];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        frag_b_split([&](int m, int cc) { return s.cx[m] * s.dY[cc * PC + m]; }, k0, 8 * h2, g, t, xh[h2],
                                     xr[h2]);
                        frag_b_split([&](int m, int cc) { return s.co[m] * s.OJ[cc * PC + m]; }, k0, 8 * h2, g, t, oh[h2],
                                     orr[h2]);
                    }
#pragma unroll
                    for (int mi = 0; mi < MTW; ++mi) {
                        const int dp = colp<KD>(kb + 16 * mi) + g;
                        const uint32_t ak[4] = {fbits(s.Kr[(k0 + t) * PK + dp]), fbits(s.Kr[(k0 + t) * PK + dp + 8]),
                                                fbits(s.Kr[(k0 + t + 4) * PK + dp]), fbits(s.Kr[(k0 + t + 4) * PK + dp + 8])};
                        const uint32_t aq[4] = {fbits(s.Qr[(k0 + t) * PK + dp]), fbits(s.Qr[(k0 + t) * PK + dp + 8]),
                                                fbits(s.Qr[(k0 + t + 4) * PK + dp]), fbits(s.Qr[(k0 + t + 4) * PK + dp + 8])};
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            mma2a(cs[mi][h2], ak, xh[h2], xr[h2]);
                            mma2a(cs[mi][h2], aq, oh[h2], orr[h2]);
                        }
                    }
                }
#pragma unroll
                for (int mi = 0; mi < MTW; ++mi)
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int d = kb + 16 * mi + g + 8 * hh;
                            *reinterpret_cast<float2*>(dSg + static_cast<int64_t>(d) * VD + j0 + 8 * h2 + 2 * t) =
                                make_float2(cs[mi][h2][2 * hh], cs[mi][h2][2 * hh + 1]);
                        }
            }
            pb ^= 1;
        }
        __syncthreads();
        if (so) continue;  // the state gradient is all this mode computes
        if (tid == 0) {
            float p = 0.f, wsum = 0.f;
            for (int x = 0; x < kBT / 32; ++x) p += s.red[x];
            for (int j = 0; j < kC; ++j) wsum += s.wv[j];
            s.db[n - 1] += s.gam[n - 1] * p + wsum;
        }
        if (!kwarp) {
            // the dQ_hat row factor scale gamma_i
#pragma unroll
            for (int nd = 0; nd < NT; ++nd)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nd][e] *= a.scale * s.gam[om0 + g + 8 * (e >> 1)];
        }
        __syncthreads();

        // ---- tile-independent terms: A and P backward, dbeta, db, dg, the norms
        {
            // four threads per row i (j in quarter ranges), combined by shuffles
            const int i = tid >> 2, q4 = tid & 3;
            float sb = 0.f, rowsum = 0.f, colsum = 0.f;
            for (int j = q4 * 16; j < q4 * 16 + 16; ++j) {
                if (j < i) {
                    const float x = s.dA[i * PC + j] * s.dA[j * PC + i];  // dA_ij Gk_ij
                    sb += x;
                    rowsum = fmaf(x, s.beta[i], rowsum);
                }
                if (j <= i) rowsum = fmaf(s.dP[i * PC + j], s.Pt[j * PC + i], rowsum);
                if (j > i) colsum = fmaf(s.dA[j * PC + i] * s.beta[j], s.dA[i * PC + j], colsum);  // Gk_ji at [i][j]
                if (j >= i) colsum = fmaf(s.dP[j * PC + i], s.Pt[i * PC + j], colsum);
            }
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                sb += __shfl_xor_sync(0xffffffffu, sb, off);
                rowsum += __shfl_xor_sync(0xffffffffu, rowsum, off);
                colsum += __shfl_xor_sync(0xffffffffu, colsum, off);
            }
            if (q4 == 0) {
                s.dbeta[i] += sb;
                s.db[i] += rowsum - colsum;  // log Gamma_ij = b_i - b_j
            }
        }
        __syncthreads();
        if (tid < kC) {
            // dg_j = sum_{i >= j} db_i within the chunk
            const int j = tid;
            float sacc = 0.f;
            for (int i = j; i < n; ++i) sacc += s.db[i];
            if (j < n) {
                // chain rule through the input transforms: dg, dbeta of the raw inputs
                float dgr = sacc, dbr = s.dbeta[j];
                if (a.gate_mode == LA_GATE_SOFTPLUS) {
                    const float sz = sigmoidf_(raw_gate(a, t0 + j, h) + gdt);
                    dgr = sacc * gA * sz;
                    pa_log = fmaf(sacc, s.gt[j], pa_log);
                    pa_dt += dgr;
                } else if (a.gate_mode == LA_GATE_SIGMOID_BOUND) {
                    const float sx = sigmoidf_(raw_gate(a, t0 + j, h));
                    dgr = sacc * a.gate_lb * sx * (1.f - sx);
                }
                if (a.beta_sigmoid) dbr *= s.beta[j] * (1.f - s.beta[j]);
                a.dg[(t0 + j) * a.dg_st + h * a.dg_sh] = dgr;
                a.dbeta[(t0 + j) * a.db_st + h * a.db_sh] = dbr;
            }
        }
        // M = dA (.) beta_i Gamma (strictly lower part; the upper part keeps Gk), H = dP (.) Gamma
        // (incl.), in place
        for (int e = tid; e < kC * kC; e += kBT) {
            const int i = e / kC, j = e % kC;
            const float G = j <= i ? expf(s.b[i] - s.b[j]) : 0.f;
            if (j < i) s.dA[i * PC + j] *= s.beta[i] * G;
            s.dP[i * PC + j] = j <= i ? s.dP[i * PC + j] * G : 0.f;
        }
        __syncthreads();
        if (kwarp) {
            // dK_hat += (M + M^T) K_hat + H^T Q_hat: the column scales rk_j, rq_j go into the
            // left operand so that the raw rows (exact) are the right one
            const int mt = w & 3;
#pragma unroll 1
            for (int kt = 0; kt < 8; ++kt) {
                const int k0 = 8 * kt;
                uint32_t ma[4];
                frag_a_round([&](int i, int j) { return (j <= i ? s.dA[i * PC + j] : s.dA[j * PC + i]) * s.rk[j]; }, om0, k0,
                             g, t, ma);
#pragma unroll
                for (int nd = 0; nd < NT; ++nd) {
                    const int dp = colp<KD>(8 * nd) + g;
                    const uint32_t b[2] = {fbits(s.Kr[(k0 + t) * PK + dp]), fbits(s.Kr[(k0 + t + 4) * PK + dp])};
                    mma_tf32_16x8x8(acc[nd], ma, b);
                }
            }
#pragma unroll 1
            for (int kt = 2 * mt; kt < 8; ++kt) {
                const int k0 = 8 * kt;
                uint32_t ha[4];
                frag_a_round([&](int i, int j) { return s.dP[j * PC + i] * s.rq[j]; }, om0, k0, g, t, ha);
#pragma unroll
                for (int nd = 0; nd < NT; ++nd) {
                    const int dp = colp<KD>(8 * nd) + g;
                    const uint32_t b[2] = {fbits(s.Qr[(k0 + t) * PK + dp]), fbits(s.Qr[(k0 + t + 4) * PK + dp])};
                    mma_tf32_16x8x8(acc[nd], ha, b);
                }
            }
        } else {
            // dQ_hat += H K_hat
            const int mt = w & 3;
#pragma unroll 1
            for (int kt = 0; kt <= 2 * mt + 1; ++kt) {
                const int k0 = 8 * kt;
                uint32_t ha[4];
                frag_a_round([&](int i, int j) { return s.dP[i * PC + j] * s.rk[j]; }, om0, k0, g, t, ha);
#pragma unroll
                for (int nd = 0; nd < NT; ++nd) {
                    const int dp = colp<KD>(8 * nd) + g;
                    const uint32_t b[2] = {fbits(s.Kr[(k0 + t) * PK + dp]), fbits(s.Kr[(k0 + t + 4) * PK + dp])};
                    mma_tf32_16x8x8(acc[nd], ha, b);
                }
            }
        }
        {
            // L2-norm backward of rows om0 + g and om0 + g + 8: with the raw row x and r = 1 / |x|,
            // dx = r (dy - r^2 (x . dy) x)
            const float* Xr = kwarp ? s.Kr : s.Qr;
            const float* rr = kwarp ? s.rk : s.rq;
            float pr[2] = {0.f, 0.f};
#pragma unroll
            for (int nd = 0; nd < NT; ++nd) {
                const int dp = colp<KD>(8 * nd) + 2 * t;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float* xr = Xr + (om0 + g + 8 * hh) * PK + dp;
                    pr[hh] = fmaf(xr[0], acc[nd][2 * hh], fmaf(xr[1], acc[nd][2 * hh + 1], pr[hh]));
                }
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                pr[hh] += __shfl_xor_sync(0xffffffffu, pr[hh], 1);
                pr[hh] += __shfl_xor_sync(0xffffffffu, pr[hh], 2);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = om0 + g + 8 * hh;
                if (i >= n) continue;
                const float r = rr[i], f = r * r * pr[hh];
                const int64_t tok = t0 + i;
                uint16_t* orow = nullptr;
                float* hrow = nullptr;
                if (a.group == 1) orow = kwarp ? a.dk + tok * a.dk_st + hk * a.dk_sh : a.dq + tok * a.dq_st + hk * a.dq_sh;
                else hrow = (kwarp ? a.dkh : a.dqh) + (tok * HO + h) * KD;
#pragma unroll
                for (int nd = 0; nd < NT; ++nd) {
                    const int d = 8 * nd + 2 * t;
                    float v0 = acc[nd][2 * hh], v1 = acc[nd][2 * hh + 1];
                    if (a.l2norm) {
                        const float* xr = Xr + i * PK + colp<KD>(8 * nd) + 2 * t;
                        v0 = r * (v0 - f * xr[0]);
                        v1 = r * (v1 - f * xr[1]);
                    }
                    if (a.group == 1) {
                        if (a.vec_out) {
                            *reinterpret_cast<uint32_t*>(orow + d) =
                                static_cast<uint32_t>(f2b(v0)) | (static_cast<uint32_t>(f2b(v1)) << 16);
                        } else {
                            orow[d] = f2b(v0);
                            orow[d + 1] = f2b(v1);
                        }
                    } else {
                        *reinterpret_cast<float2*>(hrow + d) = make_float2(v0, v1);
                    }
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait_all();  // nothing is in flight here (the last tile fetches nothing)
    if (a.gpart && tid < kC) {
        // this unit's d_a_log and d_dt_bias sums: a fixed-order reduction over the 64 token slots
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            pa_log += __shfl_xor_sync(0xffffffffu, pa_log, off);
            pa_dt += __shfl_xor_sync(0xffffffffu, pa_dt, off);
        }
        if (lane == 0) {
            s.red[2 * w] = pa_log;
            s.red[2 * w + 1] = pa_dt;
        }
    }
    __syncthreads();
    if (a.gpart && tid == 0) {
        const int64_t slot = static_cast<int64_t>(unit) * P + piece;
        a.gpart[2 * slot] = s.red[0] + s.red[2];
        a.gpart[2 * slot + 1] = s.red[1] + s.red[3];
    }
    if (a.ds0 && piece == 0) {
        for (int64_t e = tid; e < KV; e += kBT) a.ds0[unit * KV + e] = dSg[e];
    }
}

// d_a_log and d_dt_bias of a head: the per-range sums added in sequence and range order.
__global__ void gdn_bwd_gate_param_kernel(const BwdArgs a) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= a.HV) return;
    float sa = 0.f, sd = 0.f;
    for (int i = 0; i < a.N; ++i)
        for (int pc = 0; pc < a.pieces; ++pc) {
            const int64_t slot = (static_cast<int64_t>(i) * a.HV + h) * a.pieces + pc;
            sa += a.gpart[2 * slot];
            sd += a.gpart[2 * slot + 1];
        }
    if (a.d_a_log) a.d_a_log[h] = sa;
    if (a.d_dt_bias) a.d_dt_bias[h] = sd;
}

// dq, dk of a q/k head: the sum over its group of value heads (fixed order), rounded to bf16.
__global__ void gdn_bwd_group_sum_kernel(const BwdArgs a) {
    const int64_t total = a.T * a.HK * a.K;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int d = static_cast<int>(e % a.K);
        const int64_t th = e / a.K;
        const int hk = static_cast<int>(th % a.HK);
        const int64_t t = th / a.HK;
        float sk = 0.f, sq = 0.f;
        for (int gi = 0; gi < a.group; ++gi) {
            const int64_t src = (t * a.HV + hk * a.group + gi) * a.K + d;
            sk += a.dkh[src];
            sq += a.dqh[src];
        }
        a.dk[t * a.dk_st + hk * a.dk_sh + d] = f2b(sk);
        a.dq[t * a.dq_st + hk * a.dq_sh + d] = f2b(sq);
    }
}

// CTAs of the backward kernel resident on the whole GPU at once (one wave), per device and
// head-dimension pair; looked up on the first launch (outside any stream capture).  Host
// threads may launch concurrently: each slot is written atomically (every writer stores the
// same value).
std::atomic<int> g_bwd_wave[128][4];

template <int KD, int VD>
cudaError_t launch_bwd_kv(const BwdArgs& a0, cudaStream_t s) {
    BwdArgs a = a0;
    const int units = a.N * a.HV;
    a.pieces = 1;
    a.item_base = 0;
    if (units > 0) {
        auto* fn = gdn_bwd_kernel<KD, VD>;
        const int smem = static_cast<int>(sizeof(BwdSmem<KD>));
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        std::atomic<int>& slot = g_bwd_wave[dev & 127][(KD == 128 ? 2 : 0) + (VD == 128 ? 1 : 0)];
        int wave = slot.load(std::memory_order_relaxed);
        if (wave == 0) {
            int sms = 0, per_sm = 0;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
            if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBT, smem)) != cudaSuccess) return e;
            wave = sms * (per_sm > 0 ? per_sm : 1);
            slot.store(wave, std::memory_order_relaxed);
        }
        // more units than one wave: four ranges per unit, launched range by range in waves (a
        // range's successor in the unit is at least `units` >= `wave` items earlier, so in an
        // earlier launch)
        if (units > wave) a.pieces = kBwdPieces;
        const int items = units * a.pieces;
        const int grid = a.pieces == 1 ? units : wave;
        for (int base = 0; base < items; base += grid) {
            a.item_base = base;
            fn<<<items - base < grid ? items - base : grid, kBT, smem, s>>>(a);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
    }
    if (a.group > 1 && a.T > 0 && !a.state_only) {
        gdn_bwd_group_sum_kernel<<<1024, 256, 0, s>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.gpart && !a.state_only) {
        gdn_bwd_gate_param_kernel<<<(a.HV + 127) / 128, 128, 0, s>>>(a);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_finish(const BwdArgs& a, cudaStream_t s) {
    if (a.group > 1 && a.T > 0) {
        gdn_bwd_group_sum_kernel<<<1024, 256, 0, s>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.gpart) {
        gdn_bwd_gate_param_kernel<<<(a.HV + 127) / 128, 128, 0, s>>>(a);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s) {
    if (a.K == 128) return a.V == 128 ? launch_bwd_kv<128, 128>(a, s) : launch_bwd_kv<128, 64>(a, s);
    return a.V == 128 ? launch_bwd_kv<64, 128>(a, s) : launch_bwd_kv<64, 64>(a, s);
}

}  // namespace la
