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
// then the L2-norm backward for q and k and the sum over grouped value heads.
//
// Mapping.  One CTA of 256 threads per (sequence, head) walks the chunks in reverse and
// carries dS in a global per-unit buffer.  The value columns are independent chains (each
// column of S evolves on its own), so a chunk is processed in 16-column tiles of S, dS, V and
// dO; the tile-independent parts (normalised K and Q, A, T, P, the decays) are formed once
// per chunk in shared memory and the cross-column sums (dA, dP, dK, dQ, dbeta, db) are
// accumulated over the tiles in shared memory and registers.  The chunk entering states come
// from the forward kernel run with fp32 checkpoints every 64 tokens.  All arithmetic is fp32
// on the CUDA cores.
#include <cuda_bf16.h>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"

namespace la {
namespace {

constexpr int kBT = 256;   // threads
constexpr int kC = 64;     // chunk
constexpr int kVT = 16;    // value columns per tile

__device__ __forceinline__ uint16_t f2b(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Shared-memory layout of the key-length rows (K, Q, S^T, dS^T): the four KD/4-column slices
// that four neighbouring threads read are staggered by 4 words, and the row stride is 4 mod 8
// words, so that 16-byte reads of neighbouring rows or of the four slices hit distinct banks.
template <int KD>
__device__ __forceinline__ int colp(int d) { return d + (d / (KD / 4)) * 4; }

template <int KD>
struct BwdSmem {
    static constexpr int PK = KD + 12;  // row stride of K / Q / S^T / dS^T (4 mod 8 words)
    static constexpr int PC = kC + 4;   // row stride of the 64 x 64 matrices and of the tiles
    float Kh[kC * PK];      // normalised keys (rows past the end are zero)
    float Qh[kC * PK];      // normalised queries
    float Tm[kC * PC];      // T = (I + A)^{-1}
    float Pm[kC * PC];      // P (lower incl.)
    // strictly lower part: dA accumulated over the tiles, then M; strictly upper part: the
    // transpose of Gk_ij = (k_i . k_j) Gamma_ij (j < i) stored at [j][i]; diagonal zero
    float dA[kC * PC];
    float dP[kC * PC];      // accumulated over tiles, then H
    // value tiles, stored transposed: row = value column cc, contiguous along the token / key index;
    // S and dS are double buffered so that the next tile streams in while this one is computed
    float SJ[2][kVT * PK];  // S[:, tile]^T
    float dSJ[2][kVT * PK]; // dS_next[:, tile]^T
    float X[kVT * PC], Y[kVT * PC], D[kVT * PC], dD[kVT * PC], dY[kVT * PC];
    float VJ[kVT * PC], OJ[kVT * PC], QS[kVT * PC], KdS[kVT * PC];
    uint16_t Vb[kC * kVT], Ob[kC * kVT];  // the next tile's raw V and dO rows (bf16, token-major)
    float beta[kC], b[kC], gam[kC], GC[kC], rk[kC], rq[kC];
    float dbeta[kC], db[kC], wv[kC];
    float red[kBT / 32];
};
static_assert(sizeof(BwdSmem<128>) <= 227 * 1024, "backward shared memory exceeds the per-CTA limit");

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
}

// out[c][r] = sum_m Lt[c][m] * R[r][m] for a kVT x kC output (c = value column, r = token),
// both operands contiguous along m in groups of 4 (column map CM); each thread computes
// rows r, r + 16, r + 32, r + 48 of one column.
template <int MM, class CM, class FO>
__device__ __forceinline__ void tile_nt(const float* Lt, int ldl, const float* R, int ldr, CM cm, FO out) {
    const int tid = threadIdx.x;
    const int c = tid >> 4, r = tid & 15;
    float4 acc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int m = 0; m < MM; m += 4) {
        const int mp = cm(m);
        const float4 l = ld4(Lt + c * ldl + mp);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 rv = ld4(R + (r + 16 * e) * ldr + mp);
            acc[e].x = fmaf(l.x, rv.x, acc[e].x);
            acc[e].y = fmaf(l.y, rv.y, acc[e].y);
            acc[e].z = fmaf(l.z, rv.z, acc[e].z);
            acc[e].w = fmaf(l.w, rv.w, acc[e].w);
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) out(c, r + 16 * e, (acc[e].x + acc[e].y) + (acc[e].z + acc[e].w));
}

// out[c][r] = sum_m Lt[c][m] * R[m][r] for a kVT x kC output, R contiguous along r.
template <int MM, class FL, class FO>
__device__ __forceinline__ void tile_nn(FL Lt, const float* R, int ldr, FO out) {
    const int tid = threadIdx.x;
    const int c = tid >> 4, r0 = (tid & 15) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int m = 0; m < MM; ++m) {
        const float l = Lt(c, m);
        const float4 rv = ld4(R + m * ldr + r0);
        acc.x = fmaf(l, rv.x, acc.x);
        acc.y = fmaf(l, rv.y, acc.y);
        acc.z = fmaf(l, rv.z, acc.z);
        acc.w = fmaf(l, rv.w, acc.w);
    }
    out(c, r0 + 0, acc.x);
    out(c, r0 + 1, acc.y);
    out(c, r0 + 2, acc.z);
    out(c, r0 + 3, acc.w);
}

template <int KD, int VD>
__global__ void __launch_bounds__(kBT, 1) gdn_bwd_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BwdSmem<KD>& s = *reinterpret_cast<BwdSmem<KD>*>(smem_raw);
    constexpr int PK = BwdSmem<KD>::PK;
    constexpr int PC = BwdSmem<KD>::PC;
    const int tid = threadIdx.x;
    if (tid == 0) s.red[0] = __int_as_float(*reinterpret_cast<const volatile int32_t*>(&a.hdr->status));
    __syncthreads();
    if (__float_as_int(s.red[0]) != LA_OK) return;  // bad cu_seqlens: the forward ran nothing
    __syncthreads();
    const int HO = a.HV;
    const int unit = blockIdx.x;
    const int seq = unit / HO, h = unit % HO;
    const int hk = h / a.group;
    const int64_t ts = a.cu64 ? static_cast<const int64_t*>(a.cu)[seq] : static_cast<const int32_t*>(a.cu)[seq];
    const int64_t te = a.cu64 ? static_cast<const int64_t*>(a.cu)[seq + 1] : static_cast<const int32_t*>(a.cu)[seq + 1];
    const int64_t L = te - ts;
    const int nch = static_cast<int>((L + kC - 1) / kC);
    const int64_t KV = static_cast<int64_t>(KD) * VD;
    float* dSg = a.dS_work + static_cast<int64_t>(unit) * KV;  // carried dS (global, L2 resident)

    // dS after the last token: d_final_state or zero
    for (int64_t e = tid; e < KV; e += kBT) dSg[e] = a.dfinal ? a.dfinal[unit * KV + e] : 0.f;
    __syncthreads();

    // thread ownership for the per-row accumulators of dK and dQ: row i, KD/4-column slice
    constexpr int KSL = KD / 4;
    const int own_r = tid >> 2, own_c0 = (tid & 3) * KSL;

    // Asynchronous fetch of one value tile (chunk cc, columns j0..j0+15) into buffer pb: the
    // S and dS columns (4-byte copies, transposed into the tile layout) and the raw V and dO
    // rows (4-byte copies of bf16 pairs when the operands allow it, else plain loads).
    auto fetch_tile = [&](int cc, int j0, int pb) {
        const int64_t ft0 = ts + static_cast<int64_t>(cc) * kC;
        const int fn = static_cast<int>(L - static_cast<int64_t>(cc) * kC < kC ? L - static_cast<int64_t>(cc) * kC : kC);
        const float* Sf = a.ckpt + ((a.ckpt_off[seq] + cc) * HO + h) * KV;
        for (int e = tid; e < KD * kVT; e += kBT) {
            const int r = e / kVT, col = e % kVT;
            cp_async4(&s.SJ[pb][col * PK + colp<KD>(r)], Sf + r * VD + j0 + col);
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
                const uint16_t* vs = a.v + (ft0 + i) * a.v_st + h * a.v_sh + j0 + c2;
                const uint16_t* os = a.dout + (ft0 + i) * a.do_st + h * a.do_sh + j0 + c2;
                if (a.vo_async) {
                    cp_async4(vd, vs);
                    cp_async4(od, os);
                } else {
                    vd[0] = vs[0];
                    vd[1] = vs[1];
                    od[0] = os[0];
                    od[1] = os[1];
                }
            }
        }
        cp_async_commit();
    };
    int pb = 0;  // buffer of the current tile
    if (nch > 0) fetch_tile(nch - 1, 0, 0);

    for (int c = nch - 1; c >= 0; --c) {
        const int64_t t0 = ts + static_cast<int64_t>(c) * kC;
        const int n = static_cast<int>(L - static_cast<int64_t>(c) * kC < kC ? L - static_cast<int64_t>(c) * kC : kC);

        // ---- chunk-level quantities: normalised rows, decays, A, T, P
        for (int e = tid; e < kC * KD / 8; e += kBT) {
            // 8 bf16 (16 bytes) per load: k and q rows are 16-byte aligned (TMA operand rules)
            const int i = e / (KD / 8), d = (e % (KD / 8)) * 8;
            uint4 kw = make_uint4(0u, 0u, 0u, 0u), qw = kw;
            if (i < n) {
                kw = *reinterpret_cast<const uint4*>(a.k + (t0 + i) * a.k_st + hk * a.k_sh + d);
                qw = *reinterpret_cast<const uint4*>(a.q + (t0 + i) * a.q_st + hk * a.q_sh + d);
            }
            float* kd = &s.Kh[i * PK + colp<KD>(d)];
            float* qd = &s.Qh[i * PK + colp<KD>(d)];
            const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w}, qq[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                kd[2 * x] = __uint_as_float(kk[x] << 16);
                kd[2 * x + 1] = __uint_as_float(kk[x] & 0xFFFF0000u);
                qd[2 * x] = __uint_as_float(qq[x] << 16);
                qd[2 * x + 1] = __uint_as_float(qq[x] & 0xFFFF0000u);
            }
        }
        if (tid < kC) {
            const int i = tid;
            s.beta[i] = i < n ? a.beta[(t0 + i) * a.b_st + h * a.b_sh] : 0.f;
            s.b[i] = i < n ? a.g[(t0 + i) * a.g_st + h * a.g_sh] : 0.f;
        }
        __syncthreads();
        {
            // row norms: four threads per row (rows = tid / 4), quarter rows each
            const int i = tid >> 2, q4 = tid & 3;
            float sk = 0.f, sq = 0.f;
#pragma unroll 4
            for (int d = q4 * KSL; d < (q4 + 1) * KSL; d += 4) {
                const float4 kv = ld4(&s.Kh[i * PK + colp<KD>(d)]), qv = ld4(&s.Qh[i * PK + colp<KD>(d)]);
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
        for (int e = tid; e < kC * KD; e += kBT) {
            const int i = e / KD, d = colp<KD>(e % KD);
            s.Kh[i * PK + d] *= s.rk[i];
            s.Qh[i * PK + d] *= s.rq[i];
        }
        if (tid < kC) {
            const float bl = s.b[n - 1];
            s.gam[tid] = expf(s.b[tid]);
            s.GC[tid] = tid < n ? expf(bl - s.b[tid]) : 0.f;
            s.dbeta[tid] = 0.f;
            s.db[tid] = 0.f;
        }
        __syncthreads();
        {
            // Gk = (k_i . k_j) Gamma_ij and P = (q_i . k_j) Gamma_ij (lower incl.): 4 x 4 blocks
            // rows i = 4 bi + x, columns j = bj + 16 y (neighbouring threads read neighbouring rows)
            const int bi = tid >> 4, bj = tid & 15;
            const int i0 = 4 * bi;
            float kk[4][4], qk[4][4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) kk[x][y] = qk[x][y] = 0.f;
            if (bj <= i0 + 3) {
#pragma unroll 2
                for (int d = 0; d < KD; d += 4) {
                    const int dp = colp<KD>(d);
                    float4 ki[4], qi[4], kj[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        ki[x] = ld4(&s.Kh[(i0 + x) * PK + dp]);
                        qi[x] = ld4(&s.Qh[(i0 + x) * PK + dp]);
                        kj[x] = ld4(&s.Kh[(bj + 16 * x) * PK + dp]);
                    }
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int y = 0; y < 4; ++y) {
                            kk[x][y] = dot4(ki[x], kj[y], kk[x][y]);
                            qk[x][y] = dot4(qi[x], kj[y], qk[x][y]);
                        }
                }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    const int i = i0 + x, j = bj + 16 * y;
                    const float G = j <= i ? expf(s.b[i] - s.b[j]) : 0.f;
                    if (j <= i) s.dA[i * PC + j] = 0.f;              // dA accumulator, diagonal
                    if (j < i) s.dA[j * PC + i] = kk[x][y] * G;      // Gk_ij, transposed
                    s.Pm[i * PC + j] = qk[x][y] * G;
                    s.dP[i * PC + j] = 0.f;
                }
        }
        __syncthreads();
        {
            // T = (I + A)^{-1}, A = strict_tril(beta_i Gk_ij), in 16 x 16 blocks: the diagonal
            // blocks by substitution (warp w, lane = column), then the blocks below by
            // T[bi][bj] = -T[bi][bi] sum_{m = bj}^{bi - 1} A[bi][m] T[m][bj], one level of block
            // distance at a time (scratch: the dD tile, not yet in use)
            const int w = tid >> 5, lane = tid & 31;
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
                    float t[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) t[x] = 0.f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float tk = s.Tm[(16 * bi + r) * PC + 16 * bi + k];
#pragma unroll
                        for (int x = 0; x < 8; ++x) t[x] = fmaf(tk, Ysc[k * 16 + c0 + x], t[x]);
                    }
#pragma unroll
                    for (int x = 0; x < 8; ++x) s.Tm[(16 * bi + r) * PC + 16 * bj + c0 + x] = -t[x];
                    __syncwarp();
                }
                __syncthreads();
            }
        }
        float dKacc[KSL], dQacc[KSL];
#pragma unroll
        for (int e = 0; e < KSL; ++e) dKacc[e] = dQacc[e] = 0.f;

        // ---- the value tiles: independent columns of S and dS
        for (int j0 = 0; j0 < VD; j0 += kVT) {
            cp_async_wait_all();
            __syncthreads();  // this tile's S, dS, V, dO have landed
            float* SJ = s.SJ[pb];
            float* dSJ = s.dSJ[pb];
            {
                // V and dO of this tile into the fp32 tiles, each element by the thread that reads
                // it first below (column tid / 16, rows tid % 16 + 16 e)
                const int cc = tid >> 4, r = tid & 15;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = r + 16 * e;
                    s.VJ[cc * PC + i] = __uint_as_float(static_cast<uint32_t>(s.Vb[i * kVT + cc]) << 16);
                    s.OJ[cc * PC + i] = __uint_as_float(static_cast<uint32_t>(s.Ob[i * kVT + cc]) << 16);
                }
            }
            // x = K S_J, Q S_J, K dS_J (transposed tiles)
            auto ck = [](int m) { return colp<KD>(m); };
            auto cc_id = [](int m) { return m; };
            tile_nt<KD>(SJ, PK, s.Kh, PK, ck, [&](int cc, int r, float v) {
                s.X[cc * PC + r] = v;
                s.Y[cc * PC + r] = s.beta[r] * (s.VJ[cc * PC + r] - s.gam[r] * v);
            });
            tile_nt<KD>(SJ, PK, s.Qh, PK, ck, [&](int cc, int r, float v) { s.QS[cc * PC + r] = v; });
            tile_nt<KD>(dSJ, PK, s.Kh, PK, ck, [&](int cc, int r, float v) { s.KdS[cc * PC + r] = v; });
            __syncthreads();
            // the next tile (this chunk's next columns, else the previous chunk's first) streams
            // into the other buffer; the staged V / dO rows have been read above
            if (j0 + kVT < VD) fetch_tile(c, j0 + kVT, pb ^ 1);
            else if (c > 0) fetch_tile(c - 1, 0, pb ^ 1);
            // D = T Y;  dD = scale P^T dO + Gamma_C (K dS_J)
            tile_nt<kC>(s.Y, PC, s.Tm, PC, cc_id, [&](int cc, int r, float v) { s.D[cc * PC + r] = v; });
            tile_nn<kC>([&](int cc, int m) { return s.OJ[cc * PC + m]; }, s.Pm, PC,
                        [&](int cc, int r, float v) { s.dD[cc * PC + r] = a.scale * v + s.GC[r] * s.KdS[cc * PC + r]; });
            __syncthreads();
            // dY = T^T dD
            tile_nn<kC>([&](int cc, int m) { return s.dD[cc * PC + m]; }, s.Tm, PC,
                        [&](int cc, int r, float v) { s.dY[cc * PC + r] = v; });
            __syncthreads();
            // dV = beta dY (final): four consecutive columns of one row per thread
            {
                const int r = tid >> 2, c4 = (tid & 3) * 4;
                if (r < n) {
                    uint16_t* dst = a.dv + (t0 + r) * a.dv_st + h * a.dv_sh + j0 + c4;
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = f2b(s.beta[r] * s.dY[(c4 + e) * PC + r]);
                }
            }
            // per-row sums: dbeta (Y's beta), db (Y's gamma, O's gamma); the Gamma_Cj terms of
            // S_next, w_j = Gamma_Cj sum_v (K dS_J)_jv D_jv, move from b_j to b_last
            if (tid < kC) {
                const int i = tid;
                float sb = 0.f, sg = 0.f, so = 0.f, w = 0.f;
#pragma unroll
                for (int cc = 0; cc < kVT; ++cc) {
                    const float dy = s.dY[cc * PC + i], xv = s.X[cc * PC + i];
                    sb = fmaf(dy, s.VJ[cc * PC + i] - s.gam[i] * xv, sb);
                    sg = fmaf(dy, xv, sg);
                    so = fmaf(s.OJ[cc * PC + i], s.QS[cc * PC + i], so);
                    w = fmaf(s.KdS[cc * PC + i], s.D[cc * PC + i], w);
                }
                s.dbeta[i] += sb;
                s.db[i] += s.gam[i] * (a.scale * so - s.beta[i] * sg) - w * s.GC[i];
                s.wv[i] = w * s.GC[i];
            }
            {
                // gamma_last <dS_J, S_J>: the decay of the entering state into S_next
                float p = 0.f;
                for (int e = tid; e < KD * kVT; e += kBT) {
                    const int r = colp<KD>(e % KD), cc = e / KD;
                    p = fmaf(dSJ[cc * PK + r], SJ[cc * PK + r], p);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
                if ((tid & 31) == 0) s.red[tid >> 5] = p;
            }
            // dA += -dY D^T, dP += scale dO D^T (lower parts), 4 x 4 blocks
            {
                const int bi = tid >> 4, bj = tid & 15;
                const int i0 = 4 * bi, jj0 = 4 * bj;
                if (bj <= bi) {
                    float ad[4][4], pd[4][4];
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int y = 0; y < 4; ++y) ad[x][y] = pd[x][y] = 0.f;
#pragma unroll 4
                    for (int cc = 0; cc < kVT; ++cc) {
                        const float4 yv = ld4(&s.dY[cc * PC + i0]), ov = ld4(&s.OJ[cc * PC + i0]);
                        const float4 dv = ld4(&s.D[cc * PC + jj0]);
                        const float yy[4] = {yv.x, yv.y, yv.z, yv.w}, oo[4] = {ov.x, ov.y, ov.z, ov.w};
                        const float dd[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                        for (int x = 0; x < 4; ++x)
#pragma unroll
                            for (int y = 0; y < 4; ++y) {
                                ad[x][y] = fmaf(yy[x], dd[y], ad[x][y]);
                                pd[x][y] = fmaf(oo[x], dd[y], pd[x][y]);
                            }
                    }
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int y = 0; y < 4; ++y) {
                            const int i = i0 + x, j = jj0 + y;
                            if (j < i) s.dA[i * PC + j] -= ad[x][y];
                            if (j <= i) s.dP[i * PC + j] += a.scale * pd[x][y];
                        }
                }
            }
            {
                // dK += dx S_J^T + Gamma_C D dS_J^T (dx = -beta gamma dY); dQ += scale gamma dO S_J^T
                const int i = own_r;
                const float bx = -s.beta[i] * s.gam[i], gc = s.GC[i], sg = a.scale * s.gam[i];
#pragma unroll 2
                for (int cc = 0; cc < kVT; ++cc) {
                    const float fy = bx * s.dY[cc * PC + i], fd = gc * s.D[cc * PC + i], fo = sg * s.OJ[cc * PC + i];
#pragma unroll
                    for (int e = 0; e < KSL; e += 4) {
                        const float4 sj = ld4(&SJ[cc * PK + colp<KD>(own_c0 + e)]);
                        const float4 dsj = ld4(&dSJ[cc * PK + colp<KD>(own_c0 + e)]);
                        dKacc[e + 0] = fmaf(fy, sj.x, fmaf(fd, dsj.x, dKacc[e + 0]));
                        dKacc[e + 1] = fmaf(fy, sj.y, fmaf(fd, dsj.y, dKacc[e + 1]));
                        dKacc[e + 2] = fmaf(fy, sj.z, fmaf(fd, dsj.z, dKacc[e + 2]));
                        dKacc[e + 3] = fmaf(fy, sj.w, fmaf(fd, dsj.w, dKacc[e + 3]));
                        dQacc[e + 0] = fmaf(fo, sj.x, dQacc[e + 0]);
                        dQacc[e + 1] = fmaf(fo, sj.y, dQacc[e + 1]);
                        dQacc[e + 2] = fmaf(fo, sj.z, dQacc[e + 2]);
                        dQacc[e + 3] = fmaf(fo, sj.w, dQacc[e + 3]);
                    }
                }
            }
            __syncthreads();
            if (tid == 0) {
                float p = 0.f, w = 0.f;
                for (int x = 0; x < kBT / 32; ++x) p += s.red[x];
                for (int j = 0; j < kC; ++j) w += s.wv[j];
                s.db[n - 1] += s.gam[n - 1] * p + w;
            }
            {
                // dS_J <- gamma_last dS_J + K^T dx + scale Q^T (gamma dO): column cc of dS, keys
                // d .. d+3 per thread (KD x kVT outputs over 256 threads)
                constexpr int PER = KD * kVT / (4 * kBT);  // float4 groups per thread
#pragma unroll
                for (int e = 0; e < PER; ++e) {
                    const int idx = tid + e * kBT;
                    const int cc = idx % kVT, d = (idx / kVT) * 4;  // 16 threads: one row segment
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                    for (int m = 0; m < kC; ++m) {
                        const float fx = -s.beta[m] * s.gam[m] * s.dY[cc * PC + m];
                        const float fo = a.scale * s.gam[m] * s.OJ[cc * PC + m];
                        const float4 kv = ld4(&s.Kh[m * PK + colp<KD>(d)]), qv = ld4(&s.Qh[m * PK + colp<KD>(d)]);
                        acc.x = fmaf(fx, kv.x, fmaf(fo, qv.x, acc.x));
                        acc.y = fmaf(fx, kv.y, fmaf(fo, qv.y, acc.y));
                        acc.z = fmaf(fx, kv.z, fmaf(fo, qv.z, acc.z));
                        acc.w = fmaf(fx, kv.w, fmaf(fo, qv.w, acc.w));
                    }
                    const float gl = s.gam[n - 1];
                    float* dst = dSg + static_cast<int64_t>(d) * VD + j0 + cc;
                    const float4 old = ld4(&dSJ[cc * PK + colp<KD>(d)]);
                    dst[0] = fmaf(gl, old.x, acc.x);
                    dst[VD] = fmaf(gl, old.y, acc.y);
                    dst[2 * VD] = fmaf(gl, old.z, acc.z);
                    dst[3 * VD] = fmaf(gl, old.w, acc.w);
                }
            }
            __syncthreads();
            pb ^= 1;
        }

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
                if (j <= i) rowsum = fmaf(s.dP[i * PC + j], s.Pm[i * PC + j], rowsum);
                if (j > i) colsum = fmaf(s.dA[j * PC + i] * s.beta[j], s.dA[i * PC + j], colsum);  // Gk_ji at [i][j]
                if (j >= i) colsum = fmaf(s.dP[j * PC + i], s.Pm[j * PC + i], colsum);
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
        // M = dA (.) beta_i Gamma (strictly lower part; the upper part keeps Gk), H = dP (.) Gamma
        // (incl.), in place
        for (int e = tid; e < kC * kC; e += kBT) {
            const int i = e / kC, j = e % kC;
            const float G = j <= i ? expf(s.b[i] - s.b[j]) : 0.f;
            if (j < i) s.dA[i * PC + j] *= s.beta[i] * G;
            s.dP[i * PC + j] = j <= i ? s.dP[i * PC + j] * G : 0.f;
        }
        __syncthreads();
        {
            // dK += (M + M^T) K + H^T Q, dQ += H K
            const int i = own_r;
#pragma unroll 2
            for (int j = 0; j < kC; ++j) {
                // M_ij + M_ji with M strictly lower (its diagonal is zero)
                const float mk = j <= i ? s.dA[i * PC + j] : s.dA[j * PC + i];
                const float hq = s.dP[j * PC + i], hk = s.dP[i * PC + j];
#pragma unroll
                for (int e = 0; e < KSL; e += 4) {
                    const float4 kj = ld4(&s.Kh[j * PK + colp<KD>(own_c0 + e)]);
                    const float4 qj = ld4(&s.Qh[j * PK + colp<KD>(own_c0 + e)]);
                    dKacc[e + 0] = fmaf(mk, kj.x, fmaf(hq, qj.x, dKacc[e + 0]));
                    dKacc[e + 1] = fmaf(mk, kj.y, fmaf(hq, qj.y, dKacc[e + 1]));
                    dKacc[e + 2] = fmaf(mk, kj.z, fmaf(hq, qj.z, dKacc[e + 2]));
                    dKacc[e + 3] = fmaf(mk, kj.w, fmaf(hq, qj.w, dKacc[e + 3]));
                    dQacc[e + 0] = fmaf(hk, kj.x, dQacc[e + 0]);
                    dQacc[e + 1] = fmaf(hk, kj.y, dQacc[e + 1]);
                    dQacc[e + 2] = fmaf(hk, kj.z, dQacc[e + 2]);
                    dQacc[e + 3] = fmaf(hk, kj.w, dQacc[e + 3]);
                }
            }
        }
        __syncthreads();
        if (tid < kC) {
            // dg_j = sum_{i >= j} db_i within the chunk
            const int j = tid;
            float acc = 0.f;
            for (int i = j; i < n; ++i) acc += s.db[i];
            if (j < n) {
                a.dg[(t0 + j) * a.dg_st + h * a.dg_sh] = acc;
                a.dbeta[(t0 + j) * a.db_st + h * a.db_sh] = s.dbeta[j];
            }
        }
        {
            // L2-norm backward of row own_r: dx = r dy - r^3 (x . dy) x on the raw row
            const int i = own_r;
            float pk = 0.f, pq = 0.f;
#pragma unroll
            for (int e = 0; e < KSL; ++e) {
                pk = fmaf(s.Kh[i * PK + colp<KD>(own_c0 + e)], dKacc[e], pk);
                pq = fmaf(s.Qh[i * PK + colp<KD>(own_c0 + e)], dQacc[e], pq);
            }
            pk += __shfl_xor_sync(0xffffffffu, pk, 1);
            pk += __shfl_xor_sync(0xffffffffu, pk, 2);
            pq += __shfl_xor_sync(0xffffffffu, pq, 1);
            pq += __shfl_xor_sync(0xffffffffu, pq, 2);
            if (i < n) {
                // with the normalised row x_hat = r x: r^3 (x . dy) x = r (x_hat . dy) x_hat
                const float rkk = s.rk[i], rqq = s.rq[i];
#pragma unroll
                for (int e = 0; e < KSL; ++e) {
                    if (a.l2norm) {
                        dKacc[e] = rkk * (dKacc[e] - pk * s.Kh[i * PK + colp<KD>(own_c0 + e)]);
                        dQacc[e] = rqq * (dQacc[e] - pq * s.Qh[i * PK + colp<KD>(own_c0 + e)]);
                    }
                }
                const int64_t t = t0 + i;
                if (a.group == 1 && a.vec_out) {
                    // 8 bf16 per 16-byte store (dq, dk rows 16-byte aligned)
                    uint4* kd = reinterpret_cast<uint4*>(a.dk + t * a.dk_st + hk * a.dk_sh + own_c0);
                    uint4* qd = reinterpret_cast<uint4*>(a.dq + t * a.dq_st + hk * a.dq_sh + own_c0);
#pragma unroll
                    for (int e = 0; e < KSL; e += 8) {
                        uint32_t kw[4], qw[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            kw[x] = static_cast<uint32_t>(f2b(dKacc[e + 2 * x])) | (static_cast<uint32_t>(f2b(dKacc[e + 2 * x + 1])) << 16);
                            qw[x] = static_cast<uint32_t>(f2b(dQacc[e + 2 * x])) | (static_cast<uint32_t>(f2b(dQacc[e + 2 * x + 1])) << 16);
                        }
                        kd[e / 8] = make_uint4(kw[0], kw[1], kw[2], kw[3]);
                        qd[e / 8] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < KSL; ++e) {
                        const int d = own_c0 + e;
                        if (a.group == 1) {
                            a.dk[t * a.dk_st + hk * a.dk_sh + d] = f2b(dKacc[e]);
                            a.dq[t * a.dq_st + hk * a.dq_sh + d] = f2b(dQacc[e]);
                        } else {
                            a.dkh[(t * HO + h) * KD + d] = dKacc[e];
                            a.dqh[(t * HO + h) * KD + d] = dQacc[e];
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait_all();  // nothing is in flight here (the last tile fetches nothing)
    if (a.ds0) {
        for (int64_t e = tid; e < KV; e += kBT) a.ds0[unit * KV + e] = dSg[e];
    }
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

template <int KD, int VD>
cudaError_t launch_bwd_kv(const BwdArgs& a, cudaStream_t s) {
    const int units = a.N * a.HV;
    if (units > 0) {
        auto* fn = gdn_bwd_kernel<KD, VD>;
        const int smem = static_cast<int>(sizeof(BwdSmem<KD>));
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        fn<<<units, kBT, smem, s>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.group > 1 && a.T > 0) {
        gdn_bwd_group_sum_kernel<<<1024, 256, 0, s>>>(a);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s) {
    if (a.K == 128) return a.V == 128 ? launch_bwd_kv<128, 128>(a, s) : launch_bwd_kv<128, 64>(a, s);
    return a.V == 128 ? launch_bwd_kv<64, 128>(a, s) : launch_bwd_kv<64, 64>(a, s);
}

}  // namespace la
