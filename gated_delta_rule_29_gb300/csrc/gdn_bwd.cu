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
constexpr int kPC = kC + 1;     // padded row strides (fp32 words)
constexpr int kPT = kVT + 1;

__device__ __forceinline__ float bfv(const uint16_t* p, int64_t i) {
    return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
}
__device__ __forceinline__ uint16_t f2b(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

template <int KD>
struct BwdSmem {
    static constexpr int PK = KD + 1;
    float Kh[kC * PK];      // normalised keys (rows past the end are zero)
    float Qh[kC * PK];      // normalised queries
    float Tm[kC * kPC];     // T = (I + A)^{-1}
    float Pm[kC * kPC];     // P (incl. lower)
    float Gk[kC * kPC];     // (k_i . k_j) Gamma_ij, lower incl.
    float dA[kC * kPC];     // accumulated over tiles
    float dP[kC * kPC];
    float SJ[KD * kPT];     // tile of the entering state
    float dSJ[KD * kPT];    // tile of dS_next (then dS)
    float VJ[kC * kPT], OJ[kC * kPT], X[kC * kPT], D[kC * kPT], dD[kC * kPT], dY[kC * kPT];
    float beta[kC], b[kC], gam[kC], GC[kC], rk[kC], rq[kC];
    float dbeta[kC], db[kC], wv[kC];
    float red[kBT / 32];
};

// out[r][c] (+)= alpha * sum_m L(r, m) R(m, c) for an RxC output spread over the CTA.
template <int R, int CC, int MM, class FL, class FR, class FO>
__device__ __forceinline__ void cta_mm(FL L, FR Rm, FO out) {
    constexpr int PER = R * CC / kBT;
    static_assert(R * CC % kBT == 0, "tile");
    const int tid = threadIdx.x;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const int idx = tid + e * kBT;
        const int r = idx / CC, c = idx % CC;
        float acc = 0.f;
#pragma unroll 8
        for (int m = 0; m < MM; ++m) acc = fmaf(L(r, m), Rm(m, c), acc);
        out(r, c, acc);
    }
}

template <int KD, int VD>
__global__ void __launch_bounds__(kBT, 1) gdn_bwd_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BwdSmem<KD>& s = *reinterpret_cast<BwdSmem<KD>*>(smem_raw);
    constexpr int PK = BwdSmem<KD>::PK;
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

    // thread ownership for the per-row accumulators of dK and dQ: row i, 32-column slice
    constexpr int KSL = KD / 4;
    const int own_r = tid >> 2, own_c0 = (tid & 3) * KSL;

    for (int c = nch - 1; c >= 0; --c) {
        const int64_t t0 = ts + static_cast<int64_t>(c) * kC;
        const int n = static_cast<int>(L - static_cast<int64_t>(c) * kC < kC ? L - static_cast<int64_t>(c) * kC : kC);
        const float* Sc = a.ckpt + ((a.ckpt_off[seq] + c) * HO + h) * KV;  // state entering this chunk

        // ---- chunk-level quantities: normalised rows, decays, A, T, P
        for (int e = tid; e < kC * KD; e += kBT) {
            const int i = e / KD, d = e % KD;
            float kv = 0.f, qv = 0.f;
            if (i < n) {
                kv = bfv(a.k, (t0 + i) * a.k_st + hk * a.k_sh + d);
                qv = bfv(a.q, (t0 + i) * a.q_st + hk * a.q_sh + d);
            }
            s.Kh[i * PK + d] = kv;
            s.Qh[i * PK + d] = qv;
        }
        if (tid < kC) {
            const int i = tid;
            s.beta[i] = i < n ? a.beta[(t0 + i) * a.b_st + h * a.b_sh] : 0.f;
            s.b[i] = i < n ? a.g[(t0 + i) * a.g_st + h * a.g_sh] : 0.f;
        }
        __syncthreads();
        if (tid < kC) {
            // row norms (one thread per row; K is at most 128) and the chunk-local cumsum of g
            const int i = tid;
            float sk = 0.f, sq = 0.f;
            for (int d = 0; d < KD; ++d) {
                sk = fmaf(s.Kh[i * PK + d], s.Kh[i * PK + d], sk);
                sq = fmaf(s.Qh[i * PK + d], s.Qh[i * PK + d], sq);
            }
            s.rk[i] = (i < n && a.l2norm) ? 1.0f / sqrtf(sk + 1e-6f) : (i < n ? 1.f : 0.f);
            s.rq[i] = (i < n && a.l2norm) ? 1.0f / sqrtf(sq + 1e-6f) : (i < n ? 1.f : 0.f);
        }
        if (tid == 64) {
            float acc = 0.f;
            for (int i = 0; i < kC; ++i) {
                acc += s.b[i];
                s.b[i] = acc;  // rows past the end carry g = 0, so b stays at b_last
            }
        }
        __syncthreads();
        for (int e = tid; e < kC * KD; e += kBT) {
            const int i = e / KD, d = e % KD;
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
        // Gk = (k_i . k_j) Gamma_ij and P (lower incl.), zero dA / dP
        for (int e = tid; e < kC * kC; e += kBT) {
            const int i = e / kC, j = e % kC;
            float kk = 0.f, qk = 0.f;
            if (j <= i) {
                for (int d = 0; d < KD; ++d) {
                    kk = fmaf(s.Kh[i * PK + d], s.Kh[j * PK + d], kk);
                    qk = fmaf(s.Qh[i * PK + d], s.Kh[j * PK + d], qk);
                }
                const float G = expf(s.b[i] - s.b[j]);
                kk *= G;
                qk *= G;
            }
            s.Gk[i * kPC + j] = kk;
            s.Pm[i * kPC + j] = qk;
            s.dA[i * kPC + j] = 0.f;
            s.dP[i * kPC + j] = 0.f;
        }
        __syncthreads();
        // T = (I + A)^{-1}: column j by forward substitution, one thread per column
        if (tid < kC) {
            const int j = tid;
            for (int i = 0; i < kC; ++i) {
                float t = (i == j) ? 1.f : 0.f;
                if (i > j) {
                    float acc = 0.f;
                    for (int m = j; m < i; ++m) acc = fmaf(s.beta[i] * s.Gk[i * kPC + m], s.Tm[m * kPC + j], acc);
                    t = -acc;
                } else if (i < j) {
                    t = 0.f;
                }
                s.Tm[i * kPC + j] = t;
            }
        }
        __syncthreads();

        float dKacc[KSL], dQacc[KSL];
#pragma unroll
        for (int e = 0; e < KSL; ++e) dKacc[e] = dQacc[e] = 0.f;

        // ---- the value tiles: independent columns of S and dS
        for (int j0 = 0; j0 < VD; j0 += kVT) {
            for (int e = tid; e < KD * kVT; e += kBT) {
                const int r = e / kVT, cc = e % kVT;
                s.SJ[r * kPT + cc] = Sc[r * VD + j0 + cc];
                s.dSJ[r * kPT + cc] = dSg[r * VD + j0 + cc];
            }
            for (int e = tid; e < kC * kVT; e += kBT) {
                const int i = e / kVT, cc = e % kVT;
                float vv = 0.f, ov = 0.f;
                if (i < n) {
                    vv = bfv(a.v, (t0 + i) * a.v_st + h * a.v_sh + j0 + cc);
                    ov = bfv(a.dout, (t0 + i) * a.do_st + h * a.do_sh + j0 + cc);
                }
                s.VJ[i * kPT + cc] = vv;
                s.OJ[i * kPT + cc] = ov;
            }
            __syncthreads();
            // x = K S_J
            cta_mm<kC, kVT, KD>([&](int r, int m) { return s.Kh[r * PK + m]; },
                                [&](int m, int cc) { return s.SJ[m * kPT + cc]; },
                                [&](int r, int cc, float acc) { s.X[r * kPT + cc] = acc; });
            __syncthreads();
            // D = T Y with Y = beta V - beta gamma x; dD = scale P^T dO + Gamma_C (K dS_J)
            cta_mm<kC, kVT, kC>([&](int r, int m) { return s.Tm[r * kPC + m]; },
                                [&](int m, int cc) {
                                    return s.beta[m] * (s.VJ[m * kPT + cc] - s.gam[m] * s.X[m * kPT + cc]);
                                },
                                [&](int r, int cc, float acc) { s.D[r * kPT + cc] = acc; });
            cta_mm<kC, kVT, KD>([&](int r, int m) { return s.Kh[r * PK + m]; },
                                [&](int m, int cc) { return s.dSJ[m * kPT + cc]; },
                                [&](int r, int cc, float acc) { s.dD[r * kPT + cc] = s.GC[r] * acc; });
            __syncthreads();
            cta_mm<kC, kVT, kC>([&](int r, int m) { return s.Pm[m * kPC + r]; },
                                [&](int m, int cc) { return s.OJ[m * kPT + cc]; },
                                [&](int r, int cc, float acc) { s.dD[r * kPT + cc] += a.scale * acc; });
            __syncthreads();
            // dY = T^T dD; dV = beta dY (final)
            cta_mm<kC, kVT, kC>([&](int r, int m) { return s.Tm[m * kPC + r]; },
                                [&](int m, int cc) { return s.dD[m * kPT + cc]; },
                                [&](int r, int cc, float acc) {
                                    s.dY[r * kPT + cc] = acc;
                                    if (r < n) a.dv[(t0 + r) * a.dv_st + h * a.dv_sh + j0 + cc] = f2b(s.beta[r] * acc);
                                });
            __syncthreads();
            // per-row sums: dbeta (Y's beta), db (Y's gamma and O's gamma)
            if (tid < kC) {
                const int i = tid;
                float sb = 0.f, sg = 0.f, so = 0.f;
                for (int cc = 0; cc < kVT; ++cc) {
                    const float dy = s.dY[i * kPT + cc], xv = s.X[i * kPT + cc];
                    sb = fmaf(dy, s.VJ[i * kPT + cc] - s.gam[i] * xv, sb);
                    sg = fmaf(dy, xv, sg);
                    float qs = 0.f;
                    for (int d = 0; d < KD; ++d) qs = fmaf(s.Qh[i * PK + d], s.SJ[d * kPT + cc], qs);
                    so = fmaf(s.OJ[i * kPT + cc], qs, so);
                }
                s.dbeta[i] += sb;
                s.db[i] += s.gam[i] * (a.scale * so - s.beta[i] * sg);
            } else if (tid < 2 * kC) {
                // the Gamma_Cj terms of S_next: w_j = Gamma_Cj sum_v (K dS_J)_jv D_jv moves from b_j
                // to b_last
                const int j = tid - kC;
                float w = 0.f;
                for (int cc = 0; cc < kVT; ++cc) {
                    float kd = 0.f;
                    for (int d = 0; d < KD; ++d) kd = fmaf(s.Kh[j * PK + d], s.dSJ[d * kPT + cc], kd);
                    w = fmaf(kd, s.D[j * kPT + cc], w);
                }
                s.wv[j] = w * s.GC[j];
            }
            {
                // gamma_last <dS_J, S_J>: the decay of the entering state into S_next
                float p = 0.f;
                for (int e = tid; e < KD * kVT; e += kBT) {
                    const int r = e / kVT, cc = e % kVT;
                    p = fmaf(s.dSJ[r * kPT + cc], s.SJ[r * kPT + cc], p);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
                if ((tid & 31) == 0) s.red[tid >> 5] = p;
            }
            __syncthreads();
            if (tid < kC) s.db[tid] -= s.wv[tid];
            __syncthreads();
            if (tid == 0) {
                float p = 0.f, w = 0.f;
                for (int i = 0; i < kBT / 32; ++i) p += s.red[i];
                for (int j = 0; j < kC; ++j) w += s.wv[j];
                s.db[n - 1] += s.gam[n - 1] * p + w;
            }
            // dA += -dY D^T, dP += scale dO D^T (lower parts)
            for (int e = tid; e < kC * kC; e += kBT) {
                const int i = e / kC, j = e % kC;
                if (j > i) continue;
                float ad = 0.f, pd = 0.f;
#pragma unroll
                for (int cc = 0; cc < kVT; ++cc) {
                    ad = fmaf(s.dY[i * kPT + cc], s.D[j * kPT + cc], ad);
                    pd = fmaf(s.OJ[i * kPT + cc], s.D[j * kPT + cc], pd);
                }
                if (j < i) s.dA[i * kPC + j] -= ad;
                s.dP[i * kPC + j] += a.scale * pd;
            }
            // dK += dx S_J^T + Gamma_C D dS_J^T (dx = -beta gamma dY); dQ += scale gamma dO S_J^T
            {
                const int i = own_r;
                const float bx = -s.beta[i] * s.gam[i], gc = s.GC[i], sg = a.scale * s.gam[i];
#pragma unroll
                for (int e = 0; e < KSL; ++e) {
                    const int d = own_c0 + e;
                    float ak = 0.f, aq = 0.f;
#pragma unroll
                    for (int cc = 0; cc < kVT; ++cc) {
                        const float sj = s.SJ[d * kPT + cc];
                        ak = fmaf(bx * s.dY[i * kPT + cc], sj, ak);
                        ak = fmaf(gc * s.D[i * kPT + cc], s.dSJ[d * kPT + cc], ak);
                        aq = fmaf(s.OJ[i * kPT + cc], sj, aq);
                    }
                    dKacc[e] += ak;
                    dQacc[e] += sg * aq;
                }
            }
            __syncthreads();
            // dS_J <- gamma_last dS_J + K^T dx + scale Q^T (gamma dO); back to the global buffer
            cta_mm<KD, kVT, kC>([&](int r, int m) { return s.Kh[m * PK + r]; },
                                [&](int m, int cc) { return -s.beta[m] * s.gam[m] * s.dY[m * kPT + cc]; },
                                [&](int r, int cc, float acc) {
                                    float qo = 0.f;
                                    for (int m = 0; m < kC; ++m)
                                        qo = fmaf(s.Qh[m * PK + r], s.gam[m] * s.OJ[m * kPT + cc], qo);
                                    dSg[r * VD + j0 + cc] = s.gam[n - 1] * s.dSJ[r * kPT + cc] + acc + a.scale * qo;
                                });
            __syncthreads();
        }

        // ---- tile-independent terms: A and P backward, dbeta, db, dg, the norms
        if (tid < kC) {
            const int i = tid;
            float sb = 0.f, rowsum = 0.f, colsum = 0.f;
            for (int j = 0; j < kC; ++j) {
                if (j < i) {
                    sb = fmaf(s.dA[i * kPC + j], s.Gk[i * kPC + j], sb);
                    rowsum += s.dA[i * kPC + j] * s.beta[i] * s.Gk[i * kPC + j];
                }
                if (j <= i) rowsum += s.dP[i * kPC + j] * s.Pm[i * kPC + j];
                if (j > i) colsum += s.dA[j * kPC + i] * s.beta[j] * s.Gk[j * kPC + i];
                if (j >= i) colsum += s.dP[j * kPC + i] * s.Pm[j * kPC + i];
            }
            s.dbeta[i] += sb;
            s.db[i] += rowsum - colsum;  // log Gamma_ij = b_i - b_j
        }
        __syncthreads();
        // M = dA (.) beta_i Gamma (strict), H = dP (.) Gamma (incl.), in place
        for (int e = tid; e < kC * kC; e += kBT) {
            const int i = e / kC, j = e % kC;
            const float G = j <= i ? expf(s.b[i] - s.b[j]) : 0.f;
            s.dA[i * kPC + j] = j < i ? s.dA[i * kPC + j] * s.beta[i] * G : 0.f;
            s.dP[i * kPC + j] = j <= i ? s.dP[i * kPC + j] * G : 0.f;
        }
        __syncthreads();
        {
            // dK += M K + M^T K + H^T Q, dQ += H K
            const int i = own_r;
#pragma unroll
            for (int e = 0; e < KSL; ++e) {
                const int d = own_c0 + e;
                float ak = 0.f, aq = 0.f;
                for (int j = 0; j < kC; ++j) {
                    const float kj = s.Kh[j * PK + d];
                    ak = fmaf(s.dA[i * kPC + j] + s.dA[j * kPC + i], kj, ak);
                    ak = fmaf(s.dP[j * kPC + i], s.Qh[j * PK + d], ak);
                    aq = fmaf(s.dP[i * kPC + j], kj, aq);
                }
                dKacc[e] += ak;
                dQacc[e] += aq;
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
                pk = fmaf(s.Kh[i * PK + own_c0 + e], dKacc[e], pk);
                pq = fmaf(s.Qh[i * PK + own_c0 + e], dQacc[e], pq);
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
                    const int d = own_c0 + e;
                    float gk = dKacc[e], gq = dQacc[e];
                    if (a.l2norm) {
                        gk = rkk * (gk - pk * s.Kh[i * PK + d]);
                        gq = rqq * (gq - pq * s.Qh[i * PK + d]);
                    }
                    const int64_t t = t0 + i;
                    if (a.group == 1) {
                        a.dk[t * a.dk_st + hk * a.dk_sh + d] = f2b(gk);
                        a.dq[t * a.dq_st + hk * a.dq_sh + d] = f2b(gq);
                    } else {
                        a.dkh[(t * HO + h) * KD + d] = gk;
                        a.dqh[(t * HO + h) * KD + d] = gq;
                    }
                }
            }
        }
        __syncthreads();
    }
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
