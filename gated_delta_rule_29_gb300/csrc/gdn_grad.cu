// gdn_grad.cu -- the state-gradient pass of gdn_summary_bwd on the tensor cores (sm_103a).
//
// Method (cuDNN Linear Attention page, "Summaries": every summary op has a state-gradient
// counterpart).  With the chunked form of the forward (the chunk kernel's header), a chunk
// with entering state S maps the gradient of the state leaving it, dS_out, and the outputs'
// cotangent dO to the gradient of the state entering it:
//
//   dD    = P^T dO + diag(sd) (K dS_out)          sd_j = 2^{b_C - b_j} rk_j   (64 x V)
//   dY    = T^T dD
//   dS_in = 2^{b_C} dS_out + K^T (-sx (.) dY) + Q^T (sq (.) dO)
//                                                 sx_j = beta_j 2^{b_j} rk_j, sq_i = scale rq_i 2^{b_i}
//
// (reverse mode through D = T X, X = beta V - sx (K S), O = sq (Q S) + P D and the state update;
// K and Q are the raw rows, the norms live in the factors).  T, P and the factors are the WY
// records of the forward's WY pass, so this pass only walks each (span, head) backwards over
// its chunks with the state-dependent products.
//
// Mapping, mirrored from the forward's state pass: one persistent CTA of 256 threads per SM takes
// (span, head) units longest first; threads r and r + 128 own TMEM lane r = value column v and
// split its columns (the chunk's tokens, or the key columns of dS^T) in halves.  dS^T (fp32,
// lane v, column k) lives in TMEM for the whole span and is updated in place by the tensor core;
// every product is a tcgen05.mma (kind::f16, bf16 operands split into hi + lo parts, fp32
// accumulation, M = 128 value columns) in transposed form:
//   (K dS)^T  = dS^T K^T        A = dS^T (hi, lo)       B = K (K-major)
//   (P^T dO)^T = dO^T P         A = dO^T (MN-major)     B = P (MN-major)
//   dY^T      = dD^T T          A = dD^T (hi, lo)       B = T (MN-major)
//   dS^T     += a^T K + b^T Q   A = a^T, b^T (hi, lo)   B = K, Q (MN-major), a = -sx dY, b = sq dO
// The K/Q and dO tiles and the records arrive by TMA (128-byte swizzle), prefetched one chunk
// ahead (in reverse order); the state gradient is pre-multiplied by the decay of the chunk it is
// about to enter, so the update product accumulates onto it.  For the full backward (gdn_bwd) the
// pass also stores the gradient leaving every chunk (its bf16 hi + lo copy, the layout the chunk
// pass reads) and the gradient entering each sequence is d_initial_state.  Every wait is bounded.
#include <cuda_bf16.h>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"
#include "ptx.cuh"
#include "gdn_device.cuh"

namespace la {
namespace {

constexpr int kGT = 256;  // threads: two per TMEM lane, splitting the columns
constexpr int kGradPieces = 4;  // chunk ranges per unit when the units outnumber the SMs
constexpr float kLog2eG = 1.4426950408889634f;

// shared memory (byte offsets from the 1024-aligned base)
constexpr uint32_t G_KQ = 0;        // [region 0..1][128 rows: K 0-63, Q 64-127][128 B]
constexpr uint32_t G_DO = 32768;    // dO tile [region 0..1][64 rows][128 B]
constexpr uint32_t G_WB = 49152;    // dS^T bf16 hi [2][128][128 B] | dD^T hi, lo | a^T hi, lo
constexpr uint32_t G_SLO = 81920;   // dS^T bf16 lo, same layout
constexpr uint32_t G_B2 = 114688;   // b^T hi, lo [128][128 B] each
constexpr uint32_t G_TB = 147456;   // T bf16 [64][128 B]
constexpr uint32_t G_PB = 155648;   // P bf16 [64][128 B]
constexpr uint32_t G_SC = 163840;   // scalars
constexpr uint32_t G_SMEM = G_SC + 2048 + 1024;

// TMEM columns (fp32, 128 lanes)
constexpr uint32_t G_DS = 0;     // dS^T (K columns)
constexpr uint32_t G_R1 = 128;   // (K dS)^T, then dY^T
constexpr uint32_t G_R2 = 192;   // (P^T dO)^T
constexpr uint32_t G_TMEM = 256;

struct __align__(16) GradScalars {
    float bet[64], sx[64], sq[64], sd[64];  // one WY record's factors (contiguous: one bulk copy)
    float gsum[2];                          // per-warp sums of the next chunk's g * log2(e)
    uint64_t bar_kq, bar_do, bar_mma, bar_f;
    uint32_t tmem_base;
    int32_t unit_lo, unit_hi, status0, flag_ok;
};
static_assert(sizeof(GradScalars) <= 2048, "gradient-pass scalar area");

// Bounded wait until *f >= need (acquire, GPU scope); false after budget_ns.  One thread.
__device__ __forceinline__ bool wait_flag(const int32_t* f, int32_t need, uint64_t budget_ns) {
    uint64_t t0 = 0;
    for (int it = 0;; ++it) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
        if (v >= need) return true;
        if (it == 0) t0 = globaltimer_ns();
        else if (globaltimer_ns() - t0 > budget_ns) return false;
        __nanosleep(256);
    }
}
__device__ __forceinline__ void set_flag(int32_t* f, int32_t v) {
    __threadfence();
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

// One WY record's T, P and factors, on bar_f.  One thread.
__device__ __forceinline__ void grad_load_record(const ChunkArgs& a, const CUtensorMap& wymap, int64_t chunk, int h,
                                                 uint8_t* TB, uint8_t* PB, GradScalars& sc) {
    const int64_t item = chunk * a.HV + h;
    mbar_arrive_expect_tx(&sc.bar_f, static_cast<uint32_t>(kWyRecordBytes));
    tma_load_3d(TB, &wymap, &sc.bar_f, 0, static_cast<int>(item), 0);
    tma_load_3d(PB, &wymap, &sc.bar_f, 0, static_cast<int>(item), 64);
    bulk_load(sc.bet, a.wy + item * static_cast<int64_t>(kWyRecordBytes) + 2 * kWyTileBytes,
              static_cast<uint32_t>(kWyFactorBytes), &sc.bar_f);
}

template <int KD>
__global__ void __launch_bounds__(kGT, 1)
    gdn_grad_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap domap, const __grid_constant__ CUtensorMap wymap,
                    const ChunkArgs a) {
    constexpr int KP = KD / 16;  // 16-column pieces of the state gradient
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GradScalars& sc = *reinterpret_cast<GradScalars*>(sm + G_SC);
    uint8_t* KQ = sm + G_KQ;
    uint8_t* DO = sm + G_DO;
    uint8_t* WB = sm + G_WB;
    uint8_t* SLO = sm + G_SLO;
    uint8_t* B2 = sm + G_B2;
    uint8_t* TB = sm + G_TB;
    uint8_t* PB = sm + G_PB;
    const int tid = threadIdx.x;
    const int r = tid & 127;  // TMEM lane = value column
    const int hf = tid >> 7;  // column half: tokens 32 hf .., key columns KD / 2 hf ..
    const int HO = a.HV;

    if (tid == 0) sc.status0 = *reinterpret_cast<volatile int32_t*>(&a.hdr->status);
    __syncthreads();
    if (sc.status0 != LA_OK) return;
    if (tid < 32) {
        tmem_alloc(&sc.tmem_base, G_TMEM);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sc.bar_kq, 1);
        mbar_init(&sc.bar_do, 1);
        mbar_init(&sc.bar_mma, 1);
        mbar_init(&sc.bar_f, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sc.tmem_base;
    const uint32_t trow = tmem + (static_cast<uint32_t>(r & ~31) << 16);
    constexpr int KH = KP / 2;  // 16-column pieces of the state gradient per column half
    // operand descriptors (an operand at byte offset off from a buffer uses base + (off >> 4))
    const uint64_t d_kq = sdesc_sw128(smem_u32(KQ), 16, 1024);             // K rows, K-major
    const uint64_t d_k_mn = sdesc_sw128(smem_u32(KQ), 16384, 1024);        // K rows, MN-major
    const uint64_t d_q_mn = sdesc_sw128(smem_u32(KQ + 8192), 16384, 1024); // Q rows, MN-major
    const uint64_t d_wb = sdesc_sw128(smem_u32(WB), 16, 1024);
    const uint64_t d_slo = sdesc_sw128(smem_u32(SLO), 16, 1024);
    const uint64_t d_b2 = sdesc_sw128(smem_u32(B2), 16, 1024);
    const uint64_t d_do_mn = sdesc_sw128(smem_u32(DO), 8192, 1024);        // dO^T: value columns MN-major
    const uint64_t d_p_mn = sdesc_sw128(smem_u32(PB), 8192, 1024);         // P read MN-major
    const uint64_t d_t_mn = sdesc_sw128(smem_u32(TB), 8192, 1024);         // T read MN-major
    const uint32_t kq_bytes = KD * 256u;                                    // K and Q rows
    const uint32_t do_bytes = static_cast<uint32_t>(a.V) * 128u;
    const uint64_t budget = a.wait_budget_ns;
    const int NP = a.pieces > 1 ? a.pieces : 1;  // chunk ranges per unit
    uint32_t ph_kq = 0, ph_do = 0, ph_mma = 0, ph_f = 0;
    bool pend_kq = false, pend_do = false, pend_mma = false, pend_f = false, failed = false;

    for (;;) {
        if (tid == 0) {
            const unsigned long long u = atomicAdd(reinterpret_cast<unsigned long long*>(&a.hdr->ticket), 1ull);
            sc.unit_lo = static_cast<int32_t>(u & 0xFFFFFFFFull);
            sc.unit_hi = static_cast<int32_t>(u >> 32);
        }
        __syncthreads();
        const int64_t tk = (static_cast<int64_t>(sc.unit_hi) << 32) | static_cast<uint32_t>(sc.unit_lo);
        __syncthreads();  // every thread has read the ticket before thread 0 may take the next one
        // tickets run through the units' last ranges first, then the ranges before them: a
        // range's successor has an earlier ticket, held by a CTA that is running or done
        if (tk >= a.num_units * NP) break;
        const int64_t unit = tk % a.num_units;
        const int piece = NP - 1 - static_cast<int>(tk / a.num_units);
        const int seq = a.order[unit / HO];
        const int h = static_cast<int>(unit % HO);
        const int hk = h / a.group;
        const int64_t tok_s = cu_get(a.cu, a.cu64, seq);
        const int64_t L = cu_get(a.cu, a.cu64, seq + 1) - tok_s;
        const int nch_all = static_cast<int>((L + kChunk - 1) / kChunk);
        const int clo = static_cast<int>(static_cast<int64_t>(piece) * nch_all / NP);        // chunks clo ..
        const int chi = static_cast<int>(static_cast<int64_t>(piece + 1) * nch_all / NP);    // .. chi - 1
        const int nch = chi;  // (the walk starts at chunk chi - 1)
        const int64_t unit_state = static_cast<int64_t>(seq) * HO + h;
        // where the range starts from (d_final_state, or its successor's output) and where it ends
        const float* src = piece == NP - 1 ? static_cast<const float*>(a.s0) : a.grad_carry;
        float* dst = piece == 0 ? a.final_state : a.grad_carry;
        if (piece < NP - 1) {
            if (tid == 0) sc.flag_ok = wait_flag(a.grad_flags + unit_state, NP - 1 - piece, budget) ? 1 : 0;
            if (__syncthreads_or(tid == 0 && sc.flag_ok == 0)) { failed = true; break; }
        }
        float gA = 0.f, gdt = 0.f;
        if (a.gate_mode == LA_GATE_SOFTPLUS && tid < 64) {
            gA = -expf(a.a_log[h]);
            gdt = a.dt_bias[h];
        }
        // the total decay of the range's last chunk, the first one walked
        if (tid < 64) {
            const int64_t t_last = tok_s + static_cast<int64_t>(nch > clo ? nch - 1 : 0) * kChunk;
            float x = (nch > clo && t_last + tid < tok_s + L) ? gate_row<false>(a, t_last + tid, h, gA, gdt) * kLog2eG : 0.f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
            if ((tid & 31) == 0) sc.gsum[tid >> 5] = x;
        }
        __syncthreads();
        const float gam0 = nch > clo ? exp2f(sc.gsum[0] + sc.gsum[1]) : 1.f;

        // ---- the gradient leaving the span (d_final_state, or 0): bf16 hi + lo copy for (K dS), and
        // TMEM pre-multiplied by the last chunk's decay; an empty span passes it straight through
        {
            const int64_t base = unit_state * KD * a.V + r;
#pragma unroll 1
            for (int p = hf * KH; p < (hf + 1) * KH; ++p) {
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    x[e] = (src && r < a.V) ? src[base + static_cast<int64_t>(16 * p + e) * a.V] : 0.f;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int kc = 2 * p + hh;
                    const uint32_t off = (kc >> 3) * 16384 + sw128_off(r, kc & 7);
                    store8_split(WB + off, SLO + off, &x[8 * hh]);
                }
                if (nch == clo && r < a.V && dst) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) dst[base + static_cast<int64_t>(16 * p + e) * a.V] = x[e];
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) x[e] *= gam0;
                tmem_st16(trow + G_DS + 16 * p, x);
            }
            tmem_wait_st();
        }
        if (nch == clo) {
            // an empty range passes the gradient straight through
            __syncthreads();
            if (tid == 0 && piece > 0) set_flag(a.grad_flags + unit_state, NP - piece);
            continue;
        }

        // ---- the last chunk's tiles and record
        {
            const int64_t tl = tok_s + static_cast<int64_t>(nch - 1) * kChunk;
            if (tid == 0) {
                mbar_arrive_expect_tx(&sc.bar_kq, kq_bytes);
#pragma unroll
                for (int rg = 0; rg < KD / 64; ++rg) {
                    tma_load_3d(KQ + rg * 16384, &kmap, &sc.bar_kq, rg * 64, hk, static_cast<int>(tl));
                    tma_load_3d(KQ + rg * 16384 + 8192, &qmap, &sc.bar_kq, rg * 64, hk, static_cast<int>(tl));
                }
                mbar_arrive_expect_tx(&sc.bar_do, do_bytes);
                for (int rg = 0; rg < a.V / 64; ++rg)
                    tma_load_3d(DO + rg * 8192, &domap, &sc.bar_do, rg * 64, h, static_cast<int>(tl));
                grad_load_record(a, wymap, a.chunk_off[seq] + nch - 1, h, TB, PB, sc);
            }
            pend_kq = pend_do = pend_f = true;
        }
        for (int c = nch - 1; c >= clo; --c) {
            const bool last = c == clo;  // the last chunk walked (the range's first)
            const int64_t t0 = tok_s + static_cast<int64_t>(c) * kChunk;
            // the gates of the chunk walked next (a full chunk: only the span's last can be short)
            float g_nx = 0.f;
            if (!last && tid < 64) g_nx = gate_row<false>(a, t0 - kChunk + tid, h, gA, gdt);

            // ---- G1: (K dS)^T -> R1 (hi + lo of dS), then (P^T dO)^T -> R2 once dO and the record are in
            bool ok = mbar_wait(&sc.bar_kq, ph_kq, budget);
            if (ok) {
                ph_kq ^= 1u;
                pend_kq = false;
            }
            if (c == nch - 1) {
                // every thread has written its row of the starting gradient's bf16 copy
                fence_proxy_async_smem();
                tc_fence_before();
                if (__syncthreads_or(!ok)) { failed = true; break; }
            }
            if (tid == 0 && ok && a.ds_chunks) {
                // the full backward's chunk pass reads the gradient leaving this chunk: its bf16
                // hi + lo copy goes out by bulk copy before the dD^T tiles take its place
                const int64_t item = (a.chunk_off[seq] + c) * HO + h;
                bulk_store(a.ds_chunks + item * 65536, WB, 32768u);
                bulk_store(a.ds_chunks + item * 65536 + 32768, SLO, 32768u);
                bulk_commit_group();
            }
            if (tid == 0 && ok) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
                for (int kk = 0; kk < KD / 16; ++kk) {
                    const uint64_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    umma_bf16(tmem + G_R1, d_wb + off, d_kq + off, idesc, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < KD / 16; ++kk) {
                    const uint64_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    umma_bf16(tmem + G_R1, d_slo + off, d_kq + off, idesc, 1u);
                }
            }
            {
                const bool okd = mbar_wait(&sc.bar_do, ph_do, budget);
                if (okd) {
                    ph_do ^= 1u;
                    pend_do = false;
                }
                const bool okf = mbar_wait(&sc.bar_f, ph_f, budget);
                if (okf) {
                    ph_f ^= 1u;
                    pend_f = false;
                }
                ok = ok && okd && okf;
            }
            if (tid == 0) {
                tc_fence_after();
                if (ok) {
                    const uint32_t idesc = idesc_bf16_f32(128, 64, true, true);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + G_R2, d_do_mn + ((kk * 2048) >> 4), d_p_mn + ((kk * 2048) >> 4), idesc, kk > 0);
                }
                umma_commit(&sc.bar_mma);  // (arrives once everything this thread issued is done)
            }
            pend_mma = true;
            // b^T = sq (.) dO^T (hi + lo), from this thread's column of the dO tile, while the products run
            {
                const bool has_v = ok && r < a.V;
                const uint8_t* vcol = DO + (r >> 6) * 8192 + (r & 7) * 2;
                const uint32_t vchunk = (r & 63) >> 3;
#pragma unroll
                for (int cc = 4 * hf; cc < 4 * hf + 4; ++cc) {
                    float x[8], sqv[8];
                    ld8(sqv, &sc.sq[8 * cc]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float dov = has_v
                            ? bf16_bits_to_f(*reinterpret_cast<const uint16_t*>(vcol + sw128_off(8 * cc + e, vchunk)))
                            : 0.f;
                        x[e] = sqv[e] * dov;
                    }
                    store8_split(B2 + sw128_off(r, cc), B2 + 16384 + sw128_off(r, cc), x);
                }
            }

            // ---- G2: dD^T = (P^T dO)^T + sd (.) (K dS)^T -> WB (hi, lo)
            {
                const bool okm = mbar_wait(&sc.bar_mma, ph_mma, budget);
                if (okm) {
                    ph_mma ^= 1u;
                    pend_mma = false;
                }
                ok = ok && okm;
            }
            if (a.ds_chunks) {
                if (tid == 0) bulk_wait_read_all();
                __syncthreads();
            }
            tc_fence_after();
            {
                float k32[32], p32[32];
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    tmem_ld16(trow + G_R1 + 32 * hf + 16 * p, *reinterpret_cast<float(*)[16]>(&k32[16 * p]));
                    tmem_ld16(trow + G_R2 + 32 * hf + 16 * p, *reinterpret_cast<float(*)[16]>(&p32[16 * p]));
                }
                tmem_wait_ld();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int cc = 4 * hf + c4;
                    float x[8], sdv[8];
                    ld8(sdv, &sc.sd[8 * cc]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = p32[8 * c4 + e] + sdv[e] * k32[8 * c4 + e];
                    store8_split(WB + sw128_off(r, cc), WB + 16384 + sw128_off(r, cc), x);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }
            // the dO tile is consumed (by the product and by b): fetch the next chunk's
            if (tid == 0 && !last) {
                mbar_arrive_expect_tx(&sc.bar_do, do_bytes);
                for (int rg = 0; rg < a.V / 64; ++rg)
                    tma_load_3d(DO + rg * 8192, &domap, &sc.bar_do, rg * 64, h, static_cast<int>(t0 - kChunk));
            }
            if (!last) pend_do = true;

            // ---- G3: dY^T = dD^T T -> R1
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, 64, false, true);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + G_R1, d_wb + ((part * 16384 + kk * 32) >> 4), d_t_mn + ((kk * 2048) >> 4), idesc,
                                  (part | kk) != 0);
                umma_commit(&sc.bar_mma);
            }
            pend_mma = true;
            if (tid < 64) {
                // total gate of the chunk walked next (the decay the new gradient is pre-multiplied by)
                float x = last ? 0.f : g_nx * kLog2eG;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
                if ((tid & 31) == 0) sc.gsum[tid >> 5] = x;
            }
            {
                const bool okm = mbar_wait(&sc.bar_mma, ph_mma, budget);
                if (okm) {
                    ph_mma ^= 1u;
                    pend_mma = false;
                }
                ok = ok && okm;
            }
            tc_fence_after();

            // ---- G4: a^T = -sx (.) dY^T -> WB (hi, lo), dD^T being consumed
            {
                float d32[32];
#pragma unroll
                for (int p = 0; p < 2; ++p)
                    tmem_ld16(trow + G_R1 + 32 * hf + 16 * p, *reinterpret_cast<float(*)[16]>(&d32[16 * p]));
                tmem_wait_ld();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int cc = 4 * hf + c4;
                    float x[8], sxv[8];
                    ld8(sxv, &sc.sx[8 * cc]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = -sxv[e] * d32[8 * c4 + e];
                    store8_split(WB + sw128_off(r, cc), WB + 16384 + sw128_off(r, cc), x);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }
            // T, P and the factors are consumed: fetch the next chunk's record
            if (tid == 0 && !last) grad_load_record(a, wymap, a.chunk_off[seq] + c - 1, h, TB, PB, sc);
            if (!last) pend_f = true;

            // ---- G5: dS^T += a^T K + b^T Q (K and Q read MN-major), onto the pre-multiplied gradient
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, KD, false, true);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + G_DS, d_wb + ((part * 16384 + kk * 32) >> 4), d_k_mn + ((kk * 2048) >> 4), idesc,
                                  1u);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + G_DS, d_b2 + ((part * 16384 + kk * 32) >> 4), d_q_mn + ((kk * 2048) >> 4), idesc,
                                  1u);
                umma_commit(&sc.bar_mma);
            }
            pend_mma = true;
            {
                const bool okm = mbar_wait(&sc.bar_mma, ph_mma, budget);
                if (okm) {
                    ph_mma ^= 1u;
                    pend_mma = false;
                }
                ok = ok && okm;
            }
            tc_fence_after();
            // the K/Q tile is consumed: fetch the next chunk's
            if (tid == 0 && ok && !last) {
                mbar_arrive_expect_tx(&sc.bar_kq, kq_bytes);
#pragma unroll
                for (int rg = 0; rg < KD / 64; ++rg) {
                    tma_load_3d(KQ + rg * 16384, &kmap, &sc.bar_kq, rg * 64, hk, static_cast<int>(t0 - kChunk));
                    tma_load_3d(KQ + rg * 16384 + 8192, &qmap, &sc.bar_kq, rg * 64, hk, static_cast<int>(t0 - kChunk));
                }
            }
            if (!last) pend_kq = true;

            // ---- G6: the gradient entering this chunk: the output (span start), or its bf16 hi + lo
            // copy for the next (K dS) and TMEM pre-multiplied by the next chunk's decay
            {
                const float gnext = last ? 1.f : exp2f(sc.gsum[0] + sc.gsum[1]);
                const int64_t obase = unit_state * KD * a.V + r;
#pragma unroll 1
                for (int p0 = hf * KH; p0 < (hf + 1) * KH; p0 += 4) {
                    float s64[64];
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp)
                        if (p0 + pp < (hf + 1) * KH)
                            tmem_ld16(trow + G_DS + 16 * (p0 + pp), *reinterpret_cast<float(*)[16]>(&s64[16 * pp]));
                    tmem_wait_ld();
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        const int p = p0 + pp;
                        if (p >= (hf + 1) * KH) break;
                        float* x = &s64[16 * pp];
                        if (last) {
                            if (r < a.V && dst) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) dst[obase + static_cast<int64_t>(16 * p + e) * a.V] = x[e];
                            }
                        } else {
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const int kc = 2 * p + hh;
                                const uint32_t off = (kc >> 3) * 16384 + sw128_off(r, kc & 7);
                                store8_split(WB + off, SLO + off, &x[8 * hh]);
                            }
#pragma unroll
                            for (int e = 0; e < 16; ++e) x[e] *= gnext;
                            tmem_st16(trow + G_DS + 16 * p, *reinterpret_cast<float(*)[16]>(x));
                        }
                    }
                }
                if (!last) tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        if (failed) break;
        // the range's output (the gradient entering its first chunk) is written: its predecessor may start
        if (tid == 0 && piece > 0) set_flag(a.grad_flags + unit_state, NP - piece);
    }

    if (failed) {
        // let in-flight copies and products finish (bounded) before TMEM and shared memory go away
        if (pend_kq) mbar_wait(&sc.bar_kq, ph_kq, budget);
        if (pend_do) mbar_wait(&sc.bar_do, ph_do, budget);
        if (pend_mma) mbar_wait(&sc.bar_mma, ph_mma, budget);
        if (pend_f) mbar_wait(&sc.bar_f, ph_f, budget);
        tmem_wait_st();
        if (tid == 0) {
            atomicCAS(&a.hdr->status, LA_OK, LA_ERR_TIMEOUT);
            if (a.user_status) atomicCAS(a.user_status, LA_OK, LA_ERR_TIMEOUT);
        }
    }
    if (tid == 0 && a.ds_chunks) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tmem, G_TMEM);
}

}  // namespace

cudaError_t launch_grad(const ChunkArgs& a, const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& dom,
                        const CUtensorMap& wm, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    auto* fn = a.K == 128 ? gdn_grad_kernel<128> : gdn_grad_kernel<64>;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(G_SMEM));
    if (e != cudaSuccess) return e;
    // one CTA per SM (163 KB of shared memory), persistent over the units
    const int64_t grid = a.num_units < sms ? a.num_units : sms;
    if (grid <= 0) return cudaSuccess;
    ChunkArgs b = a;
    b.pieces = 1;
    if (a.grad_carry && a.grad_flags && a.num_units > sms) {
        // more units than SMs: four chunk ranges per unit over co-resident CTAs (a cooperative
        // launch, which guarantees them), so that the last wave is not left half empty; not under
        // stream capture (then one walk per unit, as below)
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        int coop = 0;
        if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone &&
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop) {
            e = cudaMemsetAsync(a.grad_flags, 0, static_cast<size_t>(a.num_units) * sizeof(int32_t), s);
            if (e != cudaSuccess) return e;
            b.pieces = kGradPieces;
            void* args[] = {const_cast<CUtensorMap*>(&qm), const_cast<CUtensorMap*>(&km), const_cast<CUtensorMap*>(&dom),
                            const_cast<CUtensorMap*>(&wm), &b};
            e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fn), dim3(sms), dim3(kGT), args, G_SMEM, s);
            if (e == cudaSuccess) return cudaSuccess;
            (void)cudaGetLastError();  // (not launched: one walk per unit instead)
            b.pieces = 1;
        }
    }
    fn<<<static_cast<int>(grid), kGT, G_SMEM, s>>>(qm, km, dom, wm, b);
    return cudaGetLastError();
}

}  // namespace la
